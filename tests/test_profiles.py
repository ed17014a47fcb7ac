"""The ncu summaries under profiles/: each names the command that made it
and the sources of the kernels it covers with their hash, so a summary
whose kernel changed afterwards can be told apart (the headline kernel's
traffic figure in bench.py turns null in that case)."""
import hashlib
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "gradient_sync_ddp_gb300", "csrc")
LINE = re.compile(r"source_sha256:\s*([0-9a-f]{16})(?:\s+over\s+([\w.]+(?:,\s*[\w.]+)*))?")


def _summaries():
    return sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def test_every_summary_has_a_command_and_a_source_hash():
    names = _summaries()
    assert names
    for name in names:
        txt = open(os.path.join(PROFILES, name), encoding="utf-8").read()
        assert "ncu " in txt and "--clock-control none" in txt, name
        assert LINE.search(txt), f"{name}: no source_sha256 line"


def test_hashed_sources_exist():
    for name in _summaries():
        txt = open(os.path.join(PROFILES, name), encoding="utf-8").read()
        for m in LINE.finditer(txt):
            if m.group(2):
                for f in (x.strip().rstrip(".") for x in m.group(2).split(",")):
                    assert os.path.exists(os.path.join(CSRC, f)), (name, f)


def test_headline_summary_is_current():
    """The headline kernel's summary was captured from the sources bench.py
    hashes for roofline.traffic (in that order): a change to them needs a
    new capture, else the bench line's traffic figure is null."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    txt = open(os.path.join(PROFILES, "mean_kernel_resnet50.md"), encoding="utf-8").read()
    m = re.search(r"traffic_bytes_per_element:\s*[0-9.]+\s+source_sha256:\s*([0-9a-f]+)", txt)
    assert m
    h = hashlib.sha256()
    for f in bench.kernel_source_hash():
        h.update(open(f, "rb").read())
    assert h.hexdigest()[:16] == m.group(1)
