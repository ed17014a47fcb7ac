"""Guard words around every buffer a kernel writes.

Without a memory checker on the GPU, out-of-bounds writes are caught here:
each output is the middle of a larger allocation whose first and last 256
bytes hold a sentinel byte pattern, and after the call (on ragged sizes,
every dtype and every kernel variant) both guards must be intact.  Results
are also checked against the oracle where the other tests do not already
cover the size."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_bit_exact, dev_bf16, dev_f32, load_library, sync

pytestmark = pytest.mark.gpu

GUARD = 256       # bytes on each side (a multiple of 16, so the inner buffer stays 16-byte aligned)
PATTERN = 0x5A


@pytest.fixture(scope="module")
def g():
    return load_library()


class Guarded:
    """A device buffer of n elements inside sentinel guards."""

    def __init__(self, n, dtype, shape=None, fill=None):
        self.esz = torch.empty((), dtype=dtype).element_size()
        self.k = GUARD // self.esz
        self.buf = torch.empty(n + 2 * self.k, dtype=dtype, device="cuda")
        self.buf.view(torch.uint8).fill_(PATTERN)
        self.n = n
        self.t = self.buf[self.k:self.k + n]
        if fill is not None:
            self.t.copy_(fill)
        if shape is not None:
            self.t = self.t.view(shape)

    def check(self, what):
        b = self.buf.view(torch.uint8)
        head = b[:GUARD].cpu().numpy()
        tail = b[GUARD + self.n * self.esz:].cpu().numpy()
        assert tail.size == GUARD
        assert np.all(head == PATTERN), f"{what}: bytes before the buffer overwritten"
        assert np.all(tail == PATTERN), f"{what}: bytes after the buffer overwritten"


SIZES = (1, 3, 5, 8, 9, 4099, 300_007)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_mean_all_orders(g, dtype):
    gen = np.random.Generator(np.random.PCG64(31))
    for numel in SIZES:
        for n in (1, 3, 8, 16):
            reps = [gen.standard_normal(numel).astype(np.float32) for _ in range(n)]
            if dtype == "bf16":
                reps = [workloads.f32_to_bf16_bits(r) for r in reps]
            d = [dev_f32(r) if dtype == "f32" else dev_bf16(r) for r in reps]
            for flags, want_fn in ((0, oracle.grad_mean), (g.FLAG_TREE_ORDER, oracle.grad_mean_tree),
                                   (g.FLAG_RING_ORDER, None)):
                if flags == g.FLAG_TREE_ORDER and n & (n - 1):
                    continue
                out = Guarded(numel, torch.float32)
                g.ddp_bucket_allreduce_mean(d, out.t, flags=flags)
                sync()
                out.check(f"mean {dtype} n={n} numel={numel} flags={flags}")
                if want_fn is not None:
                    assert_bit_exact(out.t, want_fn(reps, dtype=dtype), f"mean {dtype} n={n} numel={numel}")


def test_mean_write_back_all(g):
    gen = np.random.Generator(np.random.PCG64(32))
    for numel in SIZES:
        reps = [gen.standard_normal(numel).astype(np.float32) for _ in range(4)]
        bufs = [Guarded(numel, torch.float32, fill=torch.from_numpy(r).cuda()) for r in reps]
        out = Guarded(numel, torch.float32)
        g.ddp_bucket_allreduce_mean([b.t for b in bufs], out.t, flags=g.FLAG_WRITE_BACK_ALL)
        sync()
        out.check(f"write-back out numel={numel}")
        for r, b in enumerate(bufs):
            b.check(f"write-back replica {r} numel={numel}")
            assert_bit_exact(b.t, oracle.grad_mean(reps), f"write-back replica {r}")


def test_grouped_mean(g):
    gen = np.random.Generator(np.random.PCG64(33))
    sizes = [7, 4099, 1, 300_001, 16, 9, 65_537]
    offs = np.concatenate([[0], np.cumsum([(s + 63) // 64 * 64 for s in sizes])])
    total = int(offs[-1])
    for n in (2, 8):
        reps = [gen.standard_normal(total).astype(np.float32) for _ in range(n)]
        out = Guarded(total, torch.float32, fill=torch.zeros(total, device="cuda"))
        buckets = [(int(o), s) for o, s in zip(offs[:-1], sizes)]
        g.ddp_bucket_allreduce_mean_multi([dev_f32(r) for r in reps], buckets, out.t)
        sync()
        out.check(f"grouped n={n}")
        got = out.t.cpu().numpy()
        for o, s in buckets:
            assert_bit_exact(torch.from_numpy(got[o:o + s]), oracle.grad_mean([r[o:o + s] for r in reps]),
                             f"grouped bucket {o}")


def test_sgd_outputs(g):
    gen = np.random.Generator(np.random.PCG64(34))
    for numel in SIZES:
        for n in (1, 8):
            theta = (gen.standard_normal(numel) * 0.02).astype(np.float32)
            reps = [workloads.f32_to_bf16_bits((gen.standard_normal(numel) * 0.01).astype(np.float32))
                    for _ in range(n)]
            th = Guarded(numel, torch.float32, fill=torch.from_numpy(theta).cuda())
            buf = Guarded(numel, torch.float32, fill=torch.zeros(numel, device="cuda"))
            gout = Guarded(numel, torch.float32)
            low = Guarded(numel, torch.bfloat16)
            g.ddp_bucket_allreduce_sgd_cast([dev_bf16(r) for r in reps], th.t, buf.t, 0.1, 0.9, 1e-4, low.t,
                                            grad_out=gout.t)
            sync()
            for b, w in ((th, "theta"), (buf, "buffer"), (gout, "grad_out"), (low, "bf16 copy")):
                b.check(f"sgd {w} n={n} numel={numel}")
            th_w, b_w, g_w = oracle.sgd_step(reps, theta, np.zeros(numel, np.float32), 0.1, 0.9, 1e-4, dtype="bf16")
            assert_bit_exact(th.t, th_w, "theta")
            assert_bit_exact(gout.t, g_w, "grad_out")


def test_accumulate_and_norm(g):
    gen = np.random.Generator(np.random.PCG64(35))
    for numel in SIZES:
        micro = [workloads.f32_to_bf16_bits(gen.standard_normal(numel).astype(np.float32)) for _ in range(3)]
        acc0 = [gen.standard_normal(numel).astype(np.float32) for _ in range(3)]
        accs = [Guarded(numel, torch.float32, fill=torch.from_numpy(a).cuda()) for a in acc0]
        g.ddp_bucket_accumulate([dev_bf16(m) for m in micro], [a.t for a in accs])
        sync()
        for r, a in enumerate(accs):
            a.check(f"accumulate replica {r} numel={numel}")
            assert_bit_exact(a.t, oracle.accumulate(acc0[r], micro[r], dtype="bf16"), f"accumulate {r}")
        ws = Guarded(g.ddp_norm_workspace_bytes(2), torch.uint8)
        out = Guarded(numel, torch.float32)
        g.ddp_bucket_allreduce_mean_norm([a.t for a in accs], out.t, ws.t, 1)
        sync()
        ws.check(f"norm workspace numel={numel}")
        out.check(f"norm out numel={numel}")


@pytest.mark.parametrize("shape", [(2, 2, 3, 5, 7), (4, 3, 7, 7, 7), (2, 3, 5, 64, 64), (8, 2, 5, 1, 1),
                                   (1, 1, 3, 111, 111), (2, 2, 70, 3, 7), (3, 2, 260, 1, 7), (2, 1, 7, 13, 17),
                                   (3, 5, 1000, 3, 3)])
@pytest.mark.parametrize("io", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32")])
def test_syncbn_outputs(g, shape, io):
    n, B, C, H, W = shape
    xs = workloads.syncbn_input(4, n, B, C, H, W)
    if io[0] == "f32":
        xs_dev = [dev_f32(oracle.bf16_bits_to_f32(x)) for x in xs]
    else:
        xs_dev = [dev_bf16(x) for x in xs]
    odt = torch.bfloat16 if io[1] == "bf16" else torch.float32
    ys = [Guarded(B * C * H * W, odt, shape=(B, C, H, W)) for _ in range(n)]
    mean, inv = Guarded(C, torch.float32), Guarded(C, torch.float32)
    ws = Guarded(g.syncbn_workspace_bytes(n, B, C, H, W), torch.uint8)
    g.syncbn_merge_apply(xs_dev, [y.t for y in ys], mean.t, inv.t, ws.t)
    sync()
    for r, y in enumerate(ys):
        y.check(f"syncbn {shape} {io} y[{r}]")
    mean.check("syncbn mean")
    inv.check("syncbn invstd")
    ws.check("syncbn workspace")
    assert np.all(np.isfinite(inv.t.cpu().numpy())) and np.all(np.isfinite(mean.t.cpu().numpy()))


def test_sampler_outputs(g):
    for n in (1, 2, 3, 100, 100_003, 1_281_167):
        for N in (1, 3, 8):
            for rank in (-1, N - 1):
                for shuffle in (False, True):
                    ns = g.dist_sampler_num_samples(n, N, False)
                    cnt = ns * N if rank < 0 else ns
                    out = Guarded(cnt, torch.int64)
                    st = Guarded(1, torch.int32)
                    g.dist_sampler_indices(n, N, rank, 3, 1, shuffle, False, out.t, walk_status=st.t)
                    sync()
                    out.check(f"sampler n={n} N={N} rank={rank} shuffle={shuffle}")
                    st.check("sampler status")
                    assert st.t.item() == 0
                    want = oracle.dist_sampler_indices(n, N, rank, 3, 1, shuffle, False).reshape(-1)
                    np.testing.assert_array_equal(out.t.cpu().numpy(), want)
    for start in (0, 7, 20_000):
        ns = g.dist_sampler_num_samples(100_003, 3, False)
        out = Guarded((ns - start) * 3, torch.int64)
        g.dist_sampler_indices_from(100_003, 3, -1, 3, 1, True, False, start, out.t)
        sync()
        out.check(f"sampler from {start}")
        want = oracle.dist_sampler_indices(100_003, 3, -1, 3, 1, True, False)[:, start:].reshape(-1)
        np.testing.assert_array_equal(out.t.cpu().numpy(), want)
