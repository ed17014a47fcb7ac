"""Pins for the oracle's gradient average (CPU only).

Each check_* takes the implementation under test so that test_oracle_mutations
can confirm that a planted mistake in the oracle trips at least one pin.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import golden_rows


def _f(tok):
    tok = tok.strip()
    if tok in ("inf", "-inf", "nan"):
        return float(tok)
    return float.fromhex(tok)


def _same_f32(a, b):
    a = np.float32(a)
    b = np.float32(b)
    if np.isnan(a) or np.isnan(b):
        return bool(np.isnan(a) and np.isnan(b))
    return a.tobytes() == b.tobytes()


# --- pin 1: the data-parallel identity ∇L = (1/N) Σ_k g_k --------------------

def check_dp_identity(mean_fn):
    """AI_Infra notes "1.DataParallel / DDP" §一: averaging the per-shard mean
    gradients of N equal shards equals the full-batch gradient.  Model
    Linear(128, 10) + cross-entropy as in the page's §1.1 / §4.1 examples;
    gradients from torch autograd in fp64 (independent of the oracle)."""
    g = torch.Generator().manual_seed(7)
    B, N = 64, 4
    x = torch.randn(B, 128, generator=g, dtype=torch.float64)
    y = torch.randint(0, 10, (B,), generator=g)
    W = torch.randn(10, 128, generator=g, dtype=torch.float64) * 0.1
    b = torch.randn(10, generator=g, dtype=torch.float64) * 0.1

    def grad(xs, ys):
        Wp = W.clone().requires_grad_(True)
        bp = b.clone().requires_grad_(True)
        loss = torch.nn.functional.cross_entropy(xs @ Wp.T + bp, ys)
        loss.backward()
        return torch.cat([Wp.grad.reshape(-1), bp.grad]).numpy()

    full = grad(x, y)
    shards = [grad(x[k * B // N:(k + 1) * B // N], y[k * B // N:(k + 1) * B // N]) for k in range(N)]
    got = mean_fn(shards, "f64")
    assert got.shape == (1290,)
    np.testing.assert_allclose(got, full, rtol=1e-12, atol=1e-15)


def test_dp_identity():
    check_dp_identity(oracle.grad_mean)


# --- pin 2: hand-derived binary32 cases --------------------------------------

def check_golden_rank_order(mean_fn):
    rows = golden_rows("mean_rank_order.txt")
    assert len(rows) >= 10
    for n_s, vals_s, exp_s, why in rows:
        vals = [_f(t) for t in vals_s.split()]
        assert len(vals) == int(n_s)
        reps = [np.array([v], dtype=np.float32) for v in vals]
        got = mean_fn(reps, "f32")[0]
        assert _same_f32(got, _f(exp_s)), (vals_s, got, exp_s, why)


def test_golden_rank_order():
    check_golden_rank_order(oracle.grad_mean)


# --- pin 3: exact closed form on integers ------------------------------------

def check_integer_closed_form(mean_fn):
    """g_r[i] = i*N + r with small integers: every partial sum is exact, so
    the result is the exact mean i*N + (N-1)/2 for any N (a half-integer)."""
    for N in (1, 2, 3, 4, 5, 8, 16):
        i = np.arange(1000, dtype=np.float64)
        reps = [(i * N + r).astype(np.float32) for r in range(N)]
        got = mean_fn(reps, "f32")
        np.testing.assert_array_equal(got, (i * N + (N - 1) / 2.0).astype(np.float32))


def test_integer_closed_form():
    check_integer_closed_form(oracle.grad_mean)


# --- pin 4: equal replicas with few significant bits --------------------------

def check_equal_replicas(mean_fn):
    """If every replica holds the same bf16-representable value g (8
    significant bits), each partial sum k*g has at most 12 significant bits
    and is exact, so the average is exactly g for every N <= 16."""
    gen = np.random.Generator(np.random.PCG64(3))
    bits = gen.integers(0, 1 << 16, 4096).astype(np.uint16)
    g = oracle.bf16_bits_to_f32(bits)
    g = g[np.isfinite(g) & (np.abs(g) < 1e30) & (np.abs(g) > 1e-30)]
    for N in (2, 4, 8, 16):
        got = mean_fn([g.copy() for _ in range(N)], "f32")
        np.testing.assert_array_equal(got, g)


def test_equal_replicas():
    check_equal_replicas(oracle.grad_mean)


# --- pin 5: exact bf16 widening -----------------------------------------------

def test_bf16_widening_known_patterns():
    pats = {0x3F80: 1.0, 0xBF80: -1.0, 0x4049: 3.140625, 0x0001: 2.0 ** -133,
            0x7F80: float("inf"), 0xFF80: float("-inf"), 0x8000: -0.0, 0x4000: 2.0,
            0x3F00: 0.5, 0x7F7F: 3.3895313892515355e38}
    got = oracle.bf16_bits_to_f32(np.array(list(pats), dtype=np.uint16))
    for v, want in zip(got, pats.values()):
        assert _same_f32(v, want)
    assert np.isnan(oracle.bf16_bits_to_f32(np.array([0x7FC0], dtype=np.uint16))[0])


def test_bf16_widening_matches_torch():
    """torch's bf16 -> fp32 conversion (an independent library routine) on
    every one of the 65536 patterns that are not NaN."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_bits_to_f32(bits)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float32).numpy()
    fin = ~np.isnan(t)
    assert np.array_equal(ours[fin].view(np.uint32), t[fin].view(np.uint32))
    assert np.isnan(ours[~fin]).all()


def test_bf16_mean_equals_f32_mean_of_widened():
    gen = np.random.Generator(np.random.PCG64(11))
    reps = [gen.integers(0, 1 << 16, 777).astype(np.uint16) for _ in range(4)]
    a = oracle.grad_mean(reps, "bf16")
    b = oracle.grad_mean([oracle.bf16_bits_to_f32(r) for r in reps], "f32")
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_rejects_empty():
    with pytest.raises(ValueError):
        oracle.grad_mean([], "f32")
