"""Planted mistakes in the oracle must trip at least one pin (CPU only).

Each mutant is a copy of an oracle function with one plausible error (a
dropped term, a wrong sign or divisor, a reversed order, an off-by-one).  The
pins of test_oracle_* are run against it and at least one must fail; this
shows the pins would catch such a mistake in the oracle itself.
"""
import numpy as np
import pytest

import oracle
import test_oracle_accum_clip as tac
import test_oracle_mean as tm
import test_oracle_orders as to
import test_oracle_planner as tp
import test_oracle_sampler as ts
import test_oracle_sgd as tsg
import test_oracle_syncbn as tb

f32 = np.float32


def _conv(g, dtype):
    if dtype == "bf16":
        return oracle.bf16_bits_to_f32(g)
    return np.asarray(g, dtype={"f32": np.float32, "f64": np.float64, "obj": object}[dtype])


def _mean_variant(kind):
    def fn(grads, dtype="f32"):
        gs = [_conv(g, dtype) for g in grads]
        n = len(gs)
        dt = gs[0].dtype.type
        if kind == "reverse":
            gs = gs[::-1]
        if kind == "drop_last" and n > 1:
            gs = gs[:-1]
        acc = gs[0].copy() if kind == "no_zero_start" else np.zeros_like(gs[0])
        for g in (gs[1:] if kind == "no_zero_start" else gs):
            acc = acc + g
        if kind == "wide_acc" and dtype == "f32":
            acc = np.sum(np.stack(gs).astype(np.float64), axis=0).astype(np.float32)
        if kind == "div_nm1":
            return acc / dt(max(n - 1, 1))
        if kind == "mul_recip" and dtype == "f32":
            return acc * f32(f32(1) / f32(n))
        if kind == "scale_each":
            return sum((g / dt(n) for g in gs), np.zeros_like(gs[0]))
        return acc / dt(n)
    return fn


MEAN_CHECKS = [tm.check_dp_identity, tm.check_golden_rank_order, tm.check_integer_closed_form,
               tm.check_equal_replicas]


def _trips(checks, impl):
    for c in checks:
        try:
            with np.errstate(all="ignore"):
                c(impl)
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("kind", ["reverse", "drop_last", "no_zero_start", "wide_acc", "div_nm1",
                                  "mul_recip", "scale_each"])
def test_mean_mutants_are_caught(kind):
    assert _trips(MEAN_CHECKS, _mean_variant(kind)), kind


def test_unmutated_mean_passes_all():
    assert not _trips(MEAN_CHECKS, oracle.grad_mean)


def _ring_variant(kind):
    def fn(grads, dtype="f32"):
        out, b = oracle.ring_allreduce_mean(grads, dtype)
        if kind == "rank_order":
            return oracle.grad_mean(grads, dtype), b
        if kind == "backwards":
            n = len(grads)
            gs = [_conv(g, dtype) for g in grads]
            res = np.empty(gs[0].shape[0], dtype=gs[0].dtype)
            for j, (a, e) in enumerate(b):
                acc = gs[j][a:e].copy()
                for step in range(1, n):
                    acc = acc + gs[(j - step) % n][a:e]
                res[a:e] = acc / gs[0].dtype.type(n)
            return res, b
        return out, b
    return fn


@pytest.mark.parametrize("kind", ["rank_order", "backwards"])
def test_ring_mutants_are_caught(kind):
    assert _trips([to.check_ring_matches_page_tables], _ring_variant(kind))


def _sgd_variant(kind):
    def fn(grads, theta, buf, lr, momentum, wd, dtype="f32"):
        g = oracle.grad_mean(grads, dtype)
        th = np.asarray(theta, np.float32)
        d = g
        if wd != 0 and kind != "no_wd":
            d = d - f32(wd) * th if kind == "wd_sign" else d + f32(wd) * th
        b = None
        if momentum != 0:
            if kind == "lr_in_buf":
                b = f32(momentum) * np.asarray(buf, np.float32) + f32(lr) * d
                return th - b, b, g
            b = f32(momentum) * np.asarray(buf, np.float32) + d
            d = b if kind != "mom_unused" else d
        if kind == "wd_after_mom" and wd != 0:
            d = d + f32(wd) * th
        return th - f32(lr) * d, b, g
    return fn


@pytest.mark.parametrize("kind", ["wd_sign", "no_wd", "lr_in_buf", "mom_unused", "wd_after_mom"])
def test_sgd_mutants_are_caught(kind):
    assert _trips([tsg.check_sgd_golden, tsg.check_sgd_vs_torch], _sgd_variant(kind))


def _plan_variant(kind):
    def fn(numels, eb, cap, mode=oracle.PLAN_CAP, is_first=None, align_bytes=256):
        if kind == "forward":
            T = len(numels)
            rev = list(reversed(numels))
            p = oracle.plan_buckets(rev, eb, cap, mode, None if is_first is None else list(reversed(is_first)),
                                    align_bytes)
            p["order"] = [T - 1 - t for t in p["order"]]
            p["tensor_offset"] = list(reversed(p["tensor_offset"]))
            p["tensor_bucket"] = list(reversed(p["tensor_bucket"]))
            return p
        if kind == "cap_ge":
            return oracle.plan_buckets(numels, eb, cap - eb, mode, is_first, align_bytes)
        if kind == "no_align":
            return oracle.plan_buckets(numels, eb, cap, mode, is_first, eb)
        return oracle.plan_buckets(numels, eb, cap, mode, is_first, align_bytes)
    return fn


@pytest.mark.parametrize("kind", ["forward", "cap_ge", "no_align"])
def test_planner_mutants_are_caught(kind):
    def check(impl):
        tp.test_random_layouts_brute_force.__globals__["oracle"] = _Shim(impl)
        try:
            tp.test_resnet50_closed_forms()
            tp.test_tiny_cases()
            tp.test_random_layouts_brute_force()
        finally:
            tp.test_random_layouts_brute_force.__globals__["oracle"] = oracle
    assert _trips([check], _plan_variant(kind))


class _Shim:
    """The oracle module with plan_buckets replaced."""

    def __init__(self, plan):
        self.plan_buckets = plan
        self.PLAN_CAP = oracle.PLAN_CAP
        self.PLAN_DEEP_FIRST = oracle.PLAN_DEEP_FIRST


def _sampler_variant(kind):
    def fn(n, N, rank, seed, epoch, shuffle=True, drop_last=False):
        if kind == "ceil_always":
            drop_last = False
        out = oracle.dist_sampler_indices(n, N, -1, seed, epoch, shuffle, drop_last)
        ns = out.shape[1]
        if kind == "rank_shift" and N > 1:
            out = np.roll(out, 1, axis=0)
        if kind == "pad_tail" and n > 0 and n < ns * N <= 2 * n:
            flat = out.T.reshape(-1).copy()
            flat[n:] = flat[n - (ns * N - n):n]
            out = flat.reshape(ns, N).T
        if kind == "blocked":
            flat = out.T.reshape(-1)
            out = flat.reshape(N, ns)
        return out[rank] if rank >= 0 else out
    return fn


@pytest.mark.parametrize("kind", ["ceil_always", "rank_shift", "pad_tail", "blocked"])
def test_sampler_mutants_are_caught(kind):
    def check(impl):
        ts.check_partition_invariants(impl)
        g = ts.test_no_shuffle_matches_page_definition.__globals__
        g["oracle"] = _SamplerShim(impl)
        try:
            ts.test_no_shuffle_matches_page_definition()
        finally:
            g["oracle"] = oracle
    assert _trips([check], _sampler_variant(kind))


class _SamplerShim:
    def __init__(self, f):
        self.dist_sampler_indices = f


def _bn_variant(kind):
    def fn(xs, eps=1e-5, gamma=None, beta=None, dtype="bf16"):
        mean, invstd, ys = oracle.syncbn(xs, eps, gamma, beta, dtype)
        xs64 = [oracle.bf16_bits_to_f32(x).astype(np.float64) for x in xs]
        M = sum(x.shape[0] * x.shape[2] * x.shape[3] for x in xs64)
        var = 1 / invstd ** 2 - eps
        if kind == "unbiased":
            var = var * M / (M - 1)
        if kind == "eps_outside":
            invstd = 1 / np.sqrt(var) + eps
        elif kind in ("unbiased",):
            invstd = 1 / np.sqrt(var + eps)
        if kind == "local_stats":
            mean = np.mean(xs64[0], axis=(0, 2, 3))
        g = np.ones_like(mean) if gamma is None else np.asarray(gamma)
        b = np.zeros_like(mean) if beta is None else np.asarray(beta)
        ys = [(x - mean[None, :, None, None]) * invstd[None, :, None, None] * g[None, :, None, None]
              + b[None, :, None, None] for x in xs64]
        return mean, invstd, ys
    return fn


@pytest.mark.parametrize("kind", ["unbiased", "eps_outside", "local_stats"])
def test_syncbn_mutants_are_caught(kind):
    assert _trips([tb.check_syncbn_two_pass, tb.check_syncbn_vs_torch_batch_norm], _bn_variant(kind))


def test_accumulate_mutants_are_caught():
    def minus(acc, micro, dtype="f32"):
        return oracle.accumulate(acc, -np.asarray(micro) if dtype != "bf16" else micro, dtype)

    def first_only(acc, micro, dtype="f32"):
        return np.asarray(acc, np.float64 if dtype == "f64" else np.float32) * 0 + oracle.ddp_oracle._as_f32(micro, dtype)

    for bad in (minus, first_only):
        assert _trips([lambda f: tac.check_no_sync_equivalence(f, oracle.grad_mean)], bad)


@pytest.mark.parametrize("kind", ["no_sqrt", "no_clamp", "no_eps", "abs_sum"])
def test_norm_clip_mutants_are_caught(kind):
    def norm(grads):
        if kind == "no_sqrt":
            return oracle.grad_global_norm(grads) ** 2
        if kind == "abs_sum":
            return float(sum(np.abs(np.asarray(g, np.float64)).sum() for g in grads))
        return oracle.grad_global_norm(grads)

    def coef(n, m):
        if kind == "no_clamp":
            return m / (n + 1e-6) if m > 0 else 1.0
        if kind == "no_eps":
            return min(1.0, m / n) if m > 0 else 1.0
        return oracle.clip_coefficient(n, m)

    assert _trips([lambda _: tac.check_norm_and_clip(norm, coef)], None)


def test_bn_stats_mutants_are_caught():
    import test_oracle_bn_stats as tbs

    def biased(rm, rv, bm, bv, count, m):
        return oracle.bn_running_update(rm, rv, bm, bv, 2 ** 40, m)        # drops the count/(count-1) factor

    def swapped(rm, rv, bm, bv, count, m):
        return oracle.bn_running_update(rm, rv, bm, bv, count, 1.0 - m)    # momentum on the wrong side

    for bad in (biased, swapped):
        assert _trips([tbs.check_running_update], bad)

    def no_eps(rm, rv, gamma, beta, eps):
        return oracle.bn_fold_inference(rm, rv, gamma, beta, 0.0)

    def plus_mean(rm, rv, gamma, beta, eps):
        sc, bi = oracle.bn_fold_inference(rm, rv, gamma, beta, eps)
        return sc, bi + 2 * np.asarray(rm) * sc                             # sign of the mean term

    for bad in (no_eps, plus_mean):
        assert _trips([tbs.check_fold], bad)
