"""Pins for the oracle's BN running-statistics update and inference folding
(CPU only)."""
import numpy as np
import torch

import oracle


def check_running_update(update_fn):
    """Against torch.nn.functional.batch_norm in training mode (fp64), which
    updates running_mean / running_var in place from the batch it
    normalises: same batch statistics, same momentum."""
    gen = np.random.Generator(np.random.PCG64(3))
    x = gen.standard_normal((16, 6, 5, 5)) * 2 + 0.5
    rm0 = gen.standard_normal(6)
    rv0 = gen.random(6) + 0.5
    for momentum in (0.1, 0.01):
        rm_t, rv_t = torch.from_numpy(rm0.copy()), torch.from_numpy(rv0.copy())
        torch.nn.functional.batch_norm(torch.from_numpy(x), rm_t, rv_t, training=True, momentum=momentum)
        bm = x.mean(axis=(0, 2, 3))
        bv = x.var(axis=(0, 2, 3))                  # biased
        count = x.shape[0] * x.shape[2] * x.shape[3]
        rm, rv = update_fn(rm0.astype(np.float32), rv0.astype(np.float32), bm.astype(np.float32),
                           bv.astype(np.float32), count, momentum)
        np.testing.assert_allclose(rm, rm_t.numpy(), rtol=2e-6, atol=1e-7)
        np.testing.assert_allclose(rv, rv_t.numpy(), rtol=2e-6, atol=1e-7)


def test_running_update_vs_torch():
    check_running_update(oracle.bn_running_update)


def test_running_update_closed_form():
    """Dyadic values, exact in fp32: m = 0.5, count = 2 (correction 2)."""
    rm, rv = oracle.bn_running_update([1.0], [2.0], [3.0], [0.25], 2, 0.5)
    assert rm[0] == 2.0 and rv[0] == 1.25            # 0.5*1 + 0.5*3; 0.5*2 + 0.5*(0.25*2)


def check_fold(fold_fn):
    """Folded scale/bias reproduce BN in eval mode (torch, fp64)."""
    gen = np.random.Generator(np.random.PCG64(4))
    C = 7
    x = gen.standard_normal((3, C, 4, 4))
    rm, rv = gen.standard_normal(C), gen.random(C) + 0.1
    g, b = gen.standard_normal(C), gen.standard_normal(C)
    ref = torch.nn.functional.batch_norm(torch.from_numpy(x), torch.from_numpy(rm), torch.from_numpy(rv),
                                         torch.from_numpy(g), torch.from_numpy(b), training=False,
                                         eps=1e-5).numpy()
    sc, bi = fold_fn(rm, rv, g, b, 1e-5)
    np.testing.assert_allclose(x * sc[None, :, None, None] + bi[None, :, None, None], ref, rtol=1e-12, atol=1e-12)


def test_fold_vs_torch_eval_bn():
    check_fold(oracle.bn_fold_inference)


def test_fold_defaults():
    sc, bi = oracle.bn_fold_inference([2.0], [3.0], None, None, 1.0)
    assert sc[0] == 0.5 and bi[0] == -1.0
