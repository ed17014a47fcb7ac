"""The C oracle of the rank-ordered average (oracle/mean_ref.c) against the
numpy oracle, bit for bit: both are restatements of the same definition,
so every value class (subnormals, signed zeros, infinities, NaNs, ties) and
every replica count must agree, single-threaded and split over threads.
CPU only; skipped where no C compiler is available."""
import numpy as np
import pytest

import oracle
import workloads
from oracle import cref

pytestmark = pytest.mark.skipif(not cref.available(), reason="no C compiler for the C oracle")


def _bits(a):
    b = np.asarray(a, np.float32).view(np.uint32).copy()
    b[np.isnan(np.asarray(a, np.float32))] = 0x7fc00000          # NaN payloads carry no meaning
    return b


@pytest.mark.parametrize("threaded", [False, True])
def test_matches_numpy_oracle(threaded):
    gen = np.random.Generator(np.random.PCG64(61))
    for n in range(1, 17):
        for numel in (1, 3, 1290, 65_537):
            reps = [workloads.adversarial_f32(gen, numel) for _ in range(n)]
            with np.errstate(all="ignore"):
                want = oracle.grad_mean(reps)
            got = cref.grad_mean_c(reps, threaded=threaded)
            np.testing.assert_array_equal(_bits(got), _bits(want), f"n={n} numel={numel}")


def test_resnet50_bucket():
    reps = workloads.replica_grads(2, 8, 6_515_688, 0.01)
    np.testing.assert_array_equal(_bits(cref.grad_mean_c(reps, threaded=True)), _bits(oracle.grad_mean(reps)))
