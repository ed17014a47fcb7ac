"""Bucket readiness (the reducer's bookkeeping), host only: the C++ tracker
behind ddp_reducer_* against the rules of AI_Infra notes "1.DataParallel /
DDP" §3.2/§4.2 (a bucket's all-reduce is issued once all of its parameters
are ready) and §3.3 (an unused parameter leaves its bucket incomplete
unless it is marked as needing no communication).  No CUDA call."""
import threading
import time

import numpy as np
import pytest

import workloads


@pytest.fixture(scope="module")
def g():
    import __graft_entry__
    __graft_entry__.build()
    import gradient_sync_ddp_gb300 as pkg
    return pkg


def _resnet_tracker(g):
    num = workloads.numels(workloads.resnet50_layout())
    plan = g.ddp_plan_buckets(num, 4, 25 << 20)
    tb = list(plan["tensor_bucket"])
    return plan, tb, g.ddp_reducer_create(tb, len(plan["buckets"]))


def test_backward_order_completes_buckets_in_order(g):
    """Marking parameters in reverse registration order (the order backward
    produces gradients) completes bucket 0 first, then 1, ...; each bucket
    completes exactly at the mark of its last parameter."""
    plan, tb, h = _resnet_tracker(g)
    try:
        done = []
        for t in reversed(range(len(tb))):
            b = g.ddp_reducer_mark_ready(h, t)
            if b >= 0:
                members = [u for u in range(len(tb)) if tb[u] == b]
                assert t == min(members)                      # the last of its parameters to be marked
                done.append(b)
        assert done == list(range(len(plan["buckets"])))
        assert g.ddp_reducer_completed(h) == done
        assert g.ddp_reducer_wait_all(h, 0) == (True, -1)
    finally:
        g.ddp_reducer_destroy(h)


def test_random_order_matches_set_model(g):
    gen = np.random.Generator(np.random.PCG64(7))
    for trial in range(20):
        T = int(gen.integers(1, 60))
        B = int(gen.integers(1, T + 1))
        tb = list(gen.permutation(np.concatenate([np.arange(B), gen.integers(0, B, T - B)])).astype(int))
        h = g.ddp_reducer_create(tb, B)
        try:
            for it in range(2):                                # two iterations with a reset between
                missing = {b: {t for t in range(T) if tb[t] == b} for b in range(B)}
                done = []
                for t in gen.permutation(T):
                    b = g.ddp_reducer_mark_ready(h, int(t))
                    missing[tb[t]].discard(int(t))
                    want = tb[t] if not missing[tb[t]] else -1
                    assert b == want
                    if b >= 0:
                        done.append(b)
                assert sorted(done) == list(range(B))
                assert g.ddp_reducer_completed(h) == done
                g.ddp_reducer_reset(h)
        finally:
            g.ddp_reducer_destroy(h)


def test_rejects(g):
    with pytest.raises(g.DdpError):
        g.ddp_reducer_create([0, 2], 3)                      # bucket 1 empty: could never complete
    with pytest.raises(g.DdpError):
        g.ddp_reducer_create([0, 3], 3)                      # index out of range
    with pytest.raises(g.DdpError):
        g.ddp_reducer_create([], 1)
    h = g.ddp_reducer_create([0, 0, 1], 2)
    try:
        g.ddp_reducer_mark_ready(h, 1)
        with pytest.raises(g.DdpError):
            g.ddp_reducer_mark_ready(h, 1)                   # the hook fired twice
        with pytest.raises(g.DdpError):
            g.ddp_reducer_mark_unused(h, 1)
        with pytest.raises(g.DdpError):
            g.ddp_reducer_mark_ready(h, 3)
        with pytest.raises(g.DdpError):
            g.ddp_reducer_wait_all(h, -1)
    finally:
        g.ddp_reducer_destroy(h)


def test_unused_parameter_times_out_unless_marked(g):
    """[DDP] §3.3: parameter 4 is skipped by the forward pass.  Without
    find_unused_parameters its bucket never completes: the bounded wait
    returns DDP_ERR_TIMEOUT naming parameter 4 (after the time limit, not
    before).  Marking it unused completes the bucket."""
    tb = [0, 0, 1, 1, 1, 2]
    h = g.ddp_reducer_create(tb, 3)
    try:
        for t in (5, 3, 2, 1, 0):
            g.ddp_reducer_mark_ready(h, t)
        t0 = time.monotonic()
        ok, missing = g.ddp_reducer_wait_all(h, 50_000)
        waited = time.monotonic() - t0
        assert not ok and missing == 4
        assert 0.045 <= waited < 5.0
        assert sorted(g.ddp_reducer_completed(h)) == [0, 2]
        assert g.ddp_reducer_mark_unused(h, 4) == 1
        assert g.ddp_reducer_wait_all(h, 0) == (True, -1)
    finally:
        g.ddp_reducer_destroy(h)


def test_concurrent_marks_and_waiter(g):
    """Hooks firing on 4 threads at once; a waiter on a fifth thread sees
    every bucket complete, each reported exactly once."""
    plan, tb, h = _resnet_tracker(g)
    try:
        T = len(tb)
        results, reported = {}, []
        lock = threading.Lock()

        def waiter():
            results["wait"] = g.ddp_reducer_wait_all(h, 10_000_000)

        def marker(k):
            for t in range(k, T, 4):
                b = g.ddp_reducer_mark_ready(h, t)
                if b >= 0:
                    with lock:
                        reported.append(b)
        w = threading.Thread(target=waiter)
        w.start()
        ms = [threading.Thread(target=marker, args=(k,)) for k in range(4)]
        for m in ms:
            m.start()
        for m in ms:
            m.join()
        w.join(timeout=20)
        assert results["wait"] == (True, -1)
        assert sorted(reported) == list(range(len(plan["buckets"])))
        assert sorted(g.ddp_reducer_completed(h)) == sorted(reported)
    finally:
        g.ddp_reducer_destroy(h)


def test_hook_thread_that_never_fires(g):
    """One of the marking threads dies before marking its parameters (an
    exception in a hook): the waiter returns DDP_ERR_TIMEOUT with the lowest
    unmarked parameter instead of hanging."""
    tb = [i // 3 for i in range(12)]
    h = g.ddp_reducer_create(tb, 4)
    try:
        def marker(ts):
            for t in ts:
                g.ddp_reducer_mark_ready(h, t)

        def dead(ts):
            raise_in_thread = ts[0] >= 0
            if raise_in_thread:
                return                                        # never marks its parameters
        ths = [threading.Thread(target=marker, args=([0, 1, 2, 3, 4, 5],)),
               threading.Thread(target=dead, args=([6, 7, 8],)),
               threading.Thread(target=marker, args=([9, 10, 11],))]
        for t in ths:
            t.start()
        for t in ths:
            t.join()
        ok, missing = g.ddp_reducer_wait_all(h, 20_000)
        assert not ok and missing == 6
        assert sorted(g.ddp_reducer_completed(h)) == [0, 1, 3]
    finally:
        g.ddp_reducer_destroy(h)


def test_take_ready_groups_buckets_completed_together(g):
    """ddp_reducer_take_ready hands over every bucket completed since the
    previous take, in bucket order, each once per iteration ([DDP] §3.2:
    buckets fire as they fill; buckets that fill together go out together)."""
    plan, tb, h = _resnet_tracker(g)
    try:
        T, B = len(tb), len(plan["buckets"])
        assert B == 5
        order = list(reversed(range(T)))                      # backward order
        last = {b: min(t for t in range(T) if tb[t] == b) for b in range(B)}
        i = 0
        for t in order:                                       # complete buckets 0, 1 and 2 without taking
            g.ddp_reducer_mark_ready(h, t)
            i += 1
            if t == last[2]:
                break
        assert g.ddp_reducer_take_ready(h) == [0, 1, 2]
        assert g.ddp_reducer_take_ready(h) == []              # nothing new; timeout 0 does not wait
        for t in order[i:]:
            g.ddp_reducer_mark_ready(h, t)
        assert g.ddp_reducer_take_ready(h, max_out=1) == [3]  # the lowest first, the rest stays
        assert g.ddp_reducer_take_ready(h) == [4]
        t0 = time.monotonic()
        assert g.ddp_reducer_take_ready(h, 5_000_000) == []   # every bucket taken: returns at once
        assert time.monotonic() - t0 < 1.0
        g.ddp_reducer_reset(h)                                # a new iteration: nothing taken, nothing ready
        assert g.ddp_reducer_take_ready(h, 20_000) == []
        for t in order:
            g.ddp_reducer_mark_ready(h, t)
        assert g.ddp_reducer_take_ready(h) == list(range(B))
    finally:
        g.ddp_reducer_destroy(h)


def test_take_ready_random_marks_and_takes(g):
    """Random marking order with takes at random points: every take is
    sorted, holds only buckets complete at that moment and not taken
    before; together the takes hold every bucket exactly once."""
    gen = np.random.Generator(np.random.PCG64(11))
    for trial in range(30):
        T = int(gen.integers(1, 60))
        B = int(gen.integers(1, T + 1))
        tb = list(gen.permutation(np.concatenate([np.arange(B), gen.integers(0, B, T - B)])).astype(int))
        h = g.ddp_reducer_create(tb, B)
        try:
            missing = {b: {t for t in range(T) if tb[t] == b} for b in range(B)}
            taken = []
            for t in gen.permutation(T):
                g.ddp_reducer_mark_ready(h, int(t))
                missing[tb[t]].discard(int(t))
                if gen.random() < 0.3:
                    got = g.ddp_reducer_take_ready(h, max_out=int(gen.integers(1, 4)))
                    assert got == sorted(got)
                    assert all(not missing[b] and b not in taken for b in got)
                    taken += got
            while True:
                got = g.ddp_reducer_take_ready(h)
                if not got:
                    break
                taken += got
            assert sorted(taken) == list(range(B))
        finally:
            g.ddp_reducer_destroy(h)


def test_take_ready_launcher_thread(g):
    """Hooks mark on 4 threads; a launcher thread takes with a bounded wait
    until it has every bucket.  Each bucket reaches the launcher once."""
    plan, tb, h = _resnet_tracker(g)
    try:
        T, B = len(tb), len(plan["buckets"])
        got = []

        def launcher():
            deadline = time.monotonic() + 20
            while len(got) < B and time.monotonic() < deadline:
                got.extend(g.ddp_reducer_take_ready(h, 100_000))

        def marker(k):
            for t in range(k, T, 4):
                g.ddp_reducer_mark_ready(h, t)
        lt = threading.Thread(target=launcher)
        lt.start()
        ms = [threading.Thread(target=marker, args=(k,)) for k in range(4)]
        for m in ms:
            m.start()
        for m in ms:
            m.join()
        lt.join(timeout=30)
        assert sorted(got) == list(range(B))
    finally:
        g.ddp_reducer_destroy(h)


def test_take_ready_rejects(g):
    h = g.ddp_reducer_create([0, 1], 2)
    try:
        lib = g.lib_handle()
        import ctypes
        buf = (ctypes.c_int32 * 2)()
        n = ctypes.c_int32(0)
        assert lib.ddp_reducer_take_ready(h, 0, ctypes.addressof(buf), 0, ctypes.addressof(n)) == g.DDP_ERR_INVALID_ARG
        assert lib.ddp_reducer_take_ready(h, -1, ctypes.addressof(buf), 2, ctypes.addressof(n)) == g.DDP_ERR_INVALID_ARG
        assert lib.ddp_reducer_take_ready(h, 0, None, 2, ctypes.addressof(n)) == g.DDP_ERR_INVALID_ARG
        assert lib.ddp_reducer_take_ready(h, 0, ctypes.addressof(buf), 2, None) == g.DDP_ERR_INVALID_ARG
        assert lib.ddp_reducer_take_ready(None, 0, ctypes.addressof(buf), 2, ctypes.addressof(n)) == g.DDP_ERR_INVALID_ARG
    finally:
        g.ddp_reducer_destroy(h)
