"""The DDP bucket flow driven by real gradient hooks (AI_Infra notes
"1.DataParallel / DDP" §3.2/§4.2): N replicas of a small model run backward;
each parameter's hook copies its gradient into the replica's flat buffer and
marks it ready; when the readiness tracker reports a bucket complete (all N
replicas' parameters of that bucket are in), the bucket's average is launched
on a side stream.  The averaged flat gradient equals the oracle's average of
the replicas' flat buffers bit for bit.  §3.3: a layer the forward pass skips
makes the bounded wait time out naming it, until it is marked unused."""
import copy

import pytest
import torch

import oracle
from gpu_common import assert_bit_exact, load_library, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    return load_library()


class Net(torch.nn.Module):
    def __init__(self):
        super().__init__()
        self.l1 = torch.nn.Linear(64, 256)
        self.l2 = torch.nn.Linear(256, 256)
        self.l3 = torch.nn.Linear(256, 10)

    def forward(self, x, use_l2=True):
        h = torch.relu(self.l1(x))
        if use_l2:
            h = torch.relu(self.l2(h))
        return self.l3(h)


class Flow:
    """N replicas, their flat gradient buffers, a tracker over N*T
    parameters and the hooks that feed it."""

    def __init__(self, g, n=4, cap_bytes=128 << 10):
        torch.manual_seed(0)
        base = Net().cuda()
        self.g, self.n = g, n
        self.models = [copy.deepcopy(base) for _ in range(n)]
        self.params = [list(m.parameters()) for m in self.models]
        self.T = len(self.params[0])
        numels = [p.numel() for p in self.params[0]]
        self.plan = g.ddp_plan_buckets(numels, 4, cap_bytes)
        self.total = self.plan["total_elems"]
        self.flat = [torch.zeros(self.total, device="cuda") for _ in range(n)]
        self.out = torch.full((self.total,), float("nan"), device="cuda")
        tb = [self.plan["tensor_bucket"][t] for t in range(self.T)] * n
        self.h = g.ddp_reducer_create(tb, len(self.plan["buckets"]))
        self.side = torch.cuda.Stream()
        self.launched = []
        for r in range(n):
            for t, p in enumerate(self.params[r]):
                p.register_post_accumulate_grad_hook(lambda p, r=r, t=t: self.ready(r, t, p))

    def launch(self, b):
        ev = torch.cuda.Event()
        ev.record(torch.cuda.current_stream())            # the gradient copies so far
        self.side.wait_event(ev)
        off, numel = self.plan["buckets"][b][0], self.plan["buckets"][b][1]
        self.g.ddp_bucket_allreduce_mean([f[off:off + numel] for f in self.flat], self.out[off:off + numel],
                                         stream=self.side)
        self.launched.append(b)

    def ready(self, r, t, p):
        off, numel = self.plan["tensor_offset"][t], p.numel()
        self.flat[r][off:off + numel].copy_(p.grad.reshape(-1))
        b = self.g.ddp_reducer_mark_ready(self.h, r * self.T + t)
        if b >= 0:
            self.launch(b)

    def backward(self, use_l2=True):
        gen = torch.Generator(device="cuda").manual_seed(1)
        for r, m in enumerate(self.models):
            x = torch.randn(32, 64, device="cuda", generator=gen)
            y = torch.randint(0, 10, (32,), device="cuda", generator=gen)
            torch.nn.functional.cross_entropy(m(x, use_l2), y).backward()

    def check(self, what):
        """Every bucket region of out equals the oracle's average of the
        replicas' flat buffers (padding between buckets is never written)."""
        sync()
        host = [f.cpu().numpy() for f in self.flat]
        got = self.out.cpu()
        for off, numel, _, _ in self.plan["buckets"]:
            assert_bit_exact(got[off:off + numel], oracle.grad_mean([h[off:off + numel] for h in host]),
                             f"{what}, bucket at {off}")


def test_hooks_launch_each_bucket_once(g):
    f = Flow(g)
    try:
        assert len(f.plan["buckets"]) >= 3
        f.backward()
        assert g.ddp_reducer_wait_all(f.h, 2_000_000) == (True, -1)
        sync()
        assert sorted(f.launched) == list(range(len(f.plan["buckets"])))
        assert f.launched == g.ddp_reducer_completed(f.h)
        f.check("hook-driven bucket averages")
        got = f.out.clone()
        # the average of the models' own .grad, in rank order, is the same
        for t, p in enumerate(f.params[0]):
            off = f.plan["tensor_offset"][t]
            mean_t = oracle.grad_mean([f.params[r][t].grad.reshape(-1).cpu().numpy() for r in range(f.n)])
            assert_bit_exact(got[off:off + p.numel()], mean_t, f"parameter {t}")
    finally:
        g.ddp_reducer_destroy(f.h)


def test_skipped_layer_times_out_until_marked_unused(g):
    f = Flow(g)
    try:
        f.backward(use_l2=False)                          # l2's weight and bias get no gradient
        ok, missing = g.ddp_reducer_wait_all(f.h, 100_000)
        names = [n for n, _ in f.models[0].named_parameters()]
        assert not ok and names[missing % f.T].startswith("l2.")
        # find_unused_parameters: zero the skipped slices, mark them unused, launch what completes
        for r in range(f.n):
            for t, (name, p) in enumerate(f.models[r].named_parameters()):
                if p.grad is None:
                    off = f.plan["tensor_offset"][t]
                    f.flat[r][off:off + p.numel()].zero_()
                    b = g.ddp_reducer_mark_unused(f.h, r * f.T + t)
                    if b >= 0:
                        f.launch(b)
        assert g.ddp_reducer_wait_all(f.h, 2_000_000) == (True, -1)
        sync()
        assert sorted(f.launched) == list(range(len(f.plan["buckets"])))
        f.check("averages with the skipped layer zeroed")
    finally:
        g.ddp_reducer_destroy(f.h)


def test_buckets_completed_together_go_out_in_one_grouped_launch(g):
    """Small caps (4 KiB: six buckets for this model) make one launch per
    bucket latency-bound.  Here the hooks only copy and mark; the first
    time three or more buckets are complete, the hook takes every completed
    bucket from the tracker and averages them with one grouped launch
    (ddp_bucket_allreduce_mean_multi); after backward the rest go out the
    same way.  Every bucket is launched exactly once, at least one launch
    carries several buckets, and the averages equal the oracle's bit for
    bit."""
    f = Flow(g, cap_bytes=4 << 10)
    groups = []

    def launch_group(bs):
        if not bs:
            return
        ev = torch.cuda.Event()
        ev.record(torch.cuda.current_stream())
        f.side.wait_event(ev)
        g.ddp_bucket_allreduce_mean_multi(f.flat, [f.plan["buckets"][b] for b in bs], f.out, stream=f.side)
        groups.append(bs)

    def ready(r, t, p):
        off, numel = f.plan["tensor_offset"][t], p.numel()
        f.flat[r][off:off + numel].copy_(p.grad.reshape(-1))
        g.ddp_reducer_mark_ready(f.h, r * f.T + t)
        if not groups and len(g.ddp_reducer_completed(f.h)) >= 3:
            launch_group(g.ddp_reducer_take_ready(f.h))

    f.ready = ready
    try:
        nb = len(f.plan["buckets"])
        assert nb >= 4
        f.backward()
        assert g.ddp_reducer_wait_all(f.h, 2_000_000) == (True, -1)
        launch_group(g.ddp_reducer_take_ready(f.h))
        sync()
        assert sorted(b for grp in groups for b in grp) == list(range(nb))
        assert max(len(grp) for grp in groups) >= 3
        assert all(grp == sorted(grp) for grp in groups)
        f.check("grouped launches of the completed buckets")
    finally:
        g.ddp_reducer_destroy(f.h)
