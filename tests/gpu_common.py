"""Helpers for the GPU parity tests: build + import the library, move seeded
numpy inputs to the device and compare results bit for bit."""
import numpy as np
import torch


def load_library():
    """Build (if stale) and import the package; fails loudly without CUDA."""
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need CUDA")
    import __graft_entry__
    __graft_entry__.build()
    import gradient_sync_ddp_gb300 as pkg
    return pkg


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> a bf16 device tensor with those bits."""
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a device tensor (uint32 for fp32, uint16 for bf16)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(t.dtype)


def assert_bit_exact(got: torch.Tensor, want: np.ndarray, what: str = ""):
    """fp32 results equal bit for bit; NaN matches any NaN (payloads differ
    between the CPU and the GPU and carry no meaning here)."""
    g = host_bits(got)
    w = np.ascontiguousarray(want, dtype=np.float32).view(np.uint32)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    gn = np.isnan(g.view(np.float32))
    wn = np.isnan(w.view(np.float32))
    bad = (g != w) & ~(gn & wn)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} differ; first at {i}: "
                             f"gpu {g.view(np.float32)[i]!r} ({g[i]:#010x}) vs oracle {w.view(np.float32)[i]!r} "
                             f"({w[i]:#010x})")


def sync():
    torch.cuda.synchronize()
