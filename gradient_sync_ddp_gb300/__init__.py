"""Python binding of libddp_sync.so — argument marshalling only.

Every function here has the name of a C entry point declared in
include/ddp_sync.h and does nothing but turn torch tensors (or plain Python
values) into the pointers and sizes the C ABI takes, call it, and raise
``DdpError`` on a non-zero status.  All computation runs in the library's
CUDA kernels (or, for the planner, its C++ host code).  There is no fallback:
if the library is missing, importing this package raises.

torch is used for device memory and streams only: a tensor argument must
already live where the C function expects it (device tensors for device
pointers), and calls are enqueued on ``torch.cuda.current_stream()`` unless a
``stream`` is given.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libddp_sync.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libddp_sync.so is not built ({LIB_PATH}); run "
                      "`python gradient_sync_ddp_gb300/build.py` or `__graft_entry__.build()` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

MAX_REPLICAS = 16
F32, BF16 = 0, 1
PLAN_CAP, PLAN_DEEP_FIRST = 0, 1
FLAG_TREE_ORDER, FLAG_WRITE_BACK_ALL, FLAG_RING_ORDER = 1, 2, 4

DDP_OK = 0
DDP_ERR_INVALID_ARG = -1
DDP_ERR_ALIGNMENT = -2
DDP_ERR_CAPACITY = -3
DDP_ERR_CUDA = -4
DDP_ERR_UNSUPPORTED = -5
DDP_ERR_TIMEOUT = -6


class DdpBucket(ctypes.Structure):
    _fields_ = [("offset_elems", ctypes.c_int64), ("numel", ctypes.c_int64),
                ("first", ctypes.c_int32), ("count", ctypes.c_int32)]


_c = ctypes
_P = _c.c_void_p
_lib.ddp_plan_buckets.argtypes = [_c.c_int32, _P, _c.c_int32, _c.c_int64, _c.c_int32, _P, _c.c_int32,
                                  _P, _c.c_int32, _P, _P, _P, _P, _P]
_lib.ddp_plan_buckets.restype = _c.c_int
_lib.ddp_bucket_allreduce_mean.argtypes = [_P, _c.c_int32, _c.c_int32, _c.c_int64, _P, _c.c_uint32, _P]
_lib.ddp_bucket_allreduce_mean.restype = _c.c_int
_lib.ddp_bucket_allreduce_sgd.argtypes = [_P, _c.c_int32, _c.c_int32, _c.c_int64, _P, _P, _c.c_float,
                                          _c.c_float, _c.c_float, _P, _c.c_uint32, _P]
_lib.ddp_bucket_allreduce_sgd.restype = _c.c_int
_lib.syncbn_workspace_bytes.argtypes = [_c.c_int32] * 5
_lib.syncbn_workspace_bytes.restype = _c.c_size_t
_lib.syncbn_channel_parts.argtypes = [_c.c_int32] * 6
_lib.syncbn_channel_parts.restype = _c.c_int
_lib.syncbn_merge_apply.argtypes = [_P, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32,
                                    _c.c_float, _P, _P, _P, _c.c_int32, _P, _P, _P, _c.c_size_t, _P]
_lib.syncbn_merge_apply.restype = _c.c_int
_lib.dist_sampler_num_samples.argtypes = [_c.c_int64, _c.c_int32, _c.c_int32]
_lib.dist_sampler_num_samples.restype = _c.c_int64
_lib.dist_sampler_indices.argtypes = [_c.c_int64, _c.c_int32, _c.c_int32, _c.c_uint64, _c.c_uint64, _c.c_int32,
                                      _c.c_int32, _P, _c.c_int64, _P, _P, _P]
_lib.dist_sampler_indices.restype = _c.c_int
_lib.ddp_status_string.argtypes = [_c.c_int]
_lib.ddp_status_string.restype = _c.c_char_p
_lib.ddp_last_cuda_error.argtypes = []
_lib.ddp_last_cuda_error.restype = _c.c_int
_lib.ddp_sync_version.argtypes = []
_lib.ddp_sync_version.restype = _c.c_char_p


class DdpError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.ddp_status_string(status).decode()
        if status == DDP_ERR_CUDA:
            msg += f" (cudaError {_lib.ddp_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")
        self.status = status


def _check(st: int, where: str) -> int:
    if st != DDP_OK:
        raise DdpError(st, where)
    return st


def status_string(status: int) -> str:
    return _lib.ddp_status_string(status).decode()


def version() -> str:
    return _lib.ddp_sync_version().decode()


def lib_handle():
    """The loaded ctypes library (for tests that call the C ABI directly)."""
    return _lib


def _ptr(x):
    """Device/host address of a tensor, an int address, or None -> NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream_ptr(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr_array(items):
    arr = (ctypes.c_void_p * max(1, len(items)))()
    for i, t in enumerate(items):
        arr[i] = _ptr(t)
    return arr


# ---------------------------------------------------------------- planner

def ddp_plan_buckets(numels, elem_bytes: int, cap_bytes: int, mode: int = PLAN_CAP, is_first=None,
                     align_bytes: int = 256):
    """Host planner (C++).  Returns a dict like the oracle's planner:
    buckets [(offset_elems, numel, first, count)], order, tensor_offset,
    tensor_bucket, total_elems."""
    T = len(numels)
    c_num = (ctypes.c_int64 * max(1, T))(*numels)
    c_first = None
    if is_first is not None:
        c_first = (ctypes.c_uint8 * max(1, T))(*[1 if f else 0 for f in is_first])
    order = (ctypes.c_int32 * max(1, T))()
    toff = (ctypes.c_int64 * max(1, T))()
    tbk = (ctypes.c_int32 * max(1, T))()
    nb = ctypes.c_int32(0)
    total = ctypes.c_int64(0)
    cap = max(1, T)
    while True:
        bk = (DdpBucket * cap)()
        st = _lib.ddp_plan_buckets(T, ctypes.addressof(c_num), elem_bytes, cap_bytes, mode,
                                   ctypes.addressof(c_first) if c_first is not None else None, align_bytes,
                                   ctypes.addressof(bk), cap, ctypes.addressof(nb), ctypes.addressof(order),
                                   ctypes.addressof(toff), ctypes.addressof(tbk), ctypes.addressof(total))
        if st == DDP_ERR_CAPACITY and nb.value > cap:
            cap = nb.value
            continue
        _check(st, "ddp_plan_buckets")
        break
    return {"buckets": [(b.offset_elems, b.numel, b.first, b.count) for b in bk[:nb.value]],
            "order": list(order[:T]), "tensor_offset": list(toff[:T]), "tensor_bucket": list(tbk[:T]),
            "total_elems": total.value}


# ---------------------------------------------------------------- all-reduce

def ddp_bucket_allreduce_mean(replicas, out, flags: int = 0, numel=None, stream=None) -> None:
    """out[:numel] = average of replicas[r][:numel] (fp32 or bf16 tensors on one device)."""
    if not 1 <= len(replicas) <= MAX_REPLICAS:
        raise ValueError("need 1..16 replicas")
    n = int(numel if numel is not None else replicas[0].numel())
    _check(_lib.ddp_bucket_allreduce_mean(_ptr_array(replicas), len(replicas), _dtype_code(replicas[0]), n,
                                          _ptr(out), flags, _stream_ptr(stream)),
           "ddp_bucket_allreduce_mean")


def ddp_bucket_allreduce_sgd(replicas, param, momentum_buf, lr: float, momentum: float, weight_decay: float,
                             grad_out=None, flags: int = 0, numel=None, stream=None) -> None:
    """Average the replicas and apply SGD (momentum, weight decay) to param in place."""
    if not 1 <= len(replicas) <= MAX_REPLICAS:
        raise ValueError("need 1..16 replicas")
    n = int(numel if numel is not None else replicas[0].numel())
    _check(_lib.ddp_bucket_allreduce_sgd(_ptr_array(replicas), len(replicas), _dtype_code(replicas[0]), n,
                                         _ptr(param), _ptr(momentum_buf), lr, momentum, weight_decay,
                                         _ptr(grad_out), flags, _stream_ptr(stream)),
           "ddp_bucket_allreduce_sgd")


# ---------------------------------------------------------------- SyncBN

def syncbn_workspace_bytes(n_replicas: int, batch: int, C: int, H: int, W: int) -> int:
    return int(_lib.syncbn_workspace_bytes(n_replicas, batch, C, H, W))


def syncbn_channel_parts(n_replicas: int, in_dtype: int, batch: int, C: int, H: int, W: int) -> int:
    """2 when syncbn_merge_apply runs these sizes as two channel halves on
    two streams, 1 for one sequence on the caller's stream (in_dtype: F32 or
    BF16)."""
    r = int(_lib.syncbn_channel_parts(n_replicas, in_dtype, batch, C, H, W))
    _check(r if r < 0 else 0, "syncbn_channel_parts")
    return r


def syncbn_merge_apply(xs, ys, mean_out, invstd_out, workspace, eps: float = 1e-5, gamma=None, beta=None,
                       stream=None) -> None:
    """Strict SyncBatchNorm forward over replicas xs[r] ([B, C, H, W], NCHW)
    into ys[r]; mean_out/invstd_out are float32 [C]; workspace is a uint8
    device tensor of at least syncbn_workspace_bytes(...) bytes."""
    B, C, H, W = xs[0].shape
    _check(_lib.syncbn_merge_apply(_ptr_array(xs), len(xs), _dtype_code(xs[0]), B, C, H, W, eps,
                                   _ptr(gamma), _ptr(beta), _ptr_array(ys), _dtype_code(ys[0]),
                                   _ptr(mean_out), _ptr(invstd_out), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "syncbn_merge_apply")


# ---------------------------------------------------------------- sampler

def dist_sampler_num_samples(n_items: int, n_replicas: int, drop_last: bool) -> int:
    v = int(_lib.dist_sampler_num_samples(n_items, n_replicas, int(bool(drop_last))))
    if v < 0:
        raise DdpError(DDP_ERR_INVALID_ARG, "dist_sampler_num_samples")
    return v


def dist_sampler_indices(n_items: int, n_replicas: int, rank: int, seed: int, epoch: int, shuffle: bool,
                         drop_last: bool, out, walk_status=None, stream=None) -> int:
    """Fill out (int64 device tensor) with rank's indices, or all ranks'
    rank-major when rank == -1.  Returns num_samples."""
    ns = ctypes.c_int64(0)
    _check(_lib.dist_sampler_indices(n_items, n_replicas, rank, seed & (2 ** 64 - 1), epoch & (2 ** 64 - 1),
                                     int(bool(shuffle)), int(bool(drop_last)), _ptr(out),
                                     0 if out is None else out.numel(), ctypes.addressof(ns), _ptr(walk_status),
                                     _stream_ptr(stream)),
           "dist_sampler_indices")
    return ns.value


__all__ = [
    "ddp_plan_buckets", "ddp_bucket_allreduce_mean", "ddp_bucket_allreduce_sgd", "syncbn_workspace_bytes",
    "syncbn_merge_apply", "dist_sampler_num_samples", "dist_sampler_indices", "DdpError", "status_string",
    "version", "lib_handle", "F32", "BF16", "PLAN_CAP", "PLAN_DEEP_FIRST", "FLAG_TREE_ORDER",
    "FLAG_WRITE_BACK_ALL", "FLAG_RING_ORDER", "MAX_REPLICAS",
]


_lib.syncbn_merge_apply_noalloc.argtypes = [_P, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32,
                                            _c.c_int32, _c.c_float, _P, _P, _P, _c.c_int32, _P, _P, _P]
_lib.syncbn_merge_apply_noalloc.restype = _c.c_int
_lib.syncbn_noalloc_max_workspace_bytes.argtypes = []
_lib.syncbn_noalloc_max_workspace_bytes.restype = _c.c_size_t


def syncbn_merge_apply_noalloc(xs, ys, mean_out, invstd_out, eps: float = 1e-5, gamma=None, beta=None,
                               stream=None) -> None:
    """syncbn_merge_apply for callers that cannot allocate device memory: the
    statistics scratch is a fixed 1 MiB array inside the library (see
    include/ddp_sync.h for the size limit, the first-call set-up and why
    overlapping calls must not run concurrently)."""
    B, C, H, W = xs[0].shape
    _check(_lib.syncbn_merge_apply_noalloc(_ptr_array(xs), len(xs), _dtype_code(xs[0]), B, C, H, W, eps,
                                           _ptr(gamma), _ptr(beta), _ptr_array(ys), _dtype_code(ys[0]),
                                           _ptr(mean_out), _ptr(invstd_out), _stream_ptr(stream)),
           "syncbn_merge_apply_noalloc")


def syncbn_noalloc_max_workspace_bytes() -> int:
    return int(_lib.syncbn_noalloc_max_workspace_bytes())


__all__ += ["syncbn_merge_apply_noalloc", "syncbn_noalloc_max_workspace_bytes"]


# ---------------------------------------------------------------- accumulation, norm / clipping, non-finite

NORM_SLOTS = 2048
_lib.ddp_bucket_accumulate.argtypes = [_P, _P, _c.c_int32, _c.c_int32, _c.c_int64, _P]
_lib.ddp_bucket_accumulate.restype = _c.c_int
_lib.ddp_norm_workspace_bytes.argtypes = [_c.c_int32]
_lib.ddp_norm_workspace_bytes.restype = _c.c_size_t
_lib.ddp_bucket_allreduce_mean_norm.argtypes = [_P, _c.c_int32, _c.c_int32, _c.c_int64, _P, _P, _c.c_int32, _P]
_lib.ddp_bucket_allreduce_mean_norm.restype = _c.c_int
_lib.ddp_grad_norm_finalize.argtypes = [_P, _c.c_int32, _c.c_float, _P, _P, _P, _P]
_lib.ddp_grad_norm_finalize.restype = _c.c_int
_lib.ddp_bucket_sgd.argtypes = [_P, _P, _P, _c.c_int64, _c.c_float, _c.c_float, _c.c_float, _P, _P, _P]
_lib.ddp_bucket_sgd.restype = _c.c_int


def ddp_bucket_accumulate(micro, acc, numel=None, stream=None) -> None:
    """acc[r] += micro[r] for every replica r (micro fp32 or bf16, acc fp32)."""
    if len(micro) != len(acc) or not 1 <= len(micro) <= MAX_REPLICAS:
        raise ValueError("need 1..16 replicas and one accumulator per replica")
    n = int(numel if numel is not None else micro[0].numel())
    _check(_lib.ddp_bucket_accumulate(_ptr_array(micro), _ptr_array(acc), len(micro), _dtype_code(micro[0]), n,
                                      _stream_ptr(stream)), "ddp_bucket_accumulate")


def ddp_norm_workspace_bytes(n_buckets: int) -> int:
    return int(_lib.ddp_norm_workspace_bytes(n_buckets))


def ddp_bucket_allreduce_mean_norm(replicas, out, norm_ws, bucket_index: int, numel=None, stream=None) -> None:
    """Rank-ordered average into out plus bucket bucket_index's Σout² and
    non-finite flag in norm_ws (a uint8 device tensor)."""
    if not 1 <= len(replicas) <= MAX_REPLICAS:
        raise ValueError("need 1..16 replicas")
    n = int(numel if numel is not None else replicas[0].numel())
    _check(_lib.ddp_bucket_allreduce_mean_norm(_ptr_array(replicas), len(replicas), _dtype_code(replicas[0]), n,
                                               _ptr(out), _ptr(norm_ws), bucket_index, _stream_ptr(stream)),
           "ddp_bucket_allreduce_mean_norm")


def ddp_grad_norm_finalize(norm_ws, n_buckets: int, max_norm: float, norm_out=None, clip_coef_out=None,
                           nonfinite_out=None, stream=None) -> None:
    """Global norm, clip factor and non-finite flag of the step, in device memory."""
    _check(_lib.ddp_grad_norm_finalize(_ptr(norm_ws), n_buckets, max_norm, _ptr(norm_out), _ptr(clip_coef_out),
                                       _ptr(nonfinite_out), _stream_ptr(stream)), "ddp_grad_norm_finalize")


def ddp_bucket_sgd(grad, param, momentum_buf, lr: float, momentum: float, weight_decay: float, grad_scale=None,
                   param_bf16=None, numel=None, stream=None) -> None:
    """SGD on an averaged fp32 gradient, optionally multiplied by a device
    scalar first; optionally also writes θ rounded to bf16."""
    n = int(numel if numel is not None else grad.numel())
    _check(_lib.ddp_bucket_sgd(_ptr(grad), _ptr(param), _ptr(momentum_buf), n, lr, momentum, weight_decay,
                               _ptr(grad_scale), _ptr(param_bf16), _stream_ptr(stream)), "ddp_bucket_sgd")


__all__ += ["ddp_bucket_accumulate", "ddp_norm_workspace_bytes", "ddp_bucket_allreduce_mean_norm",
            "ddp_grad_norm_finalize", "ddp_bucket_sgd", "NORM_SLOTS"]


# ---------------------------------------------------------------- BN running statistics

_lib.bn_running_stats_update.argtypes = [_P, _P, _c.c_int64, _c.c_float, _P, _P, _c.c_int32, _P]
_lib.bn_running_stats_update.restype = _c.c_int
_lib.bn_fold_inference_params.argtypes = [_P, _P, _P, _P, _c.c_float, _c.c_int32, _P, _P, _P]
_lib.bn_fold_inference_params.restype = _c.c_int


def bn_running_stats_update(batch_mean, batch_var, count: int, momentum: float, running_mean, running_var,
                            stream=None) -> None:
    _check(_lib.bn_running_stats_update(_ptr(batch_mean), _ptr(batch_var), count, momentum, _ptr(running_mean),
                                        _ptr(running_var), running_mean.numel(), _stream_ptr(stream)),
           "bn_running_stats_update")


def bn_fold_inference_params(running_mean, running_var, gamma, beta, eps: float, scale_out, bias_out,
                             stream=None) -> None:
    _check(_lib.bn_fold_inference_params(_ptr(running_mean), _ptr(running_var), _ptr(gamma), _ptr(beta), eps,
                                         running_mean.numel(), _ptr(scale_out), _ptr(bias_out),
                                         _stream_ptr(stream)), "bn_fold_inference_params")


__all__ += ["bn_running_stats_update", "bn_fold_inference_params"]


_lib.ddp_bucket_allreduce_sgd_cast.argtypes = [_P, _c.c_int32, _c.c_int32, _c.c_int64, _P, _P, _c.c_float, _c.c_float,
                                               _c.c_float, _P, _P, _P]
_lib.ddp_bucket_allreduce_sgd_cast.restype = _c.c_int


def ddp_bucket_allreduce_sgd_cast(replicas, param, momentum_buf, lr: float, momentum: float, weight_decay: float,
                                  param_bf16, grad_out=None, numel=None, stream=None) -> None:
    """ddp_bucket_allreduce_sgd that also writes the updated θ rounded to bf16 into param_bf16."""
    if not 1 <= len(replicas) <= MAX_REPLICAS:
        raise ValueError("need 1..16 replicas")
    n = int(numel if numel is not None else replicas[0].numel())
    _check(_lib.ddp_bucket_allreduce_sgd_cast(_ptr_array(replicas), len(replicas), _dtype_code(replicas[0]), n,
                                              _ptr(param), _ptr(momentum_buf), lr, momentum, weight_decay,
                                              _ptr(grad_out), _ptr(param_bf16), _stream_ptr(stream)),
           "ddp_bucket_allreduce_sgd_cast")


__all__ += ["ddp_bucket_allreduce_sgd_cast"]


MULTI_MAX_BUCKETS = 1024
_lib.ddp_bucket_allreduce_mean_multi.argtypes = [_P, _c.c_int32, _c.c_int32, _P, _c.c_int32, _P, _P]
_lib.ddp_bucket_allreduce_mean_multi.restype = _c.c_int


def ddp_bucket_allreduce_mean_multi(replica_bases, buckets, out_base, stream=None) -> None:
    """Average several buckets (list of (offset_elems, numel, ...)) of one
    flat layout in one launch; same bits as one call per bucket."""
    if not 1 <= len(replica_bases) <= MAX_REPLICAS:
        raise ValueError("need 1..16 replicas")
    nb = len(buckets)
    arr = (DdpBucket * max(1, nb))()
    for i, b in enumerate(buckets):
        arr[i].offset_elems, arr[i].numel = int(b[0]), int(b[1])
    _check(_lib.ddp_bucket_allreduce_mean_multi(_ptr_array(replica_bases), len(replica_bases),
                                                _dtype_code(replica_bases[0]), ctypes.addressof(arr), nb,
                                                _ptr(out_base), _stream_ptr(stream)),
           "ddp_bucket_allreduce_mean_multi")


__all__ += ["ddp_bucket_allreduce_mean_multi", "MULTI_MAX_BUCKETS"]


# ---------------------------------------------------------------- bucket readiness (host only)

_lib.ddp_reducer_create.argtypes = [_c.c_int32, _P, _c.c_int32, _P]
_lib.ddp_reducer_create.restype = _c.c_int
_lib.ddp_reducer_destroy.argtypes = [_P]
_lib.ddp_reducer_destroy.restype = None
for _name in ("ddp_reducer_mark_ready", "ddp_reducer_mark_unused"):
    getattr(_lib, _name).argtypes = [_P, _c.c_int32, _P]
    getattr(_lib, _name).restype = _c.c_int
_lib.ddp_reducer_wait_all.argtypes = [_P, _c.c_int64, _P]
_lib.ddp_reducer_wait_all.restype = _c.c_int
_lib.ddp_reducer_reset.argtypes = [_P]
_lib.ddp_reducer_reset.restype = _c.c_int
_lib.ddp_reducer_completed.argtypes = [_P, _P, _c.c_int32, _P]
_lib.ddp_reducer_completed.restype = _c.c_int
_lib.ddp_reducer_take_ready.argtypes = [_P, _c.c_int64, _P, _c.c_int32, _P]
_lib.ddp_reducer_take_ready.restype = _c.c_int


def ddp_reducer_create(tensor_bucket, n_buckets: int) -> int:
    """Tracker handle for parameters whose buckets are tensor_bucket[t]."""
    T = len(tensor_bucket)
    arr = (ctypes.c_int32 * max(1, T))(*[int(b) for b in tensor_bucket])
    h = ctypes.c_void_p(0)
    _check(_lib.ddp_reducer_create(T, ctypes.addressof(arr), int(n_buckets), ctypes.addressof(h)),
           "ddp_reducer_create")
    return h.value


def ddp_reducer_destroy(handle) -> None:
    _lib.ddp_reducer_destroy(handle)


def ddp_reducer_mark_ready(handle, tensor: int) -> int:
    """Mark a parameter's gradient ready; returns the bucket this completed, or -1."""
    b = ctypes.c_int32(-1)
    _check(_lib.ddp_reducer_mark_ready(handle, int(tensor), ctypes.addressof(b)), "ddp_reducer_mark_ready")
    return b.value


def ddp_reducer_mark_unused(handle, tensor: int) -> int:
    """Mark a parameter unused in this iteration; returns the bucket this completed, or -1."""
    b = ctypes.c_int32(-1)
    _check(_lib.ddp_reducer_mark_unused(handle, int(tensor), ctypes.addressof(b)), "ddp_reducer_mark_unused")
    return b.value


def ddp_reducer_wait_all(handle, timeout_us: int):
    """(True, -1) when every bucket is complete; (False, first unmarked
    parameter) when the wait ran out (DDP_ERR_TIMEOUT).  Other errors raise."""
    m = ctypes.c_int32(-1)
    st = _lib.ddp_reducer_wait_all(handle, int(timeout_us), ctypes.addressof(m))
    if st == DDP_ERR_TIMEOUT:
        return False, m.value
    _check(st, "ddp_reducer_wait_all")
    return True, m.value


def ddp_reducer_reset(handle) -> None:
    _check(_lib.ddp_reducer_reset(handle), "ddp_reducer_reset")


def ddp_reducer_completed(handle) -> list:
    """Buckets completed so far in this iteration, in completion order."""
    n = ctypes.c_int32(0)
    _check(_lib.ddp_reducer_completed(handle, None, 0, ctypes.addressof(n)), "ddp_reducer_completed")
    arr = (ctypes.c_int32 * max(1, n.value))()
    _check(_lib.ddp_reducer_completed(handle, ctypes.addressof(arr), n.value, ctypes.addressof(n)),
           "ddp_reducer_completed")
    return list(arr[:n.value])


def ddp_reducer_take_ready(handle, timeout_us: int = 0, max_out: int = MULTI_MAX_BUCKETS) -> list:
    """Buckets completed since the previous take, in bucket order (waits up
    to timeout_us for one if none is waiting); each is taken once per
    iteration."""
    arr = (ctypes.c_int32 * max(1, max_out))()
    n = ctypes.c_int32(0)
    _check(_lib.ddp_reducer_take_ready(handle, int(timeout_us), ctypes.addressof(arr), max_out,
                                       ctypes.addressof(n)), "ddp_reducer_take_ready")
    return list(arr[:n.value])


__all__ += ["ddp_reducer_create", "ddp_reducer_destroy", "ddp_reducer_mark_ready", "ddp_reducer_mark_unused",
            "ddp_reducer_wait_all", "ddp_reducer_reset", "ddp_reducer_completed", "ddp_reducer_take_ready"]


# ---------------------------------------------------------------- sampler resume

_lib.dist_sampler_indices_from.argtypes = [_c.c_int64, _c.c_int32, _c.c_int32, _c.c_uint64, _c.c_uint64,
                                           _c.c_int32, _c.c_int32, _c.c_int64, _P, _c.c_int64, _P, _P, _P]
_lib.dist_sampler_indices_from.restype = _c.c_int


def dist_sampler_indices_from(n_items: int, n_replicas: int, rank: int, seed: int, epoch: int, shuffle: bool,
                              drop_last: bool, start: int, out, walk_status=None, stream=None) -> int:
    """dist_sampler_indices from list position `start` on (resuming an
    epoch); out holds num_samples - start indices per rank.  Returns num_samples."""
    ns = ctypes.c_int64(0)
    _check(_lib.dist_sampler_indices_from(n_items, n_replicas, rank, seed & (2 ** 64 - 1), epoch & (2 ** 64 - 1),
                                          int(bool(shuffle)), int(bool(drop_last)), int(start), _ptr(out),
                                          0 if out is None else out.numel(), ctypes.addressof(ns),
                                          _ptr(walk_status), _stream_ptr(stream)),
           "dist_sampler_indices_from")
    return ns.value


__all__ += ["dist_sampler_indices_from"]
