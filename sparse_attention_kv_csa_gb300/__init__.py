"""Python binding of libcsa, the GB300 (sm_103a) CSA/HCA fused Compressor.

Argument marshalling only: every step of the forward and backward runs in the
CUDA kernels of libcsa.so; this module passes device pointers, sizes and the
stream through the C ABI declared in include/csa.h and turns a non-OK status
into an exception.  There is no CPU fallback: if the library cannot be loaded
(or built), importing the package raises.

The C entry points keep their names here:
    csa_compress_fwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, n_seg, ratio,
                     coff, head_dim, capacity, out, stream=None)
    csa_compress_bwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, n_seg, ratio,
                     coff, head_dim, capacity, n_tokens, grad_out, dkv, dscore,
                     dape, stream=None)
    csa_check_support(ratio, coff, head_dim, n_tokens, capacity) -> int status
    csa_grad_ape_order(ratio, coff, head_dim, capacity) -> dict (the backward's
                     grad_ape grouping on the current device; host-side)
Tensor arguments may be torch tensors (their data_ptr() is passed) or integer
device addresses.  bf16 tensors may be torch.bfloat16 or any 16-bit dtype
holding bf16 bit patterns.  ``stream`` is a torch.cuda.Stream, a raw
cudaStream_t integer, or None for torch's current stream.

compress_forward / compress_backward allocate the outputs with torch and call
the same entry points (the layout of the "CSA Fused Compressor" wrappers).
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = [
    "csa_compress_fwd", "csa_compress_bwd", "csa_compress_bwd_noalloc", "csa_check_support", "csa_status_string",
    "csa_last_error_message", "csa_version", "csa_device_status", "csa_selftest_bounded_wait",
    "csa_selftest_reciprocal", "csa_grad_ape_order", "CSAError", "compress_forward", "compress_backward",
    "library_path", "STATUS",
]

STATUS = {
    0: "CSA_OK", 1: "CSA_ERR_INVALID_VALUE", 2: "CSA_ERR_UNSUPPORTED", 3: "CSA_ERR_MISALIGNED",
    4: "CSA_ERR_TOO_LARGE", 5: "CSA_ERR_CUDA", 6: "CSA_ERR_OUT_OF_MEMORY", 7: "CSA_ERR_DEVICE_TIMEOUT",
}


class CSAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), message))
        self.status = status


class _Grouping(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("kind", "strided", "blocks", "rows_per_block", "lanes", "cluster",
                                               "flat", "partials", "final_ranges")]


def _load():
    path = _build.build()  # no-op when up to date
    lib = ctypes.CDLL(path)
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    common = [P, P, P, P, P, i32, i32, i32, i32, i32]
    lib.csa_compress_fwd.argtypes = common + [P, P]
    lib.csa_compress_bwd.argtypes = common + [i64, P, P, P, P, P]
    lib.csa_compress_bwd_noalloc.argtypes = common + [i64, P, P, P, P, P]
    lib.csa_check_support.argtypes = [i32, i32, i32, i64, i32]
    lib.csa_device_status.argtypes = [ctypes.c_int]
    lib.csa_selftest_bounded_wait.argtypes = [i64, P]
    lib.csa_selftest_reciprocal.argtypes = [P, P, i64, P]
    lib.csa_grad_ape_order.argtypes = [i32, i32, i32, i32, ctypes.POINTER(_Grouping)]
    lib.csa_status_string.argtypes = [ctypes.c_int]
    lib.csa_status_string.restype = ctypes.c_char_p
    lib.csa_last_error_message.argtypes = []
    lib.csa_last_error_message.restype = ctypes.c_char_p
    for f in ("csa_compress_fwd", "csa_compress_bwd", "csa_compress_bwd_noalloc", "csa_check_support",
              "csa_version", "csa_device_status", "csa_selftest_bounded_wait", "csa_selftest_reciprocal",
              "csa_grad_ape_order"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


_lib = _load()


def library_path() -> str:
    return os.path.abspath(_build.LIB)


def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int):
    if rc != 0:
        raise CSAError(rc, _lib.csa_last_error_message().decode())


def csa_status_string(status: int) -> str:
    return _lib.csa_status_string(status).decode()


def csa_last_error_message() -> str:
    return _lib.csa_last_error_message().decode()


def csa_version() -> int:
    return _lib.csa_version()


def csa_device_status(clear: bool = False) -> int:
    """Synchronises and returns the device status (0 = no bounded wait expired)."""
    return _lib.csa_device_status(1 if clear else 0)


def csa_selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Launches the bounded-wait self-test kernel (see csa.h)."""
    _check(_lib.csa_selftest_bounded_wait(limit_ns, _stream(stream)))


def csa_selftest_reciprocal(d, out, n: int, stream=None) -> None:
    """The kernels' denominator reciprocal applied to n device floats (see csa.h)."""
    _check(_lib.csa_selftest_reciprocal(_addr(d), _addr(out), n, _stream(stream)))


def csa_check_support(ratio, coff, head_dim, n_tokens, capacity) -> int:
    return _lib.csa_check_support(ratio, coff, head_dim, n_tokens, capacity)


def csa_grad_ape_order(ratio, coff, head_dim, capacity) -> dict:
    """How the backward groups the grad_ape sum for this shape on the current device
    (see csa.h): kind ("row_blocks" or "chunked"), strided, blocks, rows_per_block,
    lanes, cluster, flat, partials, final_ranges."""
    g = _Grouping()
    _check(_lib.csa_grad_ape_order(ratio, coff, head_dim, capacity, ctypes.byref(g)))
    d = {n: int(getattr(g, n)) for n, _ in _Grouping._fields_}
    d["kind"] = {0: "row_blocks", 1: "chunked"}[d["kind"]]
    return d


def csa_compress_fwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, n_seg, ratio, coff, head_dim,
                     capacity, out, stream=None) -> None:
    _check(_lib.csa_compress_fwd(_addr(kv), _addr(score), _addr(ape), _addr(cu_seqlens),
                                 _addr(cu_seqlens_comp), n_seg, ratio, coff, head_dim, capacity,
                                 _addr(out), _stream(stream)))


def csa_compress_bwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, n_seg, ratio, coff, head_dim,
                     capacity, n_tokens, grad_out, dkv, dscore, dape, stream=None) -> None:
    _check(_lib.csa_compress_bwd(_addr(kv), _addr(score), _addr(ape), _addr(cu_seqlens),
                                 _addr(cu_seqlens_comp), n_seg, ratio, coff, head_dim, capacity,
                                 n_tokens, _addr(grad_out), _addr(dkv), _addr(dscore), _addr(dape),
                                 _stream(stream)))


def csa_compress_bwd_noalloc(kv, score, ape, cu_seqlens, cu_seqlens_comp, n_seg, ratio, coff, head_dim,
                             capacity, n_tokens, grad_out, dkv, dscore, dape, stream=None) -> None:
    """csa_compress_bwd for callers that cannot allocate: its scratch is a fixed
    6 MiB array of the library (shared by all calls on a device; see csa.h)."""
    _check(_lib.csa_compress_bwd_noalloc(_addr(kv), _addr(score), _addr(ape), _addr(cu_seqlens),
                                         _addr(cu_seqlens_comp), n_seg, ratio, coff, head_dim, capacity,
                                         n_tokens, _addr(grad_out), _addr(dkv), _addr(dscore), _addr(dape),
                                         _stream(stream)))


def compress_forward(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity,
                     out=None, stream=None):
    """Allocates out [capacity, head_dim] bf16 (if not given) and runs the forward."""
    import torch
    if out is None:
        out = torch.empty((capacity, head_dim), dtype=torch.bfloat16, device=kv.device)
    csa_compress_fwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, cu_seqlens.numel() - 1, ratio, coff,
                     head_dim, capacity, out, stream)
    return out


def compress_backward(kv, score, ape, cu_seqlens, cu_seqlens_comp, grad_out, ratio, coff, head_dim,
                      capacity, stream=None):
    """Allocates (uninitialised) grad_kv / grad_score and grad_ape and runs the backward."""
    import torch
    dkv = torch.empty(kv.shape, dtype=torch.bfloat16, device=kv.device)
    dsc = torch.empty(kv.shape, dtype=torch.bfloat16, device=kv.device)
    dape = torch.empty(ape.shape, dtype=torch.float32, device=kv.device)
    csa_compress_bwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, cu_seqlens.numel() - 1, ratio, coff,
                     head_dim, capacity, kv.shape[0], grad_out, dkv, dsc, dape, stream)
    return dkv, dsc, dape
