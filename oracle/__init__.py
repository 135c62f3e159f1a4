"""CPU oracle for the CSA fused Compressor -- TEST INFRASTRUCTURE.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package.  The product path (the CUDA library and its Python binding) never
imports, links or calls it, and it never imports them.

Two independent formulations of what the "CSA Fused Compressor" page (cuDNN
frontend docs, sections Semantics, Numerics and Class API) defines:

  * ``csa_oracle.c`` -- plain single-threaded loops over rows, columns and window
    positions, in an fp32 variant with one stated operation order (bf16 outputs)
    and an fp64 variant (libm exp, no intermediate rounding).
  * ``gather.py`` -- fp64 numpy: materialise every row's window by index gathers,
    softmax along the window axis, and scatter the gradients back.

Parity pins (in tests/): the oracle is checked against closed forms, invariants,
hand-worked examples, finite differences and brute force on toy sizes; see the
test files.  No function here is "parity unpinned".
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_LIB = os.path.join(_HERE, "libcsa_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra", "-Werror"]


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc) into oracle/libcsa_oracle.so if missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    lib.csa_oracle_exp_f32.argtypes = [ctypes.c_float]
    lib.csa_oracle_exp_f32.restype = ctypes.c_float
    common = [P, P, P, P, P, i32, i32, i32, i32, i32]
    lib.csa_oracle_fwd_f32.argtypes = common + [P]
    lib.csa_oracle_fwd_f64.argtypes = common + [P]
    lib.csa_oracle_bwd_f32.argtypes = common + [i64, P, P, P, P]
    lib.csa_oracle_bwd_f64.argtypes = common + [i64, P, P, P, P, P]
    lib.csa_oracle_consumers.argtypes = [P, P, i32, i32, i32, i32, i32, i64, P]
    lib.csa_oracle_dape_leaves_f32.argtypes = common + [P, P, i32, P]
    for f in ("csa_oracle_fwd_f32", "csa_oracle_fwd_f64", "csa_oracle_bwd_f32",
              "csa_oracle_bwd_f64", "csa_oracle_consumers", "csa_oracle_dape_leaves_f32"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Test hook: run the oracle functions on another build of csa_oracle.c (the
    mutation tests plant mistakes in a copy and check that the pins catch them)."""
    global _lib
    prev = _load()
    with _lock:
        _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = prev


def compile_source(src_path: str, lib_path: str) -> str:
    """Compile a (copy of) csa_oracle.c with the oracle's arithmetic flags (warnings
    off: a planted mistake may leave a parameter unused)."""
    flags = [f for f in CFLAGS if not f.startswith("-W")] + ["-w"]
    subprocess.check_call(["gcc", *flags, "-o", lib_path, src_path, "-lm"])
    return lib_path


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def exp_f32(x) -> np.ndarray:
    """The oracle's own fp32 exp, elementwise (slow: one C call per value)."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    out = np.empty_like(x)
    flat, fo = x.reshape(-1), out.reshape(-1)
    f = lib.csa_oracle_exp_f32
    for i in range(flat.size):
        fo[i] = f(float(flat[i]))
    return out


def _args(kv, score, ape, cu, cc, ratio, coff, head_dim, capacity):
    kv = _c(kv, np.uint16)
    score = _c(score, np.uint16)
    ape = _c(ape, np.float32)
    cu = _c(cu, np.int32)
    cc = _c(cc, np.int32)
    n_seg = len(cu) - 1
    keep = (kv, score, ape, cu, cc)
    return keep, [_ptr(kv), _ptr(score), _ptr(ape), _ptr(cu), _ptr(cc), n_seg, ratio, coff,
                  head_dim, capacity]


def fwd_f32(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity):
    """fp32 forward, bf16 bits out [capacity, head_dim]."""
    keep, a = _args(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity)
    out = np.zeros((capacity, head_dim), dtype=np.uint16)
    rc = _load().csa_oracle_fwd_f32(*a, _ptr(out))
    assert rc == 0, rc
    return out


def fwd_f64(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity):
    """fp64 forward, unrounded fp64 out [capacity, head_dim]."""
    keep, a = _args(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity)
    out = np.zeros((capacity, head_dim), dtype=np.float64)
    rc = _load().csa_oracle_fwd_f64(*a, _ptr(out))
    assert rc == 0, rc
    return out


def bwd_f32(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity,
            n_tokens, grad_out):
    """fp32 backward: (dkv bf16 bits, dscore bf16 bits, dape fp32)."""
    keep, a = _args(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity)
    g = _c(grad_out, np.uint16)
    C = coff * head_dim
    dkv = np.empty((n_tokens, C), dtype=np.uint16)
    ds = np.empty((n_tokens, C), dtype=np.uint16)
    dape = np.empty((ratio, C), dtype=np.float32)
    rc = _load().csa_oracle_bwd_f32(*a, n_tokens, _ptr(g), _ptr(dkv), _ptr(ds), _ptr(dape))
    assert rc == 0, rc
    return dkv, ds, dape


def bwd_f64(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity,
            n_tokens, grad_out, with_abs=False):
    """fp64 backward: (dkv, dscore, dape[, dape_abs]) as fp64."""
    keep, a = _args(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity)
    g = _c(grad_out, np.uint16)
    C = coff * head_dim
    dkv = np.empty((n_tokens, C), dtype=np.float64)
    ds = np.empty((n_tokens, C), dtype=np.float64)
    dape = np.empty((ratio, C), dtype=np.float64)
    dabs = np.empty((ratio, C), dtype=np.float64) if with_abs else None
    rc = _load().csa_oracle_bwd_f64(*a, n_tokens, _ptr(g), _ptr(dkv), _ptr(ds), _ptr(dape),
                                    _ptr(dabs) if with_abs else None)
    assert rc == 0, rc
    return (dkv, ds, dape, dabs) if with_abs else (dkv, ds, dape)


def dape_leaves_f32(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity,
                    grad_out, leaf_of_row, n_leaves):
    """[n_leaves, ratio, coff*head_dim] fp32: leaf i = the fp32 sum, from +0 in ascending
    row order, of the ds of the real rows r with leaf_of_row[r] == i."""
    keep, a = _args(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity)
    g = _c(grad_out, np.uint16)
    lor = _c(leaf_of_row, np.int32)
    assert lor.shape == (capacity,)
    leaves = np.empty((n_leaves, ratio, coff * head_dim), dtype=np.float32)
    rc = _load().csa_oracle_dape_leaves_f32(*a, _ptr(g), _ptr(lor), n_leaves, _ptr(leaves))
    assert rc == 0, rc
    return leaves


def leaf_of_row(grouping, capacity, n_real_rows):
    """Row -> leaf map of a row-block grouping (the rules stated for csa_grad_ape_order
    in include/csa.h): rows of block b strided (b, b + blocks, ...) or contiguous
    ([b * rows_per_block, ...)), the i-th row of a block in lane i % lanes, leaf
    b * lanes + lane.  Padding rows (>= n_real_rows) map to -1."""
    B, L = grouping["blocks"], grouping["lanes"]
    leaf = np.full(capacity, -1, dtype=np.int32)
    for r in range(min(n_real_rows, capacity)):
        if grouping["strided"]:
            b, i = r % B, r // B
        else:
            b = r // grouping["rows_per_block"]
            i = r - b * grouping["rows_per_block"]
        assert b < B, (r, b, B)
        leaf[r] = b * L + i % L
    return leaf


def combine_leaves(leaves, grouping):
    """grad_ape from the leaves [blocks * lanes, ...] of a row-block grouping, in fp32,
    following the stated combination: leaves into partials (one left-to-right pass
    over (block, lane) when flat, else lanes within each block and then blocks),
    then the partials cut into 32 contiguous ranges summed from +0, then the range
    sums added in pairs (t, t ^ m) for m = 1, 2, 4, 8, 16."""
    B, L, CL = grouping["blocks"], grouping["lanes"], grouping["cluster"]
    P = B // CL
    assert P == grouping["partials"] and grouping["final_ranges"] == 32
    assert leaves.shape[0] == B * L and leaves.dtype == np.float32

    def fold(xs):
        s = xs[0].copy()
        for v in xs[1:]:
            s = s + v
        return s

    partials = []
    for q in range(P):
        blocks = range(q * CL, (q + 1) * CL)
        if grouping["flat"]:
            partials.append(fold([leaves[b * L + l] for b in blocks for l in range(L)]))
        else:
            partials.append(fold([fold([leaves[b * L + l] for l in range(L)]) for b in blocks]))
    sub = []
    for t in range(32):
        s = np.zeros(leaves.shape[1:], dtype=np.float32)
        for b in range(t * P // 32, (t + 1) * P // 32):
            s = s + partials[b]
        sub.append(s)
    m = 1
    while m < 32:
        sub = [sub[t] + sub[t ^ m] for t in range(32)]
        m *= 2
    return sub[0]


def case_dape_grouped_f32(c, grouping):
    """The fp32 grad_ape of a csa_workloads.Case summed in a row-block grouping."""
    assert grouping["kind"] == "row_blocks"
    lor = leaf_of_row(grouping, c.capacity, c.n_real_rows)
    leaves = dape_leaves_f32(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, c.ratio, c.coff,
                             c.head_dim, c.capacity, c.grad_out, lor, grouping["blocks"] * grouping["lanes"])
    return combine_leaves(leaves, grouping)


def consumers(cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity, n_tokens):
    """[n_tokens, coff*head_dim] int64: the real row reading each slot, -1 none, -2 several."""
    cu = _c(cu_seqlens, np.int32)
    cc = _c(cu_seqlens_comp, np.int32)
    owner = np.empty((n_tokens, coff * head_dim), dtype=np.int64)
    rc = _load().csa_oracle_consumers(_ptr(cu), _ptr(cc), len(cu) - 1, ratio, coff, head_dim,
                                      capacity, n_tokens, _ptr(owner))
    assert rc == 0, rc
    return owner


# Convenience: run a csa_workloads.Case through the oracle.

def case_fwd_f32(c):
    return fwd_f32(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, c.ratio, c.coff,
                   c.head_dim, c.capacity)


def case_fwd_f64(c):
    return fwd_f64(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, c.ratio, c.coff,
                   c.head_dim, c.capacity)


def case_bwd_f32(c):
    return bwd_f32(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, c.ratio, c.coff,
                   c.head_dim, c.capacity, c.n_tokens, c.grad_out)


def case_bwd_f64(c, with_abs=False):
    return bwd_f64(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, c.ratio, c.coff,
                   c.head_dim, c.capacity, c.n_tokens, c.grad_out, with_abs)
