"""Second, independent fp64 formulation of the CSA fused Compressor -- TEST INFRASTRUCTURE.

Where csa_oracle.c loops over (row, column, window position) and skips invalid
positions, this module follows the eager description on the "CSA Fused
Compressor" page (cuDNN frontend docs, Overview and Semantics): it materialises
every row's (capacity, window, head_dim) window by index gathers, marks invalid
positions as score -inf / kv 0, takes the softmax along the window axis, and
scatters the gradients back with an add-at (the adjoint of the gather).  Rows
are mapped to segments with a sorted search instead of a scan.  Agreement of
the two formulations on every toy layout pins the window map, the tail drop, the
padding rows and the zero slots.

Small inputs only: memory is capacity * coff * ratio * head_dim doubles.
"""
from __future__ import annotations

import numpy as np


def _bf16(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def window_index(cu_seqlens, cu_seqlens_comp, ratio, coff, capacity):
    """Per row r and window position k: token, column offset (0 or head_dim units of
    the half), APE row, validity; plus which rows are real."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cc = np.asarray(cu_seqlens_comp, dtype=np.int64)
    R = int(cc[-1]) if len(cc) else 0
    r = np.arange(capacity, dtype=np.int64)
    real = r < R
    seg = np.searchsorted(cc, r, side="right") - 1
    seg = np.clip(seg, 0, max(len(cu) - 2, 0))
    blk = np.where(real, r - (cc[seg] if len(cc) > 1 else 0), 0)
    base = np.where(real, (cu[seg] if len(cu) > 1 else 0) + blk * ratio, 0)
    first = np.where(real, blk == 0, True)
    W = coff * ratio
    k = np.arange(W, dtype=np.int64)
    if coff == 2:
        prev = k < ratio
        token = np.where(prev[None, :], base[:, None] - ratio + k[None, :], base[:, None] + k[None, :] - ratio)
        half = np.where(prev, 0, 1)
        ape_row = np.where(prev, k, k - ratio)
        valid = np.where(prev[None, :], ~first[:, None], True)
    else:
        token = base[:, None] + k[None, :]
        half = np.zeros(W, dtype=np.int64)
        ape_row = k
        valid = np.ones((capacity, W), dtype=bool)
    return token, half, ape_row, valid, real


def forward_float(kvf, sf, apef, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity):
    """fp64 out [capacity, head_dim] and softmax weights p [capacity, W, head_dim] from
    real-valued kv / score / ape arrays (float64)."""
    token, half, ape_row, valid, real = window_index(cu_seqlens, cu_seqlens_comp, ratio, coff, capacity)
    j = np.arange(head_dim)
    col = half[None, :, None] * head_dim + j[None, None, :]           # [1, W, D]
    tok = np.where(valid, token, 0)[:, :, None]                        # [cap, W, 1]
    kvw = np.where(valid[:, :, None], kvf[tok, col], 0.0)
    logit = np.where(valid[:, :, None], sf[tok, col] + apef[ape_row[None, :, None], col], -np.inf)
    m = logit.max(axis=1, keepdims=True)
    e = np.exp(logit - m)
    p = e / e.sum(axis=1, keepdims=True)
    out = (p * kvw).sum(axis=1)
    return out, p


def backward_float(kvf, sf, apef, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity,
                   n_tokens, g):
    """fp64 (dkv, dscore, dape) by the adjoint of the gather (scatter-add), from
    real-valued inputs and grad_out g [capacity, head_dim]."""
    token, half, ape_row, valid, real = window_index(cu_seqlens, cu_seqlens_comp, ratio, coff, capacity)
    out, p = forward_float(kvf, sf, apef, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity)
    g = np.where(real[:, None], g, 0.0)                                # padding rows: no gradient
    j = np.arange(head_dim)
    col = half[None, :, None] * head_dim + j[None, None, :]
    tok = np.where(valid, token, 0)[:, :, None]
    use = np.broadcast_to(valid[:, :, None] & real[:, None, None], (capacity, coff * ratio, head_dim))
    kvw = np.where(use, kvf[tok, col], 0.0)
    d_kvw = np.where(use, g[:, None, :] * p, 0.0)
    d_logit = np.where(use, p * g[:, None, :] * (kvw - out[:, None, :]), 0.0)
    C = coff * head_dim
    dkv = np.zeros((n_tokens, C))
    dsc = np.zeros((n_tokens, C))
    dape = np.zeros((ratio, C))
    tt = np.broadcast_to(tok, d_kvw.shape)[use]
    cc = np.broadcast_to(col, d_kvw.shape)[use]
    np.add.at(dkv, (tt, cc), d_kvw[use])
    np.add.at(dsc, (tt, cc), d_logit[use])
    ar = np.broadcast_to(ape_row[None, :, None], d_kvw.shape)[use]
    np.add.at(dape, (ar, cc), d_logit[use])
    return dkv, dsc, dape


def forward(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity):
    """fp64 out and weights from bf16 kv / score bits and fp32 ape."""
    return forward_float(_bf16(kv), _bf16(score), np.asarray(ape, dtype=np.float32).astype(np.float64),
                         cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity)


def backward(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity,
             n_tokens, grad_out):
    """fp64 (dkv, dscore, dape) from bf16 bits / fp32 ape / bf16 grad_out bits."""
    return backward_float(_bf16(kv), _bf16(score), np.asarray(ape, dtype=np.float32).astype(np.float64),
                          cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim, capacity, n_tokens,
                          _bf16(grad_out))
