"""Helpers for the GPU tests: upload a csa_workloads.Case, run the C-ABI entry
points with NaN-canary prefilled outputs, download, compare."""
import numpy as np

import csa_workloads as w
import oracle

F = w.bf16_bits_to_f32
CANARY_BF16 = 0xFFFF  # a NaN pattern: any slot the kernel fails to write stays NaN


def torch_mod():
    import torch
    return torch


def up(a):
    torch = torch_mod()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def bits(t):
    return t.cpu().numpy().view(np.uint16)


class Dev:
    """A case resident on the GPU."""

    def __init__(self, c):
        self.c = c
        self.kv, self.score, self.ape = up(c.kv), up(c.score), up(c.ape)
        self.cu, self.cc, self.g = up(c.cu_seqlens), up(c.cu_seqlens_comp), up(c.grad_out)


def run_fwd(d, csa, canary=CANARY_BF16, capacity=None):
    torch = torch_mod()
    c = d.c
    cap = c.capacity if capacity is None else capacity
    out = torch.full((max(cap, 1), c.head_dim), np.int16(np.uint16(canary).view(np.int16)),
                     dtype=torch.int16, device="cuda")
    csa.csa_compress_fwd(d.kv, d.score, d.ape, d.cu, d.cc, c.n_seg, c.ratio, c.coff, c.head_dim, cap, out)
    torch.cuda.synchronize()
    return bits(out)[:cap]


def run_bwd(d, csa, canary=CANARY_BF16, n_tokens=None, capacity=None, dape_fill=float("nan")):
    torch = torch_mod()
    c = d.c
    C = c.coff * c.head_dim
    T = c.n_tokens
    cap = c.capacity if capacity is None else capacity
    fill = np.int16(np.uint16(canary).view(np.int16))
    dkv = torch.full((max(T, 1), C), fill, dtype=torch.int16, device="cuda")
    dsc = torch.full((max(T, 1), C), fill, dtype=torch.int16, device="cuda")
    dape = torch.full((c.ratio, C), dape_fill, dtype=torch.float32, device="cuda")
    csa.csa_compress_bwd(d.kv, d.score, d.ape, d.cu, d.cc, c.n_seg, c.ratio, c.coff, c.head_dim, cap,
                         T if n_tokens is None else n_tokens, d.g, dkv, dsc, dape)
    torch.cuda.synchronize()
    return bits(dkv)[:T], bits(dsc)[:T], dape.cpu().numpy()


def same_bits_nan_aware(a, b):
    """bf16 bit patterns equal, except that any two NaNs count as equal."""
    fa, fb = F(a), F(b)
    na, nb = np.isnan(fa), np.isnan(fb)
    return np.array_equal(na, nb) and np.array_equal(a[~na], b[~nb])


def tolerance_report(got_bits, ref64):
    """(differing bf16 elements, max_abs) of got vs the fp64 reference rounded to bf16."""
    ref_bits = w.to_bf16_bits(ref64)
    diff = got_bits != ref_bits
    return int(diff.sum()), float(np.abs(F(got_bits).astype(np.float64) - F(ref_bits)).max()) if diff.size else 0.0


def same_f32_nan_aware(a, b):
    """fp32 bit patterns equal, except that any two NaNs count as equal."""
    a, b = np.asarray(a, np.float32), np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    return np.array_equal(na, nb) and np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32))


def check_dape(c, dape, csa, grouping=None):
    """grad_ape against the oracle.  Every ratio but 128: bit for bit equal to the
    oracle's fp32 sum taken in the grouping the library reports for this shape
    (csa_grad_ape_order; the rows, leaves and combination are formed by the oracle
    from the rules stated in include/csa.h).  Ratio 128 (chunked sums, tolerance
    contract): within 1e-5 (normwise) of the fp64 oracle.  Returns the grouping."""
    g = grouping or csa.csa_grad_ape_order(c.ratio, c.coff, c.head_dim, c.capacity)
    if g["kind"] == "row_blocks":
        want = oracle.case_dape_grouped_f32(c, g)
        assert same_f32_nan_aware(dape, want), (
            "grad_ape differs from the grouped fp32 oracle in %d of %d entries (max |diff| %.3g)"
            % (int((dape.view(np.uint32) != want.view(np.uint32)).sum()), dape.size,
               float(np.nanmax(np.abs(dape.astype(np.float64) - want)))))
    else:
        _, _, d64 = oracle.case_bwd_f64(c)
        assert np.abs(dape - d64).max() <= 1e-5 * max(np.abs(d64).max(), 1e-30)
    return g


# ------------------------------------------ chunked family (tolerance contract)

def fp64_parity_ok(got_bits, ref32_bits, ref64):
    """fp64-oracle parity ("CSA Fused Compressor", Numerics): the kernel is at least
    as close to the fp64 oracle as the plain fp32 evaluation:
    err_gpu <= err_fp32 * (1 + 1e-6) + 1e-4, err = max |bf16 value - fp64|."""
    err_gpu = np.abs(F(got_bits).astype(np.float64) - ref64).max()
    err_32 = np.abs(F(ref32_bits).astype(np.float64) - ref64).max()
    return err_gpu <= err_32 * (1 + 1e-6) + 1e-4


def tolerance_counts(c, csa, scale=1.0):
    """The ratio-128 contract ("CSA Fused Compressor", Numerics: ratio == 128),
    which the library applies to every window of more than 64 positions, per case: no NaN, max_abs <= 1.6e-2 against the plain fp32 and the fp64
    oracle, fp64 parity no worse than the plain fp32 evaluation, never-consumed
    slots exact zeros, grad_ape within 1e-5 (normwise) of fp64.  Returns the outputs and the
    (differing-from-fp32, differing-from-fp64, size) counts of out / grad_kv /
    grad_score, whose max(1, 0.1%) bound the callers apply."""
    d = Dev(c)
    out = run_fwd(d, csa)
    dkv, dsc, dape = run_bwd(d, csa)
    ref32 = (oracle.case_fwd_f32(c),) + tuple(oracle.case_bwd_f32(c))
    ref64 = (oracle.case_fwd_f64(c),) + tuple(oracle.case_bwd_f64(c))
    counts = []
    for got, r32, r64, bound in ((out, ref32[0], ref64[0], 1.6e-2 * scale),
                                 (dkv, ref32[1], ref64[1], 1.6e-2 * scale),
                                 (dsc, ref32[2], ref64[2], 1.6e-2 * scale * scale)):
        assert not np.isnan(F(got)).any()
        assert np.abs(F(got).astype(np.float64) - F(r32)).max() <= bound
        n64, max_abs = tolerance_report(got, r64)
        assert max_abs <= bound
        assert fp64_parity_ok(got, r32, r64)
        counts.append((int((got != r32).sum()), n64, got.size))
    owner = oracle.consumers(c.cu_seqlens, c.cu_seqlens_comp, c.ratio, c.coff, c.head_dim, c.capacity, c.n_tokens)
    unread = owner == -1
    assert not dkv[unread].any() and not dsc[unread].any()
    assert np.abs(dape - ref64[3]).max() <= 1e-5 * np.abs(ref64[3]).max()
    return (out, dkv, dsc, dape), counts


def assert_counts(counts):
    for n32, n64, size in counts:
        assert n32 <= max(1, 0.001 * size), (n32, size)
        assert n64 <= max(1, 0.001 * size), (n64, size)
