"""Helpers for the GPU tests: upload a csa_workloads.Case, run the C-ABI entry
points with NaN-canary prefilled outputs, download, compare."""
import numpy as np

import csa_workloads as w

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
    import oracle
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
