"""Brute-force pins of the oracle's window map on toy layouts.

For every segment-length list of up to three segments over a set of lengths
that hits every boundary (0, 1, ratio-1, ratio, ratio+1, 2*ratio, 2*ratio+1),
ratio 1-4 and both window forms, with and without padding rows, leading tokens
before the first segment and token padding after the last:
  (i)   every (token, column) slot is read by at most one real row;
  (ii)  the unread slots are exactly the classes the "CSA Fused Compressor" page
        (Class API) lists as never consumed: segment tails, the last block's
        first-half columns (coff 2), segments shorter than ratio and tokens
        outside the segments -- computed here from the lengths alone;
  (iii) the loop oracle and the gather formulation agree (fp64);
  (iv)  the fp32 oracle writes exact zeros on every unread slot.
"""
import itertools

import numpy as np
import pytest

import csa_workloads as w
import oracle
from oracle import gather


def unread_slots(seqlens, ratio, coff, head_dim, leading, n_tokens):
    C = coff * head_dim
    mask = np.zeros((n_tokens, C), bool)
    mask[:leading] = True
    t = leading
    for L in seqlens:
        nb = L // ratio
        mask[t + nb * ratio:t + L] = True                       # tail (all of it if nb == 0)
        if coff == 2 and nb >= 1:
            mask[t + (nb - 1) * ratio:t + nb * ratio, :head_dim] = True   # last block, first half
        t += L
    mask[t:] = True                                             # token padding
    return mask


def layouts(ratio):
    vals = sorted({0, 1, max(ratio - 1, 0), ratio, ratio + 1, 2 * ratio, 2 * ratio + 1})
    out = [[]]
    for n in (1, 2, 3):
        out += [list(p) for p in itertools.product(vals, repeat=n)]
    return out


@pytest.mark.parametrize("coff", [1, 2])
@pytest.mark.parametrize("ratio", [1, 2, 3, 4])
def test_window_map_bruteforce(ratio, coff):
    head_dim = 2
    n = 0
    all_layouts = layouts(ratio)
    for i, lens in enumerate(all_layouts):
        extra_rows = (0, 2)[i % 2]
        leading = (0, 0, 3)[i % 3]
        pad_tokens = (0, 3)[(i // 2) % 2]
        R = sum(L // ratio for L in lens)
        T = leading + sum(lens) + pad_tokens
        if R + extra_rows > 0 and T < ratio:
            continue  # the page requires n_tokens >= ratio when rows exist
        c = w.make_case("bf", ratio, coff, head_dim, lens, extra_rows=extra_rows, n_tokens=T,
                        leading=leading, seed=i)
        owner = oracle.consumers(c.cu_seqlens, c.cu_seqlens_comp, ratio, coff, head_dim, c.capacity, T)
        assert (owner != -2).all(), lens                                          # (i)
        want_unread = unread_slots(lens, ratio, coff, head_dim, leading, T)
        assert np.array_equal(owner == -1, want_unread), (lens, leading, pad_tokens)  # (ii)
        if c.capacity == 0:
            continue
        o64 = oracle.case_fwd_f64(c)
        og, _ = gather.forward(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, ratio, coff,
                               head_dim, c.capacity)
        np.testing.assert_allclose(o64, og, rtol=1e-13, atol=1e-13)               # (iii)
        d64 = oracle.case_bwd_f64(c)
        dg = gather.backward(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, ratio, coff,
                             head_dim, c.capacity, T, c.grad_out)
        for x, y in zip(d64, dg):
            np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-13)
        dkv, dsc, _ = oracle.case_bwd_f32(c)
        assert not dkv[want_unread].any() and not dsc[want_unread].any()          # (iv)
        n += 1
    assert n > 0.8 * len(all_layouts)
