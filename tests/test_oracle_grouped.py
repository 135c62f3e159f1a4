"""Pins of the oracle's grad_ape in a stated grouping (CPU only).

The pages fix grad_ape as the sum over real rows of ds ("CSA Fused Compressor",
Semantics: the chain rule through the pooling) and ask for a deterministic result
(Numerics); the grouping of that sum is the implementation's.  The oracle evaluates
it in three plain steps -- leaves (per-leaf fp32 sums in ascending row order, in C),
the row -> leaf map, and the combination of leaves -- each pinned here against
something other than itself:

  * leaves with one row each hold that row's ds, whose bf16 rounding is the fp32
    backward's grad_score at the slot the row reads (the backward is pinned by
    test_oracle_pins.py / test_oracle_bruteforce.py / test_oracle_mutations.py);
  * those one-row leaves summed in ascending row order give the fp32 backward's
    plain grad_ape bit for bit;
  * row -> leaf maps of hand-worked strided and contiguous groupings;
  * combinations whose result depends on the order, derived by hand in fp32.
"""
import numpy as np
import pytest

import csa_workloads as w
import oracle


def _layout(ratio, coff, head_dim, seqlens, extra_rows, seed):
    return w.make_case("g", ratio, coff, head_dim, seqlens, extra_rows=extra_rows, seed=seed)


CASES = [
    (4, 2, 16, [37, 64], 3, 0),
    (4, 1, 8, [9, 0, 21], 2, 1),
    (3, 2, 8, [2, 17, 12], 1, 2),
    (1, 1, 8, [5, 3], 0, 3),
]


@pytest.mark.parametrize("ratio,coff,head_dim,seqlens,extra,seed", CASES)
def test_one_row_leaves_are_the_rows_ds(ratio, coff, head_dim, seqlens, extra, seed):
    c = _layout(ratio, coff, head_dim, seqlens, extra, seed)
    R = c.n_real_rows
    lor = np.full(c.capacity, -1, dtype=np.int32)
    lor[:R] = np.arange(R, dtype=np.int32)
    leaves = oracle.dape_leaves_f32(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, ratio, coff,
                                    head_dim, c.capacity, c.grad_out, lor, max(R, 1))
    _, dscore, dape = oracle.case_bwd_f32(c)
    C = coff * head_dim
    cu, cc = c.cu_seqlens, c.cu_seqlens_comp
    for s in range(c.n_seg):
        for b in range(cc[s + 1] - cc[s]):
            r = cc[s] + b
            base = cu[s] + b * ratio
            for k in range(coff * ratio):
                if coff == 2 and k < ratio:
                    tok, cols, arow = base - ratio + k, np.arange(head_dim), k
                    if b == 0:  # invalid for a segment's first block: nothing added
                        assert not leaves[r, arow, :head_dim].any()
                        continue
                elif coff == 2:
                    tok, cols, arow = base + k - ratio, head_dim + np.arange(head_dim), k - ratio
                else:
                    tok, cols, arow = base + k, np.arange(head_dim), k
                got = w.to_bf16_bits(leaves[r, arow, cols])
                assert np.array_equal(got, dscore[tok, cols]), (r, k)
    # ascending-row sum of the one-row leaves, from +0 = the plain fp32 grad_ape
    acc = np.zeros((ratio, C), dtype=np.float32)
    for r in range(R):
        acc = acc + leaves[r]
    assert np.array_equal(acc.view(np.uint32), dape.view(np.uint32))


def test_single_leaf_is_the_plain_sum():
    c = _layout(4, 2, 16, [37, 64], 3, 0)
    lor = np.where(np.arange(c.capacity) < c.n_real_rows, 0, -1).astype(np.int32)
    leaves = oracle.dape_leaves_f32(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, 4, 2, 16,
                                    c.capacity, c.grad_out, lor, 1)
    assert np.array_equal(leaves[0].view(np.uint32), oracle.case_bwd_f32(c)[2].view(np.uint32))


def test_unassigned_real_row_is_rejected():
    c = _layout(4, 2, 16, [37, 64], 3, 0)
    lor = np.zeros(c.capacity, dtype=np.int32)
    lor[5] = 7  # outside [0, n_leaves)
    with pytest.raises(AssertionError):
        oracle.dape_leaves_f32(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, 4, 2, 16, c.capacity,
                               c.grad_out, lor, 2)


def test_leaf_of_row_hand_examples():
    # strided, 3 blocks x 2 lanes: block r % 3, its (r // 3)-th row, lane (r // 3) % 2
    g = dict(blocks=3, lanes=2, strided=1, rows_per_block=0)
    assert oracle.leaf_of_row(g, 12, 10).tolist() == [0, 2, 4, 1, 3, 5, 0, 2, 4, 1, -1, -1]
    # contiguous, 4 rows per block x 2 lanes: block r // 4, lane (r % 4) % 2
    g = dict(blocks=3, lanes=2, strided=0, rows_per_block=4)
    assert oracle.leaf_of_row(g, 11, 10).tolist() == [0, 1, 0, 1, 2, 3, 2, 3, 4, 5, -1]


def _combine(values, blocks, lanes, cluster, flat):
    leaves = np.array(values, dtype=np.float32).reshape(-1, 1, 1)
    g = dict(blocks=blocks, lanes=lanes, cluster=cluster, flat=flat, partials=blocks // cluster,
             final_ranges=32)
    return float(oracle.combine_leaves(leaves, g)[0, 0])


def test_combination_hand_examples():
    big = 1e8  # exact in fp32; its ulp is 8, so big + 1 rounds back to big
    # Four partials [big, 1, -big, 1]: range t = [t*4//32, (t+1)*4//32) holds partial
    # t // 8 for t = 7, 15, 23, 31 and nothing else; the pairwise tree adds
    # (big + 1) + (-big + 1) = big + (-big) = 0, where a running sum would give 1.
    assert _combine([big, 1, -big, 1], blocks=4, lanes=1, cluster=1, flat=1) == 0.0
    # One partial of 2 blocks x 2 lanes, leaves [big, 1, -big, 1]:
    #   flat:   ((big + 1) + -big) + 1 = (big + -big) + 1 = 1
    #   nested: (big + 1) + (-big + 1) = big + -big = 0
    assert _combine([big, 1, -big, 1], blocks=2, lanes=2, cluster=2, flat=1) == 1.0
    assert _combine([big, 1, -big, 1], blocks=2, lanes=2, cluster=2, flat=0) == 0.0
    # 64 partials, p0 = big, p1 = -big, p32 = 1, the rest 0: contiguous ranges of two
    # give range 0 = (0 + big) + -big = 0 and range 16 = 1, total 1 (ranges taken
    # as partials t, t + 32 would give (big + 1) + -big = 0).
    p = [0.0] * 64
    p[0], p[1], p[32] = big, -big, 1.0
    assert _combine(p, blocks=64, lanes=1, cluster=1, flat=1) == 1.0
    # Empty leaves are +0: a lone -0 leaf comes out as +0 (0 + -0 = +0 in each range).
    assert np.signbit(_combine([-0.0], blocks=1, lanes=1, cluster=1, flat=1)) == False  # noqa: E712
