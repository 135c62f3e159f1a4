"""The generic-ratio kernels (every ratio in [1, 128] other than 4 and 128, except
windows of more than 64 positions with head_dim a multiple of 64, which take the
chunked kernels: test_gpu_chunked.py): the library's sequential fp32 order, so out / grad_kv / grad_score are bitwise equal to
the fp32 oracle; grad_ape bitwise equal to the oracle's fp32 sum in the grouping
the library reports (csa_grad_ape_order) and within 1e-5 (normwise) of the fp64
oracle.  Ragged packs
per ratio: tails, empty segments, segments shorter than the ratio, exact
multiples, leading tokens, token padding, padding rows."""
import numpy as np
import pytest

import csa_workloads as w
import oracle
from gpu_util import Dev, check_dape, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import sparse_attention_kv_csa_gb300 as m
    return m


def layout(ratio, i):
    r = ratio
    return [[3 * r + 1, 0, max(r - 1, 0), 2 * r],
            [5 * r + r // 2 + 1],
            [r, r, 1, 4 * r - 1, 0]][i]


def check(c, csa):
    if csa.csa_grad_ape_order(c.ratio, c.coff, c.head_dim, c.capacity)["kind"] == "chunked":
        pytest.skip("window of more than 64 positions with head_dim % 64 == 0: the chunked family, "
                    "checked by tolerance in test_gpu_chunked.py")
    d = Dev(c)
    if c.capacity > 0:
        assert np.array_equal(run_fwd(d, csa), oracle.case_fwd_f32(c))
    dkv, dsc, dape = run_bwd(d, csa)
    want = oracle.case_bwd_f32(c)
    assert np.array_equal(dkv, want[0]) and np.array_equal(dsc, want[1])
    check_dape(c, dape, csa)
    _, _, d64 = oracle.case_bwd_f64(c)
    assert np.all(np.abs(dape - d64) <= 1e-5 * max(np.abs(d64).max(), 1e-30))


@pytest.mark.parametrize("ratio", [1, 2, 3, 5, 8, 16, 31, 64, 127])
@pytest.mark.parametrize("coff", [1, 2])
@pytest.mark.parametrize("li", range(3))
def test_generic_ratio_bitwise(csa, ratio, coff, li):
    lens = layout(ratio, li)
    head_dim = (8, 64, 40)[li]
    leading = (0, 3, 0)[li]
    pad = (0, 0, 5)[li]
    T = leading + sum(lens) + pad
    c = w.make_case("gen", ratio, coff, head_dim, lens, extra_rows=(2, 0, 1)[li], n_tokens=T, leading=leading,
                    seed=100 * ratio + 10 * coff + li)
    check(c, csa)


@pytest.mark.parametrize("ratio,coff", [(16, 2), (7, 1)])
def test_generic_wide_head(csa, ratio, coff):
    c = w.make_case("genw", ratio, coff, 512, [40 * ratio + 3, 9 * ratio], extra_rows=3, seed=ratio)
    check(c, csa)


def test_generic_deterministic_and_canary_free(csa):
    c = w.make_case("gdet", 12, 2, 64, [300, 11, 97], extra_rows=2, seed=9)
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa, canary=0xFFFF), run_fwd(d, csa, canary=0x7FC1))
    b1 = run_bwd(d, csa, canary=0xFFFF, dape_fill=float("nan"))
    b2 = run_bwd(d, csa, canary=0x7FC1, dape_fill=3.0)
    assert np.array_equal(b1[0], b2[0]) and np.array_equal(b1[1], b2[1])
    assert np.array_equal(b1[2].view(np.uint32), b2[2].view(np.uint32))


def test_generic_capacity_zero_and_all_padding(csa):
    c = w.make_case("gcap0", 6, 2, 64, [5, 3], capacity=0, seed=1)
    d = Dev(c)
    dkv, dsc, dape = run_bwd(d, csa, capacity=0)
    assert not dkv.any() and not dsc.any() and not dape.any()
    c = w.make_case("gpad", 6, 2, 64, [5, 3, 4], extra_rows=2, seed=2)  # no segment reaches 6 tokens
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa), oracle.case_fwd_f32(c))
    dkv, dsc, dape = run_bwd(d, csa)
    assert not dkv.any() and not dsc.any() and not dape.any()


def test_generic_workload(csa):
    c = w.WORKLOADS["r16c2d512_8x4096"]()
    check(c, csa)
    assert csa.csa_device_status() == 0


# ------------------------------------------- shared-memory staged kernels
# head_dim a multiple of 128 and windows of at most 64 positions (coff * ratio)
# take the staged kernels (TMA boxes into a shared-memory ring); wider windows
# stay on the global-memory walk.

@pytest.mark.parametrize("ratio", [1, 2, 3, 5, 8, 16, 31, 64])
@pytest.mark.parametrize("coff", [1, 2])
@pytest.mark.parametrize("li", range(3))
def test_staged_ratio_bitwise(csa, ratio, coff, li):
    lens = layout(ratio, li)
    head_dim = (128, 256, 384)[li]
    leading = (0, 3, 0)[li]
    pad = (0, 0, 5)[li]
    T = leading + sum(lens) + pad
    c = w.make_case("gst", ratio, coff, head_dim, lens, extra_rows=(2, 0, 1)[li], n_tokens=T, leading=leading,
                    seed=200 * ratio + 10 * coff + li)
    check(c, csa)


def test_staged_many_rows_per_block(csa):
    """10000 rows on one column tile: every ring slot is reused many times."""
    c = w.make_case("gstmany", 8, 2, 128, [80003, 8 * 7 + 1], extra_rows=5, seed=31)
    check(c, csa)


def test_staged_deterministic_and_edges(csa):
    c = w.make_case("gsdet", 12, 2, 128, [3000, 11, 970], extra_rows=2, seed=19)
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa, canary=0xFFFF), run_fwd(d, csa, canary=0x7FC1))
    b1 = run_bwd(d, csa, canary=0xFFFF, dape_fill=float("nan"))
    b2 = run_bwd(d, csa, canary=0x7FC1, dape_fill=3.0)
    assert np.array_equal(b1[0], b2[0]) and np.array_equal(b1[1], b2[1])
    assert np.array_equal(b1[2].view(np.uint32), b2[2].view(np.uint32))
    c = w.make_case("gscap0", 6, 2, 128, [5, 3], capacity=0, seed=3)
    dkv, dsc, dape = run_bwd(Dev(c), csa, capacity=0)
    assert not dkv.any() and not dsc.any() and not dape.any()
    c = w.make_case("gspad", 6, 2, 256, [5, 3, 4], extra_rows=2, seed=4)
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa), oracle.case_fwd_f32(c))
    dkv, dsc, dape = run_bwd(d, csa)
    assert not dkv.any() and not dsc.any() and not dape.any()
    assert csa.csa_device_status() == 0
