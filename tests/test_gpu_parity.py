"""GPU parity: libcsa (through its C ABI) against the CPU oracle.

Contract ("CSA Fused Compressor" page, Numerics; ratio-4 family): out, grad_kv
and grad_score equal, bit for bit, the oracle's fp32 result computed in the
kernels' operation order; against the fp64 oracle they differ on at most
max(1, 0.1%) of elements with max_abs <= 1.6e-2 (x 2^k, x 2^2k under 2^k input
scaling); grad_ape equals, bit for bit, the oracle's fp32 sum taken in the
grouping the library reports (csa_grad_ape_order), and is within 1e-5 (normwise)
of the fp64 oracle and within the summation-order bound of the plain fp32 sum.  Every output is NaN-canary prefilled, so
a slot the kernels fail to write shows up as a mismatch.
"""
import numpy as np
import pytest

import csa_workloads as w
import oracle
from gpu_util import (Dev, F, assert_counts, check_dape, run_bwd, run_fwd, same_bits_nan_aware,
                      tolerance_counts, tolerance_report)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import sparse_attention_kv_csa_gb300 as m
    return m


_oracle_cache = {}


def oracle_results(c, with64=True):
    key = (c.name, with64)
    if key not in _oracle_cache:
        r = {"out": oracle.case_fwd_f32(c), "bwd": oracle.case_bwd_f32(c)}
        if with64:
            r["out64"] = oracle.case_fwd_f64(c)
            r["bwd64"] = oracle.case_bwd_f64(c, with_abs=True)
        _oracle_cache.clear()
        _oracle_cache[key] = r
    return _oracle_cache[key]


def check_against_oracle(c, csa, scale=1.0, overflow=False):
    d = Dev(c)
    out = run_fwd(d, csa)
    dkv, dsc, dape = run_bwd(d, csa)
    ref = oracle_results(c, with64=not overflow)
    assert same_bits_nan_aware(out, ref["out"]), "forward differs from the fp32 oracle"
    assert same_bits_nan_aware(dkv, ref["bwd"][0]), "grad_kv differs from the fp32 oracle"
    assert same_bits_nan_aware(dsc, ref["bwd"][1]), "grad_score differs from the fp32 oracle"
    check_dape(c, dape, csa)
    if overflow:
        assert np.isnan(F(out)).any()
        assert np.array_equal(np.isnan(dape), np.isnan(ref["bwd"][2]))
        return
    for got, ref64, bound in ((out, ref["out64"], 1.6e-2 * scale), (dkv, ref["bwd64"][0], 1.6e-2 * scale),
                              (dsc, ref["bwd64"][1], 1.6e-2 * scale * scale)):
        n_diff, max_abs = tolerance_report(got, ref64)
        assert n_diff <= max(1, 0.001 * got.size), (n_diff, got.size)
        assert max_abs <= bound, max_abs
    d64, dabs = ref["bwd64"][2], ref["bwd64"][3]
    assert np.abs(dape - d64).max() <= 1e-5 * np.abs(d64).max()
    # Same fp32 terms summed in another fixed order: |diff| <= 2 (n-1) u sum|ds|.
    n = max(c.n_real_rows, 2)
    assert np.all(np.abs(dape.astype(np.float64) - ref["bwd"][2]) <= 2 * (n - 1) * 2.0 ** -24 * dabs * 1.01 + 1e-30)


def test_tiny_bitwise(csa):
    c = w.tiny()
    d = Dev(c)
    out = run_fwd(d, csa)
    dkv, dsc, dape = run_bwd(d, csa)
    assert np.array_equal(out, oracle.case_fwd_f32(c))
    want = oracle.case_bwd_f32(c)
    assert np.array_equal(dkv, want[0]) and np.array_equal(dsc, want[1])
    g = check_dape(c, dape, csa)
    assert g["kind"] == "row_blocks"
    _, _, d64 = oracle.case_bwd_f64(c)
    assert np.abs(dape - d64).max() <= 1e-5 * np.abs(d64).max()


@pytest.mark.parametrize("name", ["r4c2d512_8x4096", "r4c2d512_ragged64", "stress_unit", "stress_x64",
                                  "r4c2d128_32x4096", "r4c2d64_32x4096"])
def test_workload_parity(csa, name):
    c = w.WORKLOADS[name]()
    check_against_oracle(c, csa, scale=64.0 if name == "stress_x64" else 1.0)


def test_overflow_nan_masks(csa):
    check_against_oracle(w.WORKLOADS["stress_overflow"](), csa, overflow=True)


@pytest.mark.parametrize("ratio", [4, 8])
@pytest.mark.parametrize("order", ["ascending", "shuffled"])
def test_every_bf16_score_pattern_bitwise(csa, ratio, order):
    """The kernels add the bf16 score to the fp32 APE with the mixed-precision add
    (bf16 operand taken as it is).  Every one of the 65536 bf16 bit patterns --
    signed zeros, subnormals, the largest finite values, infinities, NaNs -- as a
    score, against APE columns holding zeros, signed subnormals and normal values,
    gives the oracle's bits in out, grad_kv and grad_score (NaN-aware), on the
    ratio-4 stream kernels and the staged generic kernels (ratio 8)."""
    D, C = 128, 256
    T = 65536 // C
    c = w.make_case("allbf16", ratio, 2, D, [T], extra_rows=1, seed=11 + ratio)
    pat = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if order == "shuffled":
        pat = pat[np.argsort(w.uniform01(ratio, 7, 65536), kind="stable")]
    c.score = pat.reshape(T, C).copy()
    ape = c.ape.copy()
    ape[:, 0::4] = 0.0
    ape[:, 1::8] = np.float32(1e-40)
    ape[:, 5::8] = np.float32(-3e-42)
    c.ape = ape
    d = Dev(c)
    assert same_bits_nan_aware(run_fwd(d, csa), oracle.case_fwd_f32(c))
    dkv, dsc, _ = run_bwd(d, csa)
    want = oracle.case_bwd_f32(c)
    assert same_bits_nan_aware(dkv, want[0]) and same_bits_nan_aware(dsc, want[1])


def test_x64_scaling_is_exact_on_gpu(csa):
    """The kernels' outputs scale exactly 2^6 (out, grad_kv) and 2^12 (grad_score,
    grad_ape) when kv and grad_out are scaled by 64 (Numerics, point 2)."""
    c1 = w.make_case("s1", 4, 2, 512, [8192], seed=4)
    c64 = w.make_case("s64", 4, 2, 512, [8192], seed=4, kv_scale=64.0, grad_scale=64.0)
    d1, d64 = Dev(c1), Dev(c64)
    assert np.array_equal(F(run_fwd(d64, csa)), F(run_fwd(d1, csa)) * np.float32(64))
    a1, a64 = run_bwd(d1, csa), run_bwd(d64, csa)
    assert np.array_equal(F(a64[0]), F(a1[0]) * np.float32(64))
    assert np.array_equal(F(a64[1]), F(a1[1]) * np.float32(4096))
    assert np.array_equal(a64[2], a1[2] * np.float32(4096))


def test_bitwise_run_to_run_with_different_canaries(csa):
    c = w.WORKLOADS["r4c2d512_ragged64"]()
    d = Dev(c)
    o1, o2 = run_fwd(d, csa, canary=0xFFFF), run_fwd(d, csa, canary=0x7FC1)
    assert np.array_equal(o1, o2)
    b1 = run_bwd(d, csa, canary=0xFFFF, dape_fill=float("nan"))
    b2 = run_bwd(d, csa, canary=0x7FC1, dape_fill=12345.0)
    assert np.array_equal(b1[0], b2[0]) and np.array_equal(b1[1], b2[1])
    assert np.array_equal(b1[2].view(np.uint32), b2[2].view(np.uint32))


# ---------------------------------------------------------------- edge cases

LAYOUTS = [
    [37, 64], [1, 2, 3], [4], [5], [8, 0, 0, 9], [0, 0, 4], [3, 4, 5, 6, 7, 8], [64] * 5 + [3],
    [4, 1, 4, 2, 4, 3], [17, 0, 33, 2],
]


@pytest.mark.parametrize("coff", [1, 2])
@pytest.mark.parametrize("head_dim", [8, 24, 64, 96])
@pytest.mark.parametrize("li", range(len(LAYOUTS)))
def test_small_layouts_bitwise(csa, coff, head_dim, li):
    lens = LAYOUTS[li]
    extra = (0, 1, 5)[li % 3]
    leading = (0, 3)[li % 2]
    pad = (0, 2)[(li // 2) % 2]
    T = leading + sum(lens) + pad
    R = sum(L // 4 for L in lens)
    if T < 4 and R + extra > 0:
        pytest.skip("needs at least ratio tokens")
    c = w.make_case("lay", 4, coff, head_dim, lens, extra_rows=extra, n_tokens=T, leading=leading, seed=li)
    d = Dev(c)
    if c.capacity > 0:
        assert np.array_equal(run_fwd(d, csa), oracle.case_fwd_f32(c))
    dkv, dsc, dape = run_bwd(d, csa)
    want = oracle.case_bwd_f32(c)
    assert np.array_equal(dkv, want[0]) and np.array_equal(dsc, want[1])
    check_dape(c, dape, csa)
    _, _, d64 = oracle.case_bwd_f64(c)
    assert np.all(np.abs(dape - d64) <= 1e-5 * max(np.abs(d64).max(), 1e-30))


@pytest.mark.parametrize("coff", [1, 2])
@pytest.mark.parametrize("head_dim", [128, 256, 640, 1024])
@pytest.mark.parametrize("li", [0, 2, 4, 6, 7, 9])
def test_stream_row_lanes_bitwise(csa, coff, head_dim, li):
    """Tiles of 128 and 256 columns (head_dim 128, 640: 128; 256: 256; the coff-1
    backward at head_dim 1024: four tiles of 256) run two rows of a block side by
    side, and single-tile heads stage whole token rows; any layout, any number of
    rows per block, gives the oracle's bits."""
    lens = LAYOUTS[li] + [4 * 777 + 2]
    extra = (0, 1, 5)[li % 3]
    leading = (0, 3)[li % 2]
    T = leading + sum(lens) + 2
    c = w.make_case("lanes", 4, coff, head_dim, lens, extra_rows=extra, n_tokens=T, leading=leading, seed=li + 60)
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa), oracle.case_fwd_f32(c))
    dkv, dsc, dape = run_bwd(d, csa)
    want = oracle.case_bwd_f32(c)
    assert np.array_equal(dkv, want[0]) and np.array_equal(dsc, want[1])
    check_dape(c, dape, csa)
    _, _, d64 = oracle.case_bwd_f64(c)
    assert np.all(np.abs(dape - d64) <= 1e-5 * max(np.abs(d64).max(), 1e-30))


@pytest.mark.parametrize("coff", [1, 2])
def test_wide_tiles_past_the_ring_fill_bitwise(csa, coff):
    """Tiles of 512 columns (head_dim 1024: two per row) with enough rows per block
    (about 16) that most rows come after the ring's first fill: coff 2 stages them
    with 3-D boxes at both tiles' chunk offsets, coff 1 with per-token copies; ragged
    segments put first blocks and segment tails among them."""
    lens = [8192 + 3, 4096 + 1, 4, 2047, 6]
    c = w.make_case("wide_tiles", 4, coff, 1024, lens, extra_rows=3, seed=71 + coff)
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa), oracle.case_fwd_f32(c))
    dkv, dsc, dape = run_bwd(d, csa)
    want = oracle.case_bwd_f32(c)
    assert np.array_equal(dkv, want[0]) and np.array_equal(dsc, want[1])
    check_dape(c, dape, csa)


@pytest.mark.parametrize("head_dim", [1024, 8192])
def test_wide_heads_bitwise(csa, head_dim):
    c = w.make_case("wide", 4, 2, head_dim, [13, 8], extra_rows=2, seed=8)
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa), oracle.case_fwd_f32(c))
    dkv, dsc, dape = run_bwd(d, csa)
    want = oracle.case_bwd_f32(c)
    assert np.array_equal(dkv, want[0]) and np.array_equal(dsc, want[1])
    check_dape(c, dape, csa)


def test_capacity_zero(csa):
    """No rows: the forward launches nothing (out untouched); the backward still
    writes zeros to every grad_kv / grad_score slot and grad_ape = 0."""
    c = w.make_case("cap0", 4, 2, 64, [3, 2], capacity=0, seed=1)
    d = Dev(c)
    assert run_fwd(d, csa, capacity=0).shape[0] == 0
    dkv, dsc, dape = run_bwd(d, csa, capacity=0)
    assert not dkv.any() and not dsc.any() and not dape.any()


def test_all_padding_rows(csa):
    c = w.make_case("pad", 4, 2, 64, [3, 2, 1], extra_rows=3, seed=2)
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa), oracle.case_fwd_f32(c))
    dkv, dsc, dape = run_bwd(d, csa)
    assert not dkv.any() and not dsc.any() and not dape.any()


def test_negative_n_tokens_leaves_token_padding_untouched(csa):
    c = w.make_case("ntok", 4, 2, 64, [13, 9], extra_rows=1, n_tokens=30, seed=3)
    d = Dev(c)
    dkv, dsc, _ = run_bwd(d, csa, n_tokens=-1)
    want = oracle.case_bwd_f32(c)
    T0 = int(c.cu_seqlens[-1])
    assert np.array_equal(dkv[:T0], want[0][:T0]) and np.array_equal(dsc[:T0], want[1][:T0])
    assert (dkv[T0:] == 0xFFFF).all() and (dsc[T0:] == 0xFFFF).all()


def test_misaligned_view_is_rejected_and_nothing_written(csa):
    import torch
    c = w.make_case("mis", 4, 2, 64, [16], seed=5)
    d = Dev(c)
    out = torch.full((c.capacity + 1, c.head_dim), -1, dtype=torch.int16, device="cuda")
    view = out.view(-1)[1:1 + c.capacity * c.head_dim]
    with pytest.raises(csa.CSAError) as ei:
        csa.csa_compress_fwd(d.kv, d.score, d.ape, d.cu, d.cc, c.n_seg, 4, 2, 64, c.capacity, view)
    assert ei.value.status == 3
    torch.cuda.synchronize()
    assert (out == -1).all()


def test_both_kernel_families_agree_bitwise(csa):
    """head_dim 384 (a multiple of 128: the bulk-copy pipeline, two column pairs per
    thread), 320 (a multiple of 64: the pipeline, one pair) and 392 (neither: the
    register kernels) on the same rows give the oracle's bits in all three."""
    for D in (384, 320, 392):
        c = w.make_case("fam", 4, 2, D, [57, 4, 130], extra_rows=2, seed=12)
        d = Dev(c)
        assert np.array_equal(run_fwd(d, csa), oracle.case_fwd_f32(c))
        dkv, dsc, _ = run_bwd(d, csa)
        want = oracle.case_bwd_f32(c)
        assert np.array_equal(dkv, want[0]) and np.array_equal(dsc, want[1])


def test_zz_no_bounded_wait_expired(csa):
    """No kernel of this module recorded a timeout in the device status word."""
    assert csa.csa_device_status(clear=True) == 0


# ------------------------------------------------------------ ratio 128 family

def test_r128_workload_tolerance_and_determinism(csa):
    c = w.WORKLOADS["r128c1d512_4x32768"]()
    (out, dkv, dsc, dape), counts = tolerance_counts(c, csa)
    assert_counts(counts)
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa, canary=0x7FC1), out)
    b = run_bwd(d, csa, canary=0x7FC1, dape_fill=7.0)
    assert np.array_equal(b[0], dkv) and np.array_equal(b[1], dsc)
    assert np.array_equal(b[2].view(np.uint32), dape.view(np.uint32))


def test_r128_overlapping_window_workload(csa):
    """ratio 128, coff 2 (window 256), 4 x 32768 tokens, head_dim 512."""
    c = w.WORKLOADS["r128c2d512_4x32768"]()
    (out, dkv, dsc, dape), counts = tolerance_counts(c, csa)
    assert_counts(counts)
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa, canary=0x7FC1), out)


R128_LAYOUTS = [[2400, 128, 5, 8000], [127], [128], [129, 0, 2048], [5120], [3, 5600, 2]]


@pytest.mark.parametrize("coff", [1, 2])
@pytest.mark.parametrize("head_dim", [64, 128, 192])
def test_r128_small_layouts(csa, coff, head_dim):
    """Ragged ratio-128 packs (segments shorter than ratio, tails, empty segments,
    padding rows, token padding): per-case checks, and the differing-element
    bound over the union of the cases (each case is too small for a 0.1% bound)."""
    total = [[0, 0, 0] for _ in range(3)]
    for li, lens in enumerate(R128_LAYOUTS):
        T = sum(lens) + (0, 7)[li % 2]
        R = sum(L // 128 for L in lens)
        extra = (0, 2, 1)[li % 3]
        if (T < 128 and R + extra > 0) or R + extra == 0:
            continue
        c = w.make_case("r128lay", 128, coff, head_dim, lens, extra_rows=extra, n_tokens=T, seed=li + 40)
        _, counts = tolerance_counts(c, csa)
        for t, (a, b, n) in zip(total, counts):
            t[0] += a
            t[1] += b
            t[2] += n
    assert_counts([tuple(t) for t in total])


def test_interleaved_head_dims_keep_working(csa):
    """Plans of different head_dims need different shared memory on the same
    kernel; launching a larger one after a smaller one must still work (the
    kernel's shared-memory limit is a per-function attribute)."""
    for i, head_dim in enumerate([512, 128, 384, 512, 128, 1024]):
        c = w.make_case("inter", 4, 2, head_dim, [70, 33], extra_rows=1, seed=40 + i)
        d = Dev(c)
        assert np.array_equal(run_fwd(d, csa), oracle.case_fwd_f32(c))
        dkv, dsc, _ = run_bwd(d, csa)
        want = oracle.case_bwd_f32(c)
        assert np.array_equal(dkv, want[0]) and np.array_equal(dsc, want[1])
