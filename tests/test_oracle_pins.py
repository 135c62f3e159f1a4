"""Pins of the CPU oracle against what the "CSA Fused Compressor" page and the
mathematics fix (page sections Semantics, Numerics, Class API).

Each test would fail on a plausible slip in the oracle: a wrong window token,
column or APE row; a dropped or extra term; a sign error in the gradient; a
padding row that contributes gradient; a tail that is read; a missing
non-finite propagation.
"""
import json
import os

import numpy as np
import pytest

import csa_workloads as w
import oracle
from oracle import gather

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")
F = w.bf16_bits_to_f32


def golden_examples():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


def golden_case(ex):
    cu, cc = w.offsets(ex["seqlens"], ex["ratio"])
    T, C = ex["n_tokens"], ex["coff"] * ex["head_dim"]
    kv = w.to_bf16_bits(np.array(ex["kv"], dtype=np.float64))
    score = (np.zeros((T, C), np.uint16) if ex["score"] == "zeros"
             else w.to_bf16_bits(np.array(ex["score"], dtype=np.float64)))
    ape = np.array(ex["ape"], dtype=np.float32)
    g = w.to_bf16_bits(np.array(ex["grad_out"], dtype=np.float64))
    return w.Case(ex["name"], ex["ratio"], ex["coff"], ex["head_dim"], ex["seqlens"], ex["capacity"], T,
                  cu, cc, kv, score, ape, g)


# ------------------------------------------------------------------ golden

@pytest.mark.parametrize("ex", golden_examples(), ids=lambda e: e["name"])
def test_hand_worked_forward(ex):
    c = golden_case(ex)
    want = np.array(ex["out"], dtype=np.float64)
    assert np.array_equal(F(oracle.case_fwd_f32(c)), want.astype(np.float32))
    np.testing.assert_allclose(oracle.case_fwd_f64(c), want, rtol=1e-14, atol=1e-14)
    out_g, _ = gather.forward(c.kv, c.score, c.ape, c.cu_seqlens, c.cu_seqlens_comp, c.ratio, c.coff,
                              c.head_dim, c.capacity)
    np.testing.assert_allclose(out_g, want, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("ex", [e for e in golden_examples() if "grad_kv" in e or "grad_kv_at" in e],
                         ids=lambda e: e["name"])
def test_hand_worked_backward(ex):
    c = golden_case(ex)
    dkv, dsc, dape = oracle.case_bwd_f32(c)
    dkv64, dsc64, dape64 = oracle.case_bwd_f64(c)
    if "grad_kv" in ex:
        for got32, got64, key in ((dkv, dkv64, "grad_kv"), (dsc, dsc64, "grad_score")):
            want = np.array(ex[key], dtype=np.float64)
            assert np.array_equal(F(got32), want.astype(np.float32)), key
            np.testing.assert_allclose(got64, want, rtol=0, atol=1e-14)
        want = np.array(ex["grad_ape"], dtype=np.float64)
        assert np.array_equal(dape, want.astype(np.float32))
        np.testing.assert_allclose(dape64, want, rtol=0, atol=1e-14)
    for t, col, v in ex.get("grad_kv_at", []):
        assert F(dkv)[t, col] == v
        assert abs(dkv64[t, col] - v) <= 1e-14
    for t in ex.get("zero_tokens", []):
        assert not F(dkv)[t].any() and not F(dsc)[t].any()
        assert not dkv64[t].any() and not dsc64[t].any()


# -------------------------------------------------------------- invariants

def random_case(ratio=4, coff=2, head_dim=16, seqlens=(13, 8, 3, 17), extra_rows=2, seed=3, **kw):
    return w.make_case("rand", ratio, coff, head_dim, list(seqlens), extra_rows=extra_rows, seed=seed, **kw)


@pytest.mark.parametrize("coff", [1, 2])
def test_constant_kv_windows_return_the_constant(coff):
    c = random_case(coff=coff)
    D = c.head_dim
    const = w.to_bf16_bits(np.linspace(-3.0, 5.0, D))
    for h in range(coff):
        c.kv[:, h * D:(h + 1) * D] = const[None, :]
    out32 = F(oracle.case_fwd_f32(c))
    assert np.array_equal(out32, np.broadcast_to(F(const), out32.shape))
    out64 = oracle.case_fwd_f64(c)
    np.testing.assert_allclose(out64, np.broadcast_to(F(const).astype(np.float64), out64.shape), rtol=1e-15)


@pytest.mark.parametrize("coff", [1, 2])
def test_uniform_logits_give_block_means(coff):
    ratio, D = 4, 8
    lens = [23]  # 5 blocks, tail of 3
    c = w.make_case("uniform", ratio, coff, D, lens, extra_rows=1, seed=5)
    c.score[:] = 0
    c.ape[:] = 0
    kvf = F(c.kv).astype(np.float64)
    nb = lens[0] // ratio
    own = kvf[:nb * ratio].reshape(nb, ratio, coff * D)
    want = np.empty((nb + 1, D))
    if coff == 1:
        want[:nb] = own.mean(axis=1)
    else:
        want[0] = own[0, :, D:].mean(axis=0)
        want[1:nb] = np.concatenate([own[:-1, :, :D], own[1:, :, D:]], axis=1).mean(axis=1)
    want[nb] = want[0]  # padding row: a first block from token 0
    np.testing.assert_allclose(oracle.case_fwd_f64(c), want, rtol=1e-14, atol=1e-14)
    got32 = F(oracle.case_fwd_f32(c)).astype(np.float64)
    assert np.all(np.abs(got32 - want) <= np.abs(want) * 2.0 ** -8 + 1e-30)


def test_ratio_one_own_block_is_identity():
    c = w.make_case("id", 1, 1, 8, [5, 7], extra_rows=2, seed=9)
    R = c.n_real_rows
    out = oracle.case_fwd_f32(c)
    assert np.array_equal(out[:R], c.kv[:R])
    dkv, dsc, dape = oracle.case_bwd_f32(c)
    assert np.array_equal(dkv[:R], c.grad_out[:R])
    assert not dsc.any() and not dape.any()


def test_softmax_weights_sum_to_one():
    c = random_case()
    c.kv[:] = w.to_bf16_bits(np.ones(1))[0]
    assert np.all(F(oracle.case_fwd_f32(c)) == 1.0)
    np.testing.assert_allclose(oracle.case_fwd_f64(c), 1.0, rtol=0, atol=1e-15 * 8)


def test_first_block_equals_own_block_form_on_second_half():
    c2 = random_case(coff=2)
    D = c2.head_dim
    c1 = w.Case("own", c2.ratio, 1, D, c2.seqlens, c2.capacity, c2.n_tokens, c2.cu_seqlens,
                c2.cu_seqlens_comp, np.ascontiguousarray(c2.kv[:, D:]), np.ascontiguousarray(c2.score[:, D:]),
                np.ascontiguousarray(c2.ape[:, D:]), c2.grad_out)
    firsts = sorted(set(int(x) for x in c2.cu_seqlens_comp[:-1]
                        if x < c2.cu_seqlens_comp[-1]) | set(range(c2.n_real_rows, c2.capacity)))
    firsts = [r for r in firsts if r < c2.capacity and (r >= c2.n_real_rows or
              any(c2.cu_seqlens_comp[s] == r < c2.cu_seqlens_comp[s + 1] for s in range(c2.n_seg)))]
    assert len(firsts) >= 3
    a, b = oracle.case_fwd_f32(c2), oracle.case_fwd_f32(c1)
    assert np.array_equal(a[firsts], b[firsts])
    a, b = oracle.case_fwd_f64(c2), oracle.case_fwd_f64(c1)
    assert np.array_equal(a[firsts], b[firsts])
    others = [r for r in range(c2.n_real_rows) if r not in firsts]
    assert not np.array_equal(a[others], b[others])  # the overlap matters elsewhere


def test_padding_rows_are_first_blocks_from_token_zero_and_carry_no_gradient():
    c = random_case(extra_rows=4)
    R = c.n_real_rows
    out32, out64 = oracle.case_fwd_f32(c), oracle.case_fwd_f64(c)
    for r in range(R, c.capacity):
        assert np.array_equal(out32[r], out32[0]) and np.array_equal(out64[r], out64[0])
    base = oracle.case_bwd_f32(c)
    c.grad_out[R:] = w.to_bf16_bits(np.full((c.capacity - R, c.head_dim), 1e30))
    again = oracle.case_bwd_f32(c)
    for x, y in zip(base, again):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("k", [6, -3])
def test_power_of_two_scaling_is_exact(k):
    s = 2.0 ** k
    c0 = w.tiny()
    ck = w.make_case("tiny_s", 4, 2, 64, [37, 64], extra_rows=3, seed=0, kv_scale=s, grad_scale=s)
    o0, ok = F(oracle.case_fwd_f32(c0)), F(oracle.case_fwd_f32(ck))
    assert np.array_equal(ok, o0 * np.float32(s))
    (a0, b0, d0), (ak, bk, dk) = oracle.case_bwd_f32(c0), oracle.case_bwd_f32(ck)
    assert np.array_equal(F(ak), F(a0) * np.float32(s))
    assert np.array_equal(F(bk), F(b0) * np.float32(s * s))
    assert np.array_equal(dk, d0 * np.float32(s * s))


def _overflow_toy(poison_col):
    """ratio 2, coff 2, head_dim 2, one 8-token segment (rows 0-3), one padding row;
    score = bf16 max and ape = FLT_MAX on one packed column: fp32 score+ape = +inf."""
    c = w.make_case("ovf", 2, 2, 2, [8], extra_rows=1, seed=11)
    w.poison_columns(c, [poison_col])
    return c


def test_nonfinite_propagation_first_half_column():
    c = _overflow_toy(0)
    out = F(oracle.case_fwd_f32(c))
    want = np.zeros(out.shape, bool)
    want[1:4, 0] = True  # rows with a previous block read column 0; first blocks do not
    assert np.array_equal(np.isnan(out), want)
    dkv, dsc, dape = oracle.case_bwd_f32(c)
    grad_nan = np.zeros((8, 4), bool)
    grad_nan[0:6, 0] = True  # previous-block slots of rows 1-3
    grad_nan[2:8, 2] = True  # own-block slots of rows 1-3
    assert np.array_equal(np.isnan(F(dkv)), grad_nan)
    assert np.array_equal(np.isnan(F(dsc)), grad_nan)
    ape_nan = np.zeros((2, 4), bool)
    ape_nan[:, [0, 2]] = True
    assert np.array_equal(np.isnan(dape), ape_nan)
    # the fp64 oracle has no fp32 overflow: it stays finite
    assert np.isfinite(oracle.case_fwd_f64(c)).all()
    assert all(np.isfinite(x).all() for x in oracle.case_bwd_f64(c))


def test_nonfinite_propagation_second_half_column():
    c = _overflow_toy(3)
    out = F(oracle.case_fwd_f32(c))
    want = np.zeros(out.shape, bool)
    want[:, 1] = True  # every row (padding included) reads column 3 for output column 1
    assert np.array_equal(np.isnan(out), want)
    dkv, dsc, dape = oracle.case_bwd_f32(c)
    grad_nan = np.zeros((8, 4), bool)
    grad_nan[0:8, 3] = True
    grad_nan[0:6, 1] = True
    assert np.array_equal(np.isnan(F(dkv)), grad_nan)
    assert np.array_equal(np.isnan(F(dsc)), grad_nan)
    ape_nan = np.zeros((2, 4), bool)
    ape_nan[:, [1, 3]] = True
    assert np.array_equal(np.isnan(dape), ape_nan)


@pytest.mark.parametrize("coff", [1, 2])
def test_backward_matches_central_finite_differences(coff):
    ratio, D = 2, 2
    c = w.make_case("fd", ratio, coff, D, [5, 3, 1], extra_rows=1, seed=21)
    cu, cc = c.cu_seqlens, c.cu_seqlens_comp
    kv = F(c.kv).astype(np.float64)
    sc = F(c.score).astype(np.float64)
    ap = c.ape.astype(np.float64)
    g = F(c.grad_out).astype(np.float64)
    R = c.n_real_rows

    def loss(kv_, sc_, ap_):
        out, _ = gather.forward_float(kv_, sc_, ap_, cu, cc, ratio, coff, D, c.capacity)
        return float((out[:R] * g[:R]).sum())

    dkv, dsc, dape = gather.backward_float(kv, sc, ap, cu, cc, ratio, coff, D, c.capacity, c.n_tokens, g)
    for arr, grad, which in ((kv, dkv, 0), (sc, dsc, 1), (ap, dape, 2)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            h = 1e-6 * max(1.0, abs(arr[idx]))
            args_p = [kv.copy(), sc.copy(), ap.copy()]
            args_m = [kv.copy(), sc.copy(), ap.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)
    # and the loop oracle's fp64 backward is the same gradient
    for x, y in zip(oracle.case_bwd_f64(c), (dkv, dsc, dape)):
        np.testing.assert_allclose(x, y, rtol=1e-13, atol=1e-14)


def test_fp32_order_is_within_the_pages_tolerance_of_fp64():
    """The fp32 oracle against the fp64 one on the page's gate distribution:
    differing bf16 elements <= max(1, 0.1%), max_abs <= 1.6e-2; grad_ape within
    1e-5 (normwise) of fp64."""
    c = w.make_case("mid", 4, 2, 64, [512] * 6 + [37, 3], extra_rows=16, seed=2)
    out32, out64 = oracle.case_fwd_f32(c), oracle.case_fwd_f64(c)
    dkv, dsc, dape = oracle.case_bwd_f32(c)
    dkv64, dsc64, dape64 = oracle.case_bwd_f64(c)
    for got, ref in ((out32, out64), (dkv, dkv64), (dsc, dsc64)):
        diff = got != w.to_bf16_bits(ref)
        assert diff.sum() <= max(1, 0.001 * diff.size)
        assert np.abs(F(got) - F(w.to_bf16_bits(ref))).max() <= 1.6e-2
    assert np.abs(dape - dape64).max() <= 1e-5 * np.abs(dape64).max()


def test_output_rounding_is_nearest_even():
    """One final bf16 rounding, to nearest with ties to even (IEEE 754 default):
    a two-token uniform window whose fp32 mean lies exactly halfway between two bf16
    values rounds to the even one."""
    c = w.make_case("tie", 2, 1, 2, [2], seed=1)
    c.score[:] = 0
    c.ape[:] = 0
    # column 0: mean(1, 1 + 2^-7) = 1 + 2^-8, halfway between 1 and 1 + 2^-7 -> 1 (even)
    # column 1: mean(1 + 2^-7, 1 + 2^-6) = 1 + 3*2^-8, halfway -> 1 + 2^-6 (even)
    c.kv[:] = w.to_bf16_bits(np.array([[1.0, 1.0 + 2 ** -7], [1.0 + 2 ** -7, 1.0 + 2 ** -6]]))
    out = F(oracle.case_fwd_f32(c))
    assert out[0, 0] == 1.0 and out[0, 1] == 1.0 + 2 ** -6
