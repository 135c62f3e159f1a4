"""csa_compress_bwd_noalloc: the backward for callers that cannot allocate device
memory inside the call (its scratch is a fixed array in the library's device
code).  Checked through the C ABI against csa_compress_bwd on the same inputs,
for two calls in a row (the second on different data, so that anything the
first call left in the shared scratch would show), in every kernel family.  For
every ratio but 128 the grid, and so the grad_ape grouping, is the regular call's:
all four outputs are compared bit for bit.  Ratio 128 may run fewer row blocks
(its grad_ape is then the same sum in another grouping).

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import csa_workloads as w
from gpu_util import Dev, F, check_dape, run_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import sparse_attention_kv_csa_gb300 as m
    return m


def run_noalloc(d, csa, canary, n_tokens=None, capacity=None):
    import torch
    c = d.c
    C = c.coff * c.head_dim
    cap = c.capacity if capacity is None else capacity
    fill = np.int16(np.uint16(canary).view(np.int16))
    dkv = torch.full((c.n_tokens, C), fill, dtype=torch.int16, device="cuda")
    dsc = torch.full((c.n_tokens, C), fill, dtype=torch.int16, device="cuda")
    dape = torch.full((c.ratio, C), float("nan"), dtype=torch.float32, device="cuda")
    csa.csa_compress_bwd_noalloc(d.kv, d.score, d.ape, d.cu, d.cc, c.n_seg, c.ratio, c.coff, c.head_dim,
                                 cap, c.n_tokens if n_tokens is None else n_tokens, d.g, dkv, dsc, dape)
    torch.cuda.synchronize()
    return dkv.cpu().numpy().view(np.uint16), dsc.cpu().numpy().view(np.uint16), dape.cpu().numpy()


@pytest.mark.parametrize("head_dim", [512, 64, 96])  # bulk-copy pipeline (two / one pairs) / register kernels
def test_noalloc_matches_backward_two_calls_in_a_row(csa, head_dim):
    cases = [w.make_case("na%d" % s, 4, 2, head_dim, [4096, 37, 2, 1100], extra_rows=16, seed=s)
             for s in (31, 32)]
    for c, canary in zip(cases, (0xFFFF, 0x7FC1)):
        d = Dev(c)
        want_dkv, want_dsc, want_dape = run_bwd(d, csa)
        got_dkv, got_dsc, got_dape = run_noalloc(d, csa, canary)
        assert np.array_equal(got_dkv, want_dkv)
        assert np.array_equal(got_dsc, want_dsc)
        assert np.array_equal(got_dape.view(np.uint32), want_dape.view(np.uint32))
        check_dape(c, got_dape, csa)
    assert csa.csa_device_status() == 0


def test_noalloc_large_shape_then_small_shape(csa):
    """A large call fills many partials of the shared array; a smaller call right
    after it must read none of them (it writes every partial it reads)."""
    big = w.make_case("na_big4", 4, 2, 512, [4096] * 8, extra_rows=64, seed=41)
    small = w.make_case("na_small4", 4, 2, 512, [37, 9], extra_rows=1, seed=42)
    run_noalloc(Dev(big), csa, 0xFFFF)
    d = Dev(small)
    want = run_bwd(d, csa)
    got = run_noalloc(d, csa, 0x7FC1)
    for a, b in zip(got[:2], want[:2]):
        assert np.array_equal(a, b)
    assert np.array_equal(got[2].view(np.uint32), want[2].view(np.uint32))
    check_dape(small, got[2], csa)


def test_noalloc_capacity_zero_and_device_token_count(csa):
    """capacity 0: grad_kv / grad_score all +0 and grad_ape = 0, as the regular call.
    n_tokens = -1: the token count cu_seqlens[n_seg] is read on the device; token
    padding rows past it are left untouched (their canary survives)."""
    c0 = w.make_case("na_cap0", 4, 2, 64, [3, 2], capacity=0, seed=43)  # no real rows
    dkv, dsc, dape = run_noalloc(Dev(c0), csa, 0xFFFF, capacity=0)
    assert not dkv.any() and not dsc.any() and not dape.any()
    c = w.make_case("na_tok", 4, 2, 64, [9, 14], extra_rows=2, n_tokens=27, seed=43)
    d = Dev(c)
    T = int(c.cu_seqlens[-1])
    want = run_bwd(d, csa)
    got = run_noalloc(d, csa, 0x7FC1, n_tokens=-1)
    assert np.array_equal(got[0][:T], want[0][:T]) and np.array_equal(got[1][:T], want[1][:T])
    assert (got[0][T:] == 0x7FC1).all() and (got[1][T:] == 0x7FC1).all()
    assert np.array_equal(got[2].view(np.uint32), want[2].view(np.uint32))


def test_noalloc_timeouts_reach_the_device_status(csa):
    """The no-alloc call launches its kernels with the one per-device status word
    that csa_device_status() reads (a word of the library's device code, so that no
    allocation is needed to hold it).  After a no-alloc call, a bounded wait that
    runs out (the self-test kernel, given the same word) is reported by
    csa_device_status() as CSA_ERR_DEVICE_TIMEOUT; clearing it resets it."""
    c = w.make_case("na_st", 4, 2, 512, [64, 9], extra_rows=1, seed=44)
    run_noalloc(Dev(c), csa, 0xFFFF)
    assert csa.csa_device_status() == 0
    csa.csa_selftest_bounded_wait(20_000_000)
    assert csa.csa_device_status(clear=True) == 7
    assert csa.csa_device_status() == 0


def test_noalloc_rejects_bad_arguments_before_launch(csa):
    import torch
    c = w.make_case("na_bad", 4, 2, 512, [64], seed=3)
    d = Dev(c)
    dkv = torch.zeros((c.n_tokens, 1024), dtype=torch.int16, device="cuda")
    dape = torch.zeros((4, 1024), dtype=torch.float32, device="cuda")
    with pytest.raises(csa.CSAError) as ei:
        csa.csa_compress_bwd_noalloc(d.kv, d.score, d.ape, d.cu, d.cc, c.n_seg, 4, 2, 512, c.capacity,
                                     c.n_tokens, d.g, dkv, dkv, dape.view(-1)[1:].data_ptr())
    assert ei.value.status == 3  # misaligned dape
    torch.cuda.synchronize()
    assert not dkv.any()


def test_noalloc_ratio128_matches_backward(csa):
    c = w.make_case("na128", 128, 1, 512, [4096, 300], extra_rows=3, seed=5)
    d = Dev(c)
    want = run_bwd(d, csa)
    for canary in (0xFFFF, 0x7FC1):
        got = run_noalloc(d, csa, canary)
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
        assert np.abs(got[2] - want[2]).max() <= 1e-5 * np.abs(want[2]).max()


def test_noalloc_ratio128_overlapping_window_fits_with_fewer_blocks(csa):
    """ratio 128, coff 2, head_dim 512: the regular backward's grid (19 row blocks
    per column tile) would need 19 grad_ape partials of 128 x 1024 floats, more
    than the fixed array; the no-alloc call runs 12 row blocks instead.  grad_kv
    and grad_score keep their bits; grad_ape is the same sum in another grouping."""
    c = w.make_case("na128c2", 128, 2, 512, [4096, 1500], extra_rows=3, seed=9)
    d = Dev(c)
    want = run_bwd(d, csa)
    for canary in (0xFFFF, 0x7FC1):
        got = run_noalloc(d, csa, canary)
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
        assert np.abs(got[2] - want[2]).max() <= 1e-5 * np.abs(want[2]).max()


def test_noalloc_rejects_shape_beyond_its_scratch(csa):
    """ratio 128, coff 2, head_dim 8192: one grad_ape partial is 128 x 16384 floats
    (8 MiB), more than the fixed 6 MiB array holds: rejected before launch."""
    import torch
    c = w.make_case("na_big", 128, 2, 8192, [256], seed=6)
    d = Dev(c)
    C = 2 * 8192
    dkv = torch.zeros((c.n_tokens, C), dtype=torch.int16, device="cuda")
    dape = torch.zeros((128, C), dtype=torch.float32, device="cuda")
    with pytest.raises(csa.CSAError) as ei:
        csa.csa_compress_bwd_noalloc(d.kv, d.score, d.ape, d.cu, d.cc, c.n_seg, 128, 2, 8192, c.capacity,
                                     c.n_tokens, d.g, dkv, dkv, dape)
    assert ei.value.status == 4  # CSA_ERR_TOO_LARGE
    assert "scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert not dkv.any()


def test_noalloc_generic_ratio_matches_backward(csa):
    c = w.make_case("na_gen", 16, 2, 512, [4000, 37, 600], extra_rows=5, seed=8)
    d = Dev(c)
    want = run_bwd(d, csa)
    for canary in (0xFFFF, 0x7FC1):
        got = run_noalloc(d, csa, canary)
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
        assert np.array_equal(got[2].view(np.uint32), want[2].view(np.uint32))
