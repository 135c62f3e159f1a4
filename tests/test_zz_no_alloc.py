"""csa_compress_bwd_noalloc: the backward for callers that cannot allocate device
memory inside the call (its scratch is a fixed array in the library's device
code).  Checked through the C ABI against csa_compress_bwd on the same inputs,
for two calls in a row (the second on different data, so that anything the
first call left in the shared scratch would show), in both kernel families.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import csa_workloads as w
from gpu_util import Dev, F, run_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import sparse_attention_kv_csa_gb300 as m
    return m


def run_noalloc(d, csa, canary):
    import torch
    c = d.c
    C = c.coff * c.head_dim
    fill = np.int16(np.uint16(canary).view(np.int16))
    dkv = torch.full((c.n_tokens, C), fill, dtype=torch.int16, device="cuda")
    dsc = torch.full((c.n_tokens, C), fill, dtype=torch.int16, device="cuda")
    dape = torch.full((c.ratio, C), float("nan"), dtype=torch.float32, device="cuda")
    csa.csa_compress_bwd_noalloc(d.kv, d.score, d.ape, d.cu, d.cc, c.n_seg, c.ratio, c.coff, c.head_dim,
                                 c.capacity, c.n_tokens, d.g, dkv, dsc, dape)
    torch.cuda.synchronize()
    return dkv.cpu().numpy().view(np.uint16), dsc.cpu().numpy().view(np.uint16), dape.cpu().numpy()


@pytest.mark.parametrize("head_dim", [512, 64])  # bulk-copy pipeline / register kernels
def test_noalloc_matches_backward_two_calls_in_a_row(csa, head_dim):
    cases = [w.make_case("na%d" % s, 4, 2, head_dim, [4096, 37, 2, 1100], extra_rows=16, seed=s)
             for s in (31, 32)]
    for c, canary in zip(cases, (0xFFFF, 0x7FC1)):
        d = Dev(c)
        want_dkv, want_dsc, want_dape = run_bwd(d, csa)
        got_dkv, got_dsc, got_dape = run_noalloc(d, csa, canary)
        assert np.array_equal(got_dkv, want_dkv)
        assert np.array_equal(got_dsc, want_dsc)
        assert np.isfinite(got_dape).all()
        assert np.abs(got_dape - want_dape).max() <= 1e-5 * np.abs(want_dape).max()
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
