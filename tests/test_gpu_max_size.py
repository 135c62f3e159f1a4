"""Largest supported packs: n_tokens * coff * head_dim just below 2^31, the limit of
the int32 flat offsets the C ABI checks.  The packs are one segment of zeros
(cheap to create on the device); a few rows spread over it, including the last
real row and the padding row, get random windows and gradients from small seeded
cases, and those rows, their tokens' gradients, the zero-filled tail and grad_ape
are compared.  Rows with a zero
gradient contribute exact zeros to grad_ape, so it equals the sum of the small
cases' grad_ape.  The reference for the sampled rows is the same small case run
alone (bitwise: same kernels and orders, only the offsets differ), itself checked
bit for bit against the fp32 oracle for every ratio but 128 (whose contract is a
tolerance, tested elsewhere)."""
import numpy as np
import pytest

import csa_workloads as w
import oracle
from gpu_util import Dev, run_bwd, run_fwd, up

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import sparse_attention_kv_csa_gb300 as m
    return m


@pytest.mark.parametrize("ratio,coff,head_dim", [(4, 2, 512), (128, 1, 512), (16, 2, 512)])
def test_largest_pack(csa, ratio, coff, head_dim):
    import torch
    C = coff * head_dim
    T = (2 ** 31 - 1) // C
    R = T // ratio
    cap = R + 1
    assert csa.csa_check_support(ratio, coff, head_dim, T, cap) == 0
    assert csa.csa_check_support(ratio, coff, head_dim, T + 1, cap) == 4  # one more token overflows
    dev = "cuda"
    kv = torch.zeros((T, C), dtype=torch.int16, device=dev)
    sc = torch.zeros((T, C), dtype=torch.int16, device=dev)
    g = torch.zeros((cap, head_dim), dtype=torch.int16, device=dev)
    ape_np = w.normal(7, w.STREAM_APE, ratio * C, 0.25).astype(np.float32).reshape(ratio, C)
    ape = up(ape_np)
    cu = up(np.array([0, T], np.int32))
    cc = up(np.array([0, R], np.int32))

    # sampled rows: the first block (a one-block case), and blocks whose windows do
    # not overlap (two-block cases whose second block is the sampled row)
    sampled = [0, 2, R // 2, R - 1]
    cases = {}
    for i, r in enumerate(sampled):
        nblk = 1 if r == 0 else 2
        c = w.make_case("max%d" % i, ratio, coff, head_dim, [nblk * ratio], seed=50 + i)
        c.ape[:] = ape_np
        c.grad_out[: nblk - 1] = 0  # the preceding block's row carries no gradient
        t0 = (r - nblk + 1) * ratio
        kv[t0:t0 + nblk * ratio] = up(c.kv)
        sc[t0:t0 + nblk * ratio] = up(c.score)
        g[r] = up(c.grad_out[nblk - 1])
        cases[r] = (c, t0, nblk)

    out = torch.empty((cap, head_dim), dtype=torch.int16, device=dev)
    csa.csa_compress_fwd(kv, sc, ape, cu, cc, 1, ratio, coff, head_dim, cap, out)
    dkv = torch.full((T, C), -1, dtype=torch.int16, device=dev)
    dsc = torch.full((T, C), -1, dtype=torch.int16, device=dev)
    dape = torch.full((ratio, C), float("nan"), dtype=torch.float32, device=dev)
    csa.csa_compress_bwd(kv, sc, ape, cu, cc, 1, ratio, coff, head_dim, cap, T, g, dkv, dsc, dape)
    torch.cuda.synchronize()
    assert csa.csa_device_status() == 0

    bits = lambda t: t.cpu().numpy().view(np.uint16)
    want_dape = np.zeros((ratio, C), np.float64)
    for r, (c, t0, nblk) in cases.items():
        # the same rows computed on the small case alone: bitwise what the big pack
        # gives (same kernels, same orders, offsets apart); for every ratio but 128
        # that is also the fp32 oracle bit for bit
        d = Dev(c)
        small_out = run_fwd(d, csa)
        small_dkv, small_dsc, small_dape = run_bwd(d, csa)
        if ratio != 128:
            assert np.array_equal(small_out, oracle.case_fwd_f32(c))
            dk, ds, _ = oracle.case_bwd_f32(c)
            assert np.array_equal(small_dkv, dk) and np.array_equal(small_dsc, ds)
        n = nblk * ratio
        assert np.array_equal(bits(out[r]), small_out[nblk - 1]), r
        # slots that rows with a zero gradient write are +-0 depending on the signs in
        # their (different) windows: compare with the sign of zero ignored
        z = lambda a: np.where((a & 0x7FFF) == 0, 0, a)
        assert np.array_equal(z(bits(dkv[t0:t0 + n])), z(small_dkv)), r
        assert np.array_equal(z(bits(dsc[t0:t0 + n])), z(small_dsc)), r
        want_dape += small_dape
        if r == 0:  # the padding row is a first block from token 0: row 0's window
            assert np.array_equal(bits(out[R]), small_out[0])
    got_dape = dape.cpu().numpy().astype(np.float64)
    assert np.abs(got_dape - want_dape).max() <= 1e-5 * np.abs(want_dape).max()
    # the dropped tail at the highest offsets and a zero region get exact zeros
    tail = T - R * ratio
    if tail:
        assert not bits(dkv[R * ratio:]).any() and not bits(dsc[R * ratio:]).any()
    mid = (R // 4) * ratio
    assert not bits(dkv[mid:mid + 2 * ratio]).any()
    del kv, sc, dkv, dsc, out
    torch.cuda.empty_cache()
