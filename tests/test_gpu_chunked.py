"""The chunked kernels at ratios other than 128: every window of more than 64
positions (ratio 33-127 with coff 2, 65-127 with coff 1) with head_dim a multiple
of 64.  The page gives its chunked, fast-exp evaluation a tolerance contract of its
own at ratio 128 ("CSA Fused Compressor", Numerics and section ratio=128); the
library applies that contract to every window of this length: per case no NaN,
max_abs <= 1.6e-2 against the plain fp32 and the fp64 oracles, fp64 parity no
worse than the plain fp32 evaluation, never-consumed slots exact zeros, grad_ape
within 1e-5 (normwise) of fp64; at most max(1, 0.1%) differing elements over the
union of each ratio's ragged cases; bitwise run-to-run determinism."""
import numpy as np
import pytest

import csa_workloads as w
from gpu_util import Dev, assert_counts, run_bwd, run_fwd, tolerance_counts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import sparse_attention_kv_csa_gb300 as m
    return m


def layouts(r):
    """Ragged packs in units of the ratio: tails, segments shorter than the ratio,
    exact multiples, empty segments, one long segment."""
    return [[19 * r + 3, r, 5, 30 * r + 1], [r - 1], [r], [r + 1, 0, 16 * r], [24 * r], [3, 21 * r + 7, 2]]


# every chunk-count bucket and its edges: coff 2 with windows up to 96 / 128 / 160 /
# 192 / 224 / 256 positions (12 ... 32 chunks), coff 1 up to 96 / 128 (12 / 16)
CASES = [(2, 33), (2, 40), (2, 48), (2, 49), (2, 63), (2, 64), (2, 65), (2, 80), (2, 81), (2, 96),
         (2, 100), (2, 112), (2, 113), (2, 127),
         (1, 65), (1, 80), (1, 96), (1, 97), (1, 100), (1, 127)]


@pytest.mark.parametrize("coff,ratio", CASES)
@pytest.mark.parametrize("head_dim", [64, 192])
def test_chunked_ratio_layouts(csa, coff, ratio, head_dim):
    assert csa.csa_grad_ape_order(ratio, coff, head_dim, 8)["kind"] == "chunked"
    total = [[0, 0, 0] for _ in range(3)]
    for li, lens in enumerate(layouts(ratio)):
        T = sum(lens) + (0, 7)[li % 2]
        R = sum(L // ratio for L in lens)
        extra = (0, 2, 1)[li % 3]
        if (T < ratio and R + extra > 0) or R + extra == 0:
            continue
        c = w.make_case("chk", ratio, coff, head_dim, lens, extra_rows=extra, n_tokens=T,
                        seed=1000 * coff + 10 * ratio + li)
        _, counts = tolerance_counts(c, csa)
        for t, (a, b, n) in zip(total, counts):
            t[0] += a
            t[1] += b
            t[2] += n
    assert_counts([tuple(t) for t in total])


@pytest.mark.parametrize("name", ["r64c2d512_8x4096", "r96c1d512_8x6144"])
def test_chunked_workload_tolerance_and_determinism(csa, name):
    c = w.WORKLOADS[name]()
    (out, dkv, dsc, dape), counts = tolerance_counts(c, csa)
    assert_counts(counts)
    d = Dev(c)
    assert np.array_equal(run_fwd(d, csa, canary=0x7FC1), out)
    b = run_bwd(d, csa, canary=0x7FC1, dape_fill=7.0)
    assert np.array_equal(b[0], dkv) and np.array_equal(b[1], dsc)
    assert np.array_equal(b[2].view(np.uint32), dape.view(np.uint32))


def test_zz_no_bounded_wait_expired(csa):
    """No kernel of this module recorded a timeout in the device status word."""
    assert csa.csa_device_status(clear=True) == 0
