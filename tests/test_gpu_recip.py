"""The kernels' softmax-denominator reciprocal on the GPU (through the C ABI's
self-test hook) against numpy's IEEE round-to-nearest 1/d: every float in [1, 2),
samples of every binade from 2^-8 to 2^8, the all-ones significands, and NaN."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _run(d):
    import torch
    import sparse_attention_kv_csa_gb300 as csa
    x = torch.from_numpy(d).cuda()
    y = torch.empty_like(x)
    csa.csa_selftest_reciprocal(x, y, x.numel())
    torch.cuda.synchronize()
    return y.cpu().numpy()


def test_reciprocal_every_float_in_one_binade():
    d = (np.arange(1 << 23, dtype=np.uint32) + np.uint32(0x3F800000)).view(np.float32)
    got = _run(d)
    want = np.float32(1) / d
    bad = got.view(np.uint32) != want.view(np.uint32)
    assert not bad.any(), (d[bad][:4], got[bad][:4], want[bad][:4])


def test_reciprocal_other_binades_and_edges():
    rng = np.random.default_rng(11)
    parts = []
    for k in range(-8, 8):
        m = rng.integers(0, 1 << 23, 1 << 20, dtype=np.uint32)
        parts.append((m | np.uint32((127 + k) << 23)).view(np.float32))
        parts.append(np.array([(np.uint32((127 + k) << 23) | np.uint32(0x7FFFFF))], dtype=np.uint32).view(np.float32))
    parts.append(np.array([2.0 ** -8, 0.99999994, 1.0, 2.0, 3.0, 7.0, 8.0, 255.99998, 256.0], dtype=np.float32))
    d = np.concatenate(parts)
    got = _run(d)
    want = np.float32(1) / d
    bad = got.view(np.uint32) != want.view(np.uint32)
    assert not bad.any(), (d[bad][:4], got[bad][:4], want[bad][:4])
    assert np.isnan(_run(np.array([np.nan, -np.nan], dtype=np.float32))).all()


def test_reciprocal_hook_rejects_bad_arguments():
    import sparse_attention_kv_csa_gb300 as csa
    with pytest.raises(csa.CSAError):
        csa.csa_selftest_reciprocal(None, None, 4)
    with pytest.raises(csa.CSAError):
        csa.csa_selftest_reciprocal(None, None, -1)
    csa.csa_selftest_reciprocal(None, None, 0)
