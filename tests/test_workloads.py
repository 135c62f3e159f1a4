"""The seeded input generators (csa_workloads), pinned to their published
definitions: both the oracle and the GPU tests draw every input from them."""
import numpy as np

import csa_workloads as w


def test_splitmix64_matches_its_published_sequence():
    """Key 0 gives the plain SplitMix64 sequence from state 0 (state += 0x9E3779B97F4A7C15,
    then the finaliser), whose first outputs are the generator's well-known test values."""
    got = [int(x) for x in w.splitmix64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_is_counter_based():
    """Value i of a stream does not depend on how the stream is cut into calls."""
    a = w.splitmix64(7, w.STREAM_KV, 1000)
    b = np.concatenate([w.splitmix64(7, w.STREAM_KV, 300), w.splitmix64(7, w.STREAM_KV, 700, offset=300)])
    assert np.array_equal(a, b)
    assert not np.array_equal(a, w.splitmix64(7, w.STREAM_SCORE, 1000))


def test_uniforms_in_the_open_unit_interval():
    u = w.uniform01(3, 1, 100000)
    assert u.min() > 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 5e-3


def test_normals_have_the_stated_moments():
    z = w.normal(0, w.STREAM_SCORE, 400000, sigma=1.5)
    assert abs(z.mean()) < 1e-2 and abs(z.std() - 1.5) < 1e-2


def test_bf16_rounding_matches_torch():
    """Round to nearest, ties to even, against PyTorch's own float32 -> bfloat16
    conversion: random values, exact ties, values near the overflow threshold and
    the specials."""
    import torch
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        # exact ties between two bf16 neighbours (low 16 bits 0x8000), both parities
        (np.arange(0x3F800000, 0x3F800000 + 64 * 0x10000, 0x10000, dtype=np.uint32) + 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1e-40, -1e-40, 3.3895e38, -3.3895e38, 3.4e38, np.inf, -np.inf], np.float32),
    ])
    ours = w.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert w.to_bf16_bits(np.array([np.nan], np.float32))[0] & 0x7F80 == 0x7F80  # stays a NaN
