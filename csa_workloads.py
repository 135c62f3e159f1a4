"""Seeded synthetic inputs for the CSA fused Compressor.

This module only draws inputs: segment lengths, packed ``cu_seqlens`` /
``cu_seqlens_comp`` offsets and the random kv / score / ape / grad_out tensors.
It holds none of the Compressor's arithmetic, so the CPU oracle and the CUDA
library can both be fed from it without sharing any of the method.

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) run as a counter-based generator
(value i of stream ``seed`` is the SplitMix64 finaliser of ``seed*GOLDEN +
(i+1)*GOLDEN``), turned into normals with the Box-Muller transform and rounded
to bf16 with round-to-nearest-even.  The uniform draws are bit-identical on
every platform; the normals go through the platform's log/sqrt/cos/sin, which
may differ in a last fp64 ulp between machines (rarely moving a bf16 rounding).
Tests always draw oracle and GPU inputs in the same process.

Distributions follow the Numerics section of the "CSA Fused Compressor" page
(cuDNN frontend docs): kv, grad_out ~ N(0, 1) bf16, score ~ N(0, 1.5^2) bf16,
ape ~ N(0, 0.25^2) fp32.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Per-tensor stream ids, so that each tensor of a case has its own stream.
STREAM_KV = 1
STREAM_SCORE = 2
STREAM_APE = 3
STREAM_GRAD = 4
STREAM_LENGTHS = 5


def splitmix64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n uint64 values of the counter-based SplitMix64 stream (seed, stream)."""
    key = np.uint64((seed * 0x100000001B3 + stream * 0x9E3779B1) & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = key * _GOLDEN + ctr * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n doubles in (0, 1): the top 53 bits of each draw, shifted off zero."""
    z = splitmix64(seed, stream, n, offset)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, n: int, sigma: float = 1.0, chunk: int = 1 << 18) -> np.ndarray:
    """n N(0, sigma^2) doubles by Box-Muller: draws 2i and 2i+1 of the stream give
    normals 2i (cosine) and 2i+1 (sine).  Computed in cache-sized chunks; the
    generator is counter-based, so the chunks are independent and run on a pool of
    threads (numpy releases the interpreter lock in its array operations), with the
    same values as a sequential pass."""
    m = (n + 1) // 2
    z = np.empty(2 * m, dtype=np.float64)

    def one(s0):
        s1 = min(m, s0 + chunk)
        u = uniform01(seed, stream, 2 * (s1 - s0), offset=2 * s0)
        rad = np.sqrt(-2.0 * np.log(u[0::2]))
        ang = 2.0 * np.pi * u[1::2]
        z[2 * s0:2 * s1:2] = rad * np.cos(ang)
        z[2 * s0 + 1:2 * s1:2] = rad * np.sin(ang)

    starts = range(0, m, chunk)
    if len(starts) > 1:
        with concurrent.futures.ThreadPoolExecutor(min(len(starts), os.cpu_count() or 1, 32)) as ex:
            list(ex.map(one, starts))
    elif m:
        one(0)
    z = z[:n]
    if sigma != 1.0:
        z *= sigma
    return z


def _bf16_chunk(x: np.ndarray) -> np.ndarray:
    f = np.array(x, dtype=np.float32, copy=True, order="C")
    u = f.view(np.uint32)
    nan = np.isnan(f)
    lsb = u >> np.uint32(16)
    lsb &= np.uint32(1)
    lsb += np.uint32(0x7FFF)
    u += lsb  # no wrap: the largest non-NaN pattern is 0xFF800000 (-inf)
    u >>= np.uint32(16)
    r = u.astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def to_bf16_bits(x: np.ndarray, chunk: int = 1 << 20) -> np.ndarray:
    """Round float values to bf16 (nearest, ties to even); returns uint16 bit patterns.
    Elementwise, so large arrays are cut into chunks converted on a pool of threads."""
    x = np.asarray(x)
    if x.size <= chunk:
        return _bf16_chunk(x)
    flat = x.reshape(-1)
    out = np.empty(flat.size, dtype=np.uint16)

    def one(s0):
        out[s0:s0 + chunk] = _bf16_chunk(flat[s0:s0 + chunk])

    with concurrent.futures.ThreadPoolExecutor(min(os.cpu_count() or 1, 32)) as ex:
        list(ex.map(one, range(0, flat.size, chunk)))
    return out.reshape(x.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Case:
    """One Compressor problem: THD offsets plus the random tensors (host numpy)."""
    name: str
    ratio: int
    coff: int
    head_dim: int
    seqlens: list
    capacity: int
    n_tokens: int
    cu_seqlens: np.ndarray       # int32 [n_seg+1]
    cu_seqlens_comp: np.ndarray  # int32 [n_seg+1]
    kv: np.ndarray               # uint16 (bf16 bits) [n_tokens, coff*head_dim]
    score: np.ndarray            # uint16 (bf16 bits) [n_tokens, coff*head_dim]
    ape: np.ndarray              # float32 [ratio, coff*head_dim]
    grad_out: np.ndarray         # uint16 (bf16 bits) [capacity, head_dim]

    @property
    def n_seg(self) -> int:
        return len(self.seqlens)

    @property
    def n_real_rows(self) -> int:
        return int(self.cu_seqlens_comp[-1])

    @property
    def width(self) -> int:
        return self.coff * self.head_dim


def offsets(seqlens, ratio: int, leading: int = 0):
    """cu_seqlens (cumulative lengths, starting at ``leading``) and cu_seqlens_comp
    (cumulative floor(len/ratio): each segment's tail tokens form no row)."""
    cu = np.zeros(len(seqlens) + 1, dtype=np.int64)
    cu[0] = leading
    cu[1:] = leading + np.cumsum(np.asarray(seqlens, dtype=np.int64))
    cc = np.zeros(len(seqlens) + 1, dtype=np.int64)
    cc[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64) // ratio)
    return cu.astype(np.int32), cc.astype(np.int32)


def make_case(name, ratio, coff, head_dim, seqlens, capacity=None, extra_rows=0,
              n_tokens=None, leading=0, seed=0, kv_scale=1.0, grad_scale=1.0,
              score_sigma=1.5, ape_sigma=0.25) -> Case:
    """Draw one case.  ``capacity`` defaults to the real row count + ``extra_rows``;
    ``n_tokens`` defaults to cu_seqlens[-1] (no token padding)."""
    cu, cc = offsets(seqlens, ratio, leading)
    rows = int(cc[-1])
    cap = rows + extra_rows if capacity is None else int(capacity)
    T = int(cu[-1]) if n_tokens is None else int(n_tokens)
    C = coff * head_dim
    kv = to_bf16_bits(normal(seed, STREAM_KV, T * C) * kv_scale).reshape(T, C)
    score = to_bf16_bits(normal(seed, STREAM_SCORE, T * C, score_sigma)).reshape(T, C)
    ape = normal(seed, STREAM_APE, ratio * C, ape_sigma).astype(np.float32).reshape(ratio, C)
    grad = to_bf16_bits(normal(seed, STREAM_GRAD, cap * head_dim) * grad_scale).reshape(cap, head_dim)
    return Case(name, ratio, coff, head_dim, list(seqlens), cap, T, cu, cc, kv, score, ape, grad)


# --- the workloads ---------------------------------------------------------

def ragged_lengths(seed: int, n_seg: int = 64, max_len: int = 8192, ratio: int = 4,
                   n_short: int = 4) -> list:
    """Lengths uniform in [1, max_len]; then ``n_short`` distinct segments (chosen from
    the same stream) are redrawn uniform in [1, ratio-1], so that some segments are
    shorter than ratio (uniform draws alone almost never give one)."""
    u = iter(uniform01(seed, STREAM_LENGTHS, n_seg + 64 * n_short + 64))
    lens = [1 + int(next(u) * max_len) for _ in range(n_seg)]
    picked = []
    while len(picked) < min(n_short, n_seg):
        idx = int(next(u) * n_seg)
        if idx not in picked:
            picked.append(idx)
    for p in picked:
        lens[p] = 1 + int(next(u) * (ratio - 1))
    return lens


# Each workload as make_case keyword arguments (shapes only, no data drawn).
SPECS = {
    # ratio 4, coff 2, head_dim 64, segments [37, 64], 3 padding rows
    "tiny": lambda seed=0: dict(name="tiny", ratio=4, coff=2, head_dim=64, seqlens=[37, 64], extra_rows=3),
    # ratio 4, coff 2, head_dim 512, 8 segments of 4096 tokens, capacity 8256
    "r4c2d512_8x4096": lambda seed=0: dict(name="r4c2d512_8x4096", ratio=4, coff=2, head_dim=512,
                                           seqlens=[4096] * 8, capacity=8256),
    # ratio 4, coff 2, head_dim 512, 64 ragged segments, capacity = rows + 128
    "r4c2d512_ragged64": lambda seed=0: dict(name="r4c2d512_ragged64", ratio=4, coff=2, head_dim=512,
                                             seqlens=ragged_lengths(seed), extra_rows=128),
    # ratio 128, coff 1, head_dim 512, 4 segments of 32768 tokens (1024 rows)
    "r128c1d512_4x32768": lambda seed=0: dict(name="r128c1d512_4x32768", ratio=128, coff=1, head_dim=512,
                                              seqlens=[32768] * 4),
    # ratio 4, coff 2, head_dim 512, one 131072-token segment: unit scale, kv and
    # grad_out x64, and fp32 overflow (see poison_columns)
    "stress_unit": lambda seed=0: dict(name="stress_unit", ratio=4, coff=2, head_dim=512, seqlens=[131072]),
    "stress_x64": lambda seed=0: dict(name="stress_x64", ratio=4, coff=2, head_dim=512, seqlens=[131072],
                                      kv_scale=64.0, grad_scale=64.0),
    "stress_overflow": lambda seed=0: dict(name="stress_overflow", ratio=4, coff=2, head_dim=512,
                                           seqlens=[131072]),
    # ratio 128 with the overlapping window (coff 2, window 256), head_dim 512
    "r128c2d512_4x32768": lambda seed=0: dict(name="r128c2d512_4x32768", ratio=128, coff=2, head_dim=512,
                                              seqlens=[32768] * 4),
    # a head_dim that is not a multiple of 128 (register-window kernels): ratio 4,
    # coff 2, head_dim 64, 32 segments of 4096 tokens
    "r4c2d64_32x4096": lambda seed=0: dict(name="r4c2d64_32x4096", ratio=4, coff=2, head_dim=64,
                                           seqlens=[4096] * 32),
    # head_dim 128 (the page's other head size), ratio 4, coff 2, 32 x 4096 tokens
    "r4c2d128_32x4096": lambda seed=0: dict(name="r4c2d128_32x4096", ratio=4, coff=2, head_dim=128,
                                            seqlens=[4096] * 32),
    # head_dim 256, ratio 4, coff 2, 16 x 4096 tokens
    "r4c2d256_16x4096": lambda seed=0: dict(name="r4c2d256_16x4096", ratio=4, coff=2, head_dim=256,
                                            seqlens=[4096] * 16),
    # the own-block window (coff 1): ratio 4, head_dim 512, 16 x 4096 tokens
    "r4c1d512_16x4096": lambda seed=0: dict(name="r4c1d512_16x4096", ratio=4, coff=1, head_dim=512,
                                            seqlens=[4096] * 16),
    # head_dim 128 at ratio 128, coff 1, 4 x 131072 tokens
    "r128c1d128_4x131072": lambda seed=0: dict(name="r128c1d128_4x131072", ratio=128, coff=1, head_dim=128,
                                               seqlens=[131072] * 4),
    # ratio 8 (generic kernels), coff 2, head_dim 512, 8 segments of 4096 tokens
    "r8c2d512_8x4096": lambda seed=0: dict(name="r8c2d512_8x4096", ratio=8, coff=2, head_dim=512,
                                           seqlens=[4096] * 8),
    # a ratio served by the generic kernels: ratio 16, coff 2, head_dim 512,
    # 8 segments of 4096 tokens (2048 rows), 64 padding rows
    "r16c2d512_8x4096": lambda seed=0: dict(name="r16c2d512_8x4096", ratio=16, coff=2, head_dim=512,
                                            seqlens=[4096] * 8, extra_rows=64),
    # windows of more than 64 positions at ratios other than 128 (chunked kernels):
    # ratio 64 with the overlapping window (128 positions), 8 x 4096 tokens, 16
    # padding rows; ratio 96 with the own-block window, 8 x 6144 tokens
    "r64c2d512_8x4096": lambda seed=0: dict(name="r64c2d512_8x4096", ratio=64, coff=2, head_dim=512,
                                            seqlens=[4096] * 8, extra_rows=16),
    "r96c1d512_8x6144": lambda seed=0: dict(name="r96c1d512_8x6144", ratio=96, coff=1, head_dim=512,
                                            seqlens=[6144] * 8),
    # head_dims that are not multiples of 64: ratio 4 (register-window kernels,
    # head_dim 96) and ratio 16 (the generic kernel that walks the window from
    # global memory, head_dim 200)
    "r4c2d96_32x4096": lambda seed=0: dict(name="r4c2d96_32x4096", ratio=4, coff=2, head_dim=96,
                                           seqlens=[4096] * 32),
    "r16c2d200_8x4096": lambda seed=0: dict(name="r16c2d200_8x4096", ratio=16, coff=2, head_dim=200,
                                            seqlens=[4096] * 8),
}


# The shapes the Compressor page publishes kernel times for (B200; context for
# the same shapes here): ratio 4, coff 2 packs of 8192-token sequences, and
# ratio-128 single sequences -- (ratio, coff, head_dim, segments, tokens each).
PAGE_SHAPES = [(4, 2, 128, 1, 8192), (4, 2, 128, 3, 8192), (4, 2, 512, 1, 8192), (4, 2, 512, 3, 8192),
               (128, 1, 128, 1, 8192), (128, 1, 128, 1, 131072), (128, 2, 128, 1, 8192), (128, 2, 128, 1, 65536),
               (128, 1, 512, 1, 65536), (128, 2, 512, 1, 65536), (128, 2, 512, 1, 131072)]


def _page_spec(nm, r, c, d, n, length):
    return lambda seed=0: dict(name=nm, ratio=r, coff=c, head_dim=d, seqlens=[length] * n)


for _shape in PAGE_SHAPES:
    _nm = "r%dc%dd%d_%dx%d" % _shape
    SPECS[_nm] = _page_spec(_nm, *_shape)

def build(name: str, seed: int = 0) -> Case:
    kw = SPECS[name](seed)
    nm = kw.pop("name")
    c = make_case(nm, seed=seed, **kw)
    if name == "stress_overflow":
        poison_columns(c, [0, 1, c.head_dim, c.head_dim + 1])
    return c


def tiny(seed=0) -> Case:
    return build("tiny", seed)


def uniform8x4096(seed=0) -> Case:
    return build("r4c2d512_8x4096", seed)


def ragged64(seed=0) -> Case:
    return build("r4c2d512_ragged64", seed)


def r128_4x32768(seed=0) -> Case:
    return build("r128c1d512_4x32768", seed)


def poison_columns(c: Case, cols) -> None:
    """Overflow inputs: score = largest finite bf16 (0x7F7F) and ape = FLT_MAX in the
    given packed columns, so that fp32 score + ape is +inf there."""
    for col in cols:
        c.score[:, col] = 0x7F7F
        c.ape[:, col] = np.finfo(np.float32).max
    c.name += "_cols" + "-".join(str(x) for x in cols)


class _Workloads(dict):
    """name -> callable(seed=0) drawing that workload."""


WORKLOADS = _Workloads({name: (lambda name: (lambda seed=0: build(name, seed)))(name) for name in SPECS})
