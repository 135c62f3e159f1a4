// Device helpers shared by the Compressor kernels: packed fp32 pair arithmetic,
// the library's own exp, bf16 conversion and the row -> segment map.
//
// Numerics ("CSA Fused Compressor", cuDNN frontend docs, section Numerics): all
// window arithmetic is fp32 with one final bf16 rounding, and every add, multiply
// and fused multiply-add is an explicit round-to-nearest instruction, so nothing
// depends on the compiler contracting a*b+c.  The library is built without
// --use_fast_math: no flush-to-zero; the one reciprocal per output (recip_den)
// is correctly rounded.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

// ------------------------------------------------------------ fp32 pairs
// Two fp32 lanes in one float2, computed with the sm_100+ packed instructions
// (two results per issue slot).  Each lane rounds exactly like the scalar op.

__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 splat(float v) { return make_float2(v, v); }

// max that returns NaN when either input is NaN.
__device__ __forceinline__ float max_nan(float a, float b)
{
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Three-input form (sm_100 and later): NaN if any input is NaN, else the largest.
// The maximum of a set does not depend on the grouping, so a window's max may be
// taken three values at a time (a zero's sign may differ, which no use of the
// max can see: s - m and EXP treat +0 and -0 alike).
__device__ __forceinline__ float max3_nan(float a, float b, float c)
{
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ----------------------------------------------------------- reciprocal
// 1/d rounded to nearest for d in [2^-8, 2^8], which holds every softmax
// denominator here: at most 256 terms, the largest 1 or within a few ulp of it
// (NaN stays NaN).
// Seed: the hardware approximation rcp.approx, within one ulp of 1/d by the PTX
// ISA.  One Newton-Raphson correction in Markstein's fused form (P. Markstein,
// IBM J. Res. Dev. 34(1), 1990): the residual r = 1 - d*y is exact in one FMA, and
// y + y*r rounded once is the correctly rounded 1/d for every seed within one ulp,
// except when the significand of d is all ones, d = 2^k (2 - 2^-23).  There 1/d
// lies just above a rounding tie, the seed 2^(-k-1) lands on the tie, and the
// correctly rounded result 2^(-k-1) (1 + 2^-23) is the step's result with its
// lowest bit set.  Both statements hold exhaustively over one binade, and the step
// commutes with scaling by a power of two on this range (no intermediate leaves
// the normal range).
__device__ __forceinline__ float recip_den(float d)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(d));
    const float r = __fmaf_rn(-d, y, 1.0f);
    const uint32_t b = __float_as_uint(__fmaf_rn(y, r, y));
    const uint32_t tie = (~__float_as_uint(d) & 0x7fffffu) == 0u ? 1u : 0u;
    return __uint_as_float(b | tie);
}

// ------------------------------------------------------------------ exp
// e^x for x <= 0 (or NaN), the library's own: Cody-Waite reduction (Cody and
// Waite, "Software Manual for the Elementary Functions", 1980) x = n ln2 + r with
// ln2 split in two parts, |r| <= h = ln2/2; e^r by a degree-6 polynomial in Horner
// form; 2^n put into the exponent field.  Results below 2^-126.5 are +0 (n = -127
// gives a zero scale); NaN propagates.  Constants from their definitions:
//   kLog2e = 1/ln2 to fp32; kLn2Hi = ln2 cut to a 16-bit significand (so n*kLn2Hi
//   is exact); kLn2Lo = ln2 - kLn2Hi to fp32; kRound = 1.5*2^23 (adding it leaves
//   nearest(y) in the low significand bits).
// The polynomial is the degree-7 Taylor polynomial of e^r with its r^7 term
// economized over |r| <= h (Lanczos, "Applied Analysis", 1956): with x = r/h and
// the Chebyshev polynomial T7(x) = 64x^7 - 112x^5 + 56x^3 - 7x,
//   r^7 = h^7 (T7(x) + 112x^5 - 56x^3 + 7x) / 64,
// and dropping T7 (|T7| <= 1) moves 1/7! onto r^5, r^3 and r:
//   kC5 = 1/5! + (1/7!)(112/64)h^2,  kC3 = 1/3! - (1/7!)(56/64)h^4,
//   c1 = 1 + (1/7!)(7/64)h^6 = 1 in fp32 (the change is below half an ulp),
// the others 1/k!; computed in double, rounded to fp32.  Error about 7e-9
// relative (h^7/(64 7!) + h^8/8!), as small as the degree-7 Taylor polynomial's.
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2Hi = 0.693145751953125f;
constexpr float kLn2Lo = 1.42860682030941723212e-6f;
constexpr float kRound = 12582912.0f;
constexpr float kExpFloor = -88.0f;
constexpr double kHalfLn2 = 0.69314718055994530942 / 2.0;
constexpr double kHalfLn2Sq = kHalfLn2 * kHalfLn2;
constexpr float kC2 = (float)(1.0 / 2.0);
constexpr float kC3 = (float)(1.0 / 6.0 - (1.0 / 5040.0) * (56.0 / 64.0) * (kHalfLn2Sq * kHalfLn2Sq));
constexpr float kC4 = (float)(1.0 / 24.0);
constexpr float kC5 = (float)(1.0 / 120.0 + (1.0 / 5040.0) * (112.0 / 64.0) * kHalfLn2Sq);
constexpr float kC6 = (float)(1.0 / 720.0);

__device__ __forceinline__ float2 exp2lanes(float2 x)
{
    x.x = max_nan(x.x, kExpFloor);
    x.y = max_nan(x.y, kExpFloor);
    const float2 t = fma2(x, splat(kLog2e), splat(kRound));   // kRound + n
    const float2 n = add2(t, splat(-kRound));                  // n, exact
    float2 r = fma2(n, splat(-kLn2Hi), x);
    r = fma2(n, splat(-kLn2Lo), r);
    float2 p = fma2(splat(kC6), r, splat(kC5));
    p = fma2(p, r, splat(kC4));
    p = fma2(p, r, splat(kC3));
    p = fma2(p, r, splat(kC2));
    p = fma2(p, r, splat(1.0f));
    p = fma2(p, r, splat(1.0f));
    // bits(t) = bits(kRound) + n; bits(kRound) << 23 vanishes mod 2^32, so
    // (bits(t) << 23) + bias is the bit pattern of 2^n (and +0 for n = -127).
    const float2 scale = make_float2(__uint_as_float((__float_as_uint(t.x) << 23) + 0x3f800000u),
                                     __uint_as_float((__float_as_uint(t.y) << 23) + 0x3f800000u));
    return mul2(p, scale);
}

// ----------------------------------------------------------------- bf16
// Mixed-precision forms (sm_100 and later) that take bf16 operands as they are.
// Widening bf16 to fp32 is exact, so each equals its fp32 counterpart on the
// widened values bit for bit, without the two unpacking permutes per word.
// w, gw, kw: words of two bf16 (low half = lower column).

// f32(w) + a, each lane rounded once to nearest: add2(bf16x2_to_f2(w), a).
__device__ __forceinline__ float2 add2_bf16x2(uint32_t w, float2 a)
{
    float2 d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %4;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "r"(w), "f"(a.x), "f"(a.y));
    return d;
}

// f32(gw) * f32(kw) + c, each lane rounded once: fma2(bf16x2_to_f2(gw), bf16x2_to_f2(kw), c).
__device__ __forceinline__ float2 fma2_bf16x2(uint32_t gw, uint32_t kw, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b16 g0, g1, k0, k1;\n\tmov.b32 {g0, g1}, %2;\n\tmov.b32 {k0, k1}, %3;\n\t"
        "fma.rn.f32.bf16 %0, g0, k0, %4;\n\tfma.rn.f32.bf16 %1, g1, k1, %5;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "r"(gw), "r"(kw), "f"(c.x), "f"(c.y));
    return d;
}

// A 32-bit word holding two bf16 (low half = lower column) <-> an fp32 pair.
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w)
{
    // byte permutes: (w.b1 w.b0 0 0) and (w.b3 w.b2 0 0)
    return make_float2(__uint_as_float(__byte_perm(w, 0u, 0x1044u)), __uint_as_float(__byte_perm(w, 0u, 0x3244u)));
}

// Round an fp32 pair to bf16, nearest-even (cvt.rn), lower column in the low half.
__device__ __forceinline__ uint32_t f2_to_bf16x2(float2 v)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<uint32_t *>(&h);
}

// ------------------------------------------------------------- row map
// Output row r is block b = r - cu_seqlens_comp[s] of the segment s with
// cu_seqlens_comp[s] <= r < cu_seqlens_comp[s+1]; its own tokens start at
// cu_seqlens[s] + b*ratio.  Rows outside [cu_seqlens_comp[0], cu_seqlens_comp[n_seg])
// are padding rows: a first block starting at token 0 ("CSA Fused Compressor",
// Semantics: rows beyond cu_seqlens_comp[-1] use first-in-segment semantics from
// token 0).
struct RowMap {
    int64_t base;
    int seg;
    bool real;
    bool first;
};

__device__ __forceinline__ int find_segment(const int32_t *__restrict__ cc, int n_seg, int r)
{
    int lo = 0, hi = n_seg;  // cc[lo] <= r < cc[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(cc + mid) <= r)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

__device__ __forceinline__ RowMap map_row(int r, const int32_t *__restrict__ cu,
                                          const int32_t *__restrict__ cc, int n_seg, int ratio)
{
    RowMap m;
    m.base = 0;
    m.seg = -1;
    m.real = false;
    m.first = true;
    if (n_seg <= 0)
        return m;
    const int r0 = __ldg(cc), r1 = __ldg(cc + n_seg);
    if (r < r0 || r >= r1)
        return m;
    const int s = find_segment(cc, n_seg, r);
    const int b = r - __ldg(cc + s);
    m.base = (int64_t)__ldg(cu + s) + (int64_t)b * ratio;
    m.seg = s;
    m.real = true;
    m.first = (b == 0);
    return m;
}

// Row -> window map for one thread's increasing rows.  The offsets of the
// current segment stay in registers, so the next row of the same segment costs
// no load; a row a few segments further costs one load per boundary stepped
// over; only a longer jump takes the binary search (dependent loads, slow under a
// full memory system).  Same result as map_row.
struct RowCursor {
    int r0, r1;            // real rows: [cc[0], cc[n_seg])
    int lo, hi, tok;       // current segment: rows [lo, hi), first token tok
    int seg;
};

__device__ __forceinline__ void cursor_init(RowCursor &c, const int32_t *__restrict__ cc, int n_seg)
{
    c.r0 = n_seg > 0 ? __ldg(cc) : 0;
    c.r1 = n_seg > 0 ? __ldg(cc + n_seg) : 0;
    c.lo = c.hi = 0;
    c.tok = 0;
    c.seg = -1;
}

__device__ __forceinline__ RowMap cursor_map(RowCursor &c, int r, const int32_t *__restrict__ cu,
                                             const int32_t *__restrict__ cc, int n_seg, int ratio)
{
    RowMap m;
    m.base = 0;
    m.seg = -1;
    m.real = false;
    m.first = true;
    if (r < c.r0 || r >= c.r1)
        return m;
    if (c.seg < 0 || r < c.lo || r >= c.hi) {
        // Rows only increase: step over up to four segment boundaries (one load
        // each) before falling back to the binary search.  r < r1 = cc[n_seg]
        // keeps every load inside cc.
        int s = c.seg, lo = c.lo, hi = c.hi;
        if (s >= 0 && r >= hi)
            for (int k = 0; k < 4 && r >= hi; ++k) {
                ++s;
                lo = hi;
                hi = __ldg(cc + s + 1);
            }
        if (s >= 0 && r >= lo && r < hi) {
            c.seg = s;
            c.lo = lo;
            c.hi = hi;
        } else {
            c.seg = find_segment(cc, n_seg, r);
            c.lo = __ldg(cc + c.seg);
            c.hi = __ldg(cc + c.seg + 1);
        }
        c.tok = __ldg(cu + c.seg);
    }
    const int b = r - c.lo;
    m.base = (int64_t)c.tok + (int64_t)b * ratio;
    m.seg = c.seg;
    m.real = true;
    m.first = (b == 0);
    return m;
}

// 16-byte streaming load (read once: evict-first in L1 and L2).
__device__ __forceinline__ uint4 ld_stream(const void *p) { return __ldcs(reinterpret_cast<const uint4 *>(p)); }

}  // namespace csa

// ----------------------------------------- programmatic dependent launch
// Every compute kernel of the library is launched so that its blocks may become
// resident while the previous kernel in the stream is still finishing.  pdl_wait()
// holds the grid until that kernel has completed and its memory operations are
// visible (it returns at once after any other predecessor); a kernel reads and
// writes no global memory before it.  pdl_trigger() then lets the next such
// launch do the same.
namespace csa {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------- async copies, barriers
// Shared-memory mbarriers and raw bulk copies (cp.async.bulk: contiguous global
// bytes -> shared memory, completion counted on an mbarrier in bytes).

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Status codes a kernel records in the caller-visible status word.
constexpr unsigned kStatusTimeout = 1u;

// Waits for the phase with the given parity of an mbarrier, for at most about
// kWaitLimitNs (and a bounded number of polls).  On expiry records a timeout in
// *status and returns false; the caller then stops its loop instead of hanging.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned *status,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1; it < (1u << 28); ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 255u) == 0 && global_ns() - t0 > limit_ns)
            break;
    }
    atomicCAS(status, 0u, kStatusTimeout);
    return false;
}

// Next slot of a row lane: `step` slots on, the phase flipping on each wrap
// (stages is a multiple of step).
__device__ __forceinline__ void ring_next(int &st, uint32_t &ph, int step, int stages)
{
    st += step;
    if (st >= stages) {
        st -= stages;
        ph ^= 1u;
    }
}

// Contiguous global -> shared copy of `bytes` (16-byte aligned ends), completing
// `bytes` of transaction count on the mbarrier `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 2-D tiled tensor copy global -> shared through a tensor map (TMA): the box at
// element coordinates (x = column, y = row), completing its bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// The same for a 3-D tensor map: box origin (x, y, z), x the innermost coordinate.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int x, int y, int z, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Barrier over a subset of the block's warps (id > 0; nthreads a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// The same barrier, returning to every participant the AND of their predicates.
__device__ __forceinline__ bool named_barrier_and(int id, int nthreads, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

}  // namespace csa
