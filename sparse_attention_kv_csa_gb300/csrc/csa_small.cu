// Compressor kernels for small ratios (the whole window fits in registers).
//
// Semantics follow the "CSA Fused Compressor" page (cuDNN frontend docs):
//   coff == 2 (overlapping form, window 2*ratio): position k < ratio reads the
//   previous block's token on first-half column j with APE row k and is invalid
//   for a segment's first block; k >= ratio reads the own block's token on column
//   head_dim + j with APE row k - ratio.  coff == 1: the own block only.
//   out[b, j] = sum_k kv * softmax_k(score + ape), fp32, one final bf16 rounding.
//
// Work split: a thread owns a group of 2*NW consecutive output columns of one row
// (NW 32-bit words of bf16 per window row and array, one 8- or 16-byte vector
// load each).  Columns
// are processed as fp32 pairs with the packed .f32x2 instructions.  Both kernels
// are persistent and keep the next unit's window loads in flight (a second
// register buffer) while the current unit is computed.
//
// Operation order (the same in the forward and in the backward's recompute;
// invalid positions are skipped, valid ones taken in ascending k):
//   s_k = score + ape;  m = max_k s_k (NaN-propagating);  e_k = exp(s_k - m)
//   den = ((+0 + e_0) + e_1) + ...;  num = fma(e_k, kv_k, num) from +0
//   inv = 1/den rounded to nearest (recip_den);  o = num * inv;  out = bf16_rn(o)
// Backward, per valid k, with g = grad_out:
//   go = g*o;  p = e_k*inv;  grad_kv = bf16(g*p);  ds = p*(g*kv - go);
//   grad_score = bf16(ds);  ds is summed into this thread's grad_ape partial.
#include <cooperative_groups.h>

#include "csa_device.cuh"
#include "csa_launch.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

struct SmallArgs {
    const uint16_t *kv;
    const uint16_t *score;
    const float *ape;
    const int32_t *cu;
    const int32_t *cc;
    int n_seg;
    int head_dim;
    int capacity;
};

// ------------------------------------------------------------ vectors

template <int NW>
__device__ __forceinline__ void ld_words(uint32_t (&w)[NW], const uint16_t *p)
{
    if constexpr (NW == 4) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(p));
        w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
    } else if constexpr (NW == 2) {
        const uint2 v = __ldcs(reinterpret_cast<const uint2 *>(p));
        w[0] = v.x, w[1] = v.y;
    } else {
        static_assert(NW == 1, "NW is 1, 2 or 4");
        w[0] = __ldcs(reinterpret_cast<const unsigned int *>(p));
    }
}

template <int NW>
__device__ __forceinline__ void st_words(uint16_t *p, const uint32_t (&w)[NW])
{
    if constexpr (NW == 4)
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    else if constexpr (NW == 2)
        *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
    else
        *reinterpret_cast<uint32_t *>(p) = w[0];
}

template <int NW>
__device__ __forceinline__ void st_zero(uint16_t *p)
{
    if constexpr (NW == 4)
        *reinterpret_cast<uint4 *>(p) = make_uint4(0u, 0u, 0u, 0u);
    else if constexpr (NW == 2)
        *reinterpret_cast<uint2 *>(p) = make_uint2(0u, 0u);
    else
        *reinterpret_cast<uint32_t *>(p) = 0u;
}

// NW fp32 pairs of APE (read through the read-only cache; the table is small).
template <int NW>
__device__ __forceinline__ void ld_ape(float2 (&a)[NW], const float *p)
{
    if constexpr (NW == 1) {
        a[0] = __ldg(reinterpret_cast<const float2 *>(p));
    } else {
#pragma unroll
        for (int h = 0; h < NW / 2; ++h) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p) + h);
            a[2 * h] = make_float2(v.x, v.y);
            a[2 * h + 1] = make_float2(v.z, v.w);
        }
    }
}

// ------------------------------------------------------------- window

// Window position k of a row: token and packed column for column group j.
template <int RATIO, int COFF>
__device__ __forceinline__ void window_slot(int k, const RowMap &rm, int j, int head_dim,
                                            int64_t &tok, int &col)
{
    if (COFF == 2 && k < RATIO) {
        tok = rm.base - RATIO + k;
        col = j;
    } else if (COFF == 2) {
        tok = rm.base + (k - RATIO);
        col = head_dim + j;
    } else {
        tok = rm.base + k;
        col = j;
    }
}

// grad_ape entry (APE row, packed column) of window position k for column group j.
template <int RATIO, int COFF>
__device__ __forceinline__ void ape_slot(int k, int j, int head_dim, int &arow, int &col)
{
    if (COFF == 2 && k < RATIO) {
        arow = k;
        col = j;
    } else if (COFF == 2) {
        arow = k - RATIO;
        col = head_dim + j;
    } else {
        arow = k;
        col = j;
    }
}

template <int RATIO, int COFF>
__device__ __forceinline__ bool slot_valid(int k, const RowMap &rm)
{
    return !(COFF == 2 && k < RATIO && rm.first);
}

template <int RATIO, int COFF, int NW>
struct Window {
    uint32_t kv[COFF * RATIO][NW];
    uint32_t sc[COFF * RATIO][NW];
};

template <int RATIO, int COFF, int NW>
__device__ __forceinline__ void load_window(const SmallArgs &a, const RowMap &rm, int j,
                                            Window<RATIO, COFF, NW> &w)
{
    const int64_t C = (int64_t)COFF * a.head_dim;
#pragma unroll
    for (int k = 0; k < COFF * RATIO; ++k) {
        if (!slot_valid<RATIO, COFF>(k, rm))
            continue;
        int64_t tok;
        int col;
        window_slot<RATIO, COFF>(k, rm, j, a.head_dim, tok, col);
        ld_words<NW>(w.kv[k], a.kv + tok * C + col);
        ld_words<NW>(w.sc[k], a.score + tok * C + col);
    }
}

// The softmax pooling of one (row, column group) up to den and num; e[k] holds e_k
// for the valid positions.
template <int RATIO, int COFF, int NW>
__device__ __forceinline__ void pool_window(const SmallArgs &a, const RowMap &rm, int j,
                                            const Window<RATIO, COFF, NW> &w,
                                            float2 (&e)[COFF * RATIO][NW], float2 (&den)[NW],
                                            float2 (&num)[NW])
{
    constexpr int W = COFF * RATIO;
    const int64_t C = (int64_t)COFF * a.head_dim;
    float2 m[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q)
        m[q] = make_float2(-INFINITY, -INFINITY);
#pragma unroll
    for (int k = 0; k < W; ++k) {
        if (!slot_valid<RATIO, COFF>(k, rm))
            continue;
        int arow, col;
        ape_slot<RATIO, COFF>(k, j, a.head_dim, arow, col);
        float2 ap[NW];
        ld_ape<NW>(ap, a.ape + (int64_t)arow * C + col);
#pragma unroll
        for (int q = 0; q < NW; ++q) {
            // unpacked and added as a pair: with the mixed-precision add (same bits) this
            // kernel's forward measured slower (22.6 against 21.4 us at head_dim 64)
            e[k][q] = add2(bf16x2_to_f2(w.sc[k][q]), ap[q]);
            m[q].x = max_nan(m[q].x, e[k][q].x);
            m[q].y = max_nan(m[q].y, e[k][q].y);
        }
    }
    float2 negm[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) {
        negm[q] = make_float2(-m[q].x, -m[q].y);
        den[q] = make_float2(0.0f, 0.0f);
        num[q] = make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int k = 0; k < W; ++k) {
        if (!slot_valid<RATIO, COFF>(k, rm))
            continue;
#pragma unroll
        for (int q = 0; q < NW; ++q) {
            const float2 ek = exp2lanes(add2(e[k][q], negm[q]));
            e[k][q] = ek;
            den[q] = add2(den[q], ek);
            num[q] = fma2(ek, bf16x2_to_f2(w.kv[k][q]), num[q]);
        }
    }
}

// -------------------------------------------------------------- forward

// Tile choices: words of bf16 per window row per thread and the minimum resident
// blocks per SM the register budget is sized for (two: head_dim 96 forward 30.7
// -> 29.6 us at 32 x 4096 tokens against three; one or four words a row, 256
// threads a block, or four blocks measured slower).
constexpr int kFwdNW = 2;
constexpr int kFwdMinBlocks = 2;
constexpr int kFwdThreads = 128;

template <int RATIO, int COFF>
struct FwdUnit {
    Window<RATIO, COFF, kFwdNW> w;
    RowMap rm;
    int r, j;
};

template <int RATIO, int COFF>
__device__ __forceinline__ void fwd_fetch(const SmallArgs &a, int u, int groups, FwdUnit<RATIO, COFF> &f)
{
    f.r = u / groups;
    f.j = (u - f.r * groups) * (2 * kFwdNW);
    f.rm = map_row(f.r, a.cu, a.cc, a.n_seg, RATIO);
    load_window<RATIO, COFF, kFwdNW>(a, f.rm, f.j, f.w);
}

template <int RATIO, int COFF>
__device__ __forceinline__ void fwd_compute(const SmallArgs &a, const FwdUnit<RATIO, COFF> &f,
                                            uint16_t *__restrict__ out)
{
    constexpr int NW = kFwdNW;
    float2 e[COFF * RATIO][NW], den[NW], num[NW];
    pool_window<RATIO, COFF, NW>(a, f.rm, f.j, f.w, e, den, num);
    uint32_t o[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) {
        const float2 inv = make_float2(recip_den(den[q].x), recip_den(den[q].y));
        o[q] = f2_to_bf16x2(mul2(num[q], inv));
    }
    st_words<NW>(out + (int64_t)f.r * a.head_dim + f.j, o);
}

// Persistent: thread t takes units t, t + stride, ... (unit = row x column group,
// consecutive threads on consecutive column groups, so loads coalesce).  Two unit
// buffers alternate: the next unit's loads are issued before the current one is
// computed.
template <int RATIO, int COFF>
__global__ void __launch_bounds__(kFwdThreads, kFwdMinBlocks) fwd_small_kernel(SmallArgs a, uint16_t *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int groups = a.head_dim / (2 * kFwdNW);
    const int total = a.capacity * groups;
    const int stride = gridDim.x * blockDim.x;
    int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= total)
        return;
    FwdUnit<RATIO, COFF> A, B;
    fwd_fetch<RATIO, COFF>(a, u, groups, A);
    for (;;) {
        int un = u + stride;
        if (un < total)
            fwd_fetch<RATIO, COFF>(a, un, groups, B);
        fwd_compute<RATIO, COFF>(a, A, out);
        if (un >= total)
            break;
        u = un;
        un = u + stride;
        if (un < total)
            fwd_fetch<RATIO, COFF>(a, un, groups, A);
        fwd_compute<RATIO, COFF>(a, B, out);
        if (un >= total)
            break;
        u = un;
    }
}

// ------------------------------------------------------------- backward

constexpr int kBwdNW = 1;
constexpr int kBwdMinBlocks = 4;  // resident blocks per SM the register budget is sized for
constexpr int kBwdCluster = 2;    // blocks per cluster (grad_ape merged in DSMEM; 4: head_dim 96 76.7 -> 70.9 us)
constexpr int kBwdThreads = 128;

template <int RATIO, int COFF>
struct BwdRow {
    Window<RATIO, COFF, kBwdNW> w;
    uint32_t g[kBwdNW];
    RowMap rm;
};

template <int RATIO, int COFF>
__device__ __forceinline__ void bwd_fetch(const SmallArgs &a, int r, int j, const uint16_t *__restrict__ grad_out,
                                          BwdRow<RATIO, COFF> &f)
{
    f.rm = map_row(r, a.cu, a.cc, a.n_seg, RATIO);
    if (!f.rm.real)
        return;
    load_window<RATIO, COFF, kBwdNW>(a, f.rm, j, f.w);
    ld_words<kBwdNW>(f.g, grad_out + (int64_t)r * a.head_dim + j);
}

struct BwdOut {
    uint16_t *dkv;
    uint16_t *dscore;
    int64_t n_tokens;
};

// Zero the gradient slots of tokens [t0, t1) in this thread's columns.
template <int COFF>
__device__ __forceinline__ void zero_tokens(const BwdOut &o, int64_t C, int head_dim, int j, int64_t t0,
                                            int64_t t1)
{
    t1 = t1 < o.n_tokens ? t1 : o.n_tokens;
    for (int64_t t = t0 < 0 ? 0 : t0; t < t1; ++t) {
        st_zero<kBwdNW>(o.dkv + t * C + j);
        st_zero<kBwdNW>(o.dscore + t * C + j);
        if (COFF == 2) {
            st_zero<kBwdNW>(o.dkv + t * C + head_dim + j);
            st_zero<kBwdNW>(o.dscore + t * C + head_dim + j);
        }
    }
}

template <int RATIO, int COFF>
__device__ __forceinline__ void bwd_compute(const SmallArgs &a, const BwdRow<RATIO, COFF> &f, int r, int j,
                                            int R, const BwdOut &o, float2 (&acc)[COFF * RATIO][kBwdNW])
{
    constexpr int W = COFF * RATIO;
    constexpr int NW = kBwdNW;
    if (!f.rm.real)
        return;
    const int64_t C = (int64_t)COFF * a.head_dim;
    float2 e[W][NW], den[NW], num[NW];
    pool_window<RATIO, COFF, NW>(a, f.rm, j, f.w, e, den, num);
    float2 g[NW], inv[NW], ngo[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) {
        g[q] = bf16x2_to_f2(f.g[q]);
        inv[q] = make_float2(recip_den(den[q].x), recip_den(den[q].y));
        const float2 go = mul2(g[q], mul2(num[q], inv[q]));
        ngo[q] = make_float2(-go.x, -go.y);
    }
#pragma unroll
    for (int k = 0; k < W; ++k) {
        if (!slot_valid<RATIO, COFF>(k, f.rm))
            continue;
        int64_t tok;
        int col;
        window_slot<RATIO, COFF>(k, f.rm, j, a.head_dim, tok, col);
        uint32_t dk[NW], dsw[NW];
#pragma unroll
        for (int q = 0; q < NW; ++q) {
            const float2 p = mul2(e[k][q], inv[q]);
            dk[q] = f2_to_bf16x2(mul2(g[q], p));
            const float2 ds = mul2(p, add2(mul2(g[q], bf16x2_to_f2(f.w.kv[k][q])), ngo[q]));
            dsw[q] = f2_to_bf16x2(ds);
            acc[k][q] = add2(acc[k][q], ds);
        }
        if (tok < o.n_tokens) {
            st_words<NW>(o.dkv + tok * C + col, dk);
            st_words<NW>(o.dscore + tok * C + col, dsw);
        }
    }
    // Last block of its segment: its own first-half columns are read by no row
    // (coff 2), and the tokens up to the next real block form a gap.
    if (r + 1 == __ldg(a.cc + f.rm.seg + 1)) {
        if (COFF == 2) {
            for (int i = 0; i < RATIO; ++i) {
                const int64_t tok = f.rm.base + i;
                if (tok < o.n_tokens) {
                    st_zero<NW>(o.dkv + tok * C + j);
                    st_zero<NW>(o.dscore + tok * C + j);
                }
            }
        }
        int64_t next = o.n_tokens;
        if (r + 1 < R)
            next = map_row(r + 1, a.cu, a.cc, a.n_seg, RATIO).base;
        zero_tokens<COFF>(o, C, a.head_dim, j, f.rm.base + RATIO, next);
    }
}

// Backward.  Block = (threads_x column groups of 4 columns) x (lanes); blockIdx.y
// picks a slice of columns for wide heads.  Block b owns output rows
// [b*rows_per_block, (b+1)*rows_per_block) of the static capacity; lane y takes rows
// y, y + lanes, ... of that range in ascending order, prefetching its next row.
// Each thread keeps the grad_ape sums of its columns and window positions in
// registers.  At the end the lanes are added in ascending lane order in shared
// memory; then the blocks of a thread-block cluster add their shared-memory
// partials in ascending cluster rank through distributed shared memory and the
// cluster writes one [ratio, coff*head_dim] partial.  dape_finalize_kernel adds the
// partials in a fixed order.  No atomics, fixed orders: grad_ape is bitwise
// reproducible run to run.
//
// Gradient coverage ("CSA Fused Compressor", Class API: every never-consumed slot
// gets an exact zero from one owner).  A real row writes the slots it reads; the
// last block of a segment also zeroes its own first-half columns (coff == 2) and
// the gap of tokens after its block up to the next real row's block (or up to
// n_tokens): the segment's tail, segments shorter than ratio, token padding.  The
// threads of row 0 zero the tokens before the first real block.  Every token of
// [0, n_tokens) is thus written exactly once.
template <int RATIO, int COFF>
__global__ void __launch_bounds__(kBwdThreads, kBwdMinBlocks)
    bwd_small_kernel(SmallArgs a, int rows_per_block, int64_t n_tokens_arg,
                     const uint16_t *__restrict__ grad_out, uint16_t *__restrict__ dkv,
                     uint16_t *__restrict__ dscore, float *__restrict__ partial)
{
    constexpr int W = COFF * RATIO;
    constexpr int NW = kBwdNW;
    extern __shared__ float red[];
    pdl_wait();
    pdl_trigger();  // the grad_ape finalisation may launch; it waits for this grid's end
    const int lanes = blockDim.y;
    const int x = threadIdx.x, y = threadIdx.y;
    const int j = (blockIdx.y * blockDim.x + x) * (2 * NW);
    const bool col_ok = j < a.head_dim;  // the last column slice may be partial
    const int64_t C = (int64_t)COFF * a.head_dim;
    BwdOut o{dkv, dscore, n_tokens_arg >= 0 ? n_tokens_arg : (int64_t)__ldg(a.cu + a.n_seg)};
    const int R = a.n_seg > 0 ? __ldg(a.cc + a.n_seg) : 0;
    const int R0 = a.n_seg > 0 ? __ldg(a.cc) : 0;

    // Leading gap: tokens before the first real block.
    if (blockIdx.x == 0 && y == 0 && col_ok) {
        int64_t lead = o.n_tokens;
        if (R0 < R)
            lead = map_row(R0, a.cu, a.cc, a.n_seg, RATIO).base;  // a first block
        zero_tokens<COFF>(o, C, a.head_dim, j, 0, lead);
    }

    float2 acc[W][NW];
#pragma unroll
    for (int k = 0; k < W; ++k)
#pragma unroll
        for (int q = 0; q < NW; ++q)
            acc[k][q] = make_float2(0.0f, 0.0f);

    const int r_begin = blockIdx.x * rows_per_block;
    int r_end = r_begin + rows_per_block;
    r_end = r_end < a.capacity ? r_end : a.capacity;
    r_end = r_end < R ? r_end : R;  // padding rows carry no gradient
    if (!col_ok)
        r_end = r_begin;
    int r = r_begin + y;
    if (r < r_end) {
        BwdRow<RATIO, COFF> A, B;
        bwd_fetch<RATIO, COFF>(a, r, j, grad_out, A);
        for (;;) {
            int rn = r + lanes;
            if (rn < r_end)
                bwd_fetch<RATIO, COFF>(a, rn, j, grad_out, B);
            bwd_compute<RATIO, COFF>(a, A, r, j, R, o, acc);
            if (rn >= r_end)
                break;
            r = rn;
            rn = r + lanes;
            if (rn < r_end)
                bwd_fetch<RATIO, COFF>(a, rn, j, grad_out, A);
            bwd_compute<RATIO, COFF>(a, B, r, j, R, o, acc);
            if (rn >= r_end)
                break;
            r = rn;
        }
    }

    // Lanes -> shared memory [ape row][half][slice column], ascending lane order.
    const int SW = blockDim.x * 2 * NW;  // columns per half in this block's slice
    const int c0 = blockIdx.y * SW;
    for (int l = 0; l < lanes; ++l) {
        if (y == l && col_ok) {
#pragma unroll
            for (int k = 0; k < W; ++k) {
                int arow, col;
                ape_slot<RATIO, COFF>(k, j, a.head_dim, arow, col);
                const int half = col >= a.head_dim ? 1 : 0;
                float *sp = red + (arow * COFF + half) * SW + (j - c0);
#pragma unroll
                for (int q = 0; q < NW; ++q) {
                    if (l == 0) {
                        sp[2 * q] = acc[k][q].x;
                        sp[2 * q + 1] = acc[k][q].y;
                    } else {
                        sp[2 * q] = __fadd_rn(sp[2 * q], acc[k][q].x);
                        sp[2 * q + 1] = __fadd_rn(sp[2 * q + 1], acc[k][q].y);
                    }
                }
            }
        }
        __syncthreads();
    }

    // Cluster: block ranks' partials added in ascending rank order; each block of
    // the cluster reduces and writes a share of the entries.
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int rank = (int)cluster.block_rank();
    const int nrank = (int)cluster.num_blocks();
    const int per_row4 = SW / 4;
    const int n4 = RATIO * COFF * per_row4;
    const int share = (n4 + nrank - 1) / nrank;
    const int i_lo = rank * share;
    const int i_hi = i_lo + share < n4 ? i_lo + share : n4;
    float *dst = partial + (int64_t)(blockIdx.x / nrank) * RATIO * C;
    const int tid = y * blockDim.x + x;
    const int nthreads = blockDim.x * blockDim.y;
    for (int i = i_lo + tid; i < i_hi; i += nthreads) {
        const int rh = i / per_row4, lc = (i - rh * per_row4) * 4;
        const int arow = rh / COFF, half = rh - arow * COFF;
        if (c0 + lc >= a.head_dim)
            continue;
        float4 s = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(red, 0) + rh * SW + lc);
        for (int q = 1; q < nrank; ++q) {
            const float4 v = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(red, q) + rh * SW + lc);
            s.x = __fadd_rn(s.x, v.x);
            s.y = __fadd_rn(s.y, v.y);
            s.z = __fadd_rn(s.z, v.z);
            s.w = __fadd_rn(s.w, v.w);
        }
        *reinterpret_cast<float4 *>(dst + (int64_t)arow * C + half * a.head_dim + c0 + lc) = s;
    }
    cluster.sync();  // keep this block's shared memory alive until all ranks read it
}

}  // namespace

// grad_ape = the partials summed in a fixed order: range t of the 32 contiguous
// ranges [t*P/32, (t+1)*P/32) is summed in ascending order from +0, then the 32
// range sums are added pairwise, t with t^1, then with t^2, t^4, t^8, t^16.
// A block takes kFinCols 4-float columns: a warp holds four ranges of them, eight
// lanes per range on consecutive columns, so that each load of a partial is one
// contiguous 128-byte piece; the range sums meet in shared memory, where one warp
// runs the pairwise tree (a lane per float column).
// Launched as a programmatic dependent of the backward kernel: griddepcontrol.wait
// holds it until that grid has finished and its partials are visible (a plain
// launch returns from the wait at once).
constexpr int kFinCols = 8;
constexpr int kFinThreads = 256;  // 8 warps x 4 ranges = 32 ranges
static_assert(kFinThreads / 32 * (32 / kFinCols) == 32, "one range per thread");

__global__ void __launch_bounds__(kFinThreads) dape_finalize_kernel(const float *__restrict__ partial,
                                                                    int n_partials, int64_t n,
                                                                    float *__restrict__ dape)
{
    __shared__ __align__(16) float sums[32 * kFinCols * 4];  // [range][float column]
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = warp * (32 / kFinCols) + lane / kFinCols;  // range
    const int64_t stride = n / 4;
    const int64_t i = (int64_t)blockIdx.x * kFinCols + lane % kFinCols;  // 4-float column
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (i < stride) {
        const int lo = (int)((int64_t)t * n_partials / 32), hi = (int)((int64_t)(t + 1) * n_partials / 32);
        const float4 *p = reinterpret_cast<const float4 *>(partial) + i;
        int b = lo;
        for (; b + 4 <= hi; b += 4) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = __ldcg(p + (int64_t)(b + u) * stride);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc.x = __fadd_rn(acc.x, v[u].x);
                acc.y = __fadd_rn(acc.y, v[u].y);
                acc.z = __fadd_rn(acc.z, v[u].z);
                acc.w = __fadd_rn(acc.w, v[u].w);
            }
        }
        for (; b < hi; ++b) {
            const float4 v = __ldcg(p + (int64_t)b * stride);
            acc.x = __fadd_rn(acc.x, v.x);
            acc.y = __fadd_rn(acc.y, v.y);
            acc.z = __fadd_rn(acc.z, v.z);
            acc.w = __fadd_rn(acc.w, v.w);
        }
    }
    // consecutive threads store consecutive 16-byte slots: no bank conflicts
    reinterpret_cast<float4 *>(sums)[t * kFinCols + lane % kFinCols] = acc;
    __syncthreads();
    if (warp == 0 && lane < kFinCols * 4) {
        float v[32];
#pragma unroll
        for (int r = 0; r < 32; ++r)
            v[r] = sums[r * kFinCols * 4 + lane];
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1)  // level m: sums t and t^m (adjacent after the levels before)
#pragma unroll
            for (int r = 0; r < w; ++r)
                v[r] = __fadd_rn(v[2 * r], v[2 * r + 1]);
        const int64_t f = (int64_t)blockIdx.x * kFinCols * 4 + lane;
        if (f < stride * 4)
            dape[f] = v[0];
    }
}

// ------------------------------------------------------------ launchers

cudaError_t launch_dape_finalize(const float *partial, int n_partials, int64_t n, float *dape, cudaStream_t st)
{
    const int64_t blocks = (n / 4 + kFinCols - 1) / kFinCols;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(blocks > 0 ? blocks : 1), 1, 1);
    cfg.blockDim = dim3(kFinThreads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dape_finalize_kernel, partial, n_partials, n, dape);
}

template <int RATIO, int COFF>
static cudaError_t launch_fwd_small_t(const FwdParams &p, int num_sms, cudaStream_t st)
{
    SmallArgs a{static_cast<const uint16_t *>(p.kv), static_cast<const uint16_t *>(p.score), p.ape,
                p.cu_seqlens, p.cu_seqlens_comp, p.n_seg, p.head_dim, p.capacity};
    const int64_t units = (int64_t)p.capacity * (p.head_dim / (2 * kFwdNW));
    static int cached_per_sm[64] = {0};  // per device; occupancy is a slow host query
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    int per_sm = (dev >= 0 && dev < 64) ? cached_per_sm[dev] : 0;
    if (per_sm == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fwd_small_kernel<RATIO, COFF>, kFwdThreads, 0);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            cached_per_sm[dev] = per_sm;
    }
    int64_t grid = (units + kFwdThreads - 1) / kFwdThreads;
    const int64_t resident = (int64_t)(per_sm > 0 ? per_sm : 1) * num_sms;
    if (grid > resident)
        grid = resident;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kFwdThreads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fwd_small_kernel<RATIO, COFF>, a, static_cast<uint16_t *>(p.out));
}

cudaError_t launch_fwd_small(const FwdParams &p, int num_sms, cudaStream_t st)
{
    if (p.ratio == 4 && p.coff == 2)
        return launch_fwd_small_t<4, 2>(p, num_sms, st);
    if (p.ratio == 4 && p.coff == 1)
        return launch_fwd_small_t<4, 1>(p, num_sms, st);
    return cudaErrorInvalidValue;
}

SmallBwdPlan plan_bwd_small(int ratio, int coff, int head_dim, int capacity, int num_sms)
{
    SmallBwdPlan pl;
    const int groups = head_dim / (2 * kBwdNW);
    pl.threads_x = groups < kBwdThreads ? groups : kBwdThreads;
    pl.col_slices = (groups + pl.threads_x - 1) / pl.threads_x;
    pl.lanes = kBwdThreads / pl.threads_x > 1 ? kBwdThreads / pl.threads_x : 1;
    pl.cluster = kBwdCluster;
    const int resident = kBwdMinBlocks * num_sms;  // blocks the register budget is sized for
    int max_blocks = resident / pl.col_slices;
    max_blocks = max_blocks / pl.cluster * pl.cluster;
    if (max_blocks < pl.cluster)
        max_blocks = pl.cluster;
    const int rows = capacity > 0 ? capacity : 1;
    int blocks = (rows + pl.lanes - 1) / pl.lanes;
    if (blocks > max_blocks)
        blocks = max_blocks;
    pl.rows_per_block = (rows + blocks - 1) / blocks;
    blocks = (rows + pl.rows_per_block - 1) / pl.rows_per_block;
    pl.blocks = (blocks + pl.cluster - 1) / pl.cluster * pl.cluster;
    pl.smem = (size_t)ratio * coff * pl.threads_x * 2 * kBwdNW * sizeof(float);
    pl.partials = pl.blocks / pl.cluster;
    pl.partial_floats = (int64_t)pl.partials * ratio * coff * head_dim;
    return pl;
}

template <int RATIO, int COFF>
static cudaError_t launch_bwd_small_t(const BwdParams &p, const SmallBwdPlan &pl, float *partial,
                                      cudaStream_t st)
{
    SmallArgs a{static_cast<const uint16_t *>(p.kv), static_cast<const uint16_t *>(p.score), p.ape,
                p.cu_seqlens, p.cu_seqlens_comp, p.n_seg, p.head_dim, p.capacity};
    auto kern = bwd_small_kernel<RATIO, COFF>;
    if (pl.smem > 48 * 1024) {
        cudaError_t e = allow_max_smem(reinterpret_cast<const void *>(kern));
        if (e != cudaSuccess)
            return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.blocks, pl.col_slices, 1);
    cfg.blockDim = dim3(pl.threads_x, pl.lanes, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pl.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, pl.rows_per_block, p.n_tokens,
                                       static_cast<const uint16_t *>(p.grad_out), static_cast<uint16_t *>(p.dkv),
                                       static_cast<uint16_t *>(p.dscore), partial);
    if (e != cudaSuccess)
        return e;
    return launch_dape_finalize(partial, pl.partials, (int64_t)RATIO * COFF * p.head_dim, p.dape, st);
}

cudaError_t launch_bwd_small(const BwdParams &p, const SmallBwdPlan &pl, float *partial, cudaStream_t st)
{
    if (p.ratio == 4 && p.coff == 2)
        return launch_bwd_small_t<4, 2>(p, pl, partial, st);
    if (p.ratio == 4 && p.coff == 1)
        return launch_bwd_small_t<4, 1>(p, pl, partial, st);
    return cudaErrorInvalidValue;
}

}  // namespace csa
