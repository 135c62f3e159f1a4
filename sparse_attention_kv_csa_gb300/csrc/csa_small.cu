// Compressor kernels for small ratios (the whole window fits in registers).
//
// Semantics follow the "CSA Fused Compressor" page (cuDNN frontend docs):
//   coff == 2 (overlapping form, window 2*ratio): position k < ratio reads the
//   previous block's token on first-half column j with APE row k and is invalid
//   for a segment's first block; k >= ratio reads the own block's token on column
//   head_dim + j with APE row k - ratio.  coff == 1: the own block only.
//   out[b, j] = sum_k kv * softmax_k(score + ape), fp32, one final bf16 rounding.
//
// Work split: one thread owns 8 consecutive output columns j of one row, so
// every window row it touches is one 16-byte vector of kv and one of score.  The
// 8 columns are processed as 4 fp32 pairs with the packed .f32x2 instructions.
//
// Operation order (the same in the forward and in the backward's recompute;
// invalid positions are skipped, valid ones taken in ascending k):
//   s_k = score + ape;  m = max_k s_k (NaN-propagating);  e_k = exp(s_k - m)
//   den = ((+0 + e_0) + e_1) + ...;  num = fma(e_k, kv_k, num) from +0
//   inv = rcp.rn(den);  o = num * inv;  out = bf16_rn(o)
// Backward, per valid k, with g = grad_out:
//   go = g*o;  p = e_k*inv;  grad_kv = bf16(g*p);  ds = p*(g*kv - go);
//   grad_score = bf16(ds);  ds is summed into this thread's grad_ape partial.
#include "csa_device.cuh"
#include "csa_launch.h"

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

// Window position k of a row: token and packed column of its 8-column group j.
template <int RATIO, int COFF>
__device__ __forceinline__ void window_slot(int k, const RowMap &rm, int j, int head_dim,
                                            int64_t &tok, int &col, int &arow)
{
    if (COFF == 2 && k < RATIO) {
        tok = rm.base - RATIO + k;
        col = j;
        arow = k;
    } else if (COFF == 2) {
        tok = rm.base + (k - RATIO);
        col = head_dim + j;
        arow = k - RATIO;
    } else {
        tok = rm.base + k;
        col = j;
        arow = k;
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

// Loads the window of (row, 8 columns) and runs the pooling up to den/num.
// On return: e[k][q] holds e_k for column pair q (valid k only), num/den per pair,
// kvv[k] holds the raw kv vector.
template <int RATIO, int COFF>
__device__ __forceinline__ void pool_window(const SmallArgs &a, const RowMap &rm, int j,
                                            uint4 (&kvv)[COFF * RATIO], float2 (&e)[COFF * RATIO][4],
                                            float2 (&den)[4], float2 (&num)[4])
{
    constexpr int W = COFF * RATIO;
    const int64_t C = (int64_t)COFF * a.head_dim;
    const bool has_prev = (COFF == 2) && !rm.first;
    uint4 scv[W];
#pragma unroll
    for (int k = 0; k < W; ++k) {
        if (COFF == 2 && k < RATIO && !has_prev)
            continue;
        int64_t tok;
        int col, arow;
        window_slot<RATIO, COFF>(k, rm, j, a.head_dim, tok, col, arow);
        kvv[k] = ld_stream(a.kv + tok * C + col);
        scv[k] = ld_stream(a.score + tok * C + col);
    }
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        m[i] = -INFINITY;
#pragma unroll
    for (int k = 0; k < W; ++k) {
        if (COFF == 2 && k < RATIO && !has_prev)
            continue;
        int64_t tok;
        int col, arow;
        window_slot<RATIO, COFF>(k, rm, j, a.head_dim, tok, col, arow);
        const float4 *ap = reinterpret_cast<const float4 *>(a.ape + (int64_t)arow * C + col);
        const float4 a0 = __ldg(ap), a1 = __ldg(ap + 1);
        e[k][0] = add2(bf16x2_to_f2(scv[k].x), make_float2(a0.x, a0.y));
        e[k][1] = add2(bf16x2_to_f2(scv[k].y), make_float2(a0.z, a0.w));
        e[k][2] = add2(bf16x2_to_f2(scv[k].z), make_float2(a1.x, a1.y));
        e[k][3] = add2(bf16x2_to_f2(scv[k].w), make_float2(a1.z, a1.w));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            m[2 * q] = max_nan(m[2 * q], e[k][q].x);
            m[2 * q + 1] = max_nan(m[2 * q + 1], e[k][q].y);
        }
    }
    float2 negm[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        negm[q] = make_float2(-m[2 * q], -m[2 * q + 1]);
        den[q] = make_float2(0.0f, 0.0f);
        num[q] = make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int k = 0; k < W; ++k) {
        if (COFF == 2 && k < RATIO && !has_prev)
            continue;
        const uint32_t kw[4] = {kvv[k].x, kvv[k].y, kvv[k].z, kvv[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 ek = exp2lanes(add2(e[k][q], negm[q]));
            e[k][q] = ek;
            den[q] = add2(den[q], ek);
            num[q] = fma2(ek, bf16x2_to_f2(kw[q]), num[q]);
        }
    }
}

template <int RATIO, int COFF>
__global__ void __launch_bounds__(256) fwd_small_kernel(SmallArgs a, uint16_t *__restrict__ out)
{
    constexpr int W = COFF * RATIO;
    const int groups = a.head_dim >> 3;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)a.capacity * groups)
        return;
    const int r = (int)(t / groups);
    const int j = (int)(t - (int64_t)r * groups) * 8;
    const RowMap rm = map_row(r, a.cu, a.cc, a.n_seg, RATIO);

    uint4 kvv[W];
    float2 e[W][4], den[4], num[4];
    pool_window<RATIO, COFF>(a, rm, j, kvv, e, den, num);

    uint4 o;
    uint32_t ow[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 inv = make_float2(__frcp_rn(den[q].x), __frcp_rn(den[q].y));
        ow[q] = f2_to_bf16x2(mul2(num[q], inv));
    }
    o.x = ow[0];
    o.y = ow[1];
    o.z = ow[2];
    o.w = ow[3];
    *reinterpret_cast<uint4 *>(out + (int64_t)r * a.head_dim + j) = o;
}

// Backward.  Block = (up to 64 threads along x, 8 columns each) x (lanes along y);
// blockIdx.y picks the block's slice of columns when head_dim > 512.  Block p owns
// output rows [p*rows_per_block, ...) of the static capacity; lane y takes rows
// y, y + lanes, ... of that range in ascending order.  Each thread keeps the
// grad_ape sums of its 8 columns and all window positions in registers; at the
// end the lanes are added in ascending lane order through shared memory and the
// block writes one [ratio, coff*head_dim] partial.  dape_finalize_kernel then adds
// the partials in ascending block order: no atomics, a fixed order, so grad_ape is
// bitwise reproducible run to run.
//
// Gradient coverage ("CSA Fused Compressor", Class API: every never-consumed slot
// gets an exact zero from one owner).  A real row writes the slots it reads; the
// last block of a segment also zeroes its own first-half columns (coff == 2) and
// the gap of tokens after its block up to the next real row's block (or up to
// n_tokens): the segment's tail, segments shorter than ratio, token padding.  The
// thread group of row 0 zeroes the tokens before the first real block.  Every
// token of [0, n_tokens) is thus written exactly once.
template <int RATIO, int COFF>
__global__ void __launch_bounds__(256) bwd_small_kernel(SmallArgs a, int rows_per_block,
                                                        int64_t n_tokens_arg,
                                                        const uint16_t *__restrict__ grad_out,
                                                        uint16_t *__restrict__ dkv,
                                                        uint16_t *__restrict__ dscore,
                                                        float *__restrict__ partial)
{
    constexpr int W = COFF * RATIO;
    extern __shared__ float red[];
    const int lanes = blockDim.y;
    const int x = threadIdx.x, y = threadIdx.y;
    const int j = (blockIdx.y * blockDim.x + x) * 8;
    const bool col_ok = j < a.head_dim;  // the last column slice may be partial
    const int64_t C = (int64_t)COFF * a.head_dim;
    const int64_t n_tokens = n_tokens_arg >= 0 ? n_tokens_arg : (int64_t)__ldg(a.cu + a.n_seg);
    const int R = a.n_seg > 0 ? __ldg(a.cc + a.n_seg) : 0;
    const int R0 = a.n_seg > 0 ? __ldg(a.cc) : 0;
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);

    // Zero the gradient slots of tokens [t0, t1) in this thread's columns.
    auto zero_tokens = [&](int64_t t0, int64_t t1) {
        t1 = t1 < n_tokens ? t1 : n_tokens;
        for (int64_t t = t0 < 0 ? 0 : t0; t < t1; ++t) {
            *reinterpret_cast<uint4 *>(dkv + t * C + j) = zero4;
            *reinterpret_cast<uint4 *>(dscore + t * C + j) = zero4;
            if (COFF == 2) {
                *reinterpret_cast<uint4 *>(dkv + t * C + a.head_dim + j) = zero4;
                *reinterpret_cast<uint4 *>(dscore + t * C + a.head_dim + j) = zero4;
            }
        }
    };

    // Leading gap: tokens before the first real block.
    if (blockIdx.x == 0 && y == 0 && col_ok) {
        int64_t lead = n_tokens;
        if (R0 < R)
            lead = map_row(R0, a.cu, a.cc, a.n_seg, RATIO).base;  // a first block
        zero_tokens(0, lead);
    }

    float2 acc[W][4];
#pragma unroll
    for (int k = 0; k < W; ++k)
#pragma unroll
        for (int q = 0; q < 4; ++q)
            acc[k][q] = make_float2(0.0f, 0.0f);

    const int r_begin = blockIdx.x * rows_per_block;
    int r_end = r_begin + rows_per_block;
    r_end = r_end < a.capacity ? r_end : a.capacity;
    r_end = r_end < R ? r_end : R;  // padding rows carry no gradient
    if (!col_ok)
        r_end = r_begin;
    for (int r = r_begin + y; r < r_end; r += lanes) {
        const RowMap rm = map_row(r, a.cu, a.cc, a.n_seg, RATIO);
        if (!rm.real)
            continue;
        uint4 kvv[W];
        float2 e[W][4], den[4], num[4];
        pool_window<RATIO, COFF>(a, rm, j, kvv, e, den, num);

        const uint4 gv = ld_stream(grad_out + (int64_t)r * a.head_dim + j);
        const float2 g[4] = {bf16x2_to_f2(gv.x), bf16x2_to_f2(gv.y), bf16x2_to_f2(gv.z),
                             bf16x2_to_f2(gv.w)};
        float2 inv[4], go[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            inv[q] = make_float2(__frcp_rn(den[q].x), __frcp_rn(den[q].y));
            go[q] = mul2(g[q], mul2(num[q], inv[q]));
        }
        const bool has_prev = (COFF == 2) && !rm.first;
#pragma unroll
        for (int k = 0; k < W; ++k) {
            if (COFF == 2 && k < RATIO && !has_prev)
                continue;
            int64_t tok;
            int col, arow;
            window_slot<RATIO, COFF>(k, rm, j, a.head_dim, tok, col, arow);
            const uint32_t kw[4] = {kvv[k].x, kvv[k].y, kvv[k].z, kvv[k].w};
            uint32_t dk[4], dsw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 p = mul2(e[k][q], inv[q]);
                dk[q] = f2_to_bf16x2(mul2(g[q], p));
                const float2 gvk = mul2(g[q], bf16x2_to_f2(kw[q]));
                const float2 ds = mul2(p, add2(gvk, make_float2(-go[q].x, -go[q].y)));
                dsw[q] = f2_to_bf16x2(ds);
                acc[k][q] = add2(acc[k][q], ds);
            }
            if (tok < n_tokens) {
                *reinterpret_cast<uint4 *>(dkv + tok * C + col) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
                *reinterpret_cast<uint4 *>(dscore + tok * C + col) =
                    make_uint4(dsw[0], dsw[1], dsw[2], dsw[3]);
            }
        }
        // Last block of its segment: own first-half columns are never read (coff 2),
        // and the tokens up to the next real block are a gap.
        const bool last = (r + 1 == __ldg(a.cc + rm.seg + 1));
        if (last) {
            if (COFF == 2) {
                for (int i = 0; i < RATIO; ++i) {
                    const int64_t tok = rm.base + i;
                    if (tok < n_tokens) {
                        *reinterpret_cast<uint4 *>(dkv + tok * C + j) = zero4;
                        *reinterpret_cast<uint4 *>(dscore + tok * C + j) = zero4;
                    }
                }
            }
            int64_t next = n_tokens;
            if (r + 1 < R)
                next = map_row(r + 1, a.cu, a.cc, a.n_seg, RATIO).base;
            zero_tokens(rm.base + RATIO, next);
        }
    }

    // grad_ape partial of this block: lanes added in ascending order in shared
    // memory laid out [ape row][half][slice column], then copied out.
    float *dst = partial + (int64_t)blockIdx.x * RATIO * C;
    if (lanes == 1) {
        if (!col_ok)
            return;
#pragma unroll
        for (int k = 0; k < W; ++k) {
            int col, arow;
            ape_slot<RATIO, COFF>(k, j, a.head_dim, arow, col);
            float4 *d = reinterpret_cast<float4 *>(dst + (int64_t)arow * C + col);
            d[0] = make_float4(acc[k][0].x, acc[k][0].y, acc[k][1].x, acc[k][1].y);
            d[1] = make_float4(acc[k][2].x, acc[k][2].y, acc[k][3].x, acc[k][3].y);
        }
        return;
    }
    const int SW = blockDim.x * 8;  // columns per half in this block's slice
    const int c0 = blockIdx.y * SW;
    for (int l = 0; l < lanes; ++l) {
        if (y == l && col_ok) {
#pragma unroll
            for (int k = 0; k < W; ++k) {
                int col, arow;
                ape_slot<RATIO, COFF>(k, j, a.head_dim, arow, col);
                const int half = col >= a.head_dim ? 1 : 0;
                float *sp = red + (arow * COFF + half) * SW + (j - c0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
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
    const int nthreads = blockDim.x * blockDim.y;
    const int tid = y * blockDim.x + x;
    const int per_row4 = SW / 4;  // float4 per (ape row, half)
    for (int i = tid; i < RATIO * COFF * per_row4; i += nthreads) {
        const int rh = i / per_row4, lc = (i - rh * per_row4) * 4;
        const int arow = rh / COFF, half = rh - arow * COFF;
        if (c0 + lc < a.head_dim)
            *reinterpret_cast<float4 *>(dst + (int64_t)arow * C + half * a.head_dim + c0 + lc) =
                *reinterpret_cast<const float4 *>(red + rh * SW + lc);
    }
}

}  // namespace

// grad_ape = sum of the partials in ascending order: ((p0 + p1) + p2) + ...
__global__ void __launch_bounds__(256) dape_finalize_kernel(const float *__restrict__ partial,
                                                            int n_partials, int64_t n,
                                                            float *__restrict__ dape)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (4 * i >= n)
        return;
    const float4 *p = reinterpret_cast<const float4 *>(partial) + i;
    const int64_t stride = n / 4;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int b = 0;
    constexpr int U = 16;
    for (; b + U <= n_partials; b += U) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            v[u] = __ldcg(p + (int64_t)(b + u) * stride);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            acc.x = __fadd_rn(acc.x, v[u].x);
            acc.y = __fadd_rn(acc.y, v[u].y);
            acc.z = __fadd_rn(acc.z, v[u].z);
            acc.w = __fadd_rn(acc.w, v[u].w);
        }
    }
    for (; b < n_partials; ++b) {
        const float4 v = __ldcg(p + (int64_t)b * stride);
        acc.x = __fadd_rn(acc.x, v.x);
        acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z);
        acc.w = __fadd_rn(acc.w, v.w);
    }
    reinterpret_cast<float4 *>(dape)[i] = acc;
}

// ------------------------------------------------------------ launchers

template <int RATIO, int COFF>
static cudaError_t launch_fwd_small_t(const FwdParams &p, cudaStream_t st)
{
    SmallArgs a{static_cast<const uint16_t *>(p.kv), static_cast<const uint16_t *>(p.score), p.ape,
                p.cu_seqlens, p.cu_seqlens_comp, p.n_seg, p.head_dim, p.capacity};
    const int64_t threads = (int64_t)p.capacity * (p.head_dim / 8);
    const int block = 256;
    const int64_t grid = (threads + block - 1) / block;
    fwd_small_kernel<RATIO, COFF><<<(unsigned)grid, block, 0, st>>>(a, static_cast<uint16_t *>(p.out));
    return cudaGetLastError();
}

cudaError_t launch_fwd_small(const FwdParams &p, cudaStream_t st)
{
    if (p.ratio == 4 && p.coff == 2)
        return launch_fwd_small_t<4, 2>(p, st);
    if (p.ratio == 4 && p.coff == 1)
        return launch_fwd_small_t<4, 1>(p, st);
    return cudaErrorInvalidValue;
}

SmallBwdPlan plan_bwd_small(int ratio, int coff, int head_dim, int capacity, int num_sms)
{
    SmallBwdPlan pl;
    const int groups = head_dim / 8;
    pl.threads_x = groups < 64 ? groups : 64;
    pl.col_slices = (groups + pl.threads_x - 1) / pl.threads_x;
    pl.lanes = 128 / pl.threads_x > 1 ? 128 / pl.threads_x : 1;
    const int max_blocks = (num_sms * 2 + pl.col_slices - 1) / pl.col_slices;
    const int rows = capacity > 0 ? capacity : 1;
    int blocks = (rows + pl.lanes - 1) / pl.lanes;
    if (blocks > max_blocks)
        blocks = max_blocks;
    pl.rows_per_block = (rows + blocks - 1) / blocks;
    pl.blocks = (rows + pl.rows_per_block - 1) / pl.rows_per_block;
    pl.smem = pl.lanes > 1 ? (size_t)ratio * coff * pl.threads_x * 8 * sizeof(float) : 0;
    pl.partial_floats = (int64_t)pl.blocks * ratio * coff * head_dim;
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
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
        if (e != cudaSuccess)
            return e;
    }
    dim3 block(pl.threads_x, pl.lanes);
    dim3 grid(pl.blocks, pl.col_slices);
    kern<<<grid, block, pl.smem, st>>>(a, pl.rows_per_block, p.n_tokens,
                                           static_cast<const uint16_t *>(p.grad_out),
                                           static_cast<uint16_t *>(p.dkv),
                                           static_cast<uint16_t *>(p.dscore), partial);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const int64_t n = (int64_t)RATIO * COFF * p.head_dim;
    const int64_t threads = n / 4;
    dape_finalize_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(partial, pl.blocks, n, p.dape);
    return cudaGetLastError();
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
