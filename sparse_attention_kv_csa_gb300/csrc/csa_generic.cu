// Compressor kernels for every other ratio: 1 <= ratio <= 128, windows of up to
// 256 positions ("CSA Fused Compressor", cuDNN frontend docs, section Semantics;
// the page's generic kernels are generic over the ratio as well).
//
// One thread owns four adjacent columns j .. j+3 (two fp32 pairs) of one output
// row and walks the window three times (max; exp and sums; gradients), straight
// from global memory: the window is too long for registers at large ratios and
// the re-reads of a row's window hit L1/L2, so DRAM traffic stays the algorithmic
// bytes.  A window is walked part by part (coff 2: the previous block's tokens on
// the first-half columns, then the own block's tokens on the second half; coff 1:
// the own block), token by token with a pointer stepped by the row stride, a few
// tokens' loads issued before any of them is used.  The arithmetic is the library's stated
// fp32 order, exactly as in the ratio-4 kernels (same exp, same reciprocal,
// ascending window positions), so results are bitwise equal to the fp32 oracle.
//
// Backward: a block owns a column tile of blockDim.x column groups and a contiguous
// group of rows; lane y of the block takes rows y, y + lanes, ... of the group in
// ascending order.  Each thread keeps its grad_ape sums for every window position
// in its own shared-memory slots (no sharing, no atomics); at the end the lanes are
// added in ascending lane order and the block writes the group's partial
// [ratio, coff*head_dim] entries of its columns; dape_finalize_kernel adds the
// groups in ascending order.  Gradient coverage as in the other kernels: a real row
// writes the slots it reads, the last block of a segment zeroes its own first-half
// columns (coff 2) and the tokens up to the next real block (or n_tokens), row
// group 0 zeroes the tokens before the first real block.
#include "csa_device.cuh"
#include "csa_launch.h"

namespace csa {

namespace {

constexpr int kGenFwdThreads = 256;
constexpr int kGenBwdGroups = 16;  // column groups (64 columns) per backward block
constexpr int kGenBwdMaxLanes = 8;
constexpr size_t kGenBwdSmem = 96 * 1024;      // grad_ape slots: lanes x window x groups x float4
constexpr int64_t kGenPartialFloats = 1 << 20;  // grad_ape partials budget (unless one group exceeds it)
// Tokens whose loads are issued together: 2 in the forward (fewer registers, more
// warps per SM), 8 in the backward (its blocks are few and its three passes long);
// both measured fastest on GB300.
constexpr int kFwdGB = 2;
constexpr int kBwdGB = 8;

struct GenArgs {
    const uint16_t *kv;
    const uint16_t *score;
    const float *ape;
    const int32_t *cu;
    const int32_t *cc;
    int n_seg;
    int ratio;
    int coff;
    int head_dim;
    int capacity;
};

// Part p of a row's window for the thread's columns: ratio consecutive tokens
// starting at tok0, read at packed column col; APE rows 0 .. ratio-1 at col.
// Window position k = p*ratio + i.
struct Part {
    int64_t tok0;
    int col;
};

// Part p exists unless it is the previous block's half of a segment's first block.
__device__ __forceinline__ bool part_valid(const GenArgs &a, const RowMap &rm, int p)
{
    return !(a.coff == 2 && p == 0 && rm.first);
}

__device__ __forceinline__ Part part_of(const GenArgs &a, const RowMap &rm, int p, int j)
{
    Part q;
    if (a.coff == 2) {
        q.tok0 = rm.base + (int64_t)(p - 1) * a.ratio;
        q.col = p * a.head_dim + j;
    } else {
        q.tok0 = rm.base;
        q.col = j;
    }
    return q;
}

__device__ __forceinline__ void ld4(uint32_t (&w)[2], const uint16_t *p)
{
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
    w[0] = v.x;
    w[1] = v.y;
}

__device__ __forceinline__ void ld4f(float2 (&f)[2], const float *p)
{
    const float4 v = __ldg(reinterpret_cast<const float4 *>(p));
    f[0] = make_float2(v.x, v.y);
    f[1] = make_float2(v.z, v.w);
}

// Passes 1 and 2 of one row: m (NaN-propagating max), den and num, per pair.
template <int kGB>
__device__ __forceinline__ void gen_pool(const GenArgs &a, const RowMap &rm, int j, int64_t C, float2 (&m)[2],
                                         float2 (&den)[2], float2 (&num)[2])
{
    m[0] = m[1] = make_float2(-INFINITY, -INFINITY);
    for (int p = 0; p < a.coff; ++p) {
        if (!part_valid(a, rm, p))
            continue;
        const Part q = part_of(a, rm, p, j);
        const uint16_t *sp = a.score + q.tok0 * C + q.col;
        const float *ap = a.ape + q.col;
        for (int i0 = 0; i0 < a.ratio; i0 += kGB) {
            uint32_t sw[kGB][2];
            float2 av[kGB][2];
#pragma unroll
            for (int u = 0; u < kGB; ++u)
                if (i0 + u < a.ratio) {
                    ld4(sw[u], sp + (int64_t)(i0 + u) * C);
                    ld4f(av[u], ap + (int64_t)(i0 + u) * C);
                }
#pragma unroll
            for (int u = 0; u < kGB; ++u)
                if (i0 + u < a.ratio)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float2 s = add2(bf16x2_to_f2(sw[u][h]), av[u][h]);
                        m[h].x = max_nan(m[h].x, s.x);
                        m[h].y = max_nan(m[h].y, s.y);
                    }
        }
    }
    const float2 negm[2] = {make_float2(-m[0].x, -m[0].y), make_float2(-m[1].x, -m[1].y)};
    den[0] = den[1] = num[0] = num[1] = make_float2(0.0f, 0.0f);
    for (int p = 0; p < a.coff; ++p) {
        if (!part_valid(a, rm, p))
            continue;
        const Part q = part_of(a, rm, p, j);
        const uint16_t *sp = a.score + q.tok0 * C + q.col;
        const uint16_t *kp = a.kv + q.tok0 * C + q.col;
        const float *ap = a.ape + q.col;
        for (int i0 = 0; i0 < a.ratio; i0 += kGB) {
            uint32_t sw[kGB][2], kw[kGB][2];
            float2 av[kGB][2];
#pragma unroll
            for (int u = 0; u < kGB; ++u)
                if (i0 + u < a.ratio) {
                    ld4(sw[u], sp + (int64_t)(i0 + u) * C);
                    ld4(kw[u], kp + (int64_t)(i0 + u) * C);
                    ld4f(av[u], ap + (int64_t)(i0 + u) * C);
                }
#pragma unroll
            for (int u = 0; u < kGB; ++u)
                if (i0 + u < a.ratio)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float2 e = exp2lanes(add2(add2(bf16x2_to_f2(sw[u][h]), av[u][h]), negm[h]));
                        den[h] = add2(den[h], e);
                        num[h] = fma2(e, bf16x2_to_f2(kw[u][h]), num[h]);
                    }
        }
    }
}

__global__ void __launch_bounds__(kGenFwdThreads) fwd_generic_kernel(GenArgs a, uint16_t *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int groups = a.head_dim / 4;
    const int64_t units = (int64_t)a.capacity * groups;
    const int64_t C = (int64_t)a.coff * a.head_dim;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(u / groups);
        const int j = 4 * (int)(u - (int64_t)r * groups);
        // padding rows (and rows below cu_seqlens_comp[0]) come back as a first
        // block starting at token 0
        const RowMap rm = map_row(r, a.cu, a.cc, a.n_seg, a.ratio);
        float2 m[2], den[2], num[2];
        gen_pool<kFwdGB>(a, rm, j, C, m, den, num);
        uint32_t o[2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
            o[h] = f2_to_bf16x2(mul2(num[h], make_float2(recip_den(den[h].x), recip_den(den[h].y))));
        *reinterpret_cast<uint2 *>(out + (int64_t)r * a.head_dim + j) = make_uint2(o[0], o[1]);
    }
}

// Zero the gradient slots of tokens [t0, t1) in the thread's columns (first half
// only, or every half).
__device__ __forceinline__ void gen_zero(const GenArgs &a, uint16_t *dkv, uint16_t *dscore, int64_t C, int j,
                                         int64_t t0, int64_t t1, int64_t n_tokens, bool all_halves)
{
    t1 = t1 < n_tokens ? t1 : n_tokens;
    for (int64_t t = t0 < 0 ? 0 : t0; t < t1; ++t) {
        *reinterpret_cast<uint2 *>(dkv + t * C + j) = make_uint2(0u, 0u);
        *reinterpret_cast<uint2 *>(dscore + t * C + j) = make_uint2(0u, 0u);
        if (a.coff == 2 && all_halves) {
            *reinterpret_cast<uint2 *>(dkv + t * C + a.head_dim + j) = make_uint2(0u, 0u);
            *reinterpret_cast<uint2 *>(dscore + t * C + a.head_dim + j) = make_uint2(0u, 0u);
        }
    }
}

__global__ void __launch_bounds__(kGenBwdGroups * kGenBwdMaxLanes, 2)
    bwd_generic_kernel(GenArgs a, int rows_per_group, int64_t n_tokens_arg, const uint16_t *__restrict__ grad_out,
                       uint16_t *__restrict__ dkv, uint16_t *__restrict__ dscore, float *__restrict__ partial)
{
    extern __shared__ float4 acc[];  // [lane][window position][column group]: each thread's own slots
    pdl_wait();
    pdl_trigger();  // the grad_ape finalisation may launch; it waits for this grid's end
    const int W = a.coff * a.ratio;
    const int TG = blockDim.x, lanes = blockDim.y, y = threadIdx.y;
    const int groups = a.head_dim / 4;
    const int gidx = blockIdx.y * TG + threadIdx.x;
    const bool col_ok = gidx < groups;
    const int j = 4 * gidx;
    const int64_t C = (int64_t)a.coff * a.head_dim;
    const int64_t n_tokens = n_tokens_arg >= 0 ? n_tokens_arg : (int64_t)__ldg(a.cu + a.n_seg);
    const int R = a.n_seg > 0 ? __ldg(a.cc + a.n_seg) : 0;
    const int R0 = a.n_seg > 0 ? __ldg(a.cc) : 0;
    float4 *mine = acc + (size_t)y * W * TG + threadIdx.x;  // slot k at mine[k * TG]
    for (int k = 0; k < W; ++k)
        mine[k * TG] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);

    if (col_ok && blockIdx.x == 0 && y == 0) {  // leading gap: tokens before the first real block
        int64_t lead = n_tokens;
        if (R0 < R)
            lead = map_row(R0, a.cu, a.cc, a.n_seg, a.ratio).base;
        gen_zero(a, dkv, dscore, C, j, 0, lead, n_tokens, true);
    }

    const int r0 = blockIdx.x * rows_per_group;
    int r1 = r0 + rows_per_group;
    r1 = r1 < a.capacity ? r1 : a.capacity;
    r1 = r1 < R ? r1 : R;  // padding rows carry no gradient
    for (int r = r0 + y; col_ok && r < r1; r += lanes) {
        const RowMap rm = map_row(r, a.cu, a.cc, a.n_seg, a.ratio);
        if (!rm.real)
            continue;
        float2 m[2], den[2], num[2];
        gen_pool<kBwdGB>(a, rm, j, C, m, den, num);
        uint32_t gw[2];
        ld4(gw, grad_out + (int64_t)r * a.head_dim + j);
        float2 g[2], inv[2], ngo[2], negm[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            g[h] = bf16x2_to_f2(gw[h]);
            inv[h] = make_float2(recip_den(den[h].x), recip_den(den[h].y));
            const float2 go = mul2(g[h], mul2(num[h], inv[h]));
            ngo[h] = make_float2(-go.x, -go.y);
            negm[h] = make_float2(-m[h].x, -m[h].y);
        }
        for (int p = 0; p < a.coff; ++p) {
            if (!part_valid(a, rm, p))
                continue;
            const Part q = part_of(a, rm, p, j);
            const uint16_t *sp = a.score + q.tok0 * C + q.col;
            const uint16_t *kp = a.kv + q.tok0 * C + q.col;
            const float *ap = a.ape + q.col;
            uint16_t *dkp = dkv + q.tok0 * C + q.col;
            uint16_t *dsp = dscore + q.tok0 * C + q.col;
            const int64_t lim = n_tokens - q.tok0;  // tokens i < lim exist
            float4 *slot = mine + (size_t)p * a.ratio * TG;
            for (int i0 = 0; i0 < a.ratio; i0 += kBwdGB) {
                uint32_t sw[kBwdGB][2], kw[kBwdGB][2];
                float2 av[kBwdGB][2];
#pragma unroll
                for (int u = 0; u < kBwdGB; ++u)
                    if (i0 + u < a.ratio) {
                        ld4(sw[u], sp + (int64_t)(i0 + u) * C);
                        ld4(kw[u], kp + (int64_t)(i0 + u) * C);
                        ld4f(av[u], ap + (int64_t)(i0 + u) * C);
                    }
#pragma unroll
                for (int u = 0; u < kBwdGB; ++u) {
                    const int i = i0 + u;
                    if (i >= a.ratio)
                        continue;
                    uint32_t dk[2], dsw[2];
                    float2 ds[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float2 e = exp2lanes(add2(add2(bf16x2_to_f2(sw[u][h]), av[u][h]), negm[h]));
                        const float2 pk = mul2(e, inv[h]);
                        dk[h] = f2_to_bf16x2(mul2(g[h], pk));
                        ds[h] = mul2(pk, add2(mul2(g[h], bf16x2_to_f2(kw[u][h])), ngo[h]));
                        dsw[h] = f2_to_bf16x2(ds[h]);
                    }
                    float4 &ak = slot[(size_t)i * TG];
                    const float2 lo = add2(make_float2(ak.x, ak.y), ds[0]);
                    const float2 hi = add2(make_float2(ak.z, ak.w), ds[1]);
                    ak = make_float4(lo.x, lo.y, hi.x, hi.y);
                    if (i < lim) {
                        *reinterpret_cast<uint2 *>(dkp + (int64_t)i * C) = make_uint2(dk[0], dk[1]);
                        *reinterpret_cast<uint2 *>(dsp + (int64_t)i * C) = make_uint2(dsw[0], dsw[1]);
                    }
                }
            }
        }
        if (r + 1 == __ldg(a.cc + rm.seg + 1)) {  // last block of its segment
            if (a.coff == 2)  // own block's first-half columns: read by no row
                gen_zero(a, dkv, dscore, C, j, rm.base, rm.base + a.ratio, n_tokens, false);
            int64_t next = n_tokens;
            if (r + 1 < R)
                next = map_row(r + 1, a.cu, a.cc, a.n_seg, a.ratio).base;
            gen_zero(a, dkv, dscore, C, j, rm.base + a.ratio, next, n_tokens, true);
        }
    }
    __syncthreads();
    // lanes added in ascending order (lane y takes positions k = y, y + lanes, ...),
    // then this group's partial: [ape row][packed column], the thread's four columns
    float *dst = partial + (int64_t)blockIdx.x * a.ratio * C;
    for (int k = y; col_ok && k < W; k += lanes) {
        float4 s = acc[(size_t)k * TG + threadIdx.x];
        for (int l = 1; l < lanes; ++l) {
            const float4 v = acc[((size_t)l * W + k) * TG + threadIdx.x];
            s.x = __fadd_rn(s.x, v.x);
            s.y = __fadd_rn(s.y, v.y);
            s.z = __fadd_rn(s.z, v.z);
            s.w = __fadd_rn(s.w, v.w);
        }
        const int arow = k % a.ratio, half = k / a.ratio;
        *reinterpret_cast<float4 *>(dst + (int64_t)arow * C + half * a.head_dim + j) = s;
    }
}

}  // namespace

bool generic_supported(int ratio, int coff, int head_dim)
{
    return ratio >= 1 && ratio <= 128 && (coff == 1 || coff == 2) && head_dim % 8 == 0 && head_dim <= 8192;
}

GenericPlan plan_generic(int ratio, int coff, int head_dim, int capacity, int num_sms)
{
    GenericPlan pl;
    const int groups4 = head_dim / 4;
    pl.col_tiles = (groups4 + kGenBwdGroups - 1) / kGenBwdGroups;
    const size_t lane_bytes = (size_t)coff * ratio * kGenBwdGroups * sizeof(float4);
    int lanes = (int)(kGenBwdSmem / lane_bytes);
    pl.lanes = lanes < 1 ? 1 : lanes > kGenBwdMaxLanes ? kGenBwdMaxLanes : lanes;
    const int rows = capacity > 0 ? capacity : 1;
    int groups = 8 * num_sms / pl.col_tiles;  // blocks of up to 4 warps: several per SM
    const int64_t per_group = (int64_t)ratio * coff * head_dim;
    if ((int64_t)groups * per_group > kGenPartialFloats)  // keep the grad_ape workspace within 4 MB
        groups = (int)(kGenPartialFloats / per_group);
    groups = groups < 1 ? 1 : groups;
    const int max_groups = (rows + pl.lanes - 1) / pl.lanes;  // at least one row per lane
    groups = groups < max_groups ? groups : max_groups;
    pl.rows_per_group = (rows + groups - 1) / groups;
    pl.groups = (rows + pl.rows_per_group - 1) / pl.rows_per_group;
    pl.smem = lane_bytes * pl.lanes;
    pl.partial_floats = (int64_t)pl.groups * ratio * coff * head_dim;
    pl.num_sms = num_sms;
    return pl;
}

cudaError_t launch_fwd_generic(const FwdParams &p, int num_sms, cudaStream_t st)
{
    GenArgs a{static_cast<const uint16_t *>(p.kv), static_cast<const uint16_t *>(p.score), p.ape, p.cu_seqlens,
              p.cu_seqlens_comp, p.n_seg, p.ratio, p.coff, p.head_dim, p.capacity};
    const int64_t units = (int64_t)p.capacity * (p.head_dim / 4);
    int64_t grid = (units + kGenFwdThreads - 1) / kGenFwdThreads;
    const int64_t cap = 8 * (int64_t)num_sms;
    grid = grid < cap ? grid : cap;
    grid = grid < 1 ? 1 : grid;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kGenFwdThreads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fwd_generic_kernel, a, static_cast<uint16_t *>(p.out));
}

cudaError_t launch_bwd_generic(const BwdParams &p, const GenericPlan &pl, float *partial, cudaStream_t st)
{
    GenArgs a{static_cast<const uint16_t *>(p.kv), static_cast<const uint16_t *>(p.score), p.ape, p.cu_seqlens,
              p.cu_seqlens_comp, p.n_seg, p.ratio, p.coff, p.head_dim, p.capacity};
    if (pl.smem > 48 * 1024) {
        cudaError_t e = allow_max_smem(reinterpret_cast<const void *>(bwd_generic_kernel));
        if (e != cudaSuccess)
            return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.groups, pl.col_tiles, 1);
    cfg.blockDim = dim3(kGenBwdGroups, pl.lanes, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, bwd_generic_kernel, a, pl.rows_per_group, p.n_tokens,
                                       static_cast<const uint16_t *>(p.grad_out), static_cast<uint16_t *>(p.dkv),
                                       static_cast<uint16_t *>(p.dscore), partial);
    if (e != cudaSuccess)
        return e;
    return launch_dape_finalize(partial, pl.groups, (int64_t)p.ratio * p.coff * p.head_dim, p.dape, st);
}

}  // namespace csa
