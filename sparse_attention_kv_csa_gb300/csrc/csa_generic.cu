// Compressor kernels for every other ratio: 1 <= ratio <= 128, windows of up to
// 256 positions ("CSA Fused Compressor", cuDNN frontend docs, section Semantics;
// the page's generic kernels are generic over the ratio as well).  Two families:
// the staged kernels (further down) for windows of at most 64 positions on
// head_dim a multiple of 64, and the global-memory walk below for the rest.
//
// Global-memory walk: one thread owns four adjacent columns j .. j+3 (two fp32 pairs) of one output
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
                        const float2 s = add2_bf16x2(sw[u][h], av[u][h]);
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
                        const float2 e = exp2lanes(add2(add2_bf16x2(sw[u][h], av[u][h]), negm[h]));
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
                        const float2 e = exp2lanes(add2(add2_bf16x2(sw[u][h], av[u][h]), negm[h]));
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


// ------------------------------------------------------------ staged kernels
// Windows of at most kGsMaxWindow positions on head_dim a multiple of 64: the
// window is staged through shared memory instead of walked in global memory.  A
// block owns a 64-column tile; one producer thread streams its rows' windows with
// 2-D TMA boxes (per part and array one [ratio x 64] box) into a ring of stages;
// each consumer warp takes whole rows (row lane l: the block's rows l, l + lanes,
// ...), a row's 64 columns at two per thread, and walks the window in shared
// memory: max, then exp / sums, then (backward) the gradients, with the tile's
// APE rows held in shared memory for the whole block.  Narrow tiles keep a row's
// stage small, so many rows (warps) are in flight per SM.  Same arithmetic and
// order as the rest of the library.  Backward grad_ape: each thread sums its
// rows' ds per window position in its own shared-memory slots; lanes are added
// in ascending order and the block writes one partial [ratio, C] for its columns.

constexpr int kGsTile = 64;       // columns per block tile (two per consumer thread)
constexpr int kGsMaxWindow = 64;  // coff * ratio
constexpr int kGsMaxLanes = 4;    // consumer warps per block
constexpr int kGsRingBudget = 64 * 1024;  // ring bytes of a block with four consumer warps
// Per window bucket (the plan below maximises rows in flight by shared memory;
// a short window's row tile is only 1-4 KB, so its blocks are bound by their one
// producer thread's copy issue, and more, smaller blocks help): the 16-position
// bucket takes a 48 KB ring (ratio 5 / 8 with coff 2, 12 with coff 1, backward
// 105.8 / 70.8 / 52.4 -> 78.6 / 66.6 / 40.7 us at 8 x 4096 tokens, head_dim 512),
// the 8-position bucket at most two consumer warps (ratio 2 / 3 with coff 2,
// forward 63.2 / 51.8 -> 52.7 / 42.3 us).
constexpr int kGsRingBudget16 = 48 * 1024;
constexpr int kGsMaxLanes8 = 2;
constexpr size_t kGsSmemPerSM = 228 * 1024;  // shared memory per SM, 1 KB of it reserved per block

struct GsArgs {
    GenArgs g;
    int stages;       // ring depth, a multiple of the consumer warps
    int stage_bytes;  // window (+ grad_out row), a multiple of 128
    unsigned *status;
};

struct GsMeta {
    int64_t base;
    int seg;
    int row;
    int real;
    int first;
    int last;  // the last block of its segment (from the producer's row cursor)
    int pad;
};

struct GsSmem {
    unsigned char *stages;  // [stage][array][part][ratio][kGsTile] bf16 (+ grad_out row)
    GsMeta *meta;
    uint64_t *full;
    uint64_t *empty;
    float *apet;  // [window position][kGsTile]
    float2 *acc;  // backward: [lane][window position][32 threads]
};

size_t gs_smem_bytes(int stages, int stage_bytes, int W, int lanes, bool bwd)
{
    return 128 + (size_t)stages * stage_bytes + (sizeof(GsMeta) + 16) * stages + (size_t)W * kGsTile * sizeof(float) +
           (bwd ? (size_t)lanes * W * 32 * sizeof(float2) : 0);
}

__device__ __forceinline__ GsSmem gs_carve(unsigned char *raw, int stages, int stage_bytes, int W)
{
    GsSmem s;
    // 128-byte aligned stages (TMA destinations), by an offset from the shared
    // array (no integer round trip: the pointers stay shared-memory pointers)
    unsigned char *p = raw + ((128u - (smem_addr(raw) & 127u)) & 127u);
    s.stages = p;
    p += (size_t)stages * stage_bytes;
    s.meta = reinterpret_cast<GsMeta *>(p);
    p += sizeof(GsMeta) * stages;
    s.full = reinterpret_cast<uint64_t *>(p);
    s.empty = s.full + stages;
    p = reinterpret_cast<unsigned char *>(s.empty + stages);
    s.apet = reinterpret_cast<float *>(p);
    p += (size_t)W * kGsTile * sizeof(float);
    s.acc = reinterpret_cast<float2 *>(p);
    return s;
}

// Issues the window copies of rows row0, row0 + rstride, ... < rend.  One thread.
template <bool BWD>
__device__ void gs_produce(const GsArgs &a, const GsSmem &s, const CUtensorMap *tm_kv, const CUtensorMap *tm_sc,
                           const CUtensorMap *tm_kv2, const CUtensorMap *tm_sc2, int c0, int row0, int rstride,
                           int rend, const uint16_t *__restrict__ grad_out)
{
    const GenArgs &g = a.g;
    const uint32_t part_bytes = (uint32_t)g.ratio * kGsTile * 2;
    int issued = 0, st = 0;
    uint32_t ph = 0;
    RowCursor cur;
    cursor_init(cur, g.cc, g.n_seg);
    for (int row = row0; row < rend; row += rstride) {
        // the row's map first: its loads (if any) overlap the wait for a free slot
        const RowMap rm = cursor_map(cur, row, g.cu, g.cc, g.n_seg, g.ratio);
        if (!mbar_wait(smem_addr(&s.empty[st]), ph ^ 1u, a.status))
            break;
        GsMeta &m = s.meta[st];
        m.base = rm.base;
        m.seg = rm.seg;
        m.row = row;
        m.real = rm.real;
        m.first = rm.first;
        m.last = rm.real && row + 1 == cur.hi;
        const bool load = BWD ? rm.real : true;
        const int p0 = (g.coff == 2 && rm.first) ? 1 : 0;
        const uint32_t bytes = load ? (uint32_t)(g.coff - p0) * 2u * part_bytes + (BWD ? kGsTile * 2u : 0u) : 0u;
        const uint32_t fb = smem_addr(&s.full[st]);
        mbar_arrive_expect_tx(fb, bytes);
        if (load) {
            const uint32_t dst = smem_addr(s.stages + (size_t)st * a.stage_bytes);
            if (g.coff == 2 && p0 == 0) {
                // both parts in one box per array (part 0 starts ratio tokens before
                // the row's block, which is not a segment's first: y >= 0)
                const int y = (int)(rm.base - g.ratio);
                tma_load_3d(dst, tm_kv2, c0, y, 0, fb);
                tma_load_3d(dst + 2u * part_bytes, tm_sc2, c0, y, 0, fb);
            } else {
                for (int p = p0; p < g.coff; ++p) {
                    const int y = (int)(rm.base + (int64_t)(p - (g.coff - 1)) * g.ratio);
                    const int x = p * g.head_dim + c0;
                    tma_load_2d(dst + (uint32_t)p * part_bytes, tm_kv, x, y, fb);
                    tma_load_2d(dst + (uint32_t)(g.coff + p) * part_bytes, tm_sc, x, y, fb);
                }
            }
            if (BWD)
                bulk_g2s(dst + 2u * g.coff * part_bytes, grad_out + (int64_t)row * g.head_dim + c0, kGsTile * 2, fb);
        }
        ++issued;
        if (++st == a.stages) {
            st = 0;
            ph ^= 1u;
        }
    }
    const int lo = issued > a.stages ? issued - a.stages : 0;
    for (int it = lo; it < issued; ++it)
        mbar_wait(smem_addr(&s.full[it % a.stages]), (uint32_t)(it / a.stages) & 1u, a.status);
}

// The tile's APE rows, [window position k][tile column], by the consumer threads.
__device__ __forceinline__ void gs_load_ape(const GenArgs &g, float *apet, int c0, int t, int nthreads)
{
    const int W = g.coff * g.ratio;
    const int64_t C = (int64_t)g.coff * g.head_dim;
    for (int idx = t; idx < W * (kGsTile / 4); idx += nthreads) {
        const int k = idx / (kGsTile / 4), c4 = idx % (kGsTile / 4);
        const int p = k / g.ratio, i = k % g.ratio;
        const float4 v = __ldg(reinterpret_cast<const float4 *>(g.ape + i * C + (int64_t)p * g.head_dim + c0 + 4 * c4));
        *reinterpret_cast<float4 *>(apet + k * kGsTile + 4 * c4) = v;
    }
}

// Logits of window position k for the thread's two columns (stage + APE tile).
__device__ __forceinline__ float2 gs_logits(const unsigned char *sc, const float *ap, int k)
{
    const uint32_t w = *reinterpret_cast<const uint32_t *>(sc + k * (kGsTile * 2));
    return add2_bf16x2(w, *reinterpret_cast<const float2 *>(ap + k * kGsTile));
}

// Passes 1 and 2 over the staged window (positions k0 .. W-1 of at most WMAX):
// the logits, then e = EXP(s - m) in place, in registers (the window loop is
// unrolled to WMAX, positions outside [k0, W) skipped); m, den, num.
// TREE (the forward): the maximum is taken over all WMAX slots, positions outside
// [k0, W) holding -inf, in three interleaved chains of three-input maxima joined
// at the end -- the maximum of a set does not depend on the grouping (NaN if any
// is NaN), and three short chains instead of one of W dependent steps keep the
// warp issuing.  The backward, short of registers, keeps the single chain.
template <int WMAX, bool TREE>
__device__ __forceinline__ void gs_pool(const unsigned char *kvp, const unsigned char *sc, const float *ap, int k0,
                                        int W, float2 (&e)[WMAX], float2 &m, float2 &den, float2 &num)
{
    if constexpr (TREE) {
#pragma unroll
        for (int k = 0; k < WMAX; ++k)
            e[k] = (k >= k0 && k < W) ? gs_logits(sc, ap, k) : make_float2(-INFINITY, -INFINITY);
        float2 mc[3];
#pragma unroll
        for (int i = 0; i < 3; ++i)
            mc[i] = make_float2(-INFINITY, -INFINITY);
#pragma unroll
        for (int k = 0; k < WMAX; k += 2) {
            float2 &a = mc[(k / 2) % 3];
            a.x = max3_nan(a.x, e[k].x, e[k + 1].x);
            a.y = max3_nan(a.y, e[k].y, e[k + 1].y);
        }
        m = make_float2(max3_nan(mc[0].x, mc[1].x, mc[2].x), max3_nan(mc[0].y, mc[1].y, mc[2].y));
    } else {
        m = make_float2(-INFINITY, -INFINITY);
#pragma unroll
        for (int k = 0; k < WMAX; ++k)
            if (k >= k0 && k < W) {
                e[k] = gs_logits(sc, ap, k);
                m.x = max_nan(m.x, e[k].x);
                m.y = max_nan(m.y, e[k].y);
            }
    }
    const float2 negm = make_float2(-m.x, -m.y);
    den = num = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < WMAX; ++k)
        if (k >= k0 && k < W) {
            e[k] = exp2lanes(add2(e[k], negm));
            den = add2(den, e[k]);
            num = fma2(e[k], bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(kvp + k * (kGsTile * 2))), num);
        }
}

template <int WMAX>
__global__ void __launch_bounds__((kGsMaxLanes + 1) * 32)
    fwd_gs_kernel(GsArgs a, const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_sc,
                  const __grid_constant__ CUtensorMap tm_kv2, const __grid_constant__ CUtensorMap tm_sc2,
                  uint16_t *__restrict__ out)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const GenArgs &g = a.g;
    const int W = g.coff * g.ratio;
    const int lanes = blockDim.x / 32 - 1;
    const int c0 = blockIdx.y * kGsTile;
    const GsSmem s = gs_carve(smem_raw, a.stages, a.stage_bytes, W);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(smem_addr(&s.full[i]), 1);
            mbar_init(smem_addr(&s.empty[i]), 1);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    if (warp == lanes) {
        if (lane == 0)
            gs_produce<false>(a, s, &tm_kv, &tm_sc, &tm_kv2, &tm_sc2, c0, blockIdx.x, gridDim.x, g.capacity, nullptr);
        return;
    }
    gs_load_ape(g, s.apet, c0, threadIdx.x, lanes * 32);
    named_barrier(1, lanes * 32);
    const int lc = lane * 2;
    const size_t sc_off = (size_t)g.coff * g.ratio * kGsTile * 2;
    int st = warp;
    uint32_t ph = 0;
    for (int j = warp;; j += lanes, ring_next(st, ph, lanes, a.stages)) {
        const int row = blockIdx.x + j * gridDim.x;
        if (row >= g.capacity)
            break;
        if (!mbar_wait(smem_addr(&s.full[st]), ph, a.status))
            break;
        const unsigned char *stage = s.stages + (size_t)st * a.stage_bytes + lc * 2;
        const int k0 = (g.coff == 2 && s.meta[st].first) ? g.ratio : 0;
        float2 e[WMAX], m, den, num;
        gs_pool<WMAX, true>(stage, stage + sc_off, s.apet + lc, k0, W, e, m, den, num);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&s.empty[st]));
        const uint32_t o = f2_to_bf16x2(mul2(num, make_float2(recip_den(den.x), recip_den(den.y))));
        *reinterpret_cast<uint32_t *>(out + (int64_t)row * g.head_dim + c0 + lc) = o;
    }
}

// Zero the gradient slots of tokens [t0, t1) in the thread's two columns j, j+1
// (first half only, or every half).
__device__ __forceinline__ void gs_zero(const GenArgs &a, uint16_t *dkv, uint16_t *dscore, int64_t C, int j,
                                        int64_t t0, int64_t t1, int64_t n_tokens, bool all_halves)
{
    t1 = t1 < n_tokens ? t1 : n_tokens;
    for (int64_t t = t0 < 0 ? 0 : t0; t < t1; ++t) {
        *reinterpret_cast<uint32_t *>(dkv + t * C + j) = 0u;
        *reinterpret_cast<uint32_t *>(dscore + t * C + j) = 0u;
        if (a.coff == 2 && all_halves) {
            *reinterpret_cast<uint32_t *>(dkv + t * C + a.head_dim + j) = 0u;
            *reinterpret_cast<uint32_t *>(dscore + t * C + a.head_dim + j) = 0u;
        }
    }
}

template <int WMAX>
__global__ void __launch_bounds__((kGsMaxLanes + 1) * 32)
    bwd_gs_kernel(GsArgs a, const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_sc,
                  const __grid_constant__ CUtensorMap tm_kv2, const __grid_constant__ CUtensorMap tm_sc2,
                  int64_t n_tokens_arg, const uint16_t *__restrict__ grad_out, uint16_t *__restrict__ dkv,
                  uint16_t *__restrict__ dscore, float *__restrict__ partial)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const GenArgs &g = a.g;
    const int W = g.coff * g.ratio;
    const int lanes = blockDim.x / 32 - 1;
    const int c0 = blockIdx.y * kGsTile;
    const GsSmem s = gs_carve(smem_raw, a.stages, a.stage_bytes, W);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t C = (int64_t)g.coff * g.head_dim;
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(smem_addr(&s.full[i]), 1);
            mbar_init(smem_addr(&s.empty[i]), 1);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();  // the grad_ape finalisation may launch; it waits for this grid's end
    const int R = g.n_seg > 0 ? __ldg(g.cc + g.n_seg) : 0;
    const int R0 = g.n_seg > 0 ? __ldg(g.cc) : 0;
    const int rend = R < g.capacity ? R : g.capacity;  // padding rows carry no gradient
    const int64_t n_tokens = n_tokens_arg >= 0 ? n_tokens_arg : (int64_t)__ldg(g.cu + g.n_seg);
    const int lc = lane * 2;
    const int j0 = c0 + lc;  // the thread's first-half column

    if (warp == lanes) {
        if (lane == 0)
            gs_produce<true>(a, s, &tm_kv, &tm_sc, &tm_kv2, &tm_sc2, c0, blockIdx.x, gridDim.x, rend, grad_out);
    } else {
        gs_load_ape(g, s.apet, c0, threadIdx.x, lanes * 32);
        float2 *mine = s.acc + (size_t)warp * W * 32 + lane;  // slot k at mine[k * 32]
        for (int k = 0; k < W; ++k)
            mine[k * 32] = make_float2(0.0f, 0.0f);
        named_barrier(1, lanes * 32);
        if (blockIdx.x == 0 && warp == 0) {  // leading gap: tokens before the first real block
            int64_t lead = n_tokens;
            if (R0 < R)
                lead = map_row(R0, g.cu, g.cc, g.n_seg, g.ratio).base;
            gs_zero(g, dkv, dscore, C, j0, 0, lead, n_tokens, true);
        }
        const size_t sc_off = (size_t)g.coff * g.ratio * kGsTile * 2;
        const size_t go_off = 2 * sc_off;
        int st = warp;
        uint32_t ph = 0;
        for (int j = warp;; j += lanes, ring_next(st, ph, lanes, a.stages)) {
            if (blockIdx.x + j * gridDim.x >= rend)
                break;
            if (!mbar_wait(smem_addr(&s.full[st]), ph, a.status))
                break;
            const GsMeta m = s.meta[st];
            if (!m.real) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&s.empty[st]));
                continue;
            }
            const unsigned char *stage = s.stages + (size_t)st * a.stage_bytes;
            const unsigned char *kvp = stage + lc * 2, *sc = stage + sc_off + lc * 2;
            const float *ap = s.apet + lc;
            const int k0 = (g.coff == 2 && m.first) ? g.ratio : 0;
            float2 e[WMAX], mx, den, num;
            gs_pool<WMAX, false>(kvp, sc, ap, k0, W, e, mx, den, num);
            const float2 gg = bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(stage + go_off + lc * 2));
            const float2 inv = make_float2(recip_den(den.x), recip_den(den.y));
            const float2 go = mul2(gg, mul2(num, inv));
            const float2 ngo = make_float2(-go.x, -go.y);
            // window position k reads token tok_k = base - (coff-1)*ratio + k at packed
            // column p*head_dim + j0, p = 1 for the own block's half (coff 2, k >= ratio)
            const int64_t tok_k0 = m.base - (int64_t)(g.coff - 1) * g.ratio;
            const int64_t lim = n_tokens - tok_k0;  // positions k < lim have a token
            // gradient slot of position k: token row tok_k0 + k, the part's column;
            // walked by one offset stepped per position (nothing hoisted per k)
            int64_t o = (tok_k0 + k0) * C + j0 + ((g.coff == 2 && k0 >= g.ratio) ? g.head_dim : 0);
#pragma unroll
            for (int k = 0; k < WMAX; ++k)
                if (k >= k0 && k < W) {
                    if (g.coff == 2 && k == g.ratio && k0 == 0)
                        o += g.head_dim;  // into the own block's half
                    const float2 pk = mul2(e[k], inv);
                    const float2 kvf = bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(kvp + k * (kGsTile * 2)));
                    const float2 ds = mul2(pk, add2(mul2(gg, kvf), ngo));
                    mine[k * 32] = add2(mine[k * 32], ds);
                    if (k < lim) {
                        *reinterpret_cast<uint32_t *>(dkv + o) = f2_to_bf16x2(mul2(gg, pk));
                        *reinterpret_cast<uint32_t *>(dscore + o) = f2_to_bf16x2(ds);
                    }
                    o += C;
                }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&s.empty[st]));
            if (m.last) {  // last block of its segment
                if (g.coff == 2)  // own block's first-half columns: read by no row
                    gs_zero(g, dkv, dscore, C, j0, m.base, m.base + g.ratio, n_tokens, false);
                int64_t next = n_tokens;
                if (m.row + 1 < R)
                    next = map_row(m.row + 1, g.cu, g.cc, g.n_seg, g.ratio).base;
                gs_zero(g, dkv, dscore, C, j0, m.base + g.ratio, next, n_tokens, true);
            }
        }
    }
    __syncthreads();
    // lanes added in ascending order; the block's partial [ape row][packed column]
    float *dst = partial + (int64_t)blockIdx.x * g.ratio * C;
    for (int idx = threadIdx.x; idx < W * 32; idx += blockDim.x) {
        const int k = idx / 32, t = idx % 32;
        float2 sum = s.acc[(size_t)k * 32 + t];
        for (int l = 1; l < lanes; ++l) {
            const float2 v = s.acc[((size_t)l * W + k) * 32 + t];
            sum.x = __fadd_rn(sum.x, v.x);
            sum.y = __fadd_rn(sum.y, v.y);
        }
        const int p = k / g.ratio, i = k % g.ratio;
        *reinterpret_cast<float2 *>(dst + (int64_t)i * C + (int64_t)p * g.head_dim + c0 + 2 * t) = sum;
    }
}

struct GsPlan {
    int wmax;  // register window bucket: 8, 16, 32 or 64 >= coff * ratio
    int lanes;
    int stages;
    int stage_bytes;
    int threads;
    int tiles;
    size_t smem;
};

bool gs_supported(int ratio, int coff, int head_dim)
{
    return head_dim % kGsTile == 0 && coff * ratio <= kGsMaxWindow && ratio >= 1;
}

// Consumer warps per block (1, 2 or 4, each with at least two stages of its own)
// chosen for the most rows in flight per SM by shared memory.
GsPlan gs_plan(bool bwd, int ratio, int coff, int head_dim)
{
    GsPlan best{};
    const int W = coff * ratio;
    const int wmax = W <= 8 ? 8 : W <= 16 ? 16 : W <= 32 ? 32 : 64;
    const int stage_bytes = (2 * W * kGsTile * 2 + (bwd ? kGsTile * 2 : 0) + 127) / 128 * 128;
    int best_warps = -1;
    for (int lanes = wmax == 8 ? kGsMaxLanes8 : kGsMaxLanes; lanes >= 1; lanes /= 2) {
        GsPlan pl;
        pl.wmax = wmax;
        pl.lanes = lanes;
        pl.stage_bytes = stage_bytes;
        pl.tiles = head_dim / kGsTile;
        int per_lane = (wmax == 16 ? kGsRingBudget16 : kGsRingBudget) / stage_bytes / lanes;
        per_lane = per_lane < 2 ? 2 : (per_lane > 8 ? 8 : per_lane);
        pl.stages = per_lane * lanes;
        pl.smem = gs_smem_bytes(pl.stages, stage_bytes, W, lanes, bwd);
        pl.threads = (lanes + 1) * 32;
        const int per_sm = (int)(kGsSmemPerSM / (pl.smem + 1024));
        const int warps = (per_sm > 16 ? 16 : per_sm) * lanes;
        if (warps > best_warps) {
            best_warps = warps;
            best = pl;
        }
    }
    return best;
}

template <int WMAX>
const void *gs_fn(bool bwd)
{
    return bwd ? reinterpret_cast<const void *>(bwd_gs_kernel<WMAX>) : reinterpret_cast<const void *>(fwd_gs_kernel<WMAX>);
}

const void *gs_kernel(bool bwd, int wmax)
{
    switch (wmax) {
    case 8: return gs_fn<8>(bwd);
    case 16: return gs_fn<16>(bwd);
    case 32: return gs_fn<32>(bwd);
    default: return gs_fn<64>(bwd);
    }
}

// The staged kernels' tensor maps: per-part boxes [ratio x 64] of kv and score,
// and (coff 2) boxes of both parts at once (for coff 1 the per-part maps again).
cudaError_t gs_maps(const void *kv, const void *score, int ratio, int coff, int head_dim, CUtensorMap *mk,
                    CUtensorMap *ms, CUtensorMap *mk2, CUtensorMap *ms2)
{
    const int64_t C = (int64_t)coff * head_dim;
    cudaError_t e;
    if ((e = make_tensor_map_2d(mk, kv, C, kGsTile, ratio)) != cudaSuccess ||
        (e = make_tensor_map_2d(ms, score, C, kGsTile, ratio)) != cudaSuccess)
        return e;
    if (coff != 2) {
        *mk2 = *mk;
        *ms2 = *ms;
        return cudaSuccess;
    }
    if ((e = make_tensor_map_parts(mk2, kv, C, kGsTile, ratio, head_dim)) != cudaSuccess)
        return e;
    return make_tensor_map_parts(ms2, score, C, kGsTile, ratio, head_dim);
}

// Grid width (row blocks per column tile) of a staged launch.
cudaError_t gs_blocks(bool bwd, const GsPlan &pl, int capacity, int *blocks)
{
    const void *fn = gs_kernel(bwd, pl.wmax);
    int resident = 0;
    cudaError_t e = resident_blocks(fn, pl.threads, pl.smem, 1, &resident);
    if (e != cudaSuccess)
        return e;
    int b = (resident > 0 ? resident : 1) / pl.tiles;
    b = b < 1 ? 1 : b;
    const int rows = capacity > 0 ? capacity : 1;
    *blocks = b < rows ? b : rows;
    return cudaSuccess;
}

}  // namespace

bool generic_supported(int ratio, int coff, int head_dim)
{
    return ratio >= 1 && ratio <= 128 && (coff == 1 || coff == 2) && head_dim % 8 == 0 && head_dim <= 8192;
}

cudaError_t plan_generic(int ratio, int coff, int head_dim, int capacity, int num_sms, GenericPlan *out)
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
    pl.staged_blocks = 0;
    pl.staged_lanes = 0;
    if (gs_supported(ratio, coff, head_dim)) {  // one partial per row block of the staged kernel
        const GsPlan g = gs_plan(true, ratio, coff, head_dim);
        pl.staged_lanes = g.lanes;
        cudaError_t e = gs_blocks(true, g, capacity, &pl.staged_blocks);
        if (e != cudaSuccess)
            return e;
        pl.partial_floats = (int64_t)pl.staged_blocks * ratio * coff * head_dim;
    }
    *out = pl;
    return cudaSuccess;
}

cudaError_t launch_fwd_generic(const FwdParams &p, unsigned *status, int num_sms, cudaStream_t st)
{
    GenArgs a{static_cast<const uint16_t *>(p.kv), static_cast<const uint16_t *>(p.score), p.ape, p.cu_seqlens,
              p.cu_seqlens_comp, p.n_seg, p.ratio, p.coff, p.head_dim, p.capacity};
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (gs_supported(p.ratio, p.coff, p.head_dim)) {
        const GsPlan pl = gs_plan(false, p.ratio, p.coff, p.head_dim);
        int blocks = 0;
        cudaError_t e = gs_blocks(false, pl, p.capacity, &blocks);
        if (e != cudaSuccess)
            return e;
        CUtensorMap mk, ms, mk2, ms2;
        if ((e = gs_maps(p.kv, p.score, p.ratio, p.coff, p.head_dim, &mk, &ms, &mk2, &ms2)) != cudaSuccess)
            return e;
        GsArgs ga{a, pl.stages, pl.stage_bytes, status};
        uint16_t *o = static_cast<uint16_t *>(p.out);
        void *args[] = {&ga, &mk, &ms, &mk2, &ms2, &o};
        cfg.gridDim = dim3(blocks, pl.tiles, 1);
        cfg.blockDim = dim3(pl.threads, 1, 1);
        cfg.dynamicSmemBytes = pl.smem;
        return cudaLaunchKernelExC(&cfg, gs_kernel(false, pl.wmax), args);
    }
    const int64_t units = (int64_t)p.capacity * (p.head_dim / 4);
    int64_t grid = (units + kGenFwdThreads - 1) / kGenFwdThreads;
    const int64_t cap = 8 * (int64_t)num_sms;
    grid = grid < cap ? grid : cap;
    grid = grid < 1 ? 1 : grid;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kGenFwdThreads, 1, 1);
    return cudaLaunchKernelEx(&cfg, fwd_generic_kernel, a, static_cast<uint16_t *>(p.out));
}

cudaError_t launch_bwd_generic(const BwdParams &p, const GenericPlan &pl, float *partial, unsigned *status,
                               cudaStream_t st)
{
    GenArgs a{static_cast<const uint16_t *>(p.kv), static_cast<const uint16_t *>(p.score), p.ape, p.cu_seqlens,
              p.cu_seqlens_comp, p.n_seg, p.ratio, p.coff, p.head_dim, p.capacity};
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    int n_partials = pl.groups;
    if (pl.staged_blocks > 0) {
        const GsPlan gp = gs_plan(true, p.ratio, p.coff, p.head_dim);
        CUtensorMap mk, ms, mk2, ms2;
        if ((e = allow_max_smem(gs_kernel(true, gp.wmax))) != cudaSuccess ||
            (e = gs_maps(p.kv, p.score, p.ratio, p.coff, p.head_dim, &mk, &ms, &mk2, &ms2)) != cudaSuccess)
            return e;
        GsArgs ga{a, gp.stages, gp.stage_bytes, status};
        int64_t n_tokens = p.n_tokens;
        const uint16_t *go = static_cast<const uint16_t *>(p.grad_out);
        uint16_t *dk = static_cast<uint16_t *>(p.dkv), *dsc = static_cast<uint16_t *>(p.dscore);
        void *args[] = {&ga, &mk, &ms, &mk2, &ms2, &n_tokens, &go, &dk, &dsc, &partial};
        cfg.gridDim = dim3(pl.staged_blocks, gp.tiles, 1);
        cfg.blockDim = dim3(gp.threads, 1, 1);
        cfg.dynamicSmemBytes = gp.smem;
        e = cudaLaunchKernelExC(&cfg, gs_kernel(true, gp.wmax), args);
        n_partials = pl.staged_blocks;
    } else {
        if (pl.smem > 48 * 1024) {
            e = allow_max_smem(reinterpret_cast<const void *>(bwd_generic_kernel));
            if (e != cudaSuccess)
                return e;
        }
        cfg.gridDim = dim3(pl.groups, pl.col_tiles, 1);
        cfg.blockDim = dim3(kGenBwdGroups, pl.lanes, 1);
        cfg.dynamicSmemBytes = pl.smem;
        e = cudaLaunchKernelEx(&cfg, bwd_generic_kernel, a, pl.rows_per_group, p.n_tokens,
                               static_cast<const uint16_t *>(p.grad_out), static_cast<uint16_t *>(p.dkv),
                               static_cast<uint16_t *>(p.dscore), partial);
    }
    if (e != cudaSuccess)
        return e;
    return launch_dape_finalize(partial, n_partials, (int64_t)p.ratio * p.coff * p.head_dim, p.dape, st);
}

}  // namespace csa
