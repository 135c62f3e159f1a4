// Compressor kernels for every other ratio: 1 <= ratio <= 128, windows of up to
// 256 positions ("CSA Fused Compressor", cuDNN frontend docs, section Semantics;
// the page's generic kernels are generic over the ratio as well).
//
// One thread owns a pair of adjacent columns j, j+1 of one output row and walks
// the window three times (max; exp and sums; gradients), reading each position's
// bf16 pair of score and kv and fp32 pair of APE straight from global memory, eight
// positions' loads in flight at a time: the
// window is too long for registers at large ratios and too short to amortise a
// staged pipeline at small ones.  The repeated reads of a row's window hit L1/L2,
// so DRAM traffic stays the algorithmic bytes.  The arithmetic is the library's
// stated fp32 order, exactly as in the ratio-4 kernels (same exp, same reciprocal,
// ascending window positions), so results are bitwise equal to the fp32 oracle.
//
// Backward: a block owns a column tile of blockDim.x pairs and a contiguous group
// of rows; lane y of the block takes rows y, y + lanes, ... of the group in
// ascending order.  Each thread keeps its grad_ape sums for every window position
// in its own shared-memory slots (no sharing, no atomics); at the end the lanes are
// added in ascending lane order and the block writes the group's partial
// [ratio, coff*head_dim] entries of its columns; dape_finalize_kernel adds the
// groups in ascending order.  Gradient coverage as in
// the other kernels: a real row writes the slots it reads, the last block of a
// segment zeroes its own first-half columns (coff 2) and the tokens up to the next
// real block (or n_tokens), row group 0 zeroes the tokens before the first real block.
#include "csa_device.cuh"
#include "csa_launch.h"

namespace csa {

namespace {

constexpr int kGenFwdThreads = 256;
constexpr int kGenBwdPairs = 32;  // pairs (64 columns) per backward block
constexpr int kGenBwdMaxLanes = 8;
constexpr size_t kGenBwdSmem = 96 * 1024;  // grad_ape slots: lanes x window x pairs x float2
constexpr int64_t kGenPartialFloats = 1 << 20;  // grad_ape partials budget (unless one group exceeds it)

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

// Window position k of a row: validity, token, packed column of the thread's
// first column j, and the APE row (k mod ratio).
struct Slot {
    int64_t tok;
    int col;
    int arow;
};

__device__ __forceinline__ bool gen_valid(const GenArgs &a, const RowMap &rm, int k)
{
    return !(a.coff == 2 && k < a.ratio && rm.first);
}

__device__ __forceinline__ Slot gen_slot(const GenArgs &a, const RowMap &rm, int k, int j)
{
    Slot s;
    if (a.coff == 2 && k < a.ratio) {  // previous block's token, first half
        s.tok = rm.base - a.ratio + k;
        s.col = j;
        s.arow = k;
    } else if (a.coff == 2) {          // own block's token, second half
        s.tok = rm.base + (k - a.ratio);
        s.col = a.head_dim + j;
        s.arow = k - a.ratio;
    } else {
        s.tok = rm.base + k;
        s.col = j;
        s.arow = k;
    }
    return s;
}

// A batch of kGB consecutive window positions k0 .. k0 + kGB - 1, loaded before
// any of them is used so that the loads are in flight together; the arithmetic
// then takes them in ascending order.
constexpr int kGB = 8;

struct GenBatch {
    uint32_t sw[kGB];  // score pair
    uint32_t kw[kGB];  // kv pair (when loaded)
    float2 ap[kGB];    // APE pair
    unsigned valid;    // bit u: position k0 + u exists and is valid
};

template <bool KV>
__device__ __forceinline__ void gen_fetch(const GenArgs &a, const RowMap &rm, int k0, int W, int j, int64_t C,
                                          GenBatch &b)
{
    b.valid = 0u;
#pragma unroll
    for (int u = 0; u < kGB; ++u) {
        const int k = k0 + u;
        if (k < W && gen_valid(a, rm, k)) {
            b.valid |= 1u << u;
            const Slot sl = gen_slot(a, rm, k, j);
            b.sw[u] = __ldg(reinterpret_cast<const unsigned int *>(a.score + sl.tok * C + sl.col));
            b.ap[u] = __ldg(reinterpret_cast<const float2 *>(a.ape + (int64_t)sl.arow * C + sl.col));
            if (KV)
                b.kw[u] = __ldg(reinterpret_cast<const unsigned int *>(a.kv + sl.tok * C + sl.col));
        }
    }
}

// Passes 1 and 2 of one row: m (NaN-propagating max), den and num.
__device__ __forceinline__ void gen_pool(const GenArgs &a, const RowMap &rm, int j, int64_t C, float2 &m,
                                         float2 &den, float2 &num)
{
    const int W = a.coff * a.ratio;
    m = make_float2(-INFINITY, -INFINITY);
    for (int k0 = 0; k0 < W; k0 += kGB) {
        GenBatch b;
        gen_fetch<false>(a, rm, k0, W, j, C, b);
#pragma unroll
        for (int u = 0; u < kGB; ++u) {
            if (!(b.valid >> u & 1u))
                continue;
            const float2 s = add2(bf16x2_to_f2(b.sw[u]), b.ap[u]);
            m.x = max_nan(m.x, s.x);
            m.y = max_nan(m.y, s.y);
        }
    }
    const float2 negm = make_float2(-m.x, -m.y);
    den = make_float2(0.0f, 0.0f);
    num = make_float2(0.0f, 0.0f);
    for (int k0 = 0; k0 < W; k0 += kGB) {
        GenBatch b;
        gen_fetch<true>(a, rm, k0, W, j, C, b);
#pragma unroll
        for (int u = 0; u < kGB; ++u) {
            if (!(b.valid >> u & 1u))
                continue;
            const float2 e = exp2lanes(add2(add2(bf16x2_to_f2(b.sw[u]), b.ap[u]), negm));
            den = add2(den, e);
            num = fma2(e, bf16x2_to_f2(b.kw[u]), num);
        }
    }
}

__global__ void __launch_bounds__(kGenFwdThreads) fwd_generic_kernel(GenArgs a, uint16_t *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int pairs = a.head_dim / 2;
    const int64_t units = (int64_t)a.capacity * pairs;
    const int64_t C = (int64_t)a.coff * a.head_dim;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(u / pairs);
        const int j = 2 * (int)(u - (int64_t)r * pairs);
        // padding rows (and rows below cu_seqlens_comp[0]) come back as a first
        // block starting at token 0
        const RowMap rm = map_row(r, a.cu, a.cc, a.n_seg, a.ratio);
        float2 m, den, num;
        gen_pool(a, rm, j, C, m, den, num);
        const float2 inv = make_float2(recip_den(den.x), recip_den(den.y));
        *reinterpret_cast<uint32_t *>(out + (int64_t)r * a.head_dim + j) = f2_to_bf16x2(mul2(num, inv));
    }
}

// Zero the gradient slots of tokens [t0, t1) in the thread's columns (first half
// only, or every half).
__device__ __forceinline__ void gen_zero(const GenArgs &a, uint16_t *dkv, uint16_t *dscore, int64_t C, int j,
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

__global__ void __launch_bounds__(kGenBwdPairs * kGenBwdMaxLanes, 2)
    bwd_generic_kernel(GenArgs a, int rows_per_group, int64_t n_tokens_arg, const uint16_t *__restrict__ grad_out,
                       uint16_t *__restrict__ dkv, uint16_t *__restrict__ dscore, float *__restrict__ partial)
{
    extern __shared__ float2 acc[];  // [lane][window position][pair]: each thread's own slots
    pdl_wait();
    pdl_trigger();  // the grad_ape finalisation may launch; it waits for this grid's end
    const int W = a.coff * a.ratio;
    const int TP = blockDim.x, lanes = blockDim.y, y = threadIdx.y;
    const int pairs = a.head_dim / 2;
    const int p = blockIdx.y * TP + threadIdx.x;
    const bool col_ok = p < pairs;
    const int j = 2 * p;
    const int64_t C = (int64_t)a.coff * a.head_dim;
    const int64_t n_tokens = n_tokens_arg >= 0 ? n_tokens_arg : (int64_t)__ldg(a.cu + a.n_seg);
    const int R = a.n_seg > 0 ? __ldg(a.cc + a.n_seg) : 0;
    const int R0 = a.n_seg > 0 ? __ldg(a.cc) : 0;
    float2 *mine = acc + (size_t)y * W * TP + threadIdx.x;  // slot k at mine[k * TP]
    for (int k = 0; k < W; ++k)
        mine[k * TP] = make_float2(0.0f, 0.0f);

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
        float2 m, den, num;
        gen_pool(a, rm, j, C, m, den, num);
        const float2 g = bf16x2_to_f2(__ldg(reinterpret_cast<const unsigned int *>(grad_out +
                                                                                   (int64_t)r * a.head_dim + j)));
        const float2 inv = make_float2(recip_den(den.x), recip_den(den.y));
        const float2 go = mul2(g, mul2(num, inv));
        const float2 ngo = make_float2(-go.x, -go.y), negm = make_float2(-m.x, -m.y);
        for (int k0 = 0; k0 < W; k0 += kGB) {
            GenBatch b;
            gen_fetch<true>(a, rm, k0, W, j, C, b);
#pragma unroll
            for (int u = 0; u < kGB; ++u) {
                if (!(b.valid >> u & 1u))
                    continue;
                const Slot sl = gen_slot(a, rm, k0 + u, j);
                const float2 e = exp2lanes(add2(add2(bf16x2_to_f2(b.sw[u]), b.ap[u]), negm));
                const float2 pk = mul2(e, inv);
                const float2 ds = mul2(pk, add2(mul2(g, bf16x2_to_f2(b.kw[u])), ngo));
                float2 &ak = mine[(k0 + u) * TP];
                ak = add2(ak, ds);
                if (sl.tok < n_tokens) {
                    *reinterpret_cast<uint32_t *>(dkv + sl.tok * C + sl.col) = f2_to_bf16x2(mul2(g, pk));
                    *reinterpret_cast<uint32_t *>(dscore + sl.tok * C + sl.col) = f2_to_bf16x2(ds);
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
    // then this group's partial: [ape row][packed column], the thread's two columns
    float *dst = partial + (int64_t)blockIdx.x * a.ratio * C;
    for (int k = y; col_ok && k < W; k += lanes) {
        float2 s = acc[(size_t)k * TP + threadIdx.x];
        for (int l = 1; l < lanes; ++l)
            s = add2(s, acc[((size_t)l * W + k) * TP + threadIdx.x]);
        const int arow = k % a.ratio, half = k / a.ratio;
        *reinterpret_cast<float2 *>(dst + (int64_t)arow * C + half * a.head_dim + j) = s;
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
    const int pairs = head_dim / 2;
    pl.col_tiles = (pairs + kGenBwdPairs - 1) / kGenBwdPairs;
    const size_t lane_bytes = (size_t)coff * ratio * kGenBwdPairs * sizeof(float2);
    int lanes = (int)(kGenBwdSmem / lane_bytes);
    pl.lanes = lanes < 1 ? 1 : lanes > kGenBwdMaxLanes ? kGenBwdMaxLanes : lanes;
    const int rows = capacity > 0 ? capacity : 1;
    int groups = 8 * num_sms / pl.col_tiles;  // blocks of up to 8 warps: ~2 per SM
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
    const int64_t units = (int64_t)p.capacity * (p.head_dim / 2);
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
    cfg.blockDim = dim3(kGenBwdPairs, pl.lanes, 1);
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
