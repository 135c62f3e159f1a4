// Chunked Compressor kernels for windows of more than 64 positions ("CSA Fused
// Compressor", cuDNN frontend docs, sections Semantics and "ratio=128"): ratio 128
// (window 128 with coff 1, 256 with coff 2), and every other ratio whose window
// exceeds 64 positions (33-127 with coff 2, 65-127 with coff 1), head_dim a
// multiple of 64.  A window this long is split into chunks of 8 window positions
// held by different threads and merged in a fixed order.
//
// Per thread block: a column tile of TC = 64 / coff columns, persistent over the
// rows b, b + gridDim.x, ...  One producer warp streams, per row, the window's
// [ratio tokens x TC columns] boxes of kv and score (one box per array and part)
// with 2-D TMA tensor copies into a shared-memory ring tracked by mbarriers (and,
// in the backward, the grad_out row with a bulk copy).  NC chunks (12 to 32,
// covering the window): a thread owns a group g of 4 columns and
// a chunk c, whose window positions are k = c, c + NC, c + 2*NC, ... (8 of them;
// those at or past the window's end are skipped), so that the lanes of a warp
// read consecutive box rows (no bank conflicts) and each thread's APE values stay
// in registers.  Ratio 128 is compiled with the ratio as a constant; the other
// ratios take it at run time, with the fewest chunks (a multiple of the warps'
// chunk count) that cover the window.
//
// Order of the arithmetic (the page's ratio-128 family: a deterministic chunked
// order, checked against the plain sequential oracle by tolerance; the library
// applies the same contract to every window of more than 64 positions):
//   s_k = score + ape;  m = max over all valid k (exact: chunk maxima, then over
//   the warp's chunks by shuffles, then over the consumer warps; with coff 1 each
//   warp first uses its own maximum m_w and the merge below rescales its sums by
//   2^((m_w - m) log2 e));
//   e_k = 2^(s_k*log2(e) - m*log2(e)) on the multi-function unit (ex2.approx, as
//   the page's ratio-128 kernels do: ~2^-22 relative error, far below the final
//   bf16 rounding);
//   den_c = ((+0 + e_c) + e_c+NC) + ... within chunk c, num_c = fma chain;
//   chunk sums added over the warp's chunks by a fixed xor-shuffle tree, warp sums
//   added in ascending warp order by the threads of a column and then by a fixed
//   xor-shuffle tree over those threads;  inv = 1/den rounded;  o = num * inv;
//   out = bf16(o).
// Backward per valid k: p = e_k * inv;  grad_kv = bf16(g*p);
//   ds = p*fma(g, kv, -g*o);  grad_score = bf16(ds); grad_ape as in the other kernels
//   (per-thread sums over its rows, cluster merge in rank order, fixed-order
//   finalisation).  Bitwise run-to-run deterministic: fixed chunks, fixed orders.
//
// Every barrier wait on the ring is bounded in time (timeouts are recorded in
// the status word, the kernel then stops and exits normally).
#include <cooperative_groups.h>
#include <cuda.h>

#include <mutex>

#include "csa_device.cuh"
#include "csa_launch.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

constexpr int kKC = 8;  // window positions per chunk (per thread)

// Backward layout per window form and chunk count.  Register-resident: APE and
// the kv words in registers, the stage released as soon as it is read, one block
// per SM (registers), a four-stage ring.  "Lean": APE from a shared tile, kv read
// again from the stage, which stays held until the row's gradients are written,
// so that two blocks fit per SM.  coff 2 (twice the column tiles per row) runs
// lean; coff 1 runs lean up to 12 chunks, whose register-resident block has only
// seven warps on its SM (ratio 96 at 8 x 6144 tokens, head_dim 512: 55.6 -> 46.7
// us), and register-resident at 16 (ratio 128: 98.4 against 121 us lean).
template <int COFF, int NCB>
constexpr bool kBwdLean = COFF == 2 || NCB <= 12;

// The lean layouts' kv words: loaded into registers with the scores, so that the
// stage is released as soon as it is read (coff 2 up to 28 chunks: ratio 40 / 64
// / 80 / 96 / 112 backward 72.1 / 63.8 / 64.1 / 68.4 / 66.2 -> 70.2 / 60.9 / 62.0 /
// 66.2 / 63.9 us at 8 x 4096 tokens, head_dim 512), or read from the stage again
// where needed, the stage held until the row's gradients are written (coff 2 at
// 32 chunks, whose registers would spill: ratio 128 213 against 270 us; coff 1 at
// 12 chunks: ratio 96 45.1 against 48.3 us).
template <int COFF, int NCB>
constexpr bool kBwdHold = kBwdLean<COFF, NCB> && (COFF == 1 || NCB == 32);

// Block geometry for a form and a chunk count (the window's bucket).
template <int COFF, int NCB>
struct Geo {
    static constexpr int TC = 64 / COFF;      // columns per block tile
    static constexpr int G = TC / 4;          // column groups (4 columns each)
    static constexpr int CPW = 32 / G;        // chunks per warp
    static constexpr int NC = NCB;            // chunks
    static constexpr int WMAX = kKC * NC;     // longest window of the bucket
    static constexpr int CW = NC / CPW;       // consumer warps
    static constexpr int CT = CW * 32;        // consumer threads
    static constexpr int THREADS = CT + 32;   // + one producer warp
    static constexpr int RS = TC + 4;         // row stride of the merge buffers
    // The final merge: TPC consecutive threads per tile column (a power of two, so
    // that a fixed xor tree joins them within a warp), each adding WPT warp sums;
    // the threads past MT = TPC * TC take no part in it.
    static constexpr int TPC = (CW % 8 == 0 && 8 * TC <= CT) ? 8 : (CW % 4 == 0 && 4 * TC <= CT) ? 4
                             : (CW % 2 == 0 && 2 * TC <= CT) ? 2 : 1;
    static constexpr int WPT = CW / TPC;
    static constexpr int MT = TPC * TC;
    // resident blocks per SM the registers are sized for: three of the blocks with
    // at most four consumer warps (ratio 64 with coff 2: forward 32.1 -> 29.7 us,
    // backward 66.5 -> 64.8 us at 8 x 4096 tokens, head_dim 512), else two
    static constexpr int MIN_BLOCKS = CW <= 4 ? 3 : 2;
    // coff 1: each warp's terms are taken relative to the warp's own maximum and
    // the merge rescales them to the row's (one block barrier fewer per row;
    // ratio 128 backward 100.6 -> 97.4 us, ratio 96 forward / backward 26.4 / 63.2
    // -> 24.4 / 60.5 us); coff 2 keeps the row maximum first (faster there:
    // ratio-128 backward 222 against 230 us)
    static constexpr bool LOCAL = COFF == 1;
    static_assert(CW * CPW == NC, "chunks per warp");
};

struct ChArgs {
    const uint16_t *kv;
    const uint16_t *score;
    const float *ape;
    const int32_t *cu;
    const int32_t *cc;
    int n_seg;
    int head_dim;
    int capacity;
    int ratio;
    int box_bytes;  // stride of the [ratio x TC] bf16 boxes in a stage (128-byte multiple)
    int stages;
    int stage_bytes;
    unsigned *status;
};

// The window of a row: the ratio (a constant RC, or taken at run time when RC is
// 0) and, for window position k = c + NC*i of chunk c, its part (0: the previous
// block's tokens on the first-half columns, coff 2 only; else the own block) and
// its token within the part.
template <int COFF, int NCB, int RC>
struct Win {
    int r;
    int bb;  // box bytes
    __device__ __forceinline__ Win(const ChArgs &a) : r(RC > 0 ? RC : a.ratio), bb(a.box_bytes) {}
    __device__ __forceinline__ int ratio() const { return RC > 0 ? RC : r; }
    // bytes of one box's data, and the stride between boxes in a stage (rounded up
    // to 128 bytes: TMA tensor copies write 128-byte aligned shared memory)
    __device__ __forceinline__ int box_data() const { return ratio() * Geo<COFF, NCB>::TC * 2; }
    __device__ __forceinline__ int box_bytes() const { return RC > 0 ? (RC * Geo<COFF, NCB>::TC * 2 + 127) / 128 * 128 : bb; }
    __device__ __forceinline__ int win_bytes() const { return 2 * COFF * box_bytes(); }
    // false for a position past the end of the window (the bucket may be longer)
    __device__ __forceinline__ bool pos(int c, int i, int &part, int &tok) const
    {
        const int k = c + NCB * i, rr = ratio();
        if (COFF == 1) {
            part = 0;
            tok = k;
        } else {
            part = k >= rr ? 1 : 0;
            tok = k - part * rr;
        }
        if (RC > 0 && COFF * RC == kKC * NCB)
            return true;  // the window fills the bucket
        return k < COFF * rr;
    }
    // a position the row reads: inside the window, and not a first block's
    // previous-block position (coff 2)
    __device__ __forceinline__ bool valid(int c, int i, bool first) const
    {
        int part, tok;
        return pos(c, i, part, tok) && !(COFF == 2 && part == 0 && first);
    }
    // box of array arr (0 kv, 1 score) and part p in a stage
    __device__ __forceinline__ int box_offset(int arr, int part) const { return (arr * COFF + part) * box_bytes(); }
};

struct Meta {
    int64_t base;
    int seg;
    int row;
    int real;
    int first;
    int last;  // the last block of its segment
    int pad;
};

template <int COFF, int NCB>
struct ChSmem {
    unsigned char *stages;
    float *mx;   // [2][CW][RS]  warp maxima
    float *den;  // [2][CW][RS]  warp sums
    float *num;  // [2][CW][RS]
    float *fin;  // [2][2 + CW][TC]  (inv, o, each warp's scale) for the backward
    float *apet; // [WMAX][TC]  the backward's APE tile (null in the forward)
    Meta *meta;
    uint64_t *full;
    uint64_t *empty;
};

template <int COFF, int NCB>
__host__ __device__ size_t ch_smem_bytes(int stages, int stage_bytes, bool ape_tile)
{
    using G = Geo<COFF, NCB>;
    return (size_t)stages * stage_bytes + 3 * 2 * G::CW * G::RS * 4 + 2 * (2 + G::CW) * G::TC * 4 +
           (ape_tile ? (size_t)G::WMAX * G::TC * 4 : 0) + sizeof(Meta) * stages + 16 * stages + 16;
}

template <int COFF, int NCB>
__device__ __forceinline__ ChSmem<COFF, NCB> ch_carve(unsigned char *base, int stages, int stage_bytes, bool ape_tile)
{
    using G = Geo<COFF, NCB>;
    ChSmem<COFF, NCB> s;
    s.stages = base;
    unsigned char *p = base + (size_t)stages * stage_bytes;
    s.mx = reinterpret_cast<float *>(p);
    s.den = s.mx + 2 * G::CW * G::RS;
    s.num = s.den + 2 * G::CW * G::RS;
    s.fin = s.num + 2 * G::CW * G::RS;
    s.apet = ape_tile ? s.fin + 2 * (2 + G::CW) * G::TC : nullptr;
    p = reinterpret_cast<unsigned char *>(s.fin + 2 * (2 + G::CW) * G::TC + (ape_tile ? G::WMAX * G::TC : 0));
    s.meta = reinterpret_cast<Meta *>(p);
    s.full = reinterpret_cast<uint64_t *>(s.meta + stages);
    s.empty = s.full + stages;
    return s;
}

// ----------------------------------------------------------------- producer

template <int COFF, int NCB, int RC, bool BWD>
__device__ void ch_produce(const ChArgs &a, const ChSmem<COFF, NCB> &s, const CUtensorMap *tm_kv,
                           const CUtensorMap *tm_sc, int c0, int row0, int rstride, int rend,
                           const uint16_t *__restrict__ grad_out)
{
    using G = Geo<COFF, NCB>;
    const Win<COFF, NCB, RC> w(a);
    const int R = w.ratio();
    int issued = 0, st = 0;
    uint32_t ph = 0;
    RowCursor cur;
    cursor_init(cur, a.cc, a.n_seg);
    for (int row = row0; row < rend; row += rstride) {
        // the row's map first: its loads (if any) overlap the wait for a free slot
        const RowMap rm = cursor_map(cur, row, a.cu, a.cc, a.n_seg, R);
        if (!mbar_wait(smem_addr(&s.empty[st]), ph ^ 1u, a.status))
            break;
        Meta &m = s.meta[st];
        m.base = rm.base;
        m.seg = rm.seg;
        m.row = row;
        m.real = rm.real;
        m.first = rm.first;
        m.last = rm.real && row + 1 == cur.hi;
        const bool load = BWD ? rm.real : true;
        const int p0 = (COFF == 2 && rm.first) ? 1 : 0;
        const uint32_t bytes =
            load ? (uint32_t)((COFF - p0) * 2 * w.box_data()) + (BWD ? (uint32_t)G::TC * 2u : 0u) : 0u;
        const uint32_t fb = smem_addr(&s.full[st]);
        mbar_arrive_expect_tx(fb, bytes);
        if (load) {
            const uint32_t dst = smem_addr(s.stages + (size_t)st * a.stage_bytes);
            for (int p = p0; p < COFF; ++p) {
                const int y = (int)(rm.base + (int64_t)(p - (COFF - 1)) * R);
                const int x = p * a.head_dim + c0;
                tma_load_2d(dst + w.box_offset(0, p), tm_kv, x, y, fb);
                tma_load_2d(dst + w.box_offset(1, p), tm_sc, x, y, fb);
            }
            if (BWD)
                bulk_g2s(dst + w.win_bytes(), grad_out + (int64_t)row * a.head_dim + c0, G::TC * 2, fb);
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

// ----------------------------------------------------------------- consumer

struct ChunkState {
    uint2 kv[kKC];
    float2 e[kKC][2];  // s_k, then e_k
};

// The thread's APE values, [position i][column pair] (positions past the window
// are not read).
template <int COFF, int NCB, int RC>
__device__ __forceinline__ void ch_load_ape(const ChArgs &a, const Win<COFF, NCB, RC> &w, int c, int col,
                                            float2 (&ap)[kKC][2])
{
    const int64_t C = (int64_t)COFF * a.head_dim;
#pragma unroll
    for (int i = 0; i < kKC; ++i) {
        int part, tok;
        if (!w.pos(c, i, part, tok)) {
            ap[i][0] = ap[i][1] = make_float2(0.0f, 0.0f);
            continue;
        }
        const float4 v =
            __ldg(reinterpret_cast<const float4 *>(a.ape + tok * C + (int64_t)part * a.head_dim + col));
        ap[i][0] = make_float2(v.x, v.y);
        ap[i][1] = make_float2(v.z, v.w);
    }
}

// Reads the thread's positions of one row from the stage and forms s = score + ape.
template <int COFF, int NCB, int RC>
__device__ __forceinline__ void ch_load(const Win<COFF, NCB, RC> &w, const unsigned char *stage, int c, int g,
                                        bool first, const float2 (&ap)[kKC][2], ChunkState &cs)
{
#pragma unroll
    for (int i = 0; i < kKC; ++i) {
        int part, tok;
        if (!w.pos(c, i, part, tok) || (COFF == 2 && part == 0 && first))
            continue;
        const int off = tok * Geo<COFF, NCB>::TC * 2 + 8 * g;
        cs.kv[i] = *reinterpret_cast<const uint2 *>(stage + w.box_offset(0, part) + off);
        const uint2 sw = *reinterpret_cast<const uint2 *>(stage + w.box_offset(1, part) + off);
        cs.e[i][0] = add2_bf16x2(sw.x, ap[i][0]);
        cs.e[i][1] = add2_bf16x2(sw.y, ap[i][1]);
    }
}

constexpr float kLog2eF = 1.4426950408889634f;

// 2^x on the multi-function unit (flushes results below 2^-126 to zero).
__device__ __forceinline__ float ex2_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Backward: s = score + ape for the thread's positions, APE from the block's tile;
// KV: the kv words too (else kv is read from the stage again where it is needed).
template <int COFF, int NCB, int RC, bool KV>
__device__ __forceinline__ void ch_load_s(const Win<COFF, NCB, RC> &w, const unsigned char *stage,
                                          const float *apet, int c, int g, bool first, ChunkState &cs)
{
#pragma unroll
    for (int i = 0; i < kKC; ++i) {
        int part, tok;
        if (!w.pos(c, i, part, tok) || (COFF == 2 && part == 0 && first))
            continue;
        const int off = tok * Geo<COFF, NCB>::TC * 2 + 8 * g;
        if constexpr (KV)
            cs.kv[i] = *reinterpret_cast<const uint2 *>(stage + w.box_offset(0, part) + off);
        const uint2 sw = *reinterpret_cast<const uint2 *>(stage + w.box_offset(1, part) + off);
        const float4 av = *reinterpret_cast<const float4 *>(apet + (size_t)(c + NCB * i) * Geo<COFF, NCB>::TC + 4 * g);
        // unpacked and added as a pair: here measured faster than the mixed-precision
        // add of ch_load (272 against 281 us for the ratio-128 coff-2 backward; same bits)
        cs.e[i][0] = add2(bf16x2_to_f2(sw.x), make_float2(av.x, av.y));
        cs.e[i][1] = add2(bf16x2_to_f2(sw.y), make_float2(av.z, av.w));
    }
}

// kv words of window position i of the thread: from the registers the forward
// filled, or (KV_STAGE, the backward) from the stage.
template <int COFF, int NCB, int RC, bool KV_STAGE>
__device__ __forceinline__ uint2 ch_kv(const Win<COFF, NCB, RC> &w, const ChunkState &cs, const unsigned char *stage,
                                       int c, int g, int i)
{
    if constexpr (KV_STAGE) {
        int part, tok;
        w.pos(c, i, part, tok);
        return *reinterpret_cast<const uint2 *>(stage + w.box_offset(0, part) + tok * Geo<COFF, NCB>::TC * 2 + 8 * g);
    } else {
        return cs.kv[i];
    }
}

// The two merge phases of one row.  Every consumer thread calls this once per
// row.  The first barrier also votes on `ok` (the thread's wait for the row's
// data succeeded): if any thread failed, all return false together before the
// second barrier.  `have`: the row has data (cs loaded).  On true: cs.e holds e_k
// of the thread's valid positions, and each warp's sums over its chunks are in
// the merge buffers for ch_final.
template <int COFF, int NCB, int RC, bool KV_STAGE>
__device__ __forceinline__ bool ch_pool(const Win<COFF, NCB, RC> &w, const ChSmem<COFF, NCB> &s, int buf, int c,
                                        int g, bool ok, bool have, bool first, ChunkState &cs,
                                        const unsigned char *stage)
{
    using G = Geo<COFF, NCB>;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (have) {
#pragma unroll
        for (int i = 0; i < kKC; ++i) {
            if (!w.valid(c, i, first))
                continue;
            m[0] = max_nan(m[0], cs.e[i][0].x);
            m[1] = max_nan(m[1], cs.e[i][0].y);
            m[2] = max_nan(m[2], cs.e[i][1].x);
            m[3] = max_nan(m[3], cs.e[i][1].y);
        }
    }
    // over the warp's chunks: lanes g, g + G, g + 2G, ... hold the same columns
#pragma unroll
    for (int d = G::G; d < 32; d *= 2)
#pragma unroll
        for (int q = 0; q < 4; ++q)
            m[q] = max_nan(m[q], __shfl_xor_sync(0xffffffffu, m[q], d));
    float *mx = s.mx + (size_t)buf * G::CW * G::RS;
    float4 M;
    if constexpr (G::LOCAL) {
        // the warp's maximum is its terms' reference (0 where it is -inf: those
        // terms all vanish); ch_final rescales the warp sums to the row's maximum
        M = make_float4(m[0] == -INFINITY ? 0.0f : m[0], m[1] == -INFINITY ? 0.0f : m[1],
                        m[2] == -INFINITY ? 0.0f : m[2], m[3] == -INFINITY ? 0.0f : m[3]);
    } else {
        if (lane < G::G)
            *reinterpret_cast<float4 *>(mx + warp * G::RS + 4 * g) = make_float4(m[0], m[1], m[2], m[3]);
        if (!named_barrier_and(1, G::CT, ok))
            return false;
        M = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
        for (int v = 0; v < G::CW; ++v) {
            const float4 x = *reinterpret_cast<const float4 *>(mx + v * G::RS + 4 * g);
            M.x = max_nan(M.x, x.x);
            M.y = max_nan(M.y, x.y);
            M.z = max_nan(M.z, x.z);
            M.w = max_nan(M.w, x.w);
        }
    }
    float2 den[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
    float2 num[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
    // exponent s*log2(e) - m*log2(e): one fma per element
    const float2 nml[2] = {make_float2(-__fmul_rn(M.x, kLog2eF), -__fmul_rn(M.y, kLog2eF)),
                           make_float2(-__fmul_rn(M.z, kLog2eF), -__fmul_rn(M.w, kLog2eF))};
#pragma unroll
    for (int i = 0; i < kKC; ++i) {
        if (!have || !w.valid(c, i, first))
            continue;
        const uint2 kv = ch_kv<COFF, NCB, RC, KV_STAGE>(w, cs, stage, c, g, i);
        const uint32_t kw[2] = {kv.x, kv.y};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float2 x = fma2(cs.e[i][q], splat(kLog2eF), nml[q]);
            const float2 ek = make_float2(ex2_fast(x.x), ex2_fast(x.y));
            cs.e[i][q] = ek;
            den[q] = add2(den[q], ek);
            num[q] = fma2(ek, bf16x2_to_f2(kw[q]), num[q]);
        }
    }
    // over the warp's chunks, a fixed xor tree (both partners add the same two
    // values: the sums agree bitwise)
#pragma unroll
    for (int d = G::G; d < 32; d *= 2)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            den[q] = add2(den[q], make_float2(__shfl_xor_sync(0xffffffffu, den[q].x, d),
                                              __shfl_xor_sync(0xffffffffu, den[q].y, d)));
            num[q] = add2(num[q], make_float2(__shfl_xor_sync(0xffffffffu, num[q].x, d),
                                              __shfl_xor_sync(0xffffffffu, num[q].y, d)));
        }
    if (lane < G::G) {
        float *dn = s.den + (size_t)buf * G::CW * G::RS;
        float *nm = s.num + (size_t)buf * G::CW * G::RS;
        if constexpr (G::LOCAL)
            *reinterpret_cast<float4 *>(mx + warp * G::RS + 4 * g) = make_float4(m[0], m[1], m[2], m[3]);
        *reinterpret_cast<float4 *>(dn + warp * G::RS + 4 * g) = make_float4(den[0].x, den[0].y, den[1].x, den[1].y);
        *reinterpret_cast<float4 *>(nm + warp * G::RS + 4 * g) = make_float4(num[0].x, num[0].y, num[1].x, num[1].y);
    }
    if constexpr (G::LOCAL)
        return named_barrier_and(1, G::CT, ok);
    named_barrier(1, G::CT);
    return true;
}

// The fixed-order merge of the warp sums, spread over the first MT consumer threads:
// TPC consecutive threads own tile column j; each adds its WPT warps' sums in
// ascending order, then the TPC partial sums meet in a fixed xor-shuffle tree, so
// every one of them ends with the same den and num of column j.  Only threads
// below MT may call it.
template <int COFF, int NCB>
__device__ __forceinline__ void ch_final(const ChSmem<COFF, NCB> &s, int buf, int &j, float &den, float &num,
                                         float *scale)
{
    using G = Geo<COFF, NCB>;
    constexpr int TPC = G::TPC;  // threads per column
    constexpr int WPT = G::WPT;  // warp sums per thread
    static_assert(WPT * TPC == G::CW && G::MT <= G::CT && 32 % TPC == 0, "merge split");
    j = (int)threadIdx.x / TPC;
    const int q = (int)threadIdx.x % TPC;
    const float *dn = s.den + (size_t)buf * G::CW * G::RS + q * WPT * G::RS + j;
    const float *nm = s.num + (size_t)buf * G::CW * G::RS + q * WPT * G::RS + j;
    if constexpr (G::LOCAL) {
        // the row's maximum over the warps' maxima; each warp's sums rescaled by
        // 2^((m_w - M) log2 e) (0 for a warp whose terms all vanished), added in
        // ascending warp order, then the fixed xor tree
        const float *mx = s.mx + (size_t)buf * G::CW * G::RS + q * WPT * G::RS + j;
        float M = mx[0];
#pragma unroll
        for (int v = 1; v < WPT; ++v)
            M = max_nan(M, mx[v * G::RS]);
#pragma unroll
        for (int d = 1; d < TPC; d *= 2)
            M = max_nan(M, __shfl_xor_sync(0xffffffffu, M, d));
        const float nml = -__fmul_rn(M, kLog2eF);
        den = 0.0f;
        num = 0.0f;
#pragma unroll
        for (int v = 0; v < WPT; ++v) {
            const float mw = mx[v * G::RS];
            const float sc = mw == -INFINITY ? 0.0f : ex2_fast(__fmaf_rn(mw, kLog2eF, nml));
            den = __fmaf_rn(dn[v * G::RS], sc, den);
            num = __fmaf_rn(nm[v * G::RS], sc, num);
            if (scale)
                scale[(q * WPT + v) * G::TC + j] = sc;
        }
    } else {
        den = dn[0];
        num = nm[0];
#pragma unroll
        for (int v = 1; v < WPT; ++v) {
            den = __fadd_rn(den, dn[v * G::RS]);
            num = __fadd_rn(num, nm[v * G::RS]);
        }
    }
#pragma unroll
    for (int d = 1; d < TPC; d *= 2) {
        den = __fadd_rn(den, __shfl_xor_sync(0xffffffffu, den, d));
        num = __fadd_rn(num, __shfl_xor_sync(0xffffffffu, num, d));
    }
}

// The dynamic shared memory's base aligned to 1 KB (TMA tensor destinations need
// 128 bytes; the plans reserve 1 KB of slack).  OFFSET: as an offset added to the
// shared array, so the compiler keeps shared-memory addressing for every pointer
// derived from it -- faster in the forwards and the lean backward.  Otherwise
// through an integer round trip, which the register-resident coff-1 backward
// measured faster with (it then fits its registers without a spill).
template <bool OFFSET>
__device__ __forceinline__ unsigned char *align_1k(unsigned char *raw)
{
    if constexpr (OFFSET)
        return raw + ((1024u - (smem_addr(raw) & 1023u)) & 1023u);
    else
        return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

template <int COFF, int NCB>
__device__ __forceinline__ void ch_init(const ChSmem<COFF, NCB> &s, int stages)
{
    using G = Geo<COFF, NCB>;
    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(smem_addr(&s.full[i]), 1);
            mbar_init(smem_addr(&s.empty[i]), G::CW);
        }
        mbar_init_fence();
    }
    __syncthreads();
}

// ------------------------------------------------------------------ forward

template <int COFF, int NCB, int RC>
__global__ void __launch_bounds__(Geo<COFF, NCB>::THREADS, Geo<COFF, NCB>::MIN_BLOCKS)
    fwd_chunk_kernel(ChArgs a, const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_sc,
                     uint16_t *__restrict__ out)
{
    using G = Geo<COFF, NCB>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem_base = align_1k<true>(smem_raw);
    const ChSmem<COFF, NCB> s = ch_carve<COFF, NCB>(smem_base, a.stages, a.stage_bytes, false);
    const Win<COFF, NCB, RC> w(a);
    const int c0 = blockIdx.y * G::TC;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    ch_init<COFF, NCB>(s, a.stages);
    pdl_wait();
    pdl_trigger();
    if (warp == G::CW) {
        if (lane == 0)
            ch_produce<COFF, NCB, RC, false>(a, s, &tm_kv, &tm_sc, c0, blockIdx.x, gridDim.x, a.capacity, nullptr);
        return;
    }
    const int g = lane % G::G, c = G::CPW * warp + lane / G::G;
    float2 ap[kKC][2];
    ch_load_ape<COFF, NCB, RC>(a, w, c, c0 + 4 * g, ap);
    int st = 0, buf = 0;
    uint32_t ph = 0;
    for (int row = blockIdx.x; row < a.capacity; row += gridDim.x) {
        const bool ok = mbar_wait(smem_addr(&s.full[st]), ph, a.status);
        const bool first = ok ? (bool)s.meta[st].first : true;
        ChunkState cs;
        if (ok)
            ch_load<COFF, NCB, RC>(w, s.stages + (size_t)st * a.stage_bytes, c, g, first, ap, cs);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&s.empty[st]));
        if (++st == a.stages) {
            st = 0;
            ph ^= 1u;
        }
        if (!ch_pool<COFF, NCB, RC, false>(w, s, buf, c, g, ok, ok, first, cs, nullptr))
            break;
        {
            int j;
            float den, num;
            if (threadIdx.x < G::MT) {
                ch_final<COFF, NCB>(s, buf, j, den, num, nullptr);
                if (threadIdx.x % G::TPC == 0) {
                    const __nv_bfloat16 h = __float2bfloat16_rn(__fmul_rn(num, recip_den(den)));
                    out[(int64_t)row * a.head_dim + c0 + j] = *reinterpret_cast<const uint16_t *>(&h);
                }
            }
        }
        buf ^= 1;
    }
}

// ----------------------------------------------------------------- backward

// Zero tokens [t0, t1) in the thread's 4 columns (first half only, or all halves);
// the chunks share the tokens: thread chunk c takes t0 + c, t0 + c + NC, ...
template <int COFF, int NCB>
__device__ __forceinline__ void ch_zero_tokens(uint16_t *dkv, uint16_t *dscore, int64_t C, int head_dim, int col,
                                               int64_t t0, int64_t t1, int64_t n_tokens, int c, bool all_halves)
{
    t1 = t1 < n_tokens ? t1 : n_tokens;
    for (int64_t t = (t0 < 0 ? 0 : t0) + c; t < t1; t += NCB) {
        *reinterpret_cast<uint2 *>(dkv + t * C + col) = make_uint2(0u, 0u);
        *reinterpret_cast<uint2 *>(dscore + t * C + col) = make_uint2(0u, 0u);
        if (COFF == 2 && all_halves) {
            *reinterpret_cast<uint2 *>(dkv + t * C + head_dim + col) = make_uint2(0u, 0u);
            *reinterpret_cast<uint2 *>(dscore + t * C + head_dim + col) = make_uint2(0u, 0u);
        }
    }
}

template <int COFF, int NCB, int RC>
__global__ void __launch_bounds__(Geo<COFF, NCB>::THREADS, kBwdLean<COFF, NCB> ? Geo<COFF, NCB>::MIN_BLOCKS : 1)
    bwd_chunk_kernel(ChArgs a, const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_sc,
                     int64_t n_tokens_arg, const uint16_t *__restrict__ grad_out, uint16_t *__restrict__ dkv,
                     uint16_t *__restrict__ dscore, float *__restrict__ partial)
{
    using G = Geo<COFF, NCB>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    constexpr bool LEAN = kBwdLean<COFF, NCB>;
    constexpr bool HOLD = kBwdHold<COFF, NCB>;  // kv from the stage: the stage held through the row
    unsigned char *smem_base = align_1k<LEAN>(smem_raw);
    const ChSmem<COFF, NCB> s = ch_carve<COFF, NCB>(smem_base, a.stages, a.stage_bytes, LEAN);
    const Win<COFF, NCB, RC> w(a);
    const int R = w.ratio();
    const int c0 = blockIdx.y * G::TC;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t C = (int64_t)COFF * a.head_dim;
    ch_init<COFF, NCB>(s, a.stages);
    pdl_wait();
    pdl_trigger();  // the grad_ape finalisation may launch; it waits for this grid's end
    const int Rr = a.n_seg > 0 ? __ldg(a.cc + a.n_seg) : 0;  // real rows
    const int R0 = a.n_seg > 0 ? __ldg(a.cc) : 0;
    const int rend = Rr < a.capacity ? Rr : a.capacity;
    const int64_t n_tokens = n_tokens_arg >= 0 ? n_tokens_arg : (int64_t)__ldg(a.cu + a.n_seg);

    const int g = lane % G::G, c = G::CPW * warp + lane / G::G;
    const int col = c0 + 4 * g;  // thread's first column within a half
    float2 acc[kKC][2];
#pragma unroll
    for (int i = 0; i < kKC; ++i)
        acc[i][0] = acc[i][1] = make_float2(0.0f, 0.0f);

    if (warp == G::CW) {
        if (lane == 0)
            ch_produce<COFF, NCB, RC, true>(a, s, &tm_kv, &tm_sc, c0, blockIdx.x, gridDim.x, rend, grad_out);
    } else {
        if (blockIdx.x == 0) {  // leading gap: tokens before the first real block
            int64_t lead = n_tokens;
            if (R0 < Rr)
                lead = map_row(R0, a.cu, a.cc, a.n_seg, R).base;
            ch_zero_tokens<COFF, NCB>(dkv, dscore, C, a.head_dim, col, 0, lead, n_tokens, c, true);
        }
        float2 ap[kKC][2];
        if constexpr (LEAN) {
            // the block's APE tile [window position][tile column], read once
            const int W = COFF * R;
            for (int v = threadIdx.x; v < W * G::TC / 4; v += G::CT) {
                const int k = v / (G::TC / 4), c4 = v - k * (G::TC / 4);
                const int part = k / R, tk = k - part * R;
                *reinterpret_cast<float4 *>(s.apet + (size_t)v * 4) = __ldg(reinterpret_cast<const float4 *>(
                    a.ape + (int64_t)tk * C + (int64_t)part * a.head_dim + c0 + 4 * c4));
            }
            named_barrier(1, G::CT);
        } else {
            ch_load_ape<COFF, NCB, RC>(a, w, c, col, ap);
        }
        int st = 0, buf = 0;
        uint32_t ph = 0;
        for (int row = blockIdx.x; row < rend; row += gridDim.x) {
            const bool ok = mbar_wait(smem_addr(&s.full[st]), ph, a.status);
            Meta m = Meta{0, 0, row, 0, 1, 0, 0};
            if (ok)
                m = s.meta[st];
            // rows below cu_seqlens_comp[0] are not real: no loads, no gradient
            const bool first = m.first || !m.real;
            const int st_row = st;
            const unsigned char *stage = s.stages + (size_t)st * a.stage_bytes;
            ChunkState cs;
            if (ok && m.real) {
                if constexpr (LEAN)
                    ch_load_s<COFF, NCB, RC, !HOLD>(w, stage, s.apet, c, g, first, cs);
                else
                    ch_load<COFF, NCB, RC>(w, stage, c, g, first, ap, cs);
            }
            uint2 gw = make_uint2(0u, 0u);
            if (ok && m.real)
                gw = *reinterpret_cast<const uint2 *>(stage + w.win_bytes() + 8 * g);
            if constexpr (!HOLD) {  // everything the row needs is in registers now
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&s.empty[st_row]));
            }
            if (++st == a.stages) {
                st = 0;
                ph ^= 1u;
            }
            // HOLD: the stage stays held until the gradients below have read kv from it
            if (!ch_pool<COFF, NCB, RC, HOLD>(w, s, buf, c, g, ok, ok && m.real, first, cs, stage))
                break;
            const float2 gg[2] = {bf16x2_to_f2(gw.x), bf16x2_to_f2(gw.y)};
            const uint32_t gwq[2] = {gw.x, gw.y};
            float *fin = s.fin + (size_t)buf * (2 + G::CW) * G::TC;
            {
                int j;
                float den, num;
                if (threadIdx.x < G::MT) {
                    ch_final<COFF, NCB>(s, buf, j, den, num, G::LOCAL ? fin + 2 * G::TC : nullptr);
                    if (threadIdx.x % G::TPC == 0 && m.real) {
                        const float inv = recip_den(den);
                        fin[j] = inv;
                        fin[G::TC + j] = __fmul_rn(num, inv);  // o
                    }
                }
            }
            named_barrier(1, G::CT);
            buf ^= 1;
            if (!m.real) {
                if constexpr (HOLD) {
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_addr(&s.empty[st_row]));
                }
                continue;
            }
            const float4 inv4 = *reinterpret_cast<const float4 *>(fin + 4 * g);
            const float4 o4 = *reinterpret_cast<const float4 *>(fin + G::TC + 4 * g);
            float2 inv[2] = {make_float2(inv4.x, inv4.y), make_float2(inv4.z, inv4.w)};
            if constexpr (G::LOCAL) {  // p_k = e_k * scale_w * inv: e_k is relative to the warp's maximum
                const float4 sc4 = *reinterpret_cast<const float4 *>(fin + (2 + warp) * G::TC + 4 * g);
                inv[0] = mul2(inv[0], make_float2(sc4.x, sc4.y));
                inv[1] = mul2(inv[1], make_float2(sc4.z, sc4.w));
            }
            const float2 go[2] = {mul2(gg[0], make_float2(o4.x, o4.y)), mul2(gg[1], make_float2(o4.z, o4.w))};
            const float2 ngo[2] = {make_float2(-go[0].x, -go[0].y), make_float2(-go[1].x, -go[1].y)};
            // window position k = c + NC*i sits at token t0 + k (part = k / ratio)
            const int64_t t0 = m.base - (int64_t)(COFF - 1) * R;
            const int64_t lim = n_tokens - t0;  // positions k < lim hold a real token
            uint16_t *pk_dkv = dkv + t0 * C + (int64_t)c * C + col;
            uint16_t *pk_dsc = dscore + t0 * C + (int64_t)c * C + col;
#pragma unroll
            for (int i = 0; i < kKC; ++i) {
                int part, tk;
                if (!w.pos(c, i, part, tk) || (COFF == 2 && part == 0 && first))
                    continue;
                const uint2 kv = ch_kv<COFF, NCB, RC, HOLD>(w, cs, stage, c, g, i);
                const uint32_t kw[2] = {kv.x, kv.y};
                uint32_t dk[2], dsw[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float2 pk = mul2(cs.e[i][q], inv[q]);
                    dk[q] = f2_to_bf16x2(mul2(gg[q], pk));
                    const float2 ds = mul2(pk, fma2_bf16x2(gwq[q], kw[q], ngo[q]));
                    dsw[q] = f2_to_bf16x2(ds);
                    acc[i][q] = add2(acc[i][q], ds);
                }
                if (c + NCB * i < lim) {
                    const int64_t off = (int64_t)(NCB * i) * C + (int64_t)part * a.head_dim;
                    *reinterpret_cast<uint2 *>(pk_dkv + off) = make_uint2(dk[0], dk[1]);
                    *reinterpret_cast<uint2 *>(pk_dsc + off) = make_uint2(dsw[0], dsw[1]);
                }
            }
            if constexpr (HOLD) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&s.empty[st_row]));
            }
            if (m.last) {  // last block of its segment
                if (COFF == 2)  // own block's first-half columns: read by no row
                    ch_zero_tokens<COFF, NCB>(dkv, dscore, C, a.head_dim, col, m.base, m.base + R, n_tokens, c, false);
                int64_t next = n_tokens;
                if (m.row + 1 < Rr)
                    next = map_row(m.row + 1, a.cu, a.cc, a.n_seg, R).base;
                ch_zero_tokens<COFF, NCB>(dkv, dscore, C, a.head_dim, col, m.base + R, next, n_tokens, c, true);
            }
        }
    }
    __syncthreads();  // the ring is idle: its stages become the grad_ape staging area
    // grad_ape partial [ape row][part][tile column]
    float *red = reinterpret_cast<float *>(s.stages);
    if (warp < G::CW) {
#pragma unroll
        for (int i = 0; i < kKC; ++i) {
            int part, tk;
            if (!w.pos(c, i, part, tk))
                continue;
            *reinterpret_cast<float4 *>(red + (tk * COFF + part) * G::TC + 4 * g) =
                make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
        }
    }
    __syncthreads();
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int rank = (int)cluster.block_rank();
    const int nrank = (int)cluster.num_blocks();
    const int n4 = R * COFF * G::TC / 4;
    const int share = (n4 + nrank - 1) / nrank;
    const int lo = rank * share, hi = lo + share < n4 ? lo + share : n4;
    float *dst = partial + (int64_t)(blockIdx.x / nrank) * R * C;
    for (int i4 = lo + (int)threadIdx.x; i4 < hi; i4 += blockDim.x) {
        const int rp = (i4 * 4) / G::TC, lcol = i4 * 4 - rp * G::TC;
        const int arow = rp / COFF, pp = rp - arow * COFF;
        float4 v4 = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(red, 0) + i4 * 4);
        for (int q = 1; q < nrank; ++q) {
            const float4 v = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(red, q) + i4 * 4);
            v4.x = __fadd_rn(v4.x, v.x);
            v4.y = __fadd_rn(v4.y, v.y);
            v4.z = __fadd_rn(v4.z, v.z);
            v4.w = __fadd_rn(v4.w, v.w);
        }
        *reinterpret_cast<float4 *>(dst + (int64_t)arow * C + (int64_t)pp * a.head_dim + c0 + lcol) = v4;
    }
    cluster.sync();
}

// ------------------------------------------------------------------- host

struct ChPlan {
    int stages, stage_bytes, box_bytes, threads, tiles, cluster;
    size_t smem;
};

template <int COFF, int NCB>
ChPlan ch_plan(bool bwd, int ratio, int head_dim)
{
    using G = Geo<COFF, NCB>;
    ChPlan pl;
    pl.box_bytes = (ratio * G::TC * 2 + 127) / 128 * 128;
    pl.stage_bytes = (2 * COFF * pl.box_bytes + (bwd ? G::TC * 2 : 0) + 1023) / 1024 * 1024;
    const bool tile = bwd && kBwdLean<COFF, NCB>;
    // two blocks per SM (forward, lean backward): two stages; one block per SM
    // (register-resident backward): a four-stage ring fits
    pl.stages = bwd && !tile ? 4 : 2;
    pl.threads = G::THREADS;
    pl.tiles = head_dim / G::TC;
    // no clusters: pairs of blocks would halve the grad_ape partials, but the grid
    // must then be an even number of blocks per column tile, which leaves SMs idle
    // (19 blocks per tile fill 152 SMs twice over at head_dim 512, coff 2)
    pl.cluster = 1;
    pl.smem = ch_smem_bytes<COFF, NCB>(pl.stages, pl.stage_bytes, tile) + 1024;  // + alignment slack
    if (bwd) {  // grad_ape staging reuses the stages: make sure it fits
        const size_t red = (size_t)ratio * COFF * G::TC * sizeof(float);
        if ((size_t)pl.stages * pl.stage_bytes < red)
            pl.stages = (int)((red + pl.stage_bytes - 1) / pl.stage_bytes);
        pl.smem = ch_smem_bytes<COFF, NCB>(pl.stages, pl.stage_bytes, tile) + 1024;
    }
    return pl;
}

// Row blocks per column tile: as many as are resident on the device, at most one
// per row.
cudaError_t ch_blocks(const void *fn, const ChPlan &pl, int rows, int *out)
{
    int resident = 0;
    cudaError_t e = resident_blocks(fn, pl.threads, pl.smem, pl.cluster, &resident);
    if (e != cudaSuccess)
        return e;
    int blocks = (resident > 0 ? resident : 1) / pl.tiles;
    blocks = blocks / pl.cluster * pl.cluster;
    if (blocks < pl.cluster)
        blocks = pl.cluster;
    const int need = rows > 0 ? rows : 1;
    if (blocks > need)
        blocks = (need + pl.cluster - 1) / pl.cluster * pl.cluster;
    *out = blocks;
    return cudaSuccess;
}

ChArgs ch_args(const void *kv, const void *score, const float *ape, const int32_t *cu, const int32_t *cc, int n_seg,
               int head_dim, int capacity, int ratio, const ChPlan &pl, unsigned *status)
{
    return ChArgs{static_cast<const uint16_t *>(kv), static_cast<const uint16_t *>(score), ape, cu, cc, n_seg,
                  head_dim, capacity, ratio, pl.box_bytes, pl.stages, pl.stage_bytes, status};
}

template <int COFF, int NCB, int RC>
cudaError_t launch_fwd_ch(const FwdParams &p, unsigned *status, cudaStream_t st)
{
    const ChPlan pl = ch_plan<COFF, NCB>(false, p.ratio, p.head_dim);
    auto kern = fwd_chunk_kernel<COFF, NCB, RC>;
    int blocks = 0;
    cudaError_t e = ch_blocks(reinterpret_cast<const void *>(kern), pl, p.capacity, &blocks);
    if (e != cudaSuccess)
        return e;
    CUtensorMap mk, ms;
    const int64_t C = (int64_t)COFF * p.head_dim;
    if ((e = make_tensor_map_2d(&mk, p.kv, C, Geo<COFF, NCB>::TC, p.ratio)) != cudaSuccess ||
        (e = make_tensor_map_2d(&ms, p.score, C, Geo<COFF, NCB>::TC, p.ratio)) != cudaSuccess)
        return e;
    const ChArgs a = ch_args(p.kv, p.score, p.ape, p.cu_seqlens, p.cu_seqlens_comp, p.n_seg, p.head_dim, p.capacity,
                             p.ratio, pl, status);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, pl.tiles, 1);
    cfg.blockDim = dim3(pl.threads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, mk, ms, static_cast<uint16_t *>(p.out));
}

template <int COFF, int NCB, int RC>
cudaError_t ch_bwd_blocks(int ratio, int head_dim, int capacity, int *blocks, int *cluster)
{
    const ChPlan pl = ch_plan<COFF, NCB>(true, ratio, head_dim);
    *cluster = pl.cluster;
    return ch_blocks(reinterpret_cast<const void *>(bwd_chunk_kernel<COFF, NCB, RC>), pl, capacity, blocks);
}

template <int COFF, int NCB, int RC>
cudaError_t launch_bwd_ch(const BwdParams &p, float *partial, int blocks, unsigned *status, cudaStream_t st)
{
    const ChPlan pl = ch_plan<COFF, NCB>(true, p.ratio, p.head_dim);
    auto kern = bwd_chunk_kernel<COFF, NCB, RC>;
    CUtensorMap mk, ms;
    const int64_t C = (int64_t)COFF * p.head_dim;
    cudaError_t e;
    if ((e = allow_max_smem(reinterpret_cast<const void *>(kern))) != cudaSuccess ||
        (e = make_tensor_map_2d(&mk, p.kv, C, Geo<COFF, NCB>::TC, p.ratio)) != cudaSuccess ||
        (e = make_tensor_map_2d(&ms, p.score, C, Geo<COFF, NCB>::TC, p.ratio)) != cudaSuccess)
        return e;
    const ChArgs a = ch_args(p.kv, p.score, p.ape, p.cu_seqlens, p.cu_seqlens_comp, p.n_seg, p.head_dim, p.capacity,
                             p.ratio, pl, status);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, pl.tiles, 1);
    cfg.blockDim = dim3(pl.threads, 1, 1);
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
    e = cudaLaunchKernelEx(&cfg, kern, a, mk, ms, p.n_tokens, static_cast<const uint16_t *>(p.grad_out),
                           static_cast<uint16_t *>(p.dkv), static_cast<uint16_t *>(p.dscore), partial);
    if (e != cudaSuccess)
        return e;
    return launch_dape_finalize(partial, blocks / pl.cluster, (int64_t)p.ratio * C, p.dape, st);
}

}  // namespace

bool chunked_supported(int ratio, int coff, int head_dim)
{
    if (head_dim % 64 != 0 || head_dim < 64 || head_dim > 8192 || ratio > 128)
        return false;
    return (coff == 1 && ratio > 64) || (coff == 2 && ratio > 32);
}

// The kernel instance for a shape: ratio 128 with the ratio as a constant (16
// chunks for coff 1, 32 for coff 2); other ratios at run time with the fewest
// chunks of 8 positions that cover the window, in steps of whole consumer warps
// (coff 1: 12 or 16 chunks, windows up to 96 or 128; coff 2: 12, 16, 20, 24, 28
// or 32 chunks, windows up to 96 ... 256), so that no warp holds only positions
// past the window.
#define CSA_CHUNK_DISPATCH(FN, ...)                                                         \
    do {                                                                                    \
        if (ratio == 128)                                                                   \
            return coff == 2 ? FN<2, 32, 128>(__VA_ARGS__) : FN<1, 16, 128>(__VA_ARGS__);   \
        if (coff == 1)                                                                      \
            return ratio <= 96 ? FN<1, 12, 0>(__VA_ARGS__) : FN<1, 16, 0>(__VA_ARGS__);     \
        switch ((2 * ratio + 31) / 32) {                                                    \
        case 3: return FN<2, 12, 0>(__VA_ARGS__);                                           \
        case 4: return FN<2, 16, 0>(__VA_ARGS__);                                           \
        case 5: return FN<2, 20, 0>(__VA_ARGS__);                                           \
        case 6: return FN<2, 24, 0>(__VA_ARGS__);                                           \
        case 7: return FN<2, 28, 0>(__VA_ARGS__);                                           \
        default: return FN<2, 32, 0>(__VA_ARGS__);                                          \
        }                                                                                   \
    } while (0)

cudaError_t launch_fwd_chunked(const FwdParams &p, unsigned *status, cudaStream_t st)
{
    const int ratio = p.ratio, coff = p.coff;
    CSA_CHUNK_DISPATCH(launch_fwd_ch, p, status, st);
}

// Grid width of the backward and the number of grad_ape partials it writes (the
// workspace needs that many ratio x coff*head_dim slabs).
cudaError_t chunked_bwd_partials(int ratio, int coff, int head_dim, int capacity, int *partials, int *blocks)
{
    int cluster = 1;
    cudaError_t e = [&]() -> cudaError_t { CSA_CHUNK_DISPATCH(ch_bwd_blocks, ratio, head_dim, capacity, blocks, &cluster); }();
    *partials = *blocks / cluster;
    return e;
}

cudaError_t launch_bwd_chunked(const BwdParams &p, float *partial, int blocks, unsigned *status, cudaStream_t st)
{
    const int ratio = p.ratio, coff = p.coff;
    CSA_CHUNK_DISPATCH(launch_bwd_ch, p, partial, blocks, status, st);
}

#undef CSA_CHUNK_DISPATCH

}  // namespace csa
