// Streamed Compressor kernels for small ratios: a bulk-copy pipeline into shared
// memory.  Used for ratio 4 when head_dim is a multiple of 64 (the forward from
// head_dim 128 on).
//
// Semantics and operation order are exactly those of csa_small.cu ("CSA Fused
// Compressor", cuDNN frontend docs, sections Semantics and Numerics): window
// positions in ascending k, invalid ones skipped; s = score + ape; NaN-propagating
// max; e = exp(s - m) with the library's exp; den and num accumulated in ascending
// k; inv = 1/den rounded to nearest; out = bf16(num * inv); backward p = e*inv,
// grad_kv = bf16(g*p), ds = p*(g*kv - g*o).  Results are bitwise those of
// csa_small.cu.
//
// Structure (per thread block, persistent over the rows b, b + gridDim.x, ...):
//   * one producer warp: for each row, waits for a free stage of a shared-memory
//     ring, then issues raw bulk copies (cp.async.bulk) of every window row the
//     output row reads -- each (token, half) is one contiguous run of TC*2 bytes;
//     whole token rows for a narrow single-tile head; one TMA box per array and
//     part for the tiles of a wider head -- and, in the backward,
//     the grad_out row; completion is counted in bytes on the stage's "full"
//     mbarrier;
//   * consumer warps: thread t owns columns [c0 + 2*NP*t, c0 + 2*NP*(t + 1)) of
//     the block's column tile (NP fp32 pairs: two where head_dim is a multiple of
//     128, else one) for every row, so
//     its APE values stay in registers; it waits on
//     the stage's "full" barrier, computes from shared memory, writes its outputs
//     and releases the stage on the "empty" barrier.
// Every wait is bounded in time; on expiry a timeout is recorded in the status
// word, the loops stop, copies still in flight are drained, and the kernel exits
// normally (no trap, no hang).
#include <cooperative_groups.h>

#include <mutex>

#include "csa_device.cuh"
#include "csa_launch.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

// The plan's fixed choices (each measured on GB300 against its alternatives):
constexpr int kWholeMaxD = 256;          // widest coff-2 head staged as whole token rows
constexpr int kChunkCols = 256;          // widest span of one TMA box dimension
constexpr int kFwdBudget = 64 * 1024;    // ring bytes of a forward block with four consumer warps
constexpr int kBwdBudget = 64 * 1024;    // ... of a backward block
constexpr int kBwdCluster = 2;           // backward blocks per cluster (grad_ape merged in DSMEM)
constexpr int kRowLanes1 = 2;            // rows in flight per block when a tile is one warp wide
// Register cap of the forward: at 128 registers five-warp blocks fit three to an
// SM (each SM sub-partition holds four such warps).
constexpr int kFwdMaxReg = 128;

// A consumer thread owns NP fp32 column pairs (NP = 2 where head_dim is a multiple
// of 128, else 1): CPT columns, and a warp PER_WARP columns of the tile.
template <int NP>
struct Cols {
    static_assert(NP == 1 || NP == 2, "one or two column pairs per thread");
    static constexpr int CPT = 2 * NP;
    static constexpr int PER_WARP = 32 * CPT;
    static constexpr int MAX_THREADS = (512 / PER_WARP + 1) * 32;  // 512-column tile + the producer warp
};

// NP 32-bit words (2*NP bf16): one 4- or 8-byte access.
template <int NP>
__device__ __forceinline__ void ld_np(uint32_t (&w)[NP], const void *p)
{
    if constexpr (NP == 2) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        w[0] = v.x;
        w[1] = v.y;
    } else {
        w[0] = *reinterpret_cast<const uint32_t *>(p);
    }
}

template <int NP>
__device__ __forceinline__ void st_np(void *p, const uint32_t (&w)[NP])
{
    if constexpr (NP == 2)
        *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
    else
        *reinterpret_cast<uint32_t *>(p) = w[0];
}

template <int NP>
__device__ __forceinline__ void st_np_zero(void *p)
{
    if constexpr (NP == 2)
        *reinterpret_cast<uint2 *>(p) = make_uint2(0u, 0u);
    else
        *reinterpret_cast<uint32_t *>(p) = 0u;
}

// NP fp32 pairs: one 8- or 16-byte access.
template <int NP>
__device__ __forceinline__ void ld_pairs(float2 (&v)[NP], const float *p)
{
    if constexpr (NP == 2) {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(p));
        v[0] = make_float2(f.x, f.y);
        v[1] = make_float2(f.z, f.w);
    } else {
        v[0] = __ldg(reinterpret_cast<const float2 *>(p));
    }
}

template <int NP>
__device__ __forceinline__ void st_pairs(float *p, const float2 (&v)[NP])
{
    if constexpr (NP == 2)
        *reinterpret_cast<float4 *>(p) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
    else
        *reinterpret_cast<float2 *>(p) = v[0];
}

struct StreamArgs {
    const uint16_t *kv;
    const uint16_t *score;
    const float *ape;
    const int32_t *cu;
    const int32_t *cc;
    int n_seg;
    int head_dim;
    int capacity;
    int stages;        // ring depth (a multiple of row_lanes)
    int stage_bytes;   // bytes per stage (multiple of 128)
    unsigned *status;  // caller-visible status word
    int tc;            // columns of the block's tile
    int row_lanes;     // rows in flight per block: groups of tc / (32 * 2 * NP) warps
    int rw;            // elements per staged token row: tc, or C for whole rows
    int pcol;          // whole rows: head_dim (part p's data at column p * head_dim of a row); tiled: 0
    int tma;           // tiled: 0 per-token copies; 1 one 2-D TMA box [RATIO tokens x tc] per array and
                       // part; 2 one 3-D box [RATIO tokens x tc / 256 x 256] (tiles wider than 256)
};

// Staging of a window.  Tiled (rw = tc): per token of each part, the tile's
// columns of that part, 2 * COFF * RATIO copies of tc elements -- or one TMA box
// per array and part, which lands in the same layout with 2 * COFF copies: for
// tiles of at most 256 columns (the limit of one box dimension) a 2-D box
// [RATIO tokens x tc], for wider tiles (multiples of 256) a 3-D box over the rows
// seen as [C / 256][256] chunks, [RATIO tokens x tc / 256 chunks x 256].  Whole rows (one
// column tile, rw = C): per part, the RATIO whole token rows of its block, one
// contiguous copy of RATIO * C elements per array; coff 2 then also stages the
// half of each row the window does not use (the neighbouring row reads it), in
// exchange for fewer, larger copies, which narrow heads need to keep the one
// issuing thread ahead of the consumers: the parts' blocks are consecutive token
// rows, so a row that reads both parts takes a single copy of 2 * RATIO rows per
// array.

// Consumer warp w of a block works on column group w % (tc / PER_WARP) of the
// tile and on row lane w / (tc / PER_WARP): the block's j-th row (in the
// producer's order) goes to lane j % row_lanes, in ring slot j % stages.  With
// stages a multiple of row_lanes every slot always serves the same lane, so no
// consumer ever waits on a slot more than one phase ahead.
struct Lanes {
    int cols;  // column-group warps per row
    int lane;  // this warp's row lane
    int lc;    // this thread's first column in the tile
};

template <int NP>
__device__ __forceinline__ Lanes lanes_of(const StreamArgs &a, int warp, int lane)
{
    Lanes l;
    l.cols = a.tc / Cols<NP>::PER_WARP;
    l.lane = warp / l.cols;
    l.lc = ((warp % l.cols) * 32 + lane) * Cols<NP>::CPT;
    return l;
}

struct StageMeta {
    int64_t base;
    int seg;
    int row;
    int real;
    int first;
    int last;  // the last block of its segment (from the producer's row cursor)
    int pad;
};

// Window position k reads part p = k / RATIO, token i = k % RATIO of the part.
// coff 2: part 0 = the previous block on the first-half columns, part 1 = the own
// block on the second-half columns; coff 1: part 0 = the own block.  The part's
// tokens start at base + (p - (COFF - 1)) * RATIO and its columns at p * head_dim.
template <int RATIO, int COFF>
__host__ __device__ __forceinline__ int stage_offset(int arr, int part, int i, int tc)
{
    return ((arr * COFF + part) * RATIO + i) * tc * 2;
}

template <int RATIO, int COFF>
__host__ __device__ __forceinline__ int window_bytes(int tc)
{
    return 2 * COFF * RATIO * tc * 2;
}

struct Smem {
    unsigned char *stages;
    StageMeta *meta;
    uint64_t *full;
    uint64_t *empty;
    float *red;
};

// The stages start at the shared array itself, declared 128-byte aligned (an
// alignment computed through an integer round trip costs the consumers 5-9%: the
// pointers are no longer provably shared).  Only TMA boxes need more than 16
// bytes: the producer checks the address and falls back to bulk copies (same
// layout) if it is not 128-byte aligned.
__device__ __forceinline__ Smem carve(unsigned char *base, int stages, int stage_bytes)
{
    Smem s;
    s.stages = base;
    unsigned char *p = base + (size_t)stages * stage_bytes;
    s.meta = reinterpret_cast<StageMeta *>(p);
    p += sizeof(StageMeta) * stages;
    s.full = reinterpret_cast<uint64_t *>(p);
    s.empty = s.full + stages;
    p = reinterpret_cast<unsigned char *>(s.empty + stages);
    s.red = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15));
    return s;
}

__host__ size_t smem_bytes(int stages, int stage_bytes, size_t red_bytes)
{
    return (size_t)stages * stage_bytes + (sizeof(StageMeta) + 16) * stages + 16 + red_bytes;
}

// ---------------------------------------------------------------- producer

// Issues the copies of rows row0, row0 + rstride, ... < rend.  Runs on one lane.
template <int RATIO, int COFF, bool BWD>
__device__ void produce(const StreamArgs &a, const Smem &s, const CUtensorMap *tm_kv, const CUtensorMap *tm_sc,
                        int tc, int c0, int row0, int rstride, int rend, const uint16_t *__restrict__ grad_out)
{
    const int64_t C = (int64_t)COFF * a.head_dim;
    const uint32_t run = (uint32_t)tc * 2;
    const bool tma = a.tma && (smem_addr(s.stages) & 127u) == 0u;  // TMA destinations: 128-byte aligned
    // 3-D boxes are planned for coff 2 only; for coff 1 the branch is compiled out
    // (a runtime test in its producer cost the coff-1 backward 52.5 -> 55.3 us at
    // head_dim 512, 16 x 4096 tokens)
    const bool box3 = COFF == 2 && a.tma == 2;
    int issued = 0, st = 0;
    uint32_t ph = 0;
    RowCursor cur;
    cursor_init(cur, a.cc, a.n_seg);
    for (int row = row0; row < rend; row += rstride) {
        // the row's map first: its loads (if any) overlap the wait for a free slot
        const RowMap rm = cursor_map(cur, row, a.cu, a.cc, a.n_seg, RATIO);
        if (!mbar_wait(smem_addr(&s.empty[st]), ph ^ 1u, a.status))
            break;
        StageMeta &m = s.meta[st];
        m.base = rm.base;
        m.seg = rm.seg;
        m.row = row;
        m.real = rm.real;
        m.first = rm.first;
        m.last = rm.real && row + 1 == cur.hi;
        const bool load = BWD ? rm.real : true;
        const int p0 = (COFF == 2 && rm.first) ? 1 : 0;
        const uint32_t bytes =
            load ? (uint32_t)((COFF - p0) * 2 * RATIO * a.rw * 2) + (BWD ? run : 0u) : 0u;
        const uint32_t fb = smem_addr(&s.full[st]);
        mbar_arrive_expect_tx(fb, bytes);
        if (load) {
            const uint32_t dst = smem_addr(s.stages + (size_t)st * a.stage_bytes);
            for (int p = p0; p < COFF; ++p) {
                const int64_t tok0 = rm.base + (int64_t)(p - (COFF - 1)) * RATIO;
                if (a.pcol) {
                    // whole rows: the parts' token blocks are consecutive in memory and
                    // in the stage, so a row that reads both takes one copy per array
                    // (head_dim 128, coff 2: forward 32.8 -> 31.1 us, backward 57.2 ->
                    // 52.2 us at 32 x 4096 tokens against one copy per part)
                    const int np = COFF - p;
                    const uint32_t blk = (uint32_t)(np * RATIO * C * 2);
                    bulk_g2s(dst + stage_offset<RATIO, COFF>(0, p, 0, a.rw), a.kv + tok0 * C, blk, fb);
                    bulk_g2s(dst + stage_offset<RATIO, COFF>(1, p, 0, a.rw), a.score + tok0 * C, blk, fb);
                    break;
                }
                const int64_t col = (int64_t)p * a.head_dim + c0;
                // 3-D boxes once the ring has filled: while it fills, the per-token
                // copies below deliver the first rows sooner (head_dim 512, coff 2,
                // forward: 8 x 4096 tokens 27.2 -> 26.3 us against boxes from the
                // start; 64 ragged segments 178.8 -> 170.5 us against per-token
                // copies throughout).  x = 0: 16-byte aligned by construction.
                if (tma && box3 && issued >= a.stages) {
                    tma_load_3d(dst + stage_offset<RATIO, COFF>(0, p, 0, tc), tm_kv, 0, (int)(col / kChunkCols),
                                (int)tok0, fb);
                    tma_load_3d(dst + stage_offset<RATIO, COFF>(1, p, 0, tc), tm_sc, 0, (int)(col / kChunkCols),
                                (int)tok0, fb);
                    continue;
                }
                if (tma && !box3) {
                    tma_load_2d(dst + stage_offset<RATIO, COFF>(0, p, 0, tc), tm_kv, (int)col, (int)tok0, fb);
                    tma_load_2d(dst + stage_offset<RATIO, COFF>(1, p, 0, tc), tm_sc, (int)col, (int)tok0, fb);
                    continue;
                }
#pragma unroll
                for (int i = 0; i < RATIO; ++i) {
                    const int64_t g = (tok0 + i) * C + col;
                    bulk_g2s(dst + stage_offset<RATIO, COFF>(0, p, i, tc), a.kv + g, run, fb);
                    bulk_g2s(dst + stage_offset<RATIO, COFF>(1, p, i, tc), a.score + g, run, fb);
                }
            }
            if (BWD)
                bulk_g2s(dst + window_bytes<RATIO, COFF>(a.rw), grad_out + (int64_t)row * a.head_dim + c0, run, fb);
        }
        ++issued;
        if (++st == a.stages) {
            st = 0;
            ph ^= 1u;
        }
    }
    // Copies of the last (up to) `stages` rows may still be in flight if the
    // consumers stopped early: wait for them before the block may exit.
    const int lo = issued > a.stages ? issued - a.stages : 0;
    for (int it = lo; it < issued; ++it)
        mbar_wait(smem_addr(&s.full[it % a.stages]), (uint32_t)(it / a.stages) & 1u, a.status);
}

// ---------------------------------------------------------------- consumer

template <int RATIO, int COFF, int NP>
struct ApeRegs {
    float2 v[COFF * RATIO][NP];
};

template <int RATIO, int COFF, int NP>
__device__ __forceinline__ void load_ape(const StreamArgs &a, int col0, ApeRegs<RATIO, COFF, NP> &ap)
{
    const int64_t C = (int64_t)COFF * a.head_dim;
#pragma unroll
    for (int k = 0; k < COFF * RATIO; ++k) {
        const int p = k / RATIO, i = k % RATIO;
        ld_pairs(ap.v[k], a.ape + i * C + (int64_t)p * a.head_dim + col0);
    }
}

// Reads the thread's NP words (2*NP bf16) of window position k from the stage.
// RW: the staged row width when known at compile time, with the parts at column 0
// of their rows (tiled staging, or coff 1); 0: the run-time rw and pcol.
template <int RATIO, int COFF, int NP, int RW>
__device__ __forceinline__ void stage_words(uint32_t (&w)[NP], const unsigned char *stage, int arr, int k, int rw,
                                            int pcol, int lc)
{
    const int p = k / RATIO, i = k % RATIO;
    if constexpr (RW != 0)
        ld_np(w, stage + stage_offset<RATIO, COFF>(arr, p, i, RW) + lc * 2);
    else
        ld_np(w, stage + stage_offset<RATIO, COFF>(arr, p, i, rw) + (p * pcol + lc) * 2);
}

// Max over a row's valid window positions, three values at a time: the own
// block's part, then (coff 2, unless the row is a segment's first block) the
// previous block's part folded in.
template <int RATIO, int COFF>
__device__ __forceinline__ float window_max(const float (&v)[COFF * RATIO], bool first)
{
    constexpr int W = COFF * RATIO, K0 = (COFF - 1) * RATIO;
    float a = v[K0];
#pragma unroll
    for (int k = K0 + 1; k < W; k += 2)
        a = k + 1 < W ? max3_nan(a, v[k], v[k + 1]) : max_nan(a, v[k]);
    if (COFF == 1)
        return a;
    float b = a;
#pragma unroll
    for (int i = 0; i < RATIO; i += 2)
        b = i + 1 < RATIO ? max3_nan(b, v[i], v[i + 1]) : max_nan(b, v[i]);
    return first ? a : b;
}

// Reads a row's window words (score and kv, the thread's columns) from its stage.
template <int RATIO, int COFF, int NP, int RW>
__device__ __forceinline__ void stage_load(const unsigned char *stage, int rw, int pcol, int lc,
                                           uint32_t (&sw)[COFF * RATIO][NP], uint32_t (&kvw)[COFF * RATIO][NP])
{
#pragma unroll
    for (int k = 0; k < COFF * RATIO; ++k) {
        stage_words<RATIO, COFF, NP, RW>(sw[k], stage, 1, k, rw, pcol, lc);
        stage_words<RATIO, COFF, NP, RW>(kvw[k], stage, 0, k, rw, pcol, lc);
    }
}

// The pooling of one row from its words in registers (a first block's
// previous-block positions hold stale words, which the max and the sums skip).
template <int RATIO, int COFF, int NP>
__device__ __forceinline__ void pool_regs(const uint32_t (&sw)[COFF * RATIO][NP], const uint32_t (&kvw)[COFF * RATIO][NP],
                                          bool first, const ApeRegs<RATIO, COFF, NP> &ap,
                                          float2 (&e)[COFF * RATIO][NP], float2 (&den)[NP], float2 (&num)[NP])
{
    constexpr int W = COFF * RATIO;
#pragma unroll
    for (int k = 0; k < W; ++k)
#pragma unroll
        for (int q = 0; q < NP; ++q)
            e[k][q] = add2_bf16x2(sw[k][q], ap.v[k][q]);
    float2 m[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        float vx[W], vy[W];
#pragma unroll
        for (int k = 0; k < W; ++k) {
            vx[k] = e[k][q].x;
            vy[k] = e[k][q].y;
        }
        m[q] = make_float2(window_max<RATIO, COFF>(vx, first), window_max<RATIO, COFF>(vy, first));
    }
    float2 negm[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        negm[q] = make_float2(-m[q].x, -m[q].y);
        den[q] = make_float2(0.0f, 0.0f);
        num[q] = make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int k = 0; k < W; ++k) {
        if (COFF == 2 && k < RATIO && first)
            continue;
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            const float2 ek = exp2lanes(add2(e[k][q], negm[q]));
            e[k][q] = ek;
            den[q] = add2(den[q], ek);
            num[q] = fma2(ek, bf16x2_to_f2(kvw[k][q]), num[q]);
        }
    }
}

template <int RATIO, int COFF, int NP, int RW>
__device__ __forceinline__ void pool_stage(const unsigned char *stage, int rw, int pcol, int lc, bool first,
                                           const ApeRegs<RATIO, COFF, NP> &ap, uint32_t (&kvw)[COFF * RATIO][NP],
                                           float2 (&e)[COFF * RATIO][NP], float2 (&den)[NP], float2 (&num)[NP])
{
    uint32_t sw[COFF * RATIO][NP];
    stage_load<RATIO, COFF, NP, RW>(stage, rw, pcol, lc, sw, kvw);
    pool_regs<RATIO, COFF, NP>(sw, kvw, first, ap, e, den, num);
}

// ----------------------------------------------------------------- forward

// RW: 512 where the staged rows are 512 elements wide with the parts at column 0
// (0: width and part column from the arguments) -- the stage offsets then fold
// into the shared-memory loads (head_dim 512 forward: coff 2 26.3 -> 26.1 us at
// 8 x 4096 tokens, coff 1 28.5 -> 27.9 us at 16 x 4096; the backward measured
// slower with it, 53.8 against 50.5 us, and keeps the run-time width).
template <int RATIO, int COFF, int NP, int RW>
__global__ void __maxnreg__(kFwdMaxReg)
    fwd_stream_kernel(StreamArgs a, const __grid_constant__ CUtensorMap tm_kv,
                      const __grid_constant__ CUtensorMap tm_sc, uint16_t *__restrict__ out)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int ncw = blockDim.x / 32 - 1;  // consumer warps; the last warp produces
    const int tc = a.tc;
    const int c0 = blockIdx.y * tc;
    const Smem s = carve(smem_raw, a.stages, a.stage_bytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const Lanes ln = lanes_of<NP>(a, warp, lane);
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(smem_addr(&s.full[i]), 1);
            mbar_init(smem_addr(&s.empty[i]), ln.cols);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    if (warp == ncw) {
        if (lane == 0)
            produce<RATIO, COFF, false>(a, s, &tm_kv, &tm_sc, tc, c0, blockIdx.x, gridDim.x, a.capacity, nullptr);
        return;
    }
    const int lc = ln.lc;  // local column of this thread in the tile
    ApeRegs<RATIO, COFF, NP> ap;
    load_ape<RATIO, COFF, NP>(a, c0 + lc, ap);
    int st = ln.lane;
    uint32_t ph = 0;
    for (int j = ln.lane;; j += a.row_lanes, ring_next(st, ph, a.row_lanes, a.stages)) {
        const int row = blockIdx.x + j * gridDim.x;
        if (row >= a.capacity)
            break;
        if (!mbar_wait(smem_addr(&s.full[st]), ph, a.status))
            break;
        const unsigned char *stage = s.stages + (size_t)st * a.stage_bytes;
        const bool first = s.meta[st].first;
        uint32_t kvw[COFF * RATIO][NP];
        float2 e[COFF * RATIO][NP], den[NP], num[NP];
        pool_stage<RATIO, COFF, NP, RW>(stage, a.rw, a.pcol, lc, first, ap, kvw, e, den, num);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&s.empty[st]));
        uint32_t o[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q)
            o[q] = f2_to_bf16x2(mul2(num[q], make_float2(recip_den(den[q].x), recip_den(den[q].y))));
        st_np(out + (int64_t)row * a.head_dim + c0 + lc, o);
    }
}

// ---------------------------------------------------------------- backward

struct GradOut {
    uint16_t *dkv;
    uint16_t *dscore;
    int64_t n_tokens;
};

template <int COFF, int NP>
__device__ __forceinline__ void zero_range(const GradOut &o, int64_t C, int head_dim, int col, int64_t t0,
                                           int64_t t1)
{
    t1 = t1 < o.n_tokens ? t1 : o.n_tokens;
    for (int64_t t = t0 < 0 ? 0 : t0; t < t1; ++t) {
#pragma unroll
        for (int p = 0; p < COFF; ++p) {
            st_np_zero<NP>(o.dkv + t * C + p * head_dim + col);
            st_np_zero<NP>(o.dscore + t * C + p * head_dim + col);
        }
    }
}

// Gradient coverage as in csa_small.cu: a real row writes every slot it reads; the
// last block of a segment zeroes its own first-half columns (coff 2) and the gap
// up to the next real block (or n_tokens); block 0 zeroes the leading gap.  The
// grad_ape partial of each thread block (its rows in ascending order, per thread)
// is merged across the cluster in ascending rank order through distributed shared
// memory; dape_finalize_kernel sums the cluster partials in a fixed order.
template <int RATIO, int COFF, int NP>
__global__ void __launch_bounds__(Cols<NP>::MAX_THREADS) bwd_stream_kernel(StreamArgs a, const __grid_constant__ CUtensorMap tm_kv,
                                                         const __grid_constant__ CUtensorMap tm_sc, int64_t n_tokens_arg,
                                                         const uint16_t *__restrict__ grad_out,
                                                         uint16_t *__restrict__ dkv, uint16_t *__restrict__ dscore,
                                                         float *__restrict__ partial)
{
    constexpr int W = COFF * RATIO;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int ncw = blockDim.x / 32 - 1;
    const int tc = a.tc;
    const int c0 = blockIdx.y * tc;
    const Smem s = carve(smem_raw, a.stages, a.stage_bytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const Lanes ln = lanes_of<NP>(a, warp, lane);
    const int64_t C = (int64_t)COFF * a.head_dim;
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(smem_addr(&s.full[i]), 1);
            mbar_init(smem_addr(&s.empty[i]), ln.cols);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();  // the grad_ape finalisation may launch; it waits for this grid's end
    const int R = a.n_seg > 0 ? __ldg(a.cc + a.n_seg) : 0;
    const int R0 = a.n_seg > 0 ? __ldg(a.cc) : 0;
    const int rend = R < a.capacity ? R : a.capacity;  // padding rows carry no gradient
    GradOut o{dkv, dscore, n_tokens_arg >= 0 ? n_tokens_arg : (int64_t)__ldg(a.cu + a.n_seg)};

    float2 acc[W][NP];
#pragma unroll
    for (int k = 0; k < W; ++k)
#pragma unroll
        for (int q = 0; q < NP; ++q)
            acc[k][q] = make_float2(0.0f, 0.0f);
    const int lc = ln.lc;
    const int col = c0 + lc;

    if (warp == ncw) {
        if (lane == 0)
            produce<RATIO, COFF, true>(a, s, &tm_kv, &tm_sc, tc, c0, blockIdx.x, gridDim.x, rend, grad_out);
    } else {
        if (blockIdx.x == 0 && ln.lane == 0) {  // leading gap: tokens before the first real block
            int64_t lead = o.n_tokens;
            if (R0 < R)
                lead = map_row(R0, a.cu, a.cc, a.n_seg, RATIO).base;
            zero_range<COFF, NP>(o, C, a.head_dim, col, 0, lead);
        }
        ApeRegs<RATIO, COFF, NP> ap;
        load_ape<RATIO, COFF, NP>(a, col, ap);
        int st_used = ln.lane;
        uint32_t ph = 0;
        for (int j = ln.lane;; j += a.row_lanes, ring_next(st_used, ph, a.row_lanes, a.stages)) {
            if (blockIdx.x + j * gridDim.x >= rend)
                break;
            if (!mbar_wait(smem_addr(&s.full[st_used]), ph, a.status))
                break;
            const StageMeta m = s.meta[st_used];
            if (!m.real) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&s.empty[st_used]));
                continue;
            }
            const unsigned char *stage = s.stages + (size_t)st_used * a.stage_bytes;
            uint32_t kvw[W][NP];
            float2 e[W][NP], den[NP], num[NP];
            pool_stage<RATIO, COFF, NP, 0>(stage, a.rw, a.pcol, lc, m.first, ap, kvw, e, den, num);
            uint32_t gw[NP];
            ld_np(gw, stage + window_bytes<RATIO, COFF>(a.rw) + lc * 2);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&s.empty[st_used]));
            float2 g[NP], inv[NP], ngo[NP];
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                g[q] = bf16x2_to_f2(gw[q]);
                inv[q] = make_float2(recip_den(den[q].x), recip_den(den[q].y));
                const float2 go = mul2(g[q], mul2(num[q], inv[q]));
                ngo[q] = make_float2(-go.x, -go.y);
            }
#pragma unroll
            for (int k = 0; k < W; ++k) {
                if (COFF == 2 && k < RATIO && m.first)
                    continue;
                const int p = k / RATIO, i = k % RATIO;
                const int64_t tok = m.base + (int64_t)(p - (COFF - 1)) * RATIO + i;
                uint32_t dk[NP], dsw[NP];
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float2 pk = mul2(e[k][q], inv[q]);
                    dk[q] = f2_to_bf16x2(mul2(g[q], pk));
                    const float2 ds = mul2(pk, add2(mul2(g[q], bf16x2_to_f2(kvw[k][q])), ngo[q]));
                    dsw[q] = f2_to_bf16x2(ds);
                    acc[k][q] = add2(acc[k][q], ds);
                }
                if (tok < o.n_tokens) {
                    const int64_t gi = tok * C + (int64_t)p * a.head_dim + col;
                    st_np(dkv + gi, dk);
                    st_np(dscore + gi, dsw);
                }
            }
            if (m.last) {  // last block of its segment
                if (COFF == 2) {
                    for (int i = 0; i < RATIO; ++i) {
                        const int64_t tok = m.base + i;
                        if (tok < o.n_tokens) {
                            st_np_zero<NP>(dkv + tok * C + col);
                            st_np_zero<NP>(dscore + tok * C + col);
                        }
                    }
                }
                int64_t next = o.n_tokens;
                if (m.row + 1 < R)
                    next = map_row(m.row + 1, a.cu, a.cc, a.n_seg, RATIO).base;
                zero_range<COFF, NP>(o, C, a.head_dim, col, m.base + RATIO, next);
            }
        }
        // this thread's grad_ape sums -> shared memory [row lane][ape row][part][tile column]
        float *red = s.red + (size_t)ln.lane * RATIO * COFF * tc;
#pragma unroll
        for (int k = 0; k < W; ++k) {
            const int p = k / RATIO, i = k % RATIO;
            st_pairs(red + (i * COFF + p) * tc + lc, acc[k]);
        }
    }
    __syncthreads();

    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int rank = (int)cluster.block_rank();
    const int nrank = (int)cluster.num_blocks();
    const int n4 = RATIO * COFF * tc / 4;
    const int share = (n4 + nrank - 1) / nrank;
    const int i_lo = rank * share;
    const int i_hi = i_lo + share < n4 ? i_lo + share : n4;
    float *dst = partial + (int64_t)(blockIdx.x / nrank) * RATIO * C;
    const int lane_floats = RATIO * COFF * tc;
    for (int i4 = i_lo + (int)threadIdx.x; i4 < i_hi; i4 += blockDim.x) {
        const int rp = (i4 * 4) / tc, lcol = i4 * 4 - rp * tc;
        const int arow = rp / COFF, p = rp - arow * COFF;
        // ranks in ascending order, within a rank its row lanes in ascending order
        float4 acc4 = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(s.red, 0) + i4 * 4);
        for (int t = 1; t < nrank * a.row_lanes; ++t) {
            const int q = t / a.row_lanes, l = t - q * a.row_lanes;
            const float4 v =
                *reinterpret_cast<const float4 *>(cluster.map_shared_rank(s.red, q) + (size_t)l * lane_floats + i4 * 4);
            acc4.x = __fadd_rn(acc4.x, v.x);
            acc4.y = __fadd_rn(acc4.y, v.y);
            acc4.z = __fadd_rn(acc4.z, v.z);
            acc4.w = __fadd_rn(acc4.w, v.w);
        }
        *reinterpret_cast<float4 *>(dst + (int64_t)arow * C + (int64_t)p * a.head_dim + c0 + lcol) = acc4;
    }
    cluster.sync();
}

// Widest tile of at most max_tc columns (whole consumer warps of cpw columns) that
// divides head_dim.
int tile_cols(int head_dim, int cpw, int max_tc)
{
    for (int w = max_tc / cpw; w >= 1; --w)
        if (head_dim % (w * cpw) == 0)
            return w * cpw;
    return 0;
}

}  // namespace

bool stream_supported(bool bwd, int ratio, int coff, int head_dim)
{
    if (ratio != 4 || (coff != 1 && coff != 2) || head_dim % 64 != 0 || head_dim > 8192)
        return false;
    // head_dim 64, forward: the register-window kernel measured faster (21.3 against
    // 32.9 us at 32 x 4096 tokens, coff 2; the backward 69.0 against 51.8 us)
    return bwd || head_dim > 64;
}

StreamPlan plan_stream(bool bwd, int ratio, int coff, int head_dim, int capacity, int num_sms)
{
    StreamPlan pl;
    pl.np = head_dim % 128 == 0 ? 2 : 1;
    const int cpw = 64 * pl.np;  // columns per consumer warp
    // tiles of up to 512 columns; 256 for the own-block backward (coff 1, head_dim
    // 512: 58.3 -> 55.6 us at 16 x 4096 tokens; the forward and the coff-2
    // backward measured slower with the narrower tile)
    pl.tc = tile_cols(head_dim, cpw, bwd && coff == 1 ? 256 : 512);
    pl.tiles = head_dim / pl.tc;
    // Up to four consumer warps per block: tiles of one or two warps take several
    // rows at once (more would leave the block's one producer behind).
    const int cols = pl.tc / cpw;
    pl.row_lanes = cols == 1 ? kRowLanes1 : cols == 2 ? 2 : 1;
    const int warps = cols * pl.row_lanes;
    pl.threads = (warps + 1) * 32;
    // One column tile: whole token rows when the head is narrow enough (coff 2
    // then also stages the unused half, in exchange for 8x fewer copies).  Other
    // tiles: one TMA box per array and part, 2-D for tiles of at most 256 columns
    // (head_dim 640, coff 1: forward 34.0 -> 28.7 us against one bulk copy per
    // token; a single coff-2 tile of 128 or 256 columns measured no faster with
    // boxes than with whole rows), 3-D for wider coff-2 tiles that are multiples of
    // 256 (the 512-column tiles of head_dim 512: four copies a row in place of
    // sixteen per-token copies, whose issue bounds the producer).
    pl.whole = pl.tiles == 1 && (coff == 1 || head_dim <= kWholeMaxD);
    pl.tma = pl.whole ? 0 : pl.tc <= kChunkCols ? 1 : (coff == 2 && pl.tc % kChunkCols == 0) ? 2 : 0;
    const int rw = pl.whole ? coff * head_dim : pl.tc;
    const int win = 2 * coff * ratio * rw * 2;
    pl.stage_bytes = ((bwd ? win + pl.tc * 2 : win) + 127) / 128 * 128;
    // ring bytes in proportion to the consumer warps (the budget is for four)
    const int budget = (bwd ? kBwdBudget : kFwdBudget) / 4 * warps;
    int per_lane = budget / pl.stage_bytes / pl.row_lanes;
    per_lane = per_lane < 2 ? 2 : (per_lane > 8 ? 8 : per_lane);
    pl.stages = per_lane * pl.row_lanes;  // a multiple of the row lanes
    pl.red_bytes = bwd ? (size_t)pl.row_lanes * ratio * coff * pl.tc * sizeof(float) : 0;
    pl.smem = smem_bytes(pl.stages, pl.stage_bytes, pl.red_bytes);
    pl.cluster = bwd ? kBwdCluster : 1;
    pl.num_sms = num_sms;
    (void)capacity;
    return pl;
}

namespace {

template <int RATIO, int COFF, int NP, int RW = 0>
cudaError_t blocks_for(const StreamPlan &pl, bool bwd, int rows, int *out)
{
    const void *fn = bwd ? reinterpret_cast<const void *>(bwd_stream_kernel<RATIO, COFF, NP>)
                         : reinterpret_cast<const void *>(fwd_stream_kernel<RATIO, COFF, NP, RW>);
    int resident = 0;
    cudaError_t e = resident_blocks(fn, pl.threads, pl.smem, pl.cluster, &resident);
    if (e != cudaSuccess)
        return e;
    int blocks = (resident > 0 ? resident : 1) / pl.tiles;
    blocks = blocks / pl.cluster * pl.cluster;
    if (blocks < 1)
        blocks = 1;
    if (blocks > rows)
        blocks = rows > 0 ? rows : 1;
    blocks = (blocks + pl.cluster - 1) / pl.cluster * pl.cluster;
    *out = blocks;
    return cudaSuccess;
}

StreamArgs stream_args(const void *kv, const void *score, const float *ape, const int32_t *cu, const int32_t *cc,
                       int n_seg, int coff, int head_dim, int capacity, const StreamPlan &pl, unsigned *status)
{
    return StreamArgs{static_cast<const uint16_t *>(kv), static_cast<const uint16_t *>(score), ape, cu, cc, n_seg,
                      head_dim, capacity, pl.stages, pl.stage_bytes, status, pl.tc, pl.row_lanes,
                      pl.whole ? coff * head_dim : pl.tc, pl.whole ? head_dim : 0, pl.tma};
}

template <int RATIO>
cudaError_t stream_maps(const StreamPlan &pl, const void *kv, const void *score, int64_t C, CUtensorMap *mk,
                        CUtensorMap *ms)
{
    if (pl.tma == 2) {
        cudaError_t e = make_tensor_map_3d(mk, kv, C, kChunkCols, pl.tc / kChunkCols, RATIO);
        if (e == cudaSuccess)
            e = make_tensor_map_3d(ms, score, C, kChunkCols, pl.tc / kChunkCols, RATIO);
        return e;
    }
    if (!pl.tma)
        return cudaSuccess;
    cudaError_t e = make_tensor_map_2d(mk, kv, C, pl.tc, RATIO);
    if (e == cudaSuccess)
        e = make_tensor_map_2d(ms, score, C, pl.tc, RATIO);
    return e;
}

template <int RATIO, int COFF, int NP, int RW = 0>
cudaError_t launch_fwd_stream_t(const FwdParams &p, const StreamPlan &pl, unsigned *status, cudaStream_t st)
{
    const StreamArgs a = stream_args(p.kv, p.score, p.ape, p.cu_seqlens, p.cu_seqlens_comp, p.n_seg, p.coff,
                                     p.head_dim, p.capacity, pl, status);
    CUtensorMap mk{}, ms{};
    cudaError_t e = stream_maps<RATIO>(pl, p.kv, p.score, (int64_t)p.coff * p.head_dim, &mk, &ms);
    if (e != cudaSuccess)
        return e;
    int blocks = 0;
    e = blocks_for<RATIO, COFF, NP, RW>(pl, false, p.capacity, &blocks);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, pl.tiles, 1);
    cfg.blockDim = dim3(pl.threads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fwd_stream_kernel<RATIO, COFF, NP, RW>, a, mk, ms, static_cast<uint16_t *>(p.out));
}

// The exact grid width of the backward: the resident blocks, at most the upper
// bound stream_bwd_partials sizes the workspace for.
template <int RATIO, int COFF, int NP>
cudaError_t stream_bwd_blocks_t(const StreamPlan &pl, int capacity, int *out)
{
    int blocks = 0;
    cudaError_t e = blocks_for<RATIO, COFF, NP>(pl, true, capacity, &blocks);
    if (e != cudaSuccess)
        return e;
    const int max_blocks = stream_bwd_partials(pl, capacity) * pl.cluster;
    *out = blocks > max_blocks ? max_blocks : blocks;
    return cudaSuccess;
}

template <int RATIO, int COFF, int NP>
cudaError_t launch_bwd_stream_t(const BwdParams &p, const StreamPlan &pl, float *partial, unsigned *status,
                                cudaStream_t st)
{
    const StreamArgs a = stream_args(p.kv, p.score, p.ape, p.cu_seqlens, p.cu_seqlens_comp, p.n_seg, p.coff,
                                     p.head_dim, p.capacity, pl, status);
    CUtensorMap mk{}, ms{};
    cudaError_t e = stream_maps<RATIO>(pl, p.kv, p.score, (int64_t)p.coff * p.head_dim, &mk, &ms);
    if (e != cudaSuccess)
        return e;
    int blocks = 0;
    e = stream_bwd_blocks_t<RATIO, COFF, NP>(pl, p.capacity, &blocks);
    if (e != cudaSuccess)
        return e;
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
    e = cudaLaunchKernelEx(&cfg, bwd_stream_kernel<RATIO, COFF, NP>, a, mk, ms, p.n_tokens,
                           static_cast<const uint16_t *>(p.grad_out), static_cast<uint16_t *>(p.dkv),
                           static_cast<uint16_t *>(p.dscore), partial);
    if (e != cudaSuccess)
        return e;
    return launch_dape_finalize(partial, blocks / pl.cluster, (int64_t)RATIO * COFF * p.head_dim, p.dape, st);
}

}  // namespace

// The kernel instance of a plan: ratio 4, the window form, the column pairs per
// thread.
#define CSA_STREAM_DISPATCH(FN, ...)                                                        \
    do {                                                                                    \
        if (ratio != 4 || (coff != 1 && coff != 2) || (pl.np != 1 && pl.np != 2))           \
            return cudaErrorInvalidValue;                                                   \
        if (coff == 2)                                                                      \
            return pl.np == 2 ? FN<4, 2, 2>(__VA_ARGS__) : FN<4, 2, 1>(__VA_ARGS__);        \
        return pl.np == 2 ? FN<4, 1, 2>(__VA_ARGS__) : FN<4, 1, 1>(__VA_ARGS__);            \
    } while (0)

cudaError_t launch_fwd_stream(const FwdParams &p, const StreamPlan &pl, unsigned *status, cudaStream_t st)
{
    const int ratio = p.ratio, coff = p.coff;
    const int rw = pl.whole ? coff * p.head_dim : pl.tc;  // the staged row width
    const bool part_col0 = !pl.whole || coff == 1;        // every part at column 0 of its staged rows
    if (ratio == 4 && pl.np == 2 && rw == 512 && part_col0)
        return coff == 2 ? launch_fwd_stream_t<4, 2, 2, 512>(p, pl, status, st)
                         : launch_fwd_stream_t<4, 1, 2, 512>(p, pl, status, st);
    CSA_STREAM_DISPATCH(launch_fwd_stream_t, p, pl, status, st);
}

// Upper bound of grad_ape partials (cluster count) for the workspace size.
int stream_bwd_partials(const StreamPlan &pl, int capacity)
{
    const int rows = capacity > 0 ? capacity : 1;
    int blocks = 8 * pl.num_sms / pl.tiles;  // never more than 8 resident per SM
    if (blocks > rows)
        blocks = rows;
    blocks = (blocks + pl.cluster - 1) / pl.cluster * pl.cluster;
    return blocks / pl.cluster;
}

cudaError_t stream_bwd_blocks(int ratio, int coff, const StreamPlan &pl, int capacity, int *blocks)
{
    CSA_STREAM_DISPATCH(stream_bwd_blocks_t, pl, capacity, blocks);
}

cudaError_t launch_bwd_stream(const BwdParams &p, const StreamPlan &pl, float *partial, unsigned *status,
                              cudaStream_t st)
{
    const int ratio = p.ratio, coff = p.coff;
    CSA_STREAM_DISPATCH(launch_bwd_stream_t, p, pl, partial, status, st);
}

#undef CSA_STREAM_DISPATCH

}  // namespace csa
