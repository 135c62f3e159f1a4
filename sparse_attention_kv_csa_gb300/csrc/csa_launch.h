// Internal interface between the C-ABI entry points (csa_api.cu) and the kernel
// files.  Not installed, not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

// Launch attribute that lets a kernel start while its stream predecessor finishes
// (the kernel itself waits for it before touching memory: pdl_wait()).
inline cudaLaunchAttribute pdl_attribute()
{
    cudaLaunchAttribute a = {};
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

struct FwdParams {
    const void *kv;
    const void *score;
    const float *ape;
    const int32_t *cu_seqlens;
    const int32_t *cu_seqlens_comp;
    int n_seg;
    int ratio;
    int coff;
    int head_dim;
    int capacity;
    void *out;
};

struct BwdParams {
    const void *kv;
    const void *score;
    const float *ape;
    const int32_t *cu_seqlens;
    const int32_t *cu_seqlens_comp;
    int n_seg;
    int ratio;
    int coff;
    int head_dim;
    int capacity;
    int64_t n_tokens;  // -1: cu_seqlens[n_seg], read on the device
    const void *grad_out;
    void *dkv;
    void *dscore;
    float *dape;
};

// Small-ratio family (window in registers).
struct SmallBwdPlan {
    int threads_x;       // threads along the columns (4 columns each)
    int col_slices;      // blocks along the columns (gridDim.y)
    int lanes;           // rows processed side by side in a block
    int cluster;         // blocks per thread-block cluster (partials merged in DSMEM)
    int blocks;          // gridDim.x, a multiple of cluster
    int partials;        // grad_ape partials = blocks / cluster
    int rows_per_block;  // contiguous output rows per block
    size_t smem;         // bytes of dynamic shared memory (lane and cluster merge)
    int64_t partial_floats;
};

cudaError_t launch_fwd_small(const FwdParams &p, int num_sms, cudaStream_t st);

// grad_ape = fixed-order sum of n_partials partials of n floats each.
cudaError_t launch_dape_finalize(const float *partial, int n_partials, int64_t n, float *dape, cudaStream_t st);

// Streamed family (bulk-copy pipeline through shared memory), ratio 4,
// head_dim % 64 == 0.
struct StreamPlan {
    int np;              // fp32 column pairs per consumer thread: 2 (head_dim % 128 == 0) or 1
    int tc;              // columns per thread block tile (consumer threads x 2 np)
    int tiles;           // head_dim / tc (gridDim.y)
    int row_lanes;       // rows in flight per block (tc / 128 column warps each)
    bool whole;          // stage whole token rows (one column tile)
    int tma;             // stage the tile with one TMA box per array and part: 0 no, 1 2-D (tc <= 256),
                         // 2 3-D (coff 2, tc a multiple of 256 above it)
    int threads;         // consumer warps + one producer warp, x 32
    int stage_bytes;     // bytes per ring stage
    int stages;          // ring depth
    size_t red_bytes;    // backward: grad_ape staging in shared memory
    size_t smem;         // dynamic shared memory per block
    int cluster;         // backward: blocks per cluster
    int num_sms;
};

bool stream_supported(bool bwd, int ratio, int coff, int head_dim);
StreamPlan plan_stream(bool bwd, int ratio, int coff, int head_dim, int capacity, int num_sms);
int stream_bwd_partials(const StreamPlan &pl, int capacity);
cudaError_t launch_fwd_stream(const FwdParams &p, const StreamPlan &pl, unsigned *status, cudaStream_t st);
cudaError_t launch_bwd_stream(const BwdParams &p, const StreamPlan &pl, float *partial, unsigned *status,
                              cudaStream_t st);
// The exact grid width launch_bwd_stream uses (partials = blocks / pl.cluster).
cudaError_t stream_bwd_blocks(int ratio, int coff, const StreamPlan &pl, int capacity, int *blocks);

// Chunked family (windows of more than 64 positions: ratio 128, and ratios 33-127
// with coff 2 / 65-127 with coff 1; 2-D TMA staging), head_dim % 64 == 0.
bool chunked_supported(int ratio, int coff, int head_dim);
cudaError_t launch_fwd_chunked(const FwdParams &p, unsigned *status, cudaStream_t st);
// grid width of the backward and the number of grad_ape partials it writes
cudaError_t chunked_bwd_partials(int ratio, int coff, int head_dim, int capacity, int *partials, int *blocks);
cudaError_t launch_bwd_chunked(const BwdParams &p, float *partial, int blocks, unsigned *status, cudaStream_t st);

// Every other shape of a ratio other than 4 and 128 (windows of up to 64 positions
// staged in shared memory, head_dim % 64 == 0; else a thread per column pair walking
// the window from global memory), head_dim % 8 == 0.
struct GenericPlan {
    int col_tiles;          // blocks along the columns (16 groups of 4 columns each)
    int lanes;              // rows walked side by side in a block (blockDim.y)
    int groups;             // row groups = gridDim.x = grad_ape partials
    int rows_per_group;     // contiguous output rows per group
    size_t smem;            // backward shared memory (grad_ape slots)
    int64_t partial_floats; // workspace floats
    int num_sms;
    int staged_blocks;      // > 0: the shared-memory staged kernels, this many row blocks (= partials)
    int staged_lanes;       // staged kernels: consumer warps per block (row lanes)
};
bool generic_supported(int ratio, int coff, int head_dim);
cudaError_t plan_generic(int ratio, int coff, int head_dim, int capacity, int num_sms, GenericPlan *pl);
cudaError_t launch_fwd_generic(const FwdParams &p, unsigned *status, int num_sms, cudaStream_t st);
cudaError_t launch_bwd_generic(const BwdParams &p, const GenericPlan &pl, float *partial, unsigned *status,
                               cudaStream_t st);

// Raises a kernel's dynamic shared-memory limit (a per-function attribute shared
// by all its launch configurations) to the current device's maximum, once per
// (device, kernel).
cudaError_t allow_max_smem(const void *fn);

// Blocks of a kernel configuration resident on the whole current device (blocks of
// `cluster`-block clusters: whole clusters only), with allow_max_smem applied to the
// kernel first; cached per (device, kernel, threads, shared memory, cluster).
cudaError_t resident_blocks(const void *fn, int threads, size_t smem, int cluster, int *resident);

// Tiled TMA map of a [rows, C] bf16 row-major tensor at ptr with [box_rows x
// box_cols] boxes (no swizzle, 256-byte L2 promotion).
cudaError_t make_tensor_map_2d(CUtensorMap *m, const void *ptr, int64_t C, int box_cols, int box_rows);
cudaError_t make_tensor_map_3d(CUtensorMap *m, const void *ptr, int64_t C, int chunk_cols, int chunks, int box_rows);
cudaError_t make_tensor_map_parts(CUtensorMap *m, const void *ptr, int64_t C, int box_cols, int ratio, int head_dim);

// The backward's kernel family and plan for one shape on the current device: one
// computation shared by csa_compress_bwd, csa_compress_bwd_noalloc and
// csa_grad_ape_order, so that the reported grad_ape grouping is the launched one.
enum BwdFamily { kBwdChunked = 0, kBwdGeneric = 1, kBwdStream = 2, kBwdSmall = 3 };
struct BwdPlan {
    BwdFamily family;
    StreamPlan sp;
    SmallBwdPlan pl;
    GenericPlan gp;
    int ch_blocks;       // chunked: grid width (row blocks per column tile)
    int ch_partials;     // chunked: grad_ape partials
    int stream_blocks;   // streamed: exact grid width (row blocks per column tile)
    int64_t floats;      // grad_ape partial floats the launch needs (an upper bound)
};
cudaError_t plan_bwd(int ratio, int coff, int head_dim, int capacity, int num_sms, BwdPlan *out);
cudaError_t launch_bwd(const BwdParams &p, const BwdPlan &plan, float *partial, unsigned *status,
                       cudaStream_t st);

// Per-device status word of the bounded waits: a word of the library's own device
// memory (zero when the device code is loaded), looked up once per device.  No
// allocation.
cudaError_t status_word(unsigned **word);

// Records a status and the thread-local message returned by csa_last_error_message().
int fail_status(int status, const char *fmt, ...);
SmallBwdPlan plan_bwd_small(int ratio, int coff, int head_dim, int capacity, int num_sms);
cudaError_t launch_bwd_small(const BwdParams &p, const SmallBwdPlan &pl, float *partial, cudaStream_t st);

}  // namespace csa
