/*
 * csa.h -- C ABI of libcsa, the GB300 (sm_103a) CSA/HCA fused Compressor.
 *
 * The operation ("CSA Fused Compressor", cuDNN frontend docs, section Semantics):
 * for each THD segment s = [cu_seqlens[s], cu_seqlens[s+1]) and each of its
 * floor(len/ratio) blocks b of ratio tokens (the segment's tail tokens are
 * dropped), output row r = cu_seqlens_comp[s] + b is
 *
 *     out[r, j] = sum_k kv[w(b,k), c(k,j)] * softmax_k(score[w(b,k), c(k,j)]
 *                                                      + ape[k % ratio, c(k,j)])
 *
 * with, for coff == 2 (overlapping form, window 2*ratio): k < ratio -> the previous
 * block's token, column c = j (first half), invalid for a segment's first block;
 * k >= ratio -> the own block's token, column c = head_dim + j (second half).
 * For coff == 1 (own-block form, window ratio): the own block's token, column j.
 * Rows r in [cu_seqlens_comp[n_seg], capacity) are padding rows computed as a
 * first block starting at token 0; the backward ignores grad_out on them.
 * Arithmetic is fp32 with a single final bf16 rounding (section Numerics).
 *
 * Layouts (THD packed, row-major, contiguous; section API Usage):
 *   kv, score      bf16  [n_tokens, coff*head_dim]
 *   ape            fp32  [ratio, coff*head_dim]
 *   cu_seqlens     int32 [n_seg + 1]  token offsets, nondecreasing
 *   cu_seqlens_comp int32 [n_seg + 1] row offsets: cu_seqlens_comp[0] == 0 and
 *                  cu_seqlens_comp[s+1] - cu_seqlens_comp[s] == floor(len_s / ratio)
 *   out, grad_out  bf16  [capacity, head_dim]
 *   dkv, dscore    bf16  [n_tokens, coff*head_dim]
 *   dape           fp32  [ratio, coff*head_dim]
 * bf16 tensors are passed as raw 16-bit patterns (void*).
 *
 * Ownership and memory: every pointer is a device pointer on the current CUDA
 * device, owned by the caller, valid until the stream has finished the call's
 * work.  Tensor bases must be 16-byte aligned (the int32 offsets 4-byte aligned);
 * this is checked on every call.  The library keeps no per-call state.  `stream`
 * is a cudaStream_t (NULL = the legacy default stream).  Calls are asynchronous:
 * no call synchronises the device or reads device memory on the host.
 *
 * Launch order: every kernel is launched as a programmatic dependent of its stream
 * predecessor (CUDA programmatic dependent launch) and waits for that predecessor
 * to complete before it reads or writes any global memory, so stream order holds
 * after any kind of predecessor.  Its blocks may become resident early, while the
 * predecessor drains.  A caller's own kernel launched with the programmatic
 * stream-serialization attribute right after a call must likewise wait
 * (griddepcontrol.wait / cudaGridDependencySynchronize) before using the call's
 * outputs; plain launches need nothing.
 *
 * Trusted device contents: the offsets in cu_seqlens / cu_seqlens_comp are not
 * validated (that would need a device-to-host read).  The caller guarantees the
 * relations above, capacity >= cu_seqlens_comp[n_seg], and that kv / score hold at
 * least cu_seqlens[n_seg] rows (and at least ratio rows when capacity > 0).
 *
 * Errors: every entry point returns CSA_OK (0) or a csa_status below.  A failed
 * validation launches nothing and touches no output.  No C++ exception crosses
 * the ABI.  csa_last_error_message() gives a thread-local description of the
 * calling thread's last non-OK return.
 *
 * Supported set (csa_check_support): coff in {1, 2}; ratio == 128 with head_dim a
 * multiple of 64 in [64, 8192]; every other ratio in [1, 128] with head_dim a
 * multiple of 8 in [8, 8192].  Numerics per window (section Numerics): a window of
 * more than 64 positions with head_dim a multiple of 64 -- ratio 128, and ratios
 * 33-127 with coff 2 or 65-127 with coff 1 -- is summed in fixed chunks with the
 * hardware exp2, the page's ratio-128 evaluation (deterministic, equal to the
 * sequential evaluation within final-bf16 rounding tolerance); every other shape
 * (ratio 4 on its own kernels, the rest on the generic ones) computes each window
 * in ascending position order with the library's exp, bitwise equal to a plain
 * sequential fp32 evaluation.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stdint.h>

#if defined(__GNUC__)
#define CSA_API __attribute__((visibility("default")))
#else
#define CSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum csa_status {
    CSA_OK = 0,
    CSA_ERR_INVALID_VALUE = 1,   /* null pointer, negative size, coff not in {1,2}, ...   */
    CSA_ERR_UNSUPPORTED = 2,     /* (ratio, coff, head_dim) outside the kernel set        */
    CSA_ERR_MISALIGNED = 3,      /* a tensor base not 16-byte (offsets: 4-byte) aligned   */
    CSA_ERR_TOO_LARGE = 4,       /* a flat element offset would not fit in int32          */
    CSA_ERR_CUDA = 5,            /* a CUDA runtime call or kernel launch failed           */
    CSA_ERR_OUT_OF_MEMORY = 6,   /* the backward's stream-ordered workspace allocation    */
    CSA_ERR_DEVICE_TIMEOUT = 7   /* a bounded device-side wait expired (see below)        */
} csa_status;

/*
 * Forward pass ("CSA Fused Compressor", sections Semantics and API Usage: the
 * forward wrapper with an explicit static total_comp = capacity).
 *
 * Writes out[0, capacity) x [0, head_dim) in full, padding rows included.
 * Reads kv / score rows of real blocks (and their previous blocks for coff == 2)
 * and rows [0, ratio) when capacity exceeds the real row count.
 * capacity == 0: nothing is launched and CSA_OK is returned; the tensor pointers
 * may then be NULL.  Bitwise deterministic.
 */
CSA_API int csa_compress_fwd(const void *kv, const void *score, const float *ape,
                     const int32_t *cu_seqlens, const int32_t *cu_seqlens_comp, int32_t n_seg,
                     int32_t ratio, int32_t coff, int32_t head_dim, int32_t capacity,
                     void *out, void *stream);

/*
 * Backward pass ("CSA Fused Compressor", Semantics: the chain rule through the
 * pooling; Class API: gradient buffers may be uninitialised because every slot
 * is written, never-consumed slots with exact zeros).
 *
 * n_tokens: rows of kv / score / dkv / dscore.  If n_tokens < 0 the library uses
 * cu_seqlens[n_seg], read on the device (token padding rows past it are then left
 * untouched).  Writes:
 *   dkv, dscore  all of [0, n_tokens) x [0, coff*head_dim): the gradient at every
 *                slot a real row reads, +0 at every other slot (segment tails,
 *                the last block's first-half columns when coff == 2, segments
 *                shorter than ratio, tokens outside the segments);
 *   dape         overwritten (not accumulated) with the sum over real rows, formed
 *                as fixed-order partial sums: no atomics, bitwise reproducible
 *                run to run.  The grouping of that sum for a given shape and
 *                device is reported by csa_grad_ape_order (below).
 * grad_out rows at or past cu_seqlens_comp[n_seg] are ignored.
 * Scratch: grad_ape partials (a few MB at most) come from a library-owned,
 * stream-ordered memory pool on the current device, allocated and released in
 * stream order inside the call.  capacity == 0 still writes dkv / dscore zeros
 * and dape = 0.  Errors as above; CSA_ERR_OUT_OF_MEMORY if the workspace cannot
 * be allocated.
 */
CSA_API int csa_compress_bwd(const void *kv, const void *score, const float *ape,
                     const int32_t *cu_seqlens, const int32_t *cu_seqlens_comp, int32_t n_seg,
                     int32_t ratio, int32_t coff, int32_t head_dim, int32_t capacity,
                     int64_t n_tokens, const void *grad_out, void *dkv, void *dscore,
                     float *dape, void *stream);

/*
 * Backward pass that allocates nothing.  The page has no counterpart of this call:
 * it is an addition of this library for callers that cannot allocate device
 * memory inside the call -- a framework that has reserved all of HBM for its own
 * arena up front, a real-time loop in which growing or trimming a memory pool
 * could block, a plug-in that may not use the CUDA allocator.
 *
 * Same arguments, results and errors as csa_compress_bwd (bitwise the same
 * outputs, but see below for the chunked windows' grad_ape), except that the
 * grad_ape partial sums go to a fixed 6 MiB array in the library's device code
 * instead of the library's memory pool.  That array
 * occupies 6 MiB on every GPU that loads the library, until the process exits.
 * Where the regular backward's grid would need more partial storage than the
 * array holds, the chunked windows (ratio 128, and other ratios with more than 64
 * window positions) run with fewer row blocks (same grad_kv / grad_score bits;
 * grad_ape summed in another fixed grouping); a shape whose single partial
 * does not fit is rejected with CSA_ERR_TOO_LARGE before anything is launched (on
 * a 152-SM GB300 every shape fits except ratio 128 with coff 2 and head_dim above
 * 6144, and other ratios with ratio * coff * head_dim above 1572864).  No
 * cudaMalloc, cudaFree or other allocating call is made.
 *
 * Every call on a device shares the array and leaves its contents behind; each
 * call writes all it reads, so nothing needs clearing, but calls that overlap on
 * the GPU (different streams or host threads) race: order them.  The first call
 * on a device (with that device current) looks up the array's device address;
 * make that first call before any stream capture.  A first call whose set-up
 * fails returns CSA_ERR_CUDA and leaves nothing behind: the next call tries the
 * set-up again.  Bounded device waits that expire in this call's kernels are
 * recorded in the same per-device status word as those of every other call, so
 * csa_device_status() reports them (CSA_ERR_DEVICE_TIMEOUT).  The grad_ape
 * grouping is csa_grad_ape_order's for every shape outside the chunked windows.
 */
CSA_API int csa_compress_bwd_noalloc(const void *kv, const void *score, const float *ape,
                             const int32_t *cu_seqlens, const int32_t *cu_seqlens_comp, int32_t n_seg,
                             int32_t ratio, int32_t coff, int32_t head_dim, int32_t capacity,
                             int64_t n_tokens, const void *grad_out, void *dkv, void *dscore,
                             float *dape, void *stream);

/*
 * Host-only support check ("CSA Fused Compressor", section Support surface):
 * CSA_OK if (ratio, coff, head_dim) has a kernel and the sizes fit the int32
 * flat-offset bounds (n_tokens * coff * head_dim < 2^31, capacity * head_dim <
 * 2^31); capacity > 0 requires n_tokens >= ratio.  n_tokens < 0 skips the
 * checks that need it.  Makes no CUDA call.
 */
CSA_API int csa_check_support(int32_t ratio, int32_t coff, int32_t head_dim, int64_t n_tokens,
                      int32_t capacity);

/* Static string naming a status code.  Never NULL. */
CSA_API const char *csa_status_string(int status);

/* Thread-local text of the calling thread's last non-OK return ("" if none). */
CSA_API const char *csa_last_error_message(void);

/*
 * How the backward groups the grad_ape sum (the pages fix only that grad_ape is
 * the sum over real rows of ds and, in this library, that it is deterministic; the
 * grouping is the implementation's choice and depends on the shape and the
 * device).  Host-side: launches nothing, reads no device memory and allocates
 * nothing, but queries the current device's SM count and the kernels' occupancy.
 *
 * kind == CSA_GRAD_APE_ROW_BLOCKS (every ratio but 128), with R = the real row
 * count (cu_seqlens_comp[n_seg], at most capacity):
 *   1. Row blocks.  strided != 0: block b (0 <= b < blocks) takes the rows
 *      b, b + blocks, b + 2*blocks, ... below R.  strided == 0: block b takes the
 *      rows [b*rows_per_block, (b+1)*rows_per_block) below R.
 *   2. Lanes.  The i-th row of a block (i = 0, 1, ... in ascending row order) goes
 *      to the block's lane i % lanes.  Each lane sums, in fp32 from +0, the ds of
 *      its rows in ascending row order: one leaf per (block, lane).
 *   3. Partials.  Partial q takes the blocks [q*cluster, (q+1)*cluster).  flat != 0:
 *      the partial is the left-to-right fp32 sum of its leaves in ascending
 *      (block, lane) order, starting with the first leaf itself.  flat == 0: each
 *      block first sums its lanes that way, then the partial sums its blocks that
 *      way.
 *   4. Final sum.  The partials are cut into final_ranges (32) contiguous ranges,
 *      range t = [t*partials/32, (t+1)*partials/32) in integer division, each summed
 *      from +0 in ascending order; then the 32 range sums are added in pairs
 *      (t, t^1), then (t, t^2), (t, t^4), (t, t^8), (t, t^16): a balanced binary
 *      tree over the ranges in order.
 * kind == CSA_GRAD_APE_CHUNKED (the chunked windows above: ratio 128, and other
 * ratios with more than 64 window positions and head_dim a multiple of 64): every
 * sum of those kernels is taken in fixed chunks (section ratio=128 of the page);
 * grad_ape is deterministic but has no bitwise contract.  blocks, partials and
 * cluster describe the grid.
 *
 * Errors: those of csa_check_support for the shape, CSA_ERR_INVALID_VALUE for a
 * NULL out, CSA_ERR_CUDA if the device cannot be queried.
 */
typedef enum csa_grad_ape_kind {
    CSA_GRAD_APE_ROW_BLOCKS = 0,
    CSA_GRAD_APE_CHUNKED = 1
} csa_grad_ape_kind;

typedef struct csa_grad_ape_grouping {
    int32_t kind;            /* csa_grad_ape_kind                                       */
    int32_t strided;         /* rows of block b: strided (b + i*blocks) or contiguous   */
    int32_t blocks;          /* row blocks                                              */
    int32_t rows_per_block;  /* contiguous row blocks: rows per block                   */
    int32_t lanes;           /* lanes per block                                         */
    int32_t cluster;         /* row blocks per partial                                  */
    int32_t flat;            /* 1: a partial sums its (block, lane) leaves in one pass  */
    int32_t partials;        /* blocks / cluster                                        */
    int32_t final_ranges;    /* 32                                                      */
} csa_grad_ape_grouping;

CSA_API int csa_grad_ape_order(int32_t ratio, int32_t coff, int32_t head_dim, int32_t capacity,
                               csa_grad_ape_grouping *out);

/*
 * Device-side status of the current device, for diagnostics.  Kernels that wait
 * on shared-memory barriers (the bulk-copy pipelines) bound every wait in time;
 * on expiry they record a code in a per-device status word, stop, and exit
 * normally, so that a wait that can never complete gives an error instead of a
 * hung GPU.  One word per device serves every entry point (csa_compress_fwd,
 * csa_compress_bwd, csa_compress_bwd_noalloc, csa_selftest_bounded_wait); it is
 * part of the library's device code, so reading it allocates nothing.  This call
 * SYNCHRONISES with the device (it reads the word back), returns CSA_OK if no
 * kernel recorded anything and CSA_ERR_DEVICE_TIMEOUT otherwise; clear != 0
 * resets the word.  Not meant for the hot path.
 */
CSA_API int csa_device_status(int clear);

/*
 * Self-test of the bounded waits (failure detection without a GPU fault): launches
 * one small kernel on `stream` that waits on a shared-memory barrier phase nothing
 * completes, giving up after limit_ns (at most 1e9) and recording a timeout in the
 * device status word exactly as the pipelined kernels would.  The kernel then
 * exits normally and the context stays usable; csa_device_status() afterwards
 * returns CSA_ERR_DEVICE_TIMEOUT (clear it with csa_device_status(1)).
 */
CSA_API int csa_selftest_bounded_wait(int64_t limit_ns, void *stream);

/*
 * Self-test of the reciprocal the kernels take of each softmax denominator (the
 * pages have no counterpart: they only fix fp32 arithmetic).  Writes, for i < n,
 * out[i] = the library's 1/d[i]; that routine is correctly rounded for d in
 * [2^-8, 2^8], which holds every denominator (NaN in, NaN out), and is
 * unspecified elsewhere.  d and out are device pointers to n floats, 4-byte
 * aligned, not overlapping; n >= 0 (n == 0 launches nothing).  Asynchronous on
 * `stream`.  Returns CSA_ERR_INVALID_VALUE for a NULL pointer with n > 0 or for
 * n < 0, CSA_ERR_CUDA when the launch fails.
 */
CSA_API int csa_selftest_reciprocal(const float *d, float *out, int64_t n, void *stream);

/* Library version as an integer: major * 10000 + minor * 100 + patch. */
CSA_API int csa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
