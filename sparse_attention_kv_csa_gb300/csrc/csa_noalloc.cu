// csa_compress_bwd_noalloc: the backward pass for callers that cannot allocate.
//
// The regular backward takes its grad_ape partial sums from a stream-ordered
// memory pool.  Some callers must not allocate device memory inside the call:
// a host framework that has handed all of HBM to its own arena before the first
// step, a real-time loop in which growing or trimming a pool could block, or a
// plug-in that is not allowed to touch the CUDA allocator at all.  This entry
// point runs the same kernels with the scratch in a fixed array of this file
// (kScratchFloats floats, 6 MiB) that lives in every GPU's memory from the moment
// the library's device code is loaded until the process exits.  It calls no
// cudaMalloc / cudaFree or allocating routine.
//
// Sharing: every call on a device uses the same array and leaves the last call's
// partials in it.  Nothing needs to start at zero: each call writes every partial
// it later reads.  Calls whose work overlaps on the GPU (two streams, or two host
// threads) race on the array; the caller must order them.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address (cudaGetSymbolAddress) and the SM count.  That first call
// should come before any stream capture.
#include <mutex>

#include "csa.h"
#include "csa_launch.h"

// Scratch for the grad_ape partials: 1572864 floats = 6 MiB per GPU.  On a
// 152-SM GB300 every shape fits except ratio 128 with coff 2 and head_dim above
// 6144, and other ratios with ratio * coff * head_dim above 1572864, which are
// rejected.  Ratio 128 runs with fewer row blocks than the regular backward
// where a full grid's partials would not fit (coff 2: 12 per column tile at
// head_dim 512 instead of 19).
static constexpr size_t kScratchFloats = 1536u * 1024u;
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

namespace {

// Per-device set-up: the array's device address and the SM count.  Marked done
// only when it succeeds, so that a failed first call (say, one made during stream
// capture) is retried by the next call instead of disabling the entry point.
struct NoAllocDevice {
    bool ready = false;
    float *scratch = nullptr;
    int num_sms = 0;
};
constexpr int kMaxDevices = 64;
NoAllocDevice g_na[kMaxDevices];
std::mutex g_na_mu;

cudaError_t noalloc_device(NoAllocDevice *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_na_mu);
    NoAllocDevice &d = g_na[dev];
    if (!d.ready) {
        // The array's name is a host-side stand-in: ask the runtime for its device
        // address on this (current) device.
        float *scratch = nullptr;
        int num_sms = 0;
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&scratch), g_noalloc_scratch);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        d.scratch = scratch;
        d.num_sms = num_sms;
        d.ready = true;
    }
    *out = d;
    return cudaSuccess;
}

int check_ptr(const void *p, const char *name, uintptr_t align)
{
    if (!p)
        return csa::fail_status(CSA_ERR_INVALID_VALUE, "%s is NULL", name);
    if ((reinterpret_cast<uintptr_t>(p) & (align - 1)) != 0)
        return csa::fail_status(CSA_ERR_MISALIGNED, "%s = %p is not %d-byte aligned", name, p, (int)align);
    return CSA_OK;
}

}  // namespace

extern "C" int csa_compress_bwd_noalloc(const void *kv, const void *score, const float *ape,
                                        const int32_t *cu_seqlens, const int32_t *cu_seqlens_comp, int32_t n_seg,
                                        int32_t ratio, int32_t coff, int32_t head_dim, int32_t capacity,
                                        int64_t n_tokens, const void *grad_out, void *dkv, void *dscore,
                                        float *dape, void *stream)
{
    if (n_seg < 0)
        return csa::fail_status(CSA_ERR_INVALID_VALUE, "n_seg must be >= 0 (got %d)", n_seg);
    int rc = csa_check_support(ratio, coff, head_dim, n_tokens, capacity);
    if (rc != CSA_OK)
        return rc;
    const void *need[] = {cu_seqlens, cu_seqlens_comp};
    const char *need_name[] = {"cu_seqlens", "cu_seqlens_comp"};
    for (int i = 0; i < 2; ++i)
        if ((rc = check_ptr(need[i], need_name[i], 4)) != CSA_OK)
            return rc;
    if (capacity > 0) {
        const void *in[] = {kv, score, ape, grad_out};
        const char *in_name[] = {"kv", "score", "ape", "grad_out"};
        for (int i = 0; i < 4; ++i)
            if ((rc = check_ptr(in[i], in_name[i], 16)) != CSA_OK)
                return rc;
    }
    if (n_tokens != 0) {
        if ((rc = check_ptr(dkv, "dkv", 16)) != CSA_OK || (rc = check_ptr(dscore, "dscore", 16)) != CSA_OK)
            return rc;
    }
    if ((rc = check_ptr(dape, "dape", 16)) != CSA_OK)
        return rc;

    NoAllocDevice nd;
    cudaError_t e = noalloc_device(&nd);
    unsigned *status = nullptr;
    if (e == cudaSuccess)  // the same word csa_device_status() reads
        e = csa::status_word(&status);
    if (e != cudaSuccess)
        return csa::fail_status(CSA_ERR_CUDA, "no-alloc set-up: %s (%s)", cudaGetErrorName(e), cudaGetErrorString(e));

    csa::BwdParams p{kv, score, ape, cu_seqlens, cu_seqlens_comp, n_seg, ratio, coff, head_dim,
                     capacity, n_tokens, grad_out, dkv, dscore, dape};
    csa::BwdPlan plan;
    e = csa::plan_bwd(ratio, coff, head_dim, capacity, nd.num_sms, &plan);
    if (e != cudaSuccess)
        return csa::fail_status(CSA_ERR_CUDA, "no-alloc plan: %s", cudaGetErrorString(e));
    int64_t floats = plan.floats;
    const int64_t per = (int64_t)ratio * coff * head_dim;
    if (plan.family == csa::kBwdChunked && floats > (int64_t)kScratchFloats && per <= (int64_t)kScratchFloats &&
        plan.ch_partials > 0) {
        // More partials than the array holds: fewer row blocks per column tile
        // (each walks more rows; one partial per cluster of blocks).
        const int cluster = plan.ch_blocks / plan.ch_partials;
        const int fit = (int)((int64_t)kScratchFloats / per);
        plan.ch_blocks = fit * cluster;
        plan.ch_partials = fit;
        floats = (int64_t)fit * per;
    } else if (plan.family == csa::kBwdStream) {
        // the exact grid's partials (the regular call sizes its pool block by an upper bound)
        floats = (int64_t)(plan.stream_blocks / plan.sp.cluster) * per;
    }
    if (floats > (int64_t)kScratchFloats)
        return csa::fail_status(CSA_ERR_TOO_LARGE,
                                "csa_compress_bwd_noalloc needs %lld floats of grad_ape scratch for this shape; "
                                "its fixed array holds %lld (use csa_compress_bwd)",
                                (long long)floats, (long long)kScratchFloats);
    e = csa::launch_bwd(p, plan, nd.scratch, status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return csa::fail_status(CSA_ERR_CUDA, "backward launch: %s (%s)", cudaGetErrorName(e), cudaGetErrorString(e));
    return CSA_OK;
}
