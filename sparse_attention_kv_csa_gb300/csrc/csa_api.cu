// C-ABI entry points of libcsa (declared in include/csa.h): argument validation,
// kernel-family dispatch and the backward's stream-ordered workspace.
//
// Validation follows the support surface of the "CSA Fused Compressor" page
// (cuDNN frontend docs, section Support surface): coff in {1, 2}, supported
// (ratio, head_dim), int32 flat offsets, total_comp > 0 requiring at least ratio
// tokens, 16-byte aligned tensor bases (4-byte for the int32 offsets) checked per
// call.  Nothing is launched and no output is touched when validation fails.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "csa.h"
#include "csa_device.cuh"
#include "csa_launch.h"

namespace {

thread_local char g_msg[512] = "";

int fail(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return status;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(e == cudaErrorMemoryAllocation ? CSA_ERR_OUT_OF_MEMORY : CSA_ERR_CUDA, "%s: %s (%s)",
                what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int64_t kInt32Limit = int64_t(1) << 31;
constexpr int kMaxDevices = 64;

// Per-device facts and the workspace pool, created on first use on that device.  A
// set-up that fails (a transient runtime error, a first call made during stream
// capture) is not remembered: the next call on that device tries again.
struct DeviceState {
    std::atomic<bool> ready{false};
    int num_sms = 0;
    cudaMemPool_t pool = nullptr;
    unsigned *status = nullptr;  // device status word written by bounded waits
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

cudaError_t device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    DeviceState &d = g_dev[dev];
    if (d.ready.load(std::memory_order_acquire)) {
        *out = &d;
        return cudaSuccess;
    }
    std::lock_guard<std::mutex> g(g_dev_mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = csa::status_word(&d.status);
        if (e == cudaSuccess && !d.pool) {
            // A pool of its own, so that the workspace stays cached between calls
            // without changing the device's default pool.
            cudaMemPoolProps props;
            memset(&props, 0, sizeof(props));
            props.allocType = cudaMemAllocationTypePinned;
            props.handleTypes = cudaMemHandleTypeNone;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            cudaMemPool_t pool = nullptr;
            e = cudaMemPoolCreate(&pool, &props);
            if (e == cudaSuccess) {
                uint64_t keep = 256ull << 20;
                e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
                if (e == cudaSuccess)
                    d.pool = pool;
                else
                    cudaMemPoolDestroy(pool);
            }
        }
        if (e != cudaSuccess)
            return e;
        d.ready.store(true, std::memory_order_release);
    }
    *out = &d;
    return cudaSuccess;
}

int check_common(int32_t n_seg, int32_t ratio, int32_t coff, int32_t head_dim, int32_t capacity)
{
    if (n_seg < 0)
        return fail(CSA_ERR_INVALID_VALUE, "n_seg must be >= 0 (got %d)", n_seg);
    if (capacity < 0)
        return fail(CSA_ERR_INVALID_VALUE, "capacity must be >= 0 (got %d)", capacity);
    if (coff != 1 && coff != 2)
        return fail(CSA_ERR_INVALID_VALUE, "coff must be 1 or 2 (got %d)", coff);
    if (ratio < 1)
        return fail(CSA_ERR_INVALID_VALUE, "ratio must be >= 1 (got %d)", ratio);
    if (head_dim < 1)
        return fail(CSA_ERR_INVALID_VALUE, "head_dim must be >= 1 (got %d)", head_dim);
    if (ratio == 4) {
        if (head_dim % 8 != 0 || head_dim > 8192)
            return fail(CSA_ERR_UNSUPPORTED,
                        "ratio 4 needs head_dim a multiple of 8 in [8, 8192] (got %d)", head_dim);
    } else if (ratio == 128) {
        if (head_dim % 64 != 0 || head_dim > 8192)
            return fail(CSA_ERR_UNSUPPORTED,
                        "ratio 128 needs head_dim a multiple of 64 in [64, 8192] (got %d)", head_dim);
    } else if (ratio > 128 || head_dim % 8 != 0 || head_dim > 8192) {
        return fail(CSA_ERR_UNSUPPORTED,
                    "ratio %d needs ratio <= 128 and head_dim a multiple of 8 in [8, 8192] (got head_dim %d)",
                    ratio, head_dim);
    }
    if ((int64_t)capacity * head_dim >= kInt32Limit)
        return fail(CSA_ERR_TOO_LARGE, "capacity * head_dim = %lld does not fit int32 offsets",
                    (long long)capacity * head_dim);
    return CSA_OK;
}

int check_tokens(int32_t ratio, int32_t coff, int32_t head_dim, int64_t n_tokens, int32_t capacity)
{
    if (n_tokens < 0)
        return CSA_OK;
    if (n_tokens * coff * (int64_t)head_dim >= kInt32Limit)
        return fail(CSA_ERR_TOO_LARGE, "n_tokens * coff * head_dim = %lld does not fit int32 offsets",
                    (long long)(n_tokens * coff * (int64_t)head_dim));
    if (capacity > 0 && n_tokens < ratio)
        return fail(CSA_ERR_INVALID_VALUE,
                    "capacity > 0 needs n_tokens >= ratio (each row reads ratio tokens); got %lld < %d",
                    (long long)n_tokens, ratio);
    return CSA_OK;
}

int check_ptr(const void *p, const char *name, uintptr_t align)
{
    if (!p)
        return fail(CSA_ERR_INVALID_VALUE, "%s is NULL", name);
    if (!aligned(p, align))
        return fail(CSA_ERR_MISALIGNED, "%s = %p is not %d-byte aligned", name, p, (int)align);
    return CSA_OK;
}

#define CSA_TRY(expr)               \
    do {                            \
        int rc_ = (expr);           \
        if (rc_ != CSA_OK)          \
            return rc_;             \
    } while (0)

}  // namespace

namespace csa {

cudaError_t allow_max_smem(const void *fn)
{
    static std::mutex mu;
    static int devs[256];
    static const void *fns[256];
    static int n = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < n; ++i)
        if (devs[i] == dev && fns[i] == fn)
            return cudaSuccess;
    int optin = 0;
    cudaFuncAttributes fa;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess)
        e = cudaFuncGetAttributes(&fa, fn);
    if (e == cudaSuccess)  // the device maximum less the kernel's static shared memory
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - static_cast<int>(fa.sharedSizeBytes));
    if (e == cudaSuccess && n < 256) {
        devs[n] = dev;
        fns[n] = fn;
        ++n;
    }
    return e;
}

// Resident blocks of a kernel configuration, computed once per (device, kernel,
// block size, shared memory, cluster) and cached: the occupancy queries and the
// shared-memory attribute are host calls too slow to repeat on every launch.
namespace {

struct ResidentKey {
    int dev;
    const void *fn;
    int threads;
    size_t smem;
    int cluster;
};

cudaError_t cached_resident(const ResidentKey &k, int *resident, cudaError_t (*query)(const ResidentKey &, int *))
{
    static std::mutex mu;
    static ResidentKey keys[64];
    static int vals[64];
    static int n = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        for (int i = 0; i < n; ++i)
            if (keys[i].dev == k.dev && keys[i].fn == k.fn && keys[i].threads == k.threads &&
                keys[i].smem == k.smem && keys[i].cluster == k.cluster) {
                *resident = vals[i];
                return cudaSuccess;
            }
    }
    cudaError_t e = query(k, resident);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> g(mu);
    if (n < 64) {
        keys[n] = k;
        vals[n] = *resident;
        ++n;
    }
    return cudaSuccess;
}

cudaError_t query_resident(const ResidentKey &k, int *resident)
{
    // The kernel's dynamic shared-memory limit is a per-function attribute shared by
    // every configuration: raise it to the device maximum (not to this plan's size,
    // which a later plan of another head_dim could undercut).
    cudaError_t e = allow_max_smem(k.fn);
    if (e != cudaSuccess)
        return e;
    if (k.cluster > 1) {
        // clusters are placed within GPCs: ask how many fit, not blocks per SM
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(k.cluster, 1, 1);
        cfg.blockDim = dim3(k.threads, 1, 1);
        cfg.dynamicSmemBytes = k.smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = k.cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, k.fn, &cfg);
        *resident = clusters * k.cluster;
        return e;
    }
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.fn, k.threads, k.smem);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, k.dev);
    *resident = per_sm * sms;
    return e;
}

}  // namespace

cudaError_t resident_blocks(const void *fn, int threads, size_t smem, int cluster, int *resident)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    return cached_resident(ResidentKey{dev, fn, threads, smem, cluster}, resident, query_resident);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn(cudaError_t *err)
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static cudaError_t e = cudaSuccess;
    std::call_once(once, []() {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q != cudaDriverEntryPointSuccess)
            e = cudaErrorNotSupported;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    *err = e;
    return fn;
}

}  // namespace

// The row extent is the int32 flat-offset bound, not the (unknown to the forward)
// token count: every box the kernels request lies inside a real block.
cudaError_t make_tensor_map_2d(CUtensorMap *m, const void *ptr, int64_t C, int box_cols, int box_rows)
{
    cudaError_t e;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn(&e);
    if (e != cudaSuccess)
        return e;
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)(((int64_t)1 << 31) / C)};
    const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// [rows][C] bf16 seen as [rows][C / chunk_cols][chunk_cols]: a box {chunk_cols,
// chunks, box_rows} at (0, col / chunk_cols, row) lands in shared memory as the
// row-major [box_rows][chunks * chunk_cols] tile -- a tile wider than the 256
// elements one box dimension may span, in one copy.  C must be a multiple of
// chunk_cols.
cudaError_t make_tensor_map_3d(CUtensorMap *m, const void *ptr, int64_t C, int chunk_cols, int chunks, int box_rows)
{
    cudaError_t e;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn(&e);
    if (e != cudaSuccess)
        return e;
    if (chunk_cols <= 0 || C % chunk_cols != 0)
        return cudaErrorInvalidValue;
    const cuuint64_t dims[3] = {(cuuint64_t)chunk_cols, (cuuint64_t)(C / chunk_cols),
                                (cuuint64_t)(((int64_t)1 << 31) / C)};
    const cuuint64_t strides[2] = {(cuuint64_t)chunk_cols * 2, (cuuint64_t)C * 2};
    const cuuint32_t box[3] = {(cuuint32_t)chunk_cols, (cuuint32_t)chunks, (cuuint32_t)box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The two parts of a coff-2 window in one box: [rows][C] bf16 seen with a third
// dimension of extent 2 whose step is ratio rows and head_dim columns (part 1 of
// a block's window starts ratio tokens and head_dim columns after part 0).  A box
// {box_cols, ratio, 2} at (col, first token of part 0, 0) lands as [part][token]
// [box_cols], the two per-part boxes' layout, in one copy.  Its origin must not
// be negative: the part-1 elements are bounds-checked against the part-0 token
// coordinate.
cudaError_t make_tensor_map_parts(CUtensorMap *m, const void *ptr, int64_t C, int box_cols, int ratio, int head_dim)
{
    cudaError_t e;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn(&e);
    if (e != cudaSuccess)
        return e;
    const cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)(((int64_t)1 << 31) / C), 2};
    const cuuint64_t strides[2] = {(cuuint64_t)C * 2, (cuuint64_t)((int64_t)ratio * C + head_dim) * 2};
    const cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)ratio, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The status word of the bounded waits, one per device: a word of this module's
// device memory, so that neither entry point has to allocate it.
static __device__ __align__(256) unsigned g_status_word[64];

cudaError_t status_word(unsigned **word)
{
    static std::mutex mu;
    static unsigned *addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(mu);
    if (!addr[dev]) {
        // The symbol's name is a host-side stand-in: ask for its address on this
        // (current) device.
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&addr[dev]), g_status_word);
        if (e != cudaSuccess) {
            addr[dev] = nullptr;
            return e;
        }
    }
    *word = addr[dev];
    return cudaSuccess;
}

cudaError_t plan_bwd(int ratio, int coff, int head_dim, int capacity, int num_sms, BwdPlan *out)
{
    BwdPlan b{};
    cudaError_t e = cudaSuccess;
    if (chunked_supported(ratio, coff, head_dim)) {
        b.family = kBwdChunked;
        e = chunked_bwd_partials(ratio, coff, head_dim, capacity, &b.ch_partials, &b.ch_blocks);
        b.floats = (int64_t)b.ch_partials * ratio * coff * head_dim;
    } else if (ratio != 4) {
        b.family = kBwdGeneric;
        e = plan_generic(ratio, coff, head_dim, capacity, num_sms, &b.gp);
        b.floats = b.gp.partial_floats;
    } else if (stream_supported(true, ratio, coff, head_dim)) {
        b.family = kBwdStream;
        b.sp = plan_stream(true, ratio, coff, head_dim, capacity, num_sms);
        e = stream_bwd_blocks(ratio, coff, b.sp, capacity, &b.stream_blocks);
        b.floats = (int64_t)stream_bwd_partials(b.sp, capacity) * ratio * coff * head_dim;
    } else {
        b.family = kBwdSmall;
        b.pl = plan_bwd_small(ratio, coff, head_dim, capacity, num_sms);
        b.floats = b.pl.partial_floats;
    }
    *out = b;
    return e;
}

cudaError_t launch_bwd(const BwdParams &p, const BwdPlan &b, float *partial, unsigned *status, cudaStream_t st)
{
    switch (b.family) {
    case kBwdChunked: return launch_bwd_chunked(p, partial, b.ch_blocks, status, st);
    case kBwdGeneric: return launch_bwd_generic(p, b.gp, partial, status, st);
    case kBwdStream: return launch_bwd_stream(p, b.sp, partial, status, st);
    default: return launch_bwd_small(p, b.pl, partial, st);
    }
}

int fail_status(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return status;
}

}  // namespace csa

extern "C" {

int csa_version(void) { return 100; }

const char *csa_status_string(int status)
{
    switch (status) {
    case CSA_OK: return "CSA_OK";
    case CSA_ERR_INVALID_VALUE: return "CSA_ERR_INVALID_VALUE";
    case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED";
    case CSA_ERR_MISALIGNED: return "CSA_ERR_MISALIGNED";
    case CSA_ERR_TOO_LARGE: return "CSA_ERR_TOO_LARGE";
    case CSA_ERR_CUDA: return "CSA_ERR_CUDA";
    case CSA_ERR_OUT_OF_MEMORY: return "CSA_ERR_OUT_OF_MEMORY";
    case CSA_ERR_DEVICE_TIMEOUT: return "CSA_ERR_DEVICE_TIMEOUT";
    default: return "CSA_ERR_UNKNOWN";
    }
}

const char *csa_last_error_message(void) { return g_msg; }

int csa_check_support(int32_t ratio, int32_t coff, int32_t head_dim, int64_t n_tokens, int32_t capacity)
{
    CSA_TRY(check_common(0, ratio, coff, head_dim, capacity));
    CSA_TRY(check_tokens(ratio, coff, head_dim, n_tokens, capacity));
    return CSA_OK;
}

int csa_compress_fwd(const void *kv, const void *score, const float *ape, const int32_t *cu_seqlens,
                     const int32_t *cu_seqlens_comp, int32_t n_seg, int32_t ratio, int32_t coff,
                     int32_t head_dim, int32_t capacity, void *out, void *stream)
{
    CSA_TRY(check_common(n_seg, ratio, coff, head_dim, capacity));
    CSA_TRY(check_ptr(cu_seqlens, "cu_seqlens", 4));
    CSA_TRY(check_ptr(cu_seqlens_comp, "cu_seqlens_comp", 4));
    if (capacity == 0)
        return CSA_OK;
    CSA_TRY(check_ptr(kv, "kv", 16));
    CSA_TRY(check_ptr(score, "score", 16));
    CSA_TRY(check_ptr(ape, "ape", 16));
    CSA_TRY(check_ptr(out, "out", 16));
    DeviceState *ds = nullptr;
    cudaError_t e = device_state(&ds);
    if (e != cudaSuccess)
        return cuda_fail(e, "device set-up");
    csa::FwdParams p{kv, score, ape, cu_seqlens, cu_seqlens_comp, n_seg, ratio, coff, head_dim, capacity, out};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (csa::chunked_supported(ratio, coff, head_dim))
        e = csa::launch_fwd_chunked(p, ds->status, st);
    else if (ratio != 4)
        e = csa::launch_fwd_generic(p, ds->status, ds->num_sms, st);
    else if (csa::stream_supported(false, ratio, coff, head_dim))
        e = csa::launch_fwd_stream(p, csa::plan_stream(false, ratio, coff, head_dim, capacity, ds->num_sms),
                                   ds->status, st);
    else
        e = csa::launch_fwd_small(p, ds->num_sms, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "forward launch");
    return CSA_OK;
}

int csa_compress_bwd(const void *kv, const void *score, const float *ape, const int32_t *cu_seqlens,
                     const int32_t *cu_seqlens_comp, int32_t n_seg, int32_t ratio, int32_t coff,
                     int32_t head_dim, int32_t capacity, int64_t n_tokens, const void *grad_out,
                     void *dkv, void *dscore, float *dape, void *stream)
{
    CSA_TRY(check_common(n_seg, ratio, coff, head_dim, capacity));
    CSA_TRY(check_tokens(ratio, coff, head_dim, n_tokens, capacity));
    CSA_TRY(check_ptr(cu_seqlens, "cu_seqlens", 4));
    CSA_TRY(check_ptr(cu_seqlens_comp, "cu_seqlens_comp", 4));
    if (capacity > 0) {
        CSA_TRY(check_ptr(kv, "kv", 16));
        CSA_TRY(check_ptr(score, "score", 16));
        CSA_TRY(check_ptr(ape, "ape", 16));
        CSA_TRY(check_ptr(grad_out, "grad_out", 16));
    }
    if (n_tokens != 0) {
        CSA_TRY(check_ptr(dkv, "dkv", 16));
        CSA_TRY(check_ptr(dscore, "dscore", 16));
    }
    CSA_TRY(check_ptr(dape, "dape", 16));

    DeviceState *ds = nullptr;
    cudaError_t e = device_state(&ds);
    if (e != cudaSuccess)
        return cuda_fail(e, "device set-up");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    csa::BwdParams p{kv, score, ape, cu_seqlens, cu_seqlens_comp, n_seg, ratio, coff, head_dim,
                     capacity, n_tokens, grad_out, dkv, dscore, dape};
    csa::BwdPlan plan;
    e = csa::plan_bwd(ratio, coff, head_dim, capacity, ds->num_sms, &plan);
    if (e != cudaSuccess)
        return cuda_fail(e, "backward plan");
    void *partial = nullptr;
    e = cudaMallocFromPoolAsync(&partial, (size_t)plan.floats * sizeof(float), ds->pool, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "backward workspace");
    e = csa::launch_bwd(p, plan, static_cast<float *>(partial), ds->status, st);
    cudaError_t e2 = cudaFreeAsync(partial, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "backward launch");
    if (e2 != cudaSuccess)
        return cuda_fail(e2, "backward workspace release");
    return CSA_OK;
}

namespace {

// Waits for a phase of a shared-memory barrier that nothing ever completes: the
// bounded wait must give up after limit_ns and record a timeout.
__global__ void selftest_wait_kernel(unsigned *status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        csa::mbar_init(csa::smem_addr(&bar), 1);
        csa::mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        csa::mbar_wait(csa::smem_addr(&bar), 0u, status, limit_ns);
}

__global__ void selftest_recip_kernel(const float *__restrict__ d, float *__restrict__ out, int64_t n)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = csa::recip_den(d[i]);
}

}  // namespace

int csa_selftest_reciprocal(const float *d, float *out, int64_t n, void *stream)
{
    if (n < 0)
        return fail(CSA_ERR_INVALID_VALUE, "n must be >= 0 (got %lld)", (long long)n);
    if (n == 0)
        return CSA_OK;
    if (!d || !out)
        return fail(CSA_ERR_INVALID_VALUE, "d and out must not be NULL");
    DeviceState *ds = nullptr;
    cudaError_t e = device_state(&ds);
    if (e != cudaSuccess)
        return cuda_fail(e, "device set-up");
    const int64_t want = (n + 255) / 256;
    const int blocks = (int)(want < 8 * (int64_t)ds->num_sms ? want : 8 * (int64_t)ds->num_sms);
    selftest_recip_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(d, out, n);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "self-test launch");
    return CSA_OK;
}

int csa_selftest_bounded_wait(int64_t limit_ns, void *stream)
{
    if (limit_ns < 0 || limit_ns > 1000000000ll)
        return fail(CSA_ERR_INVALID_VALUE, "limit_ns must be in [0, 1e9] (got %lld)", (long long)limit_ns);
    unsigned *word = nullptr;
    cudaError_t e = csa::status_word(&word);
    if (e != cudaSuccess)
        return cuda_fail(e, "status word");
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(word, (uint64_t)limit_ns);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "self-test launch");
    return CSA_OK;
}

int csa_device_status(int clear)
{
    unsigned *status = nullptr;
    cudaError_t e = csa::status_word(&status);
    if (e != cudaSuccess)
        return cuda_fail(e, "status word");
    unsigned word = 0;
    e = cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && clear)
        e = cudaMemset(status, 0, sizeof(word));
    if (e != cudaSuccess)
        return cuda_fail(e, "status read");
    if (word != 0)
        return fail(CSA_ERR_DEVICE_TIMEOUT, "a kernel recorded device status %u (bounded wait expired)", word);
    return CSA_OK;
}

int csa_grad_ape_order(int32_t ratio, int32_t coff, int32_t head_dim, int32_t capacity, csa_grad_ape_grouping *out)
{
    CSA_TRY(check_common(0, ratio, coff, head_dim, capacity));
    if (!out)
        return fail(CSA_ERR_INVALID_VALUE, "out is NULL");
    int dev = 0, num_sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    csa::BwdPlan b;
    e = csa::plan_bwd(ratio, coff, head_dim, capacity, num_sms, &b);
    if (e != cudaSuccess)
        return cuda_fail(e, "backward plan");
    csa_grad_ape_grouping o;
    memset(&o, 0, sizeof(o));
    o.kind = CSA_GRAD_APE_ROW_BLOCKS;
    o.final_ranges = 32;
    switch (b.family) {
    case csa::kBwdChunked:
        o.kind = CSA_GRAD_APE_CHUNKED;
        o.blocks = b.ch_blocks;
        o.partials = b.ch_partials;
        o.cluster = b.ch_partials > 0 ? b.ch_blocks / b.ch_partials : 1;
        break;
    case csa::kBwdGeneric:
        if (b.gp.staged_blocks > 0) {
            o.strided = 1;
            o.blocks = b.gp.staged_blocks;
            o.lanes = b.gp.staged_lanes;
        } else {
            o.blocks = b.gp.groups;
            o.rows_per_block = b.gp.rows_per_group;
            o.lanes = b.gp.lanes;
        }
        o.cluster = 1;
        o.flat = 1;
        o.partials = o.blocks;
        break;
    case csa::kBwdStream:
        o.strided = 1;
        o.blocks = b.stream_blocks;
        o.lanes = b.sp.row_lanes;
        o.cluster = b.sp.cluster;
        o.flat = 1;
        o.partials = b.stream_blocks / b.sp.cluster;
        break;
    default:
        o.blocks = b.pl.blocks;
        o.rows_per_block = b.pl.rows_per_block;
        o.lanes = b.pl.lanes;
        o.cluster = b.pl.cluster;
        o.flat = 0;
        o.partials = b.pl.partials;
        break;
    }
    *out = o;
    return CSA_OK;
}

}  // extern "C"
