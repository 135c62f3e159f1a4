// Internal interface between the C-ABI entry points (csa_api.cu) and the kernel
// files.  Not installed, not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

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
    int threads_x;       // threads along the columns (8 columns each), <= 64
    int col_slices;      // blocks along the columns (gridDim.y)
    int lanes;           // rows processed side by side in a block
    int blocks;          // = number of grad_ape partials
    int rows_per_block;  // contiguous output rows per block
    size_t smem;         // bytes of dynamic shared memory (lane merge)
    int64_t partial_floats;
};

cudaError_t launch_fwd_small(const FwdParams &p, cudaStream_t st);
SmallBwdPlan plan_bwd_small(int ratio, int coff, int head_dim, int capacity, int num_sms);
cudaError_t launch_bwd_small(const BwdParams &p, const SmallBwdPlan &pl, float *partial, cudaStream_t st);

}  // namespace csa
