// kernels.h -- launch interfaces of the device code (internal to the library).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace pa {

cudaError_t launch_build_schedule(const ScheduleArgs& a, cudaStream_t stream);

struct SimpleParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    __nv_bfloat16* cache_k;
    __nv_bfloat16* cache_v;
    __nv_bfloat16* out;
    float* lse;
    const WorkspaceHeader* hdr;
    const SeqInfo* seqs;
    const Unit* units;
    int n_heads, n_kv_heads, group, max_cache_len;
    float scale;
    int causal;
};

cudaError_t launch_attn_simple(const SimpleParams& p, int head_dim, int grid, cudaStream_t st);

}  // namespace pa
