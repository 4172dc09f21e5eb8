// kernels.h -- launch interfaces of the device code (internal to the library).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace pa {

cudaError_t launch_build_schedule(const ScheduleArgs& a, cudaStream_t stream);

// Rotary embedding prologue: q_rot/k_rot = q/k rotated to each token's
// absolute position (runs after the scheduler, whose SeqInfo it reads).
struct RopeParams {
    const __nv_bfloat16* q;  // [T, H, d]
    const __nv_bfloat16* k;  // [T, Hk, d]
    __nv_bfloat16* q_rot;
    __nv_bfloat16* k_rot;
    const int32_t* cu_seqlens_q;
    const SeqInfo* seqs;
    int total_q, num_seqs, n_heads, n_kv_heads, head_dim;
    float inv_freq[64];  // inv_freq[i] = 1 / base^(2i / d), i < d/2
};
cudaError_t launch_rope(const RopeParams& p, cudaStream_t stream);



}  // namespace pa

#include <cuda.h>

namespace pa {

// Parameters of the warp-specialised tcgen05 attention kernel.  The tensor
// maps are encoded on the host per call.
struct FwdParams {
    CUtensorMap tm_q;        // q  [T, H, D]      viewed (D, H, T),        box (C, G, 128/G)
    CUtensorMap tm_k;        // k  [T, Hk, D]     viewed (D, Hk, T),       box (C, 1, 128)
    CUtensorMap tm_v;        // v  same as k
    CUtensorMap tm_ck;       // cache_k [B, Hk, cap, D] viewed (D, cap, B*Hk), box (C, 128, 1); paged:
                             // pool [NB, Hk, bs, D] viewed (D, bs, NB*Hk), box (C, min(bs, 128), 1)
    CUtensorMap tm_cv;       // cache_v same
    const __nv_bfloat16* k;  // raw pointers for the cache copy
    const __nv_bfloat16* v;
    __nv_bfloat16* cache_k;
    __nv_bfloat16* cache_v;
    __nv_bfloat16* out;
    float* lse;
    WorkspaceHeader* hdr;
    const SeqInfo* seqs;
    const Unit* units;
    int n_heads, n_kv_heads, group, max_cache_len;
    float scale_log2;        // scale * log2(e)
    int causal;
    int window;              // sliding window (0: none)
    // paged cache (block_table == nullptr: contiguous [B, Hk, cap, D] slots)
    const int32_t* block_table;  // [B][max_blocks]
    int block_log2;              // block_size = 1 << block_log2 (>= 8)
    int box_rows;                // min(block_size, 128): rows of one cache TMA box
    int max_blocks;
    int num_blocks;
    // int8 cache (kv_quant): cache_k/cache_v hold int8 codes, these the fp32
    // scale of each cache row ([B, Hk, cap])
    float* scale_k;
    float* scale_v;
    int kv_quant;
    int wait_timeout_test;  // test hook: CTA 0 waits on a barrier nothing completes
    // alternating variant (bf16 cache): units whose rows fit one Q tile split
    // their KV tiles between both softmax slots (even / odd) and merge the two
    // partial results; the host picks it for decode-heavy or small launches
    int alt;
    int unit_slots;  // Q tiles per unit the scheduler cut (2, or 1 in the alternating variant)
    int out_align32;  // out is 32-byte aligned: the epilogue stores whole 32-byte sectors
};

// Encodes the tensor maps of `p` (the pointer fields and sizes must be set).
// num_blocks: blocks in the pool when p.block_table is set (else unused).
cudaError_t encode_fwd_maps(FwdParams& p, const void* q, int total_q, int num_seqs, int head_dim, int num_blocks);
cudaError_t launch_attn_fwd(const FwdParams& p, int head_dim, int grid, cudaStream_t st);

}  // namespace pa
