// attn_simple.cu -- a deliberately plain CUDA kernel that proves the boundary
// (unit list, masking, GQA mapping, output/LSE layout and the cache write)
// with scalar fp32 arithmetic, one query row per thread.
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace pa {



constexpr int kSimpleKeys = 32;

template <int D>
__global__ void __launch_bounds__(128) attn_simple_kernel(SimpleParams p) {
    extern __shared__ float sm[];
    float* qs = sm;                              // [128][D + 1]
    float* ks = qs + kBlockM * (D + 1);          // [32][D]
    float* vs = ks + kSimpleKeys * D;            // [32][D]
    const int u_idx = blockIdx.x;
    if (u_idx >= p.hdr->num_units) return;
    const Unit un = p.units[u_idx];
    const SeqInfo si = p.seqs[un.b];
    const int G = p.group;
    const int tpu = kBlockM / G;
    const int r = threadIdx.x;
    const int tok = un.q0 + r / G;
    const int h = un.kvh * G + r % G;
    const bool valid = r < tpu * G && tok < si.n;
    const int Lk = si.P + si.n;
    const int last_key = valid ? (p.causal ? si.P + tok : Lk - 1) : -1;
    const int q_hi = (un.q0 + tpu < si.n ? un.q0 + tpu : si.n) - 1;
    const int kmax = p.causal ? si.P + q_hi : Lk - 1;

    for (int e = 0; e < D; ++e)
        qs[r * (D + 1) + e] = valid ? __bfloat162float(p.q[((size_t)(si.q_start + tok) * p.n_heads + h) * D + e]) : 0.f;

    float m = -INFINITY, l = 0.f;
    float acc[D];
#pragma unroll
    for (int e = 0; e < D; ++e) acc[e] = 0.f;

    for (int j0 = 0; j0 <= kmax; j0 += kSimpleKeys) {
        __syncthreads();
        for (int idx = r; idx < kSimpleKeys * D; idx += 128) {
            const int jj = idx / D, e = idx % D, j = j0 + jj;
            float kx = 0.f, vx = 0.f;
            if (j <= kmax) {
                size_t off;
                const __nv_bfloat16 *kb, *vb;
                if (j < si.P) {
                    off = (((size_t)un.b * p.n_kv_heads + un.kvh) * p.max_cache_len + j) * D + e;
                    kb = p.cache_k;
                    vb = p.cache_v;
                } else {
                    off = ((size_t)(si.q_start + j - si.P) * p.n_kv_heads + un.kvh) * D + e;
                    kb = p.k;
                    vb = p.v;
                }
                kx = __bfloat162float(kb[off]);
                vx = __bfloat162float(vb[off]);
            }
            ks[jj * D + e] = kx;
            vs[jj * D + e] = vx;
        }
        __syncthreads();
        for (int jj = 0; jj < kSimpleKeys; ++jj) {
            const int j = j0 + jj;
            if (j > last_key) break;
            float dot = 0.f;
#pragma unroll 8
            for (int e = 0; e < D; ++e) dot = fmaf(qs[r * (D + 1) + e], ks[jj * D + e], dot);
            const float s = dot * p.scale;
            const float m_new = fmaxf(m, s);
            const float corr = expf(m - m_new);
            const float pj = expf(s - m_new);
            l = l * corr + pj;
#pragma unroll
            for (int e = 0; e < D; ++e) acc[e] = acc[e] * corr + pj * vs[jj * D + e];
            m = m_new;
        }
    }
    if (valid) {
        const float inv = 1.f / l;
        __nv_bfloat16* o = p.out + ((size_t)(si.q_start + tok) * p.n_heads + h) * D;
#pragma unroll
        for (int e = 0; e < D; ++e) o[e] = __float2bfloat16_rn(acc[e] * inv);
        if (p.lse) p.lse[(size_t)(si.q_start + tok) * p.n_heads + h] = m + logf(l);
    }
    // cache write: this unit owns tokens [q0, q0 + tpu) of KV head kvh
    const int ntok = (q_hi - un.q0 + 1);
    for (int idx = r; idx < ntok * (D / 8); idx += 128) {
        const int t = un.q0 + idx / (D / 8), c = idx % (D / 8);
        const size_t src = ((size_t)(si.q_start + t) * p.n_kv_heads + un.kvh) * D + c * 8;
        const size_t dst = (((size_t)un.b * p.n_kv_heads + un.kvh) * p.max_cache_len + si.P + t) * D + c * 8;
        *reinterpret_cast<uint4*>(p.cache_k + dst) = *reinterpret_cast<const uint4*>(p.k + src);
        *reinterpret_cast<uint4*>(p.cache_v + dst) = *reinterpret_cast<const uint4*>(p.v + src);
    }
}

template <int D>
static cudaError_t launch_simple_d(const SimpleParams& p, int grid, cudaStream_t st) {
    const int smem = (kBlockM * (D + 1) + 2 * kSimpleKeys * D) * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(attn_simple_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attn_simple_kernel<D><<<grid, 128, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_attn_simple(const SimpleParams& p, int head_dim, int grid, cudaStream_t st) {
    switch (head_dim) {
        case 32: return launch_simple_d<32>(p, grid, st);
        case 64: return launch_simple_d<64>(p, grid, st);
        case 128: return launch_simple_d<128>(p, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
