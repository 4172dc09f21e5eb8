// rope.cu -- rotary position embedding prologue of the attention launch.
//
// Rotates every new query and key to its absolute position before attention
// and before the key is written to the cache ("Prefill不是热身：大模型推理的真正
// 瓶颈与优化核心" (mhpn.cn) §5.1: the token at position m has its Q/K rotated by
// theta_m = m * inv_freq, inv_freq = 1 / base^(arange(0, d, 2) / d), as in the
// Llama models the page names, whose pairing is rotate-half: dimension i turns
// with dimension i + d/2).  inv_freq comes from the host, in fp32 as the page's
// formula computes it; the angle m * inv_freq is one fp32 multiply, cos/sin
// come from sincosf, and the rotation is fp32 rounded once to bf16.
//
// The position of new token i of sequence b is cache_offsets[b] + i (the
// chunk's tokens follow its cached prefix).  A memory-bound pass (16-byte
// loads and stores, cos/sin computed once per token and frequency).
#include <cuda_bf16.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace pa {

namespace {

constexpr int kRopeThreads = 256;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One block: kRopeThreads * 2 / d tokens.  Their cos/sin (one sincosf per
// (token, frequency)) go to shared memory first; then every thread rotates
// 8-pair groups of head rows: item = (token, head of q then k, group), so that
// consecutive threads touch consecutive 16-byte pieces of a row.  Each thread
// issues the loads of kBatch items before their stores (memory-level
// parallelism for a pass that is bound by HBM bandwidth).
constexpr int kBatch = 4;

__global__ void __launch_bounds__(kRopeThreads) rope_kernel(const RopeParams p) {
    __shared__ float2 cs[kRopeThreads];  // (cos, sin) per (token of the block, frequency)
    const int half = p.head_dim / 2;
    const int tpb = kRopeThreads / half;  // tokens per block
    const int groups = half / 8;
    const int heads = p.n_heads + p.n_kv_heads;
    const long long t0 = (long long)blockIdx.x * tpb;
    griddep_wait();  // the scheduler's SeqInfo
    {
        const int tt = threadIdx.x / half, i = threadIdx.x % half;
        const long long t = t0 + tt;
        float c = 1.f, s = 0.f;
        if (t < p.total_q) {
            // the sequence owning token t: the last b with cu_seqlens_q[b] <= t
            int lo = 0, hi = p.num_seqs - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p.cu_seqlens_q[mid] <= t)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            const SeqInfo si = p.seqs[lo];  // sanitised by the scheduler (n = 0 when rejected)
            if (t >= si.q_start && t < (long long)si.q_start + si.n) {
                const float angle = __fmul_rn((float)(si.P + (int)(t - si.q_start)), p.inv_freq[i]);
                sincosf(angle, &s, &c);
            }
        }
        cs[threadIdx.x] = make_float2(c, s);
    }
    __syncthreads();
    const long long ntok = p.total_q - t0 < tpb ? p.total_q - t0 : tpb;
    const int items = (int)ntok * heads * groups;
    for (int base = threadIdx.x; base < items; base += kBatch * kRopeThreads) {
        uint4 xa[kBatch], ya[kBatch];
        __nv_bfloat16* dst[kBatch];
        int csi[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int it = base + u * kRopeThreads;
            dst[u] = nullptr;
            if (it < items) {
                const int g = it % groups, h = (it / groups) % heads, tt = it / (groups * heads);
                const long long t = t0 + tt;
                const __nv_bfloat16* src;
                if (h < p.n_heads) {
                    const size_t off = ((size_t)t * p.n_heads + h) * p.head_dim + 8 * g;
                    src = p.q + off;
                    dst[u] = p.q_rot + off;
                } else {
                    const size_t off = ((size_t)t * p.n_kv_heads + (h - p.n_heads)) * p.head_dim + 8 * g;
                    src = p.k + off;
                    dst[u] = p.k_rot + off;
                }
                xa[u] = __ldg(reinterpret_cast<const uint4*>(src));
                ya[u] = __ldg(reinterpret_cast<const uint4*>(src + half));
                csi[u] = tt * half + 8 * g;
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (!dst[u]) continue;
            const uint32_t xw[4] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w};
            const uint32_t yw[4] = {ya[u].x, ya[u].y, ya[u].z, ya[u].w};
            uint32_t ow[4], pw[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float2 c0 = cs[csi[u] + 2 * w], c1 = cs[csi[u] + 2 * w + 1];
                const float x0 = lo_f(xw[w]), x1 = hi_f(xw[w]);
                const float y0 = lo_f(yw[w]), y1 = hi_f(yw[w]);
                ow[w] = pack2(fmaf(x0, c0.x, -y0 * c0.y), fmaf(x1, c1.x, -y1 * c1.y));
                pw[w] = pack2(fmaf(y0, c0.x, x0 * c0.y), fmaf(y1, c1.x, x1 * c1.y));
            }
            *reinterpret_cast<uint4*>(dst[u]) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            *reinterpret_cast<uint4*>(dst[u] + half) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        }
    }
    // let the attention kernel launch once every block got here (it waits for
    // this kernel to finish before reading the rotated copies); triggering at
    // the end keeps its persistent blocks from taking SMs this grid still needs
    griddep_launch();
}

}  // namespace

cudaError_t launch_rope(const RopeParams& p, cudaStream_t stream) {
    const int tpb = kRopeThreads / (p.head_dim / 2);
    const long long blocks = ((long long)p.total_q + tpb - 1) / tpb;
    if (blocks == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kRopeThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rope_kernel, p);
}

}  // namespace pa
