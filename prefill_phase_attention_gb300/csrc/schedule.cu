// schedule.cu -- the longest-first tile scheduler.
//
// Reads cu_seqlens_q / cu_seqlens_k / cache_offsets on the device (the varlen
// kernel "reads cu_seqlens" itself, "大模型 Prompt Prefill 阶段的高效 Batching 与算子排布",
// §2), sanitises each sequence, cuts it into work units (query block x KV head)
// and lays the units out by descending cost (KV tiles visited) with a counting
// sort, so that the persistent attention kernel starts the longest units first
// (LPT order).  It also resets the attention kernel's work counter.
//
// One CTA of 1024 threads; its cost is a few microseconds and it keeps the whole
// launch free of host synchronisation.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "prefill_attn.h"

namespace pa {

__device__ __forceinline__ int clamp_bin(int c) { return c < kCostBins - 1 ? c : kCostBins - 1; }

__global__ void __launch_bounds__(1024) build_schedule_kernel(ScheduleArgs a) {
    __shared__ int hist[kCostBins];
    __shared__ int warp_sums[32];
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int tpu = kBlockM / a.group;  // query tokens per unit

    for (int i = tid; i < kCostBins; i += nthr) hist[i] = 0;
    __syncthreads();

    // Pass 1: sanitise each sequence and histogram the unit costs.
    for (int b = tid; b < a.num_seqs; b += nthr) {
        const int q_start = a.cu_seqlens_q[b];
        const int q_end = a.cu_seqlens_q[b + 1];
        const int lk = a.cu_seqlens_k[b + 1] - a.cu_seqlens_k[b];
        const int P = a.cache_offsets[b];
        const long long n = (long long)q_end - q_start;
        const bool ok = q_start >= 0 && n >= 0 && (long long)q_end <= a.total_q && P >= 0 &&
                        (long long)lk == (long long)P + n && (long long)P + n <= a.max_cache_len &&
                        (b > 0 || q_start == 0);
        SeqInfo si;
        si.q_start = ok ? q_start : 0;
        si.n = ok ? (int)n : 0;
        si.P = ok ? P : 0;
        si.pad = 0;
        if (!ok) atomicOr(&a.hdr->error, PA_DEVERR_METADATA);
        a.seqs[b] = si;
        for (int q0 = 0; q0 < si.n; q0 += tpu)
            atomicAdd(&hist[clamp_bin(unit_tiles(si.n, si.P, q0, tpu, a.causal))], a.n_kv_heads);
    }
    __syncthreads();

    // Exclusive scan in DESCENDING cost order: start[c] = sum of hist[c'] for c' > c.
    // Each thread owns two adjacent bins of the reversed order.
    static_assert(kCostBins == 2 * 1024, "scan assumes two bins per thread");
    const int r0 = kCostBins - 1 - 2 * tid;  // bins r0 and r0 - 1, in that order
    const int h0 = hist[r0], h1 = hist[r0 - 1];
    int x = h0 + h1;
    const int lane = tid & 31, warp = tid >> 5;
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;  // inclusive
    }
    __syncthreads();
    const int excl = x - (h0 + h1) + (warp > 0 ? warp_sums[warp - 1] : 0);
    const int total = warp_sums[31];
    __syncthreads();
    hist[r0] = excl;
    hist[r0 - 1] = excl + h0;
    if (tid == 0) {
        a.hdr->num_units = total < a.max_units ? total : a.max_units;
        a.hdr->counter = 0;
        a.hdr->max_units = a.max_units;
        if (total > a.max_units) atomicOr(&a.hdr->error, PA_DEVERR_OVERFLOW);
    }
    __syncthreads();

    // Pass 2: scatter the units to their sorted positions.
    for (int b = tid; b < a.num_seqs; b += nthr) {
        const SeqInfo si = a.seqs[b];
        for (int q0 = 0; q0 < si.n; q0 += tpu) {
            const int cost = unit_tiles(si.n, si.P, q0, tpu, a.causal);
            const int base = atomicAdd(&hist[clamp_bin(cost)], a.n_kv_heads);
            for (int kvh = 0; kvh < a.n_kv_heads; ++kvh) {
                const int pos = base + kvh;
                if (pos < a.max_units) {
                    Unit u;
                    u.b = b;
                    u.kvh = kvh;
                    u.q0 = q0;
                    u.ntiles = cost;
                    a.units[pos] = u;
                }
            }
        }
    }
}

cudaError_t launch_build_schedule(const ScheduleArgs& a, cudaStream_t stream) {
    build_schedule_kernel<<<1, 1024, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pa
