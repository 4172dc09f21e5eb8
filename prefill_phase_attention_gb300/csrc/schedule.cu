// schedule.cu -- the longest-first tile scheduler.
//
// Reads cu_seqlens_q / cu_seqlens_k / cache_offsets on the device (the varlen
// kernel takes the sequence boundaries from cu_seqlens itself, "大模型 Prompt
// Prefill 阶段的高效 Batching 与算子排布", §2), sanitises each sequence, cuts it
// into work units (query block x KV head) and lays them out for the persistent
// attention kernel, which claims them in list order: sequences by descending
// total cost (KV tiles visited, counting sort over log-spaced cost bins);
// within a sequence its KV heads in groups, and within a group the query
// blocks last to first (for a causal mask, the most expensive first) with the
// group's heads adjacent.  The longest work still starts first (LPT order
// within a group and across sequences; the last units claimed are
// the cheapest blocks of the cheapest sequences), and the CTAs running at any
// moment work on one or two sequences and few of their heads, whose K/V then
// stay in L2 (ordering by unit cost alone interleaves every sequence of a
// varlen batch, and all heads of a long prompt together outgrow L2; either
// re-reads K/V from HBM).  It also resets the attention kernel's work counter.
//
// One CTA of 1024 threads; its cost is a few microseconds and it keeps the whole
// launch free of host synchronisation.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "prefill_attn.h"

namespace pa {

constexpr long long kL2GroupBytes = 48ll << 20;
// Batches of up to this many sequences keep the per-sequence tables the passes
// below hand to one another (SeqInfo, cost bin / list position, KV-head group)
// in shared memory; larger ones go through the workspace in global memory.
constexpr int kSmemSeqs = 1024;

// Sort key of a sequence: its total cost in log-spaced bins (exact below 64,
// then 64 bins per power of two), clamped to the histogram.
__device__ __forceinline__ int cost_bin(long long c) {
    if (c < 64) return (int)c;
    const int e = 63 - __clzll(c);  // >= 6
    const long long bin = 64 + (long long)(e - 6) * 64 + ((c >> (e - 6)) & 63);
    return bin < kCostBins - 1 ? (int)bin : kCostBins - 1;
}

// Block-wide exclusive scan of one int per thread (1024 threads); returns the
// exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int x, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = x;
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = inc - x + (warp > 0 ? warp_sums[warp - 1] : 0);
    *total = warp_sums[31];
    __syncthreads();
    return excl;
}

// Sequence owning flattened query block i: the last b with seqs[b].pad <= i
// among sequences that have blocks (pad holds the first block index of b).
__device__ __forceinline__ int block_owner(const SeqInfo* seqs, int num_seqs, int i) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seqs[mid].pad <= i)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// KV heads of a sequence whose units run together.  Every unit of a head
// streams that head's K/V from the start of the sequence, so while the CTAs
// work on a group of heads, the group's K/V (keys and values of P + n tokens,
// bf16) is what they re-read from L2; groups are sized to keep it within
// kL2GroupBytes (a share of the 129 MB L2 that leaves room for the q, out and
// cache-write streams and for the next group, which starts while the last
// units of a group run).  A group must also hold at least num_ctas times the
// sequence's longest unit of work (head_cost = the KV tiles of one head's
// units, longest = the most of one unit): a group's longest unit starts when
// the group does, so a smaller last group would end the launch on that one
// unit while the other SMs idle.  That bound wins over the L2 budget.  Short
// sequences keep all their heads in one group.
__device__ __forceinline__ int kv_head_group(const SeqInfo& si, int head_dim, int n_kv_heads, int num_ctas,
                                             long long head_cost, int longest) {
    const float head_bytes = (float)(si.P + si.n) * (float)(head_dim * 4);
    float g = floorf((float)kL2GroupBytes / fmaxf(head_bytes, 1.f));
    if (head_cost > 0) g = fmaxf(g, ceilf((float)num_ctas * (float)longest / (float)head_cost));
    return g >= (float)n_kv_heads ? n_kv_heads : (g < 1.f ? 1 : (int)g);
}

__global__ void __launch_bounds__(1024) build_schedule_kernel(ScheduleArgs a) {
    __shared__ int hist[kCostBins];
    __shared__ int warp_sums[32];
    __shared__ SeqInfo s_seqs[kSmemSeqs];
    __shared__ int s_scratch[kSmemSeqs], s_group[kSmemSeqs];
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int tpu = a.unit_slots * (kBlockM / a.group);  // query tokens per unit
    // the next kernel (launched with programmatic stream serialisation) may
    // start its prologue now; it waits for this kernel before reading the list
    griddep_launch();
    // where the passes keep their per-sequence tables (the attention kernel
    // reads the sequences from a.seqs, which pass 1 always writes)
    const bool small = a.num_seqs <= kSmemSeqs;
    SeqInfo* const seqs = small ? s_seqs : a.seqs;
    int* const seq_scratch = small ? s_scratch : a.seq_scratch;
    int* const seq_group = small ? s_group : a.seq_group;

    for (int i = tid; i < kCostBins; i += nthr) hist[i] = 0;

    // Paged cache: every block a sequence touches (positions [0, P + n)) must be
    // a block of the pool; a sequence that names another is rejected below.
    // One warp per sequence; the verdict waits in SeqInfo::pad until pass 1.
    const bool paged = a.block_table != nullptr;
    if (paged) {
        const int lane = tid & 31, nwarps = nthr >> 5;
        for (int b = tid >> 5; b < a.num_seqs; b += nwarps) {
            const long long lk = (long long)a.cu_seqlens_k[b + 1] - a.cu_seqlens_k[b];
            const long long used = lk > 0 ? (lk + a.block_size - 1) / a.block_size : 0;
            const int nb = used < a.max_blocks ? (int)used : a.max_blocks;
            bool bad = false;
            for (int L = lane; L < nb; L += 32) {
                const int blk = a.block_table[(size_t)b * a.max_blocks + L];
                bad |= blk < 0 || blk >= a.num_blocks;
            }
            bad = __any_sync(0xffffffffu, bad);
            if (lane == 0) seqs[b].pad = bad ? 1 : 0;
        }
        __threadfence_block();
        __syncthreads();
    }

    // Pass 1: sanitise each sequence; number its query blocks (first block
    // index of b goes to SeqInfo::pad) with a block-wide scan per 1024 sequences.
    int blocks_before = 0;
    for (int b0 = 0; b0 < a.num_seqs; b0 += nthr) {
        const int b = b0 + tid;
        SeqInfo si{0, 0, 0, 0};
        if (b < a.num_seqs) {
            const int q_start = a.cu_seqlens_q[b];
            const int q_end = a.cu_seqlens_q[b + 1];
            const int lk = a.cu_seqlens_k[b + 1] - a.cu_seqlens_k[b];
            const int P = a.cache_offsets[b];
            const long long n = (long long)q_end - q_start;
            const bool ok = q_start >= 0 && n >= 0 && (long long)q_end <= a.total_q && P >= 0 &&
                            (long long)lk == (long long)P + n && (long long)P + n <= a.max_cache_len &&
                            (b > 0 || q_start == 0) && !(paged && seqs[b].pad != 0);
            if (!ok) atomicOr(&a.hdr->error, PA_DEVERR_METADATA);
            si.q_start = ok ? q_start : 0;
            si.n = ok ? (int)n : 0;
            si.P = ok ? P : 0;
        }
        const int nblk = (si.n + tpu - 1) / tpu;
        int chunk_total;
        const int excl = block_exclusive_scan(nblk, warp_sums, &chunk_total);
        si.pad = blocks_before + excl;
        if (b < a.num_seqs) {
            a.seqs[b] = si;
            if (small) s_seqs[b] = si;
        }
        blocks_before += chunk_total;
    }
    const int total_blocks = blocks_before;
    __threadfence_block();
    __syncthreads();

    // Pass 2 (one warp per sequence): total cost of the sequence's units; the
    // histogram counts units per cost bin, the bin waits in seq_scratch, the
    // sequence's KV-head group size in seq_group.
    {
        const int lane = tid & 31, nwarps = nthr >> 5;
        for (int b = tid >> 5; b < a.num_seqs; b += nwarps) {
            const SeqInfo si = seqs[b];
            const int nblk = (si.n + tpu - 1) / tpu;
            long long c = 0;
            int mx = 0;
            for (int i = lane; i < nblk; i += 32) {
                const int t = unit_tiles(si.n, si.P, i * tpu, tpu, a.causal, a.window, paged);
                c += t;
                mx = max(mx, t);
            }
            for (int o = 16; o > 0; o >>= 1) {
                c += __shfl_xor_sync(0xffffffffu, c, o);
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            }
            if (lane == 0 && nblk > 0) {
                const int bin = cost_bin(c * a.n_kv_heads);
                seq_scratch[b] = bin;
                seq_group[b] = kv_head_group(si, a.head_dim, a.n_kv_heads, a.num_ctas, c, mx);
                atomicAdd(&hist[bin], nblk * a.n_kv_heads);
            }
        }
    }
    __threadfence_block();
    __syncthreads();

    // Exclusive scan in DESCENDING cost order: start[c] = sum of hist[c'] for c' > c.
    static_assert(kCostBins == 2 * 1024, "scan assumes two bins per thread");
    const int r0 = kCostBins - 1 - 2 * tid;  // this thread's bins: r0, then r0 - 1
    const int h0 = hist[r0], h1 = hist[r0 - 1];
    int total;
    const int excl = block_exclusive_scan(h0 + h1, warp_sums, &total);
    hist[r0] = excl;
    hist[r0 - 1] = excl + h0;
    if (tid == 0) {
        a.hdr->num_units = total < a.max_units ? total : a.max_units;
        a.hdr->counter = 0;
        a.hdr->max_units = a.max_units;
        if (total > a.max_units) atomicOr(&a.hdr->error, PA_DEVERR_OVERFLOW);
    }
    __syncthreads();

    // Pass 3: each sequence claims its range of the list from its bin ...
    for (int b = tid; b < a.num_seqs; b += nthr) {
        const int nblk = (seqs[b].n + tpu - 1) / tpu;
        if (nblk > 0) seq_scratch[b] = atomicAdd(&hist[seq_scratch[b]], nblk * a.n_kv_heads);
    }
    __threadfence_block();
    __syncthreads();

    // ... and its units go there: its KV heads in groups whose K/V fit the L2
    // budget, and within a group the query blocks last to first with the
    // group's heads adjacent.  One unit per thread and iteration.
    const int total_units = total_blocks * a.n_kv_heads;  // < 2^31: the host bounds the units
    for (int w = tid; w < total_units; w += nthr) {
        const int i = w / a.n_kv_heads, kvh = w % a.n_kv_heads;
        const int b = block_owner(seqs, a.num_seqs, i);
        const SeqInfo si = seqs[b];
        const int blk = i - si.pad;
        const int nblk = (si.n + tpu - 1) / tpu;
        const int hg = seq_group[b];
        const int g0 = kvh - kvh % hg;                 // first head of kvh's group
        const int gsize = min(hg, a.n_kv_heads - g0);  // heads in the group
        const int pos = seq_scratch[b] + g0 * nblk + (nblk - 1 - blk) * gsize + (kvh - g0);
        if (pos < a.max_units) {
            Unit u;
            u.b = b;
            u.kvh = kvh;
            u.q0 = blk * tpu;
            u.ntiles = unit_tiles(si.n, si.P, u.q0, tpu, a.causal, a.window, paged);
            a.units[pos] = u;
        }
    }
}

cudaError_t launch_build_schedule(const ScheduleArgs& a, cudaStream_t stream) {
    build_schedule_kernel<<<1, 1024, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pa
