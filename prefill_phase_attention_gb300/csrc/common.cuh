// common.cuh -- types shared by the host shim, the tile scheduler and the
// attention kernels of the sm_103a prefill-attention library.
#pragma once

#include <cstdint>

namespace pa {

// Query rows per Q tile (one tcgen05 MMA M), Q tiles per work unit (they share
// every K/V tile), and keys per KV tile (MMA N of S = Q K^T).
constexpr int kBlockM = 128;
constexpr int kSlots = 2;
constexpr int kBlockN = 128;

// Cost histogram of the longest-first scheduler (costs above the last bin share it).
constexpr int kCostBins = 2048;

// Sanitised per-sequence metadata written by the scheduler.
struct SeqInfo {
    int q_start;  // first row of the sequence in the flattened q/k/v/out stream
    int n;        // new tokens (0 when the sequence is empty or its metadata was rejected)
    int P;        // cached prefix length = cache position of the first new token
    int pad;      // scheduler scratch: index of the sequence's first query block
};

// One work unit: query block [q0, q0 + 2 * (128/G)) of sequence b against KV
// head kvh, split into two Q tiles ("slots") of 128/G tokens; in each tile the
// G query heads of that KV head are packed into the 128 rows
// (row r <-> token q0 + slot * 128/G + r / G, head kvh * G + r % G).  With
// ScheduleArgs::unit_slots = 1 (the one-tile schedule) a unit is one Q tile,
// [q0, q0 + 128/G).
struct Unit {
    int b;
    int kvh;
    int q0;
    int ntiles;  // KV tiles the unit visits (its cost; the later slot visits all of them)
};

// Device workspace header; SeqInfo[num_seqs] and Unit[max_units] follow it.
struct WorkspaceHeader {
    int error;       // PA_DEVERR_* bits, sticky until read by prefill_attn_device_status
    int num_units;   // written by the scheduler
    int counter;     // dynamic work counter, reset by the scheduler
    int max_units;   // capacity of the unit list (informational copy)
};

struct ScheduleArgs {
    const int32_t* cu_seqlens_q;
    const int32_t* cu_seqlens_k;
    const int32_t* cache_offsets;
    WorkspaceHeader* hdr;
    SeqInfo* seqs;
    Unit* units;
    int* seq_scratch;  // [num_seqs] scheduler scratch (cost bin, then first unit of the sequence)
    int* seq_group;    // [num_seqs] scheduler scratch (KV heads per L2 group)
    int num_seqs;
    int total_q;
    int max_cache_len;
    int n_kv_heads;
    int head_dim;
    int group;      // n_heads / n_kv_heads
    int causal;
    int window;     // sliding window (0: none)
    int max_units;  // capacity of the unit list
    int num_ctas;   // CTAs of the attention launch (persistent: at most one per SM)
    int unit_slots; // Q tiles per unit: 2 (plain kernel) or 1 (alternating variant)
    // paged cache (block_table == nullptr: contiguous slots)
    const int32_t* block_table;  // [num_seqs][max_blocks]
    int block_size, max_blocks, num_blocks;
};

// KV tiles of a sequence with P cached tokens.  The new keys [P, P + n) are
// cut into tiles that START at P: tile j >= np = ceil(P / 128) covers keys
// [P + 128 (j - np), ...).  The prefix [0, P) is cut into np tiles that
//  - contiguous cache: END at P (tile j covers [P - 128 (np - j), ...); the
//    first may start below 0 and is masked there), so no tile ever reads
//    cache entries at or past P;
//  - paged cache: START at 0 (tile j covers [128 j, 128 j + 128)), so every
//    tile is a whole number of cache blocks (or a block-aligned part of one);
//    the last one is masked from P on.
__host__ __device__ inline int prefix_tiles(int P) { return (P + kBlockN - 1) / kBlockN; }

// Tile holding key position `key` (0 <= key < P + n).
__host__ __device__ inline int key_tile(int key, int P, bool paged) {
    const int np = prefix_tiles(P);
    if (key >= P) return np + (key - P) / kBlockN;
    return paged ? key / kBlockN : np - (P - key + kBlockN - 1) / kBlockN;
}

struct TileSpan {
    int lo, hi;  // tile indices [lo, hi)
};

// Tiles holding the keys that query tokens [qs, qe) (0 <= qs < qe <= n) see:
// causal -> keys up to P + qe - 1, from P + qs - window + 1 when window > 0;
// not causal -> all P + n keys.
__host__ __device__ inline TileSpan query_tiles(int n, int P, int qs, int qe, int causal, int window, bool paged) {
    int klo = 0;
    if (causal && window > 0 && P + qs - window + 1 > 0) klo = P + qs - window + 1;
    const int khi = causal ? P + qe : P + n;  // exclusive
    TileSpan t;
    t.lo = key_tile(klo, P, paged);
    t.hi = key_tile(khi - 1, P, paged) + 1;
    return t;
}

// KV tiles a work unit streams (its cost): tokens [q0, min(q0 + tokens, n)).
__host__ __device__ inline int unit_tiles(int n, int P, int q0, int tokens_per_unit, int causal, int window,
                                          bool paged) {
    const TileSpan t =
        query_tiles(n, P, q0, (q0 + tokens_per_unit < n) ? q0 + tokens_per_unit : n, causal, window, paged);
    return t.hi - t.lo;
}

}  // namespace pa
