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
// (row r <-> token q0 + slot * 128/G + r / G, head kvh * G + r % G).
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
    int num_seqs;
    int total_q;
    int max_cache_len;
    int n_kv_heads;
    int group;      // n_heads / n_kv_heads
    int causal;
    int max_units;  // capacity of the unit list
};

// Number of KV tiles of a unit.  The prefix [0, P) is cut into tiles that END
// at P (the first one may start below 0 and is masked there), and the new keys
// [P, P + n) into tiles that START at P, so no tile ever reads cache entries at
// or past P.  Causal units stop at the tile holding their last query token.
__host__ __device__ inline int unit_tiles(int n, int P, int q0, int tokens_per_unit, int causal) {
    const int prefix_tiles = (P + kBlockN - 1) / kBlockN;
    const int q_end = (q0 + tokens_per_unit < n) ? q0 + tokens_per_unit : n;
    const int new_tiles = causal ? (q_end - 1) / kBlockN + 1 : (n + kBlockN - 1) / kBlockN;
    return prefix_tiles + new_tiles;
}

}  // namespace pa
