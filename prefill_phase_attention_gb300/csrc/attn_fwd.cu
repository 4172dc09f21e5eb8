// attn_fwd.cu -- warp-specialised causal varlen prefill attention for sm_103a.
//
// Computes out = softmax(Q K^T * scale) V per work unit (128 query rows of one
// sequence sharing one KV head; GQA heads packed into the rows) over the
// unit's KV tiles -- the cached prefix read from the KV cache, then the
// sequence's own new keys -- and writes the new K/V into the cache.
//
// The method (pages, by title and section):
//  - scaled dot-product attention, each row normalised over all visible keys:
//    "大语言模型推理核心：Prefill与Decode原理及工程优化" (yfxerp.com) §2.2;
//  - tiled attention that never materialises the T x T score matrix and
//    computes only the lower-triangular blocks of the causal mask: untitled
//    page on prefill/decode compute accounting (zwxr.cn) §3.3, and
//    "Prefill不是热身：大模型推理的真正瓶颈与优化核心" (mhpn.cn) §4;
//  - varlen batches indexed by cu_seqlens, each request attending only to
//    itself: "大模型 Prompt Prefill 阶段的高效 Batching 与算子排布" (nxmr.cn) §2;
//  - chunked prefill over a cached prefix, mixed with one-token decode rows:
//    same page §3; prefill as the writer of every new token's K/V
//    (mhpn.cn §1, §4; yfxerp.com §2.1).
//
// GB300 mapping (one persistent CTA per SM, 384 threads, all 512 TMEM columns):
//   warp 0      TMA producer: fetches units from the longest-first list,
//               loads Q once per unit and K tiles into a kStages ring;
//   warp 2      TMA producer of the V tiles (a ring of its own, so K runs
//               ahead of S while V waits for the PV products);
//   warp 1      tcgen05 issuer: S = Q K^T (SS form, bf16 -> fp32 in TMEM,
//               double-buffered, issued two tiles ahead of PV) and O += P V
//               (P read from TMEM, V MN-major);
//   warps 3,12  cache writers (K, V): copy the unit's own new K/V rows out of
//               the staged tiles in shared memory into the cache (16-byte
//               stores); second releaser of every ring stage;
//   warps 4-11  softmax: two warps per TMEM sub-partition, each thread one
//               query row (TMEM lane) and one half of the key columns; online
//               max/sum in fp32 registers (partial maxima swapped through
//               shared memory), exp2 on the MUFU, P packed to bf16 into TMEM,
//               lazy O rescale, epilogue out = O / l (bf16) and LSE.
// Every wait is bounded in time; on timeout the CTA records PA_DEVERR_TIMEOUT,
// drains its in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "prefill_attn.h"
#include "ptx.cuh"

namespace pa {
using namespace ptx;

namespace {

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int kThreads = 416;  // 5 control warps + 8 softmax warps
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP0 = 384, kColP1 = 448;

template <int D>
struct Cfg {
    static constexpr int kChunkCols = D >= 64 ? 64 : 32;  // columns per swizzle atom row
    static constexpr int kChunks = D / kChunkCols;
    static constexpr int kRowBytes = kChunkCols * 2;
    static constexpr int kChunkBytes = kBlockM * kRowBytes;
    static constexpr int kTileBytes = kChunks * kChunkBytes;  // 128 rows x D bf16
    static constexpr SmemSwizzle kSw = D >= 64 ? kSwizzle128B : kSwizzle64B;
    static constexpr int kSbo = 8 * kRowBytes;  // byte distance between 8-row groups
    static constexpr int kStages = D == 128 ? 3 : 4;
    static constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
    static constexpr uint32_t kIdescO = idesc_bf16_f32(kBlockM, D, 0, 1);
};

struct UnitSlot {
    Unit u;
    SeqInfo s;
};

struct __align__(8) Ctrl {
    uint64_t q_full, q_empty;
    uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
    uint64_t s_full[2], s_empty[2], p_full[2], pv_done[2];
    uint64_t o_empty, mma_drain;
    uint64_t unit_full[2], unit_empty[2];
    uint64_t xchg[4];          // per sub-partition: the two softmax warps of the same rows
    UnitSlot slot[2];
    uint32_t tmem_base;
    int abort;
    float xbuf[2][2][kBlockM];  // [exchange parity][column half][row]
};

// Tiles first (the dynamic shared window starts 1024-byte aligned, which the
// kernel checks), control block after them.  At least 120 KB so that a second
// CTA never lands on an SM (each CTA holds all 512 TMEM columns).
template <int D>
constexpr int smem_bytes() {
    return (Cfg<D>::kTileBytes * (1 + 2 * Cfg<D>::kStages) + (int)sizeof(Ctrl)) > 120 * 1024
               ? Cfg<D>::kTileBytes * (1 + 2 * Cfg<D>::kStages) + (int)sizeof(Ctrl)
               : 120 * 1024;
}

__device__ __forceinline__ bool aborted(const Ctrl* c) { return *reinterpret_cast<const volatile int*>(&c->abort) != 0; }

// Bounded wait; gives up when the CTA has aborted or after kTimeoutNs, in
// which case it flags the CTA and the device error word.
__device__ __noinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Ctrl* c, WorkspaceHeader* hdr) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (aborted(c)) return false;
        if (globaltimer_ns() - t0 > kTimeoutNs) {
            *reinterpret_cast<volatile int*>(&c->abort) = 1;
            atomicOr(&hdr->error, PA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// Warp-uniform bounded wait: every lane polls, then the warp agrees, so the
// warp stays converged for the .sync.aligned tcgen05 instructions that follow.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, Ctrl* c, WorkspaceHeader* hdr) {
    const bool ok = wait_bar(bar, parity, c, hdr);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// First key (absolute position in the sequence) of KV tile j of a unit whose
// sequence has P cached tokens split into np = ceil(P / 128) prefix tiles.
__device__ __forceinline__ int tile_key_base(int j, int P, int np) {
    return j < np ? P - kBlockN * (np - j) : P + kBlockN * (j - np);
}

// Rows of new-key tile j (j >= np) that hold this unit's own tokens
// [q0, q_end): tile rows [lo_row, lo_row + nrows).  The unit writes exactly
// these tokens' K/V into the cache.
__device__ __forceinline__ bool own_rows(int j, int np, int q0, int q_end, int& lo_row, int& nrows) {
    if (j < np) return false;
    const int k0 = (j - np) * kBlockN;
    const int lo = max(q0, k0), hi = min(q_end, k0 + kBlockN);
    if (lo >= hi) return false;
    lo_row = lo - k0;
    nrows = hi - lo;
    return true;
}

// Copies rows [lo_row, lo_row + nrows) of a swizzled K or V tile in shared
// memory to consecutive cache rows starting at `dst` (one warp; 16-byte
// granules, the warp's stores cover contiguous cache rows).
template <int D>
__device__ __forceinline__ void copy_tile_rows(const uint8_t* tile, __nv_bfloat16* dst, int lo_row, int nrows,
                                               int lane) {
    using C = Cfg<D>;
    constexpr int kGran = D / 8;               // 16-byte granules per row
    constexpr int kChunkGran = C::kChunkCols / 8;
    const int total = nrows * kGran;
#pragma unroll 4
    for (int idx = lane; idx < total; idx += 32) {
        const int r = lo_row + idx / kGran, g = idx % kGran;
        const int c = g / kChunkGran, gg = g % kChunkGran;
        const int phys = D >= 64 ? (gg ^ (r & 7)) : (gg ^ ((r >> 1) & 3));
        const uint4 x = *reinterpret_cast<const uint4*>(tile + c * C::kChunkBytes + r * C::kRowBytes + phys * 16);
        *reinterpret_cast<uint4*>(dst + (size_t)(idx / kGran) * D + g * 8) = x;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // swizzled TMA/UMMA tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicOr(&p.hdr->error, PA_DEVERR_TIMEOUT);
        return;
    }
    uint8_t* q_smem = smem_raw;
    uint8_t* k_smem = q_smem + C::kTileBytes;
    uint8_t* v_smem = k_smem + C::kStages * C::kTileBytes;
    Ctrl* ctl = reinterpret_cast<Ctrl*>(v_smem + C::kStages * C::kTileBytes);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    WorkspaceHeader* hdr = p.hdr;
    const int G = p.group;
    const int tpu = kBlockM / G;

    if (threadIdx.x == 0) {
        mbar_init(&ctl->q_full, 1);
        mbar_init(&ctl->q_empty, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&ctl->k_full[s], 1);
            mbar_init(&ctl->k_empty[s], 2);  // MMA commit + cache writer
            mbar_init(&ctl->v_full[s], 1);
            mbar_init(&ctl->v_empty[s], 2);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->s_full[b], 1);
            mbar_init(&ctl->s_empty[b], 8);
            mbar_init(&ctl->p_full[b], 8);
            mbar_init(&ctl->pv_done[b], 1);
            mbar_init(&ctl->unit_full[b], 1);
            mbar_init(&ctl->unit_empty[b], 12);  // MMA + V loader + 2 cache writers + 8 softmax warps
        }
        for (int i = 0; i < 4; ++i) mbar_init(&ctl->xchg[i], 2);
        mbar_init(&ctl->o_empty, 8);
        mbar_init(&ctl->mma_drain, 1);
        ctl->abort = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tm_q);
        prefetch_tmap(&p.tm_k);
        prefetch_tmap(&p.tm_v);
        prefetch_tmap(&p.tm_ck);
        prefetch_tmap(&p.tm_cv);
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    // One KV ring (K or V): waits for the stage, then TMA-loads tile j of the
    // unit from the cache (prefix tiles) or from the new tokens' k/v.
    auto load_kv_tile = [&](uint8_t* ring, uint64_t* full, uint64_t* empty, const CUtensorMap* tm_cache,
                            const CUtensorMap* tm_new, int* last_parity, uint32_t t, int j, const Unit& u,
                            const SeqInfo& s, int np) -> bool {
        const int st = t % C::kStages;
        const uint32_t ph = (t / C::kStages) & 1;
        if (!wait_bar(&empty[st], ph ^ 1, ctl, hdr)) return false;
        const int kb = tile_key_base(j, s.P, np);
        mbar_arrive_expect_tx(&full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
            uint8_t* dst = ring + st * C::kTileBytes + c * C::kChunkBytes;
            if (j < np)
                tma_load_3d(dst, tm_cache, &full[st], c * C::kChunkCols, kb, u.b * p.n_kv_heads + u.kvh);
            else
                tma_load_3d(dst, tm_new, &full[st], c * C::kChunkCols, u.kvh, s.q_start + kb - s.P);
        }
        last_parity[st] = (int)ph;
        return true;
    };
    // On abort, let every copy a producer thread started land before the CTA exits.
    auto drain = [&](uint64_t* bars, const int* last_parity, int n) {
        const uint64_t t0 = globaltimer_ns();
        for (int i = 0; i < n; ++i) {
            if (last_parity[i] < 0) continue;
            while (!mbar_try_wait(&bars[i], (uint32_t)last_parity[i]) && globaltimer_ns() - t0 < kTimeoutNs) {
            }
        }
    };

    if (warp == 0) {
        // --------------------------------------------- unit fetch, Q and K loads
        if (lane == 0) {
            const int num_units = hdr->num_units;
            uint32_t t = 0;
            int last_q_parity[1] = {-1};
            int last_k_parity[4] = {-1, -1, -1, -1};
            for (int u_it = 0;; ++u_it) {
                const int sl = u_it & 1;
                if (!wait_bar(&ctl->unit_empty[sl], ((u_it >> 1) & 1) ^ 1, ctl, hdr)) break;
                const int idx = atomicAdd(&hdr->counter, 1);
                UnitSlot us;
                if (idx < num_units) {
                    us.u = p.units[idx];
                    us.s = p.seqs[us.u.b];
                } else {
                    us.u.b = -1;
                }
                ctl->slot[sl] = us;
                mbar_arrive(&ctl->unit_full[sl]);
                if (us.u.b < 0) break;
                const Unit u = us.u;
                const SeqInfo s = us.s;
                // Q tile: rows (token, head-in-group) of this unit
                if (!wait_bar(&ctl->q_empty, (u_it & 1) ^ 1, ctl, hdr)) break;
                mbar_arrive_expect_tx(&ctl->q_full, G * tpu * C::kRowBytes * C::kChunks);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(q_smem + c * C::kChunkBytes, &p.tm_q, &ctl->q_full, c * C::kChunkCols, u.kvh * G,
                                s.q_start + u.q0);
                last_q_parity[0] = u_it & 1;
                const int np = (s.P + kBlockN - 1) / kBlockN;
                bool ok = true;
                for (int j = 0; j < u.ntiles && ok; ++j, ++t)
                    ok = load_kv_tile(k_smem, ctl->k_full, ctl->k_empty, &p.tm_ck, &p.tm_k, last_k_parity, t, j, u,
                                      s, np);
                if (!ok) break;
            }
            if (aborted(ctl)) {
                drain(&ctl->q_full, last_q_parity, 1);
                drain(ctl->k_full, last_k_parity, C::kStages);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------- V loads
        // A ring of its own, so K tiles run ahead of S while V tiles wait for PV.
        if (lane == 0) {
            uint32_t t = 0;
            int last_v_parity[4] = {-1, -1, -1, -1};
            for (int u_it = 0;; ++u_it) {
                const int sl = u_it & 1;
                if (!wait_bar(&ctl->unit_full[sl], (u_it >> 1) & 1, ctl, hdr)) break;
                const UnitSlot us = ctl->slot[sl];
                mbar_arrive(&ctl->unit_empty[sl]);
                if (us.u.b < 0) break;
                const int np = (us.s.P + kBlockN - 1) / kBlockN;
                bool ok = true;
                for (int j = 0; j < us.u.ntiles && ok; ++j, ++t)
                    ok = load_kv_tile(v_smem, ctl->v_full, ctl->v_empty, &p.tm_cv, &p.tm_v, last_v_parity, t, j,
                                      us.u, us.s, np);
                if (!ok) break;
            }
            if (aborted(ctl)) drain(ctl->v_full, last_v_parity, C::kStages);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t q_addr = smem_u32(q_smem);
            const uint32_t k_addr = smem_u32(k_smem);
            const uint32_t v_addr = smem_u32(v_smem);
            uint32_t t = 0;
            bool ok = true;
            for (int u_it = 0; ok; ++u_it) {
                const int sl = u_it & 1;
                if (!wait_bar(&ctl->unit_full[sl], (u_it >> 1) & 1, ctl, hdr)) break;
                const Unit u = ctl->slot[sl].u;
                mbar_arrive(&ctl->unit_empty[sl]);
                if (u.b < 0) break;
                if (!wait_bar(&ctl->q_full, u_it & 1, ctl, hdr)) break;
                auto issue_pv = [&](uint32_t tp, bool first) -> bool {
                    const int stp = tp % C::kStages;
                    const uint32_t bp = tp & 1;
                    if (!wait_bar(&ctl->p_full[bp], (tp >> 1) & 1, ctl, hdr)) return false;
                    if (!wait_bar(&ctl->v_full[stp], (tp / C::kStages) & 1, ctl, hdr)) return false;
                    if (first && !wait_bar(&ctl->o_empty, (u_it & 1) ^ 1, ctl, hdr)) return false;
                    tc_fence_after();
                    const uint32_t vb = v_addr + stp * C::kTileBytes;
                    const uint32_t pcol = bp ? kColP1 : kColP0;
#pragma unroll
                    for (int kk = 0; kk < kBlockN / 16; ++kk) {
                        const uint64_t bd = smem_desc(vb + kk * 2 * C::kSbo, C::kChunkBytes, C::kSbo, C::kSw);
                        mma_ts(tmem + kColO, tmem + pcol + kk * 8, bd, C::kIdescO, (!first || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&ctl->pv_done[bp]);
                    mma_commit(&ctl->v_empty[stp]);
                    return true;
                };
                for (int j = 0; j < u.ntiles; ++j, ++t) {
                    const int st = t % C::kStages;
                    const uint32_t b = t & 1;
                    if (!wait_bar(&ctl->k_full[st], (t / C::kStages) & 1, ctl, hdr)) { ok = false; break; }
                    if (!wait_bar(&ctl->s_empty[b], ((t >> 1) & 1) ^ 1, ctl, hdr)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t kb = k_addr + st * C::kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int c = (kk * 16) / C::kChunkCols, w = (kk * 16) % C::kChunkCols;
                        const uint64_t ad = smem_desc(q_addr + c * C::kChunkBytes + w * 2, 16, C::kSbo, C::kSw);
                        const uint64_t bd = smem_desc(kb + c * C::kChunkBytes + w * 2, 16, C::kSbo, C::kSw);
                        mma_ss(tmem + (b ? kColS1 : kColS0), ad, bd, C::kIdescS, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&ctl->s_full[b]);
                    mma_commit(&ctl->k_empty[st]);
                    if (j == u.ntiles - 1) mma_commit(&ctl->q_empty);
                    // S runs two tiles ahead of PV: S(t+1) never waits behind
                    // the softmax of tile t-1.
                    if (j >= 2 && !issue_pv(t - 2, j == 2)) { ok = false; break; }
                }
                // the unit's last (up to two) PV products
                if (ok && u.ntiles >= 2 && !issue_pv(t - 2, u.ntiles == 2)) ok = false;
                if (ok && !issue_pv(t - 1, u.ntiles == 1)) ok = false;
            }
            // every MMA this thread issued has finished before TMEM is released
            mma_commit(&ctl->mma_drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&ctl->mma_drain, 0) && globaltimer_ns() - t0 < kTimeoutNs) {
            }
        }
    } else if (warp == 3 || warp == 12) {
        // -------------------------------------------------------- cache writers
        // Warp 3 writes K, warp 12 writes V.  Each walks every tile of its ring
        // in order and is the second releaser of every stage (with the MMA
        // commit), so it never waits on a barrier phase more than one ahead or
        // behind; on the tiles holding the unit's own tokens it first copies
        // those rows from shared memory into the cache.
        const bool is_k = warp == 3;
        uint8_t* ring = is_k ? k_smem : v_smem;
        uint64_t* full = is_k ? ctl->k_full : ctl->v_full;
        uint64_t* empty = is_k ? ctl->k_empty : ctl->v_empty;
        __nv_bfloat16* cache = is_k ? p.cache_k : p.cache_v;
        uint32_t t = 0;
        for (int u_it = 0;; ++u_it) {
            const int sl = u_it & 1;
            if (!warp_wait(&ctl->unit_full[sl], (u_it >> 1) & 1, ctl, hdr)) break;
            const UnitSlot us = ctl->slot[sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->unit_empty[sl]);
            if (us.u.b < 0) break;
            const int np = (us.s.P + kBlockN - 1) / kBlockN;
            const int q_end = min(us.u.q0 + tpu, us.s.n);
            bool ok = true;
            for (int j = 0; j < us.u.ntiles; ++j, ++t) {
                const int st = t % C::kStages;
                if (!warp_wait(&full[st], (t / C::kStages) & 1, ctl, hdr)) { ok = false; break; }
                int lo_row, nrows;
                if (own_rows(j, np, us.u.q0, q_end, lo_row, nrows)) {
                    const int first_tok = (j - np) * kBlockN + lo_row;  // token index within the sequence
                    __nv_bfloat16* dst = cache + (((size_t)us.u.b * p.n_kv_heads + us.u.kvh) * p.max_cache_len +
                                                  us.s.P + first_tok) * D;
                    copy_tile_rows<D>(ring + st * C::kTileBytes, dst, lo_row, nrows, lane);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------------- softmax
        // Warps 4-11.  Sub-partition sp = warp % 4 owns TMEM lanes (= query rows)
        // [32 sp, 32 sp + 32); half hf takes S columns [64 hf, 64 hf + 64) and
        // O columns [D/2 hf, D/2 hf + D/2).  The two warps of the same rows swap
        // their partial row max (every tile) and row sum (epilogue) through
        // shared memory.
        constexpr int kHalfN = kBlockN / 2;
        constexpr int kHalfD = D / 2;
        const int sp = warp & 3;
        const int hf = (warp - 4) >> 2;
        const int r = sp * 32 + lane;  // query row of the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
        const float sl2 = p.scale_log2;
        uint32_t t = 0, xc = 0;
        // swap one float with the partner warp; returns the partner's value
        auto exchange = [&](float mine, float& theirs) -> bool {
            ctl->xbuf[xc & 1][hf][r] = mine;
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->xchg[sp]);
            if (!warp_wait(&ctl->xchg[sp], xc & 1, ctl, hdr)) return false;
            theirs = ctl->xbuf[xc & 1][hf ^ 1][r];
            ++xc;
            return true;
        };
        for (int u_it = 0;; ++u_it) {
            const int sl = u_it & 1;
            if (!warp_wait(&ctl->unit_full[sl], (u_it >> 1) & 1, ctl, hdr)) break;
            const UnitSlot us = ctl->slot[sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->unit_empty[sl]);
            if (us.u.b < 0) break;
            const Unit u = us.u;
            const SeqInfo s = us.s;
            const int tok = u.q0 + r / G;
            const int h = u.kvh * G + r % G;
            const bool valid = r < tpu * G && tok < s.n;
            const int Lk = s.P + s.n;
            const int row_hi = p.causal ? min(s.P + tok + 1, Lk) : Lk;  // keys [0, row_hi) visible
            const int unit_hi = p.causal ? min(s.P + u.q0 + 1, Lk) : Lk;  // smallest row_hi of the unit
            const int np = (s.P + kBlockN - 1) / kBlockN;
            float m = -INFINITY, l = 0.f;  // l: this half's share of the row sum
            bool ok = true;
            for (int j = 0; j < u.ntiles; ++j, ++t) {
                const uint32_t b = t & 1;
                if (!warp_wait(&ctl->s_full[b], (t >> 1) & 1, ctl, hdr)) { ok = false; break; }
                tc_fence_after();
                float sv[kHalfN];
                {
                    uint32_t r0[32], r1[32];
                    const uint32_t sa = tmem + lane_off + (b ? kColS1 : kColS0) + hf * kHalfN;
                    tmem_ld32(sa, r0);
                    tmem_ld32(sa + 32, r1);
                    tmem_wait_ld();
                    reg_fence(r0);
                    reg_fence(r1);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        sv[i] = __uint_as_float(r0[i]);
                        sv[32 + i] = __uint_as_float(r1[i]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->s_empty[b]);

                const int kb = tile_key_base(j, s.P, np);
                if (kb < 0 || kb + kBlockN > unit_hi) {
                    const int lo = -kb - hf * kHalfN, hi = row_hi - kb - hf * kHalfN;
#pragma unroll
                    for (int c = 0; c < kHalfN; ++c)
                        if (c < lo || c >= hi) sv[c] = -INFINITY;
                }
                float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
                for (int c = 4; c < kHalfN; c += 4) {
                    mx0 = fmaxf(mx0, sv[c]);
                    mx1 = fmaxf(mx1, sv[c + 1]);
                    mx2 = fmaxf(mx2, sv[c + 2]);
                    mx3 = fmaxf(mx3, sv[c + 3]);
                }
                float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)), mx_other;
                if (!exchange(mx, mx_other)) { ok = false; break; }
                const float m_tile = fmaxf(mx, mx_other) * sl2;
                const float m_new = fmaxf(m, m_tile);
                float alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m = m_new;
                } else {
                    const bool need = m_new > m + 8.f;  // both halves of a row decide alike
                    rescale = __any_sync(0xffffffffu, need);
                    if (need) {
                        alpha = ex2(m - m_new);
                        m = m_new;
                    }
                }
                const float m_use = m == -INFINITY ? 0.f : m;
                uint32_t pk[kHalfN / 2];
                float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
                for (int c = 0; c < kHalfN; c += 2) {
                    const float p0 = ex2(fmaf(sv[c], sl2, -m_use));
                    const float p1 = ex2(fmaf(sv[c + 1], sl2, -m_use));
                    sum0 += p0;
                    sum1 += p1;
                    pk[c / 2] = pack_bf16(p0, p1);
                }
                l = l * alpha + (sum0 + sum1);
                // P buffer b was last read by the PV MMA of tile t-2
                if (j >= 2 && !warp_wait(&ctl->pv_done[b], ((t >> 1) & 1) ^ 1, ctl, hdr)) { ok = false; break; }
                tmem_st32(tmem + lane_off + (b ? kColP1 : kColP0) + hf * (kHalfN / 2), pk);
                tmem_wait_st();
                if (rescale) {
                    // O must hold the PV of tile t-1 before it is scaled
                    if (!warp_wait(&ctl->pv_done[b ^ 1], ((t - 1) >> 1) & 1, ctl, hdr)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t oa = tmem + lane_off + kColO + hf * kHalfD;
                    if constexpr (kHalfD >= 32) {
#pragma unroll
                        for (int c = 0; c < kHalfD; c += 32) {
                            uint32_t o[32];
                            tmem_ld32(oa + c, o);
                            tmem_wait_ld();
                            reg_fence(o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(oa + c, o);
                        }
                    } else {
                        uint32_t o[16];
                        tmem_ld16(oa, o);
                        tmem_wait_ld();
                        reg_fence(o);
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st16(oa, o);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->p_full[b]);
            }
            if (!ok) break;
            // epilogue: O of the unit is final once the PV of its last tile is done
            float l_other;
            if (!exchange(l, l_other)) break;
            const float l_row = l + l_other;
            const uint32_t tl = t - 1;
            if (!warp_wait(&ctl->pv_done[tl & 1], (tl >> 1) & 1, ctl, hdr)) break;
            tc_fence_after();
            const float inv_l = 1.f / l_row;
            const size_t row = (size_t)(s.q_start + tok) * p.n_heads + h;
            uint4* dst = reinterpret_cast<uint4*>(p.out + row * D + hf * kHalfD);
            const uint32_t oa = tmem + lane_off + kColO + hf * kHalfD;
            auto store8 = [&](const uint32_t* o, int v) {
                uint4 w;
                w.x = pack_bf16(__uint_as_float(o[0]) * inv_l, __uint_as_float(o[1]) * inv_l);
                w.y = pack_bf16(__uint_as_float(o[2]) * inv_l, __uint_as_float(o[3]) * inv_l);
                w.z = pack_bf16(__uint_as_float(o[4]) * inv_l, __uint_as_float(o[5]) * inv_l);
                w.w = pack_bf16(__uint_as_float(o[6]) * inv_l, __uint_as_float(o[7]) * inv_l);
                dst[v] = w;
            };
            if constexpr (kHalfD >= 32) {
#pragma unroll
                for (int c = 0; c < kHalfD; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(oa + c, o);
                    tmem_wait_ld();
                    reg_fence(o);
                    if (valid) {
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) store8(o + v4 * 8, c / 8 + v4);
                    }
                }
            } else {
                uint32_t o[16];
                tmem_ld16(oa, o);
                tmem_wait_ld();
                reg_fence(o);
                if (valid) {
                    store8(o, 0);
                    store8(o + 8, 1);
                }
            }
            if (valid && hf == 0 && p.lse) p.lse[row] = (m + lg2(l_row)) * 0.69314718055994530942f;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->o_empty);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

cudaError_t encode3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                     uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle sw,
                     CUtensorMapL2promotion l2) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_d(const FwdParams& p, int grid, cudaStream_t st) {
    constexpr int kSmem = smem_bytes<D>();
    static_assert(kSmem <= 232448, "shared memory budget");
    static int configured_for[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured_for[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        configured_for[dev] = 1;
    }
    attn_fwd_kernel<D><<<grid, kThreads, kSmem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t encode_fwd_maps(FwdParams& p, const void* q, int total_q, int num_seqs, int head_dim) {
    const uint32_t cc = head_dim >= 64 ? 64 : 32;
    const CUtensorMapSwizzle sw = head_dim >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const uint64_t D = head_dim, H = p.n_heads, Hk = p.n_kv_heads, T = total_q, cap = p.max_cache_len;
    const uint32_t G = p.group, tpu = kBlockM / G;
    cudaError_t e;
    e = encode3d(&p.tm_q, q, D, H, T, D * 2, H * D * 2, cc, G, tpu, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
    if (e != cudaSuccess) return e;
    e = encode3d(&p.tm_k, p.k, D, Hk, T, D * 2, Hk * D * 2, cc, 1, kBlockN, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e != cudaSuccess) return e;
    e = encode3d(&p.tm_v, p.v, D, Hk, T, D * 2, Hk * D * 2, cc, 1, kBlockN, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e != cudaSuccess) return e;
    e = encode3d(&p.tm_ck, p.cache_k, D, cap, (uint64_t)num_seqs * Hk, D * 2, cap * D * 2, cc, kBlockN, 1, sw,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e != cudaSuccess) return e;
    return encode3d(&p.tm_cv, p.cache_v, D, cap, (uint64_t)num_seqs * Hk, D * 2, cap * D * 2, cc, kBlockN, 1, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

cudaError_t launch_attn_fwd(const FwdParams& p, int head_dim, int grid, cudaStream_t st) {
    switch (head_dim) {
        case 32: return launch_d<32>(p, grid, st);
        case 64: return launch_d<64>(p, grid, st);
        case 128: return launch_d<128>(p, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
