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
// GB300 mapping (one persistent CTA per SM, 256 threads, all 512 TMEM columns):
//   warp 0      TMA producer: fetches units from the longest-first list,
//               loads Q once per unit and K/V tiles into a kStages ring;
//   warp 1      tcgen05 issuer: S = Q K^T (SS form, bf16 -> fp32 in TMEM,
//               double-buffered) and O += P V (P read from TMEM, V MN-major);
//   warps 2-3   copy the unit's new K/V rows into the cache (16-byte stores);
//   warps 4-7   softmax: one query row per thread (TMEM lane), online max/sum
//               in fp32 registers, exp2 on the MUFU, P packed to bf16 into
//               TMEM, lazy O rescale, epilogue out = O / l (bf16) and LSE.
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
constexpr int kThreads = 256;
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
    UnitSlot slot[2];
    uint32_t tmem_base;
    int abort;
};

// At least 120 KB so that a second CTA never lands on an SM (each CTA holds
// all 512 TMEM columns).
template <int D>
constexpr int smem_bytes() {
    return (1024 + Cfg<D>::kTileBytes * (1 + 2 * Cfg<D>::kStages) + (int)sizeof(Ctrl)) > 120 * 1024
               ? 1024 + Cfg<D>::kTileBytes * (1 + 2 * Cfg<D>::kStages) + (int)sizeof(Ctrl)
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* q_smem = base;
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
            mbar_init(&ctl->k_empty[s], 1);
            mbar_init(&ctl->v_full[s], 1);
            mbar_init(&ctl->v_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->s_full[b], 1);
            mbar_init(&ctl->s_empty[b], 4);
            mbar_init(&ctl->p_full[b], 4);
            mbar_init(&ctl->pv_done[b], 1);
            mbar_init(&ctl->unit_full[b], 1);
            mbar_init(&ctl->unit_empty[b], 7);  // MMA lane + 2 copy warps + 4 softmax warps
        }
        mbar_init(&ctl->o_empty, 4);
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

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const int num_units = hdr->num_units;
            uint32_t t = 0;
            int last_q_parity = -1;
            int last_k_parity[4] = {-1, -1, -1, -1}, last_v_parity[4] = {-1, -1, -1, -1};
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
                last_q_parity = u_it & 1;
                const int np = (s.P + kBlockN - 1) / kBlockN;
                const int cache_row = u.b * p.n_kv_heads + u.kvh;
                bool ok = true;
                for (int j = 0; j < u.ntiles; ++j, ++t) {
                    const int st = t % C::kStages;
                    const uint32_t ph = (t / C::kStages) & 1;
                    const int kb = tile_key_base(j, s.P, np);
                    const bool from_cache = j < np;
                    if (!wait_bar(&ctl->k_empty[st], ph ^ 1, ctl, hdr)) { ok = false; break; }
                    mbar_arrive_expect_tx(&ctl->k_full[st], C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        uint8_t* dst = k_smem + st * C::kTileBytes + c * C::kChunkBytes;
                        if (from_cache)
                            tma_load_3d(dst, &p.tm_ck, &ctl->k_full[st], c * C::kChunkCols, kb, cache_row);
                        else
                            tma_load_3d(dst, &p.tm_k, &ctl->k_full[st], c * C::kChunkCols, u.kvh, s.q_start + kb - s.P);
                    }
                    last_k_parity[st] = ph;
                    if (!wait_bar(&ctl->v_empty[st], ph ^ 1, ctl, hdr)) { ok = false; break; }
                    mbar_arrive_expect_tx(&ctl->v_full[st], C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        uint8_t* dst = v_smem + st * C::kTileBytes + c * C::kChunkBytes;
                        if (from_cache)
                            tma_load_3d(dst, &p.tm_cv, &ctl->v_full[st], c * C::kChunkCols, kb, cache_row);
                        else
                            tma_load_3d(dst, &p.tm_v, &ctl->v_full[st], c * C::kChunkCols, u.kvh, s.q_start + kb - s.P);
                    }
                    last_v_parity[st] = ph;
                }
                if (!ok) break;
            }
            if (aborted(ctl)) {
                // let every copy this thread started land before the CTA exits
                const uint64_t t0 = globaltimer_ns();
                auto drain = [&](uint64_t* bar, int par) {
                    if (par < 0) return;
                    while (!mbar_try_wait(bar, (uint32_t)par) && globaltimer_ns() - t0 < kTimeoutNs) {
                    }
                };
                drain(&ctl->q_full, last_q_parity);
                for (int s = 0; s < C::kStages; ++s) {
                    drain(&ctl->k_full[s], last_k_parity[s]);
                    drain(&ctl->v_full[s], last_v_parity[s]);
                }
            }
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
                    if (j > 0 && !issue_pv(t - 1, j == 1)) { ok = false; break; }
                }
                if (ok && !issue_pv(t - 1, u.ntiles == 1)) ok = false;
            }
            // every MMA this thread issued has finished before TMEM is released
            mma_commit(&ctl->mma_drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&ctl->mma_drain, 0) && globaltimer_ns() - t0 < kTimeoutNs) {
            }
        }
    } else if (warp < 4) {
        // -------------------------------------------------------- cache writers
        const int ct = (warp - 2) * 32 + lane;
        constexpr int kVec = D / 8;  // 16-byte vectors per row
        for (int u_it = 0;; ++u_it) {
            const int sl = u_it & 1;
            if (!warp_wait(&ctl->unit_full[sl], (u_it >> 1) & 1, ctl, hdr)) break;
            const UnitSlot us = ctl->slot[sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->unit_empty[sl]);
            if (us.u.b < 0) break;
            const int q_end = min(us.u.q0 + tpu, us.s.n);
            const int nvec = (q_end - us.u.q0) * kVec;
            const size_t slot_row = ((size_t)us.u.b * p.n_kv_heads + us.u.kvh) * p.max_cache_len + us.s.P;
            for (int i = ct; i < nvec; i += 64) {
                const int tk = us.u.q0 + i / kVec, c = i % kVec;
                const size_t src = ((size_t)(us.s.q_start + tk) * p.n_kv_heads + us.u.kvh) * D + c * 8;
                const size_t dst = (slot_row + tk) * D + c * 8;
                const uint4 kx = __ldg(reinterpret_cast<const uint4*>(p.k + src));
                const uint4 vx = __ldg(reinterpret_cast<const uint4*>(p.v + src));
                *reinterpret_cast<uint4*>(p.cache_k + dst) = kx;
                *reinterpret_cast<uint4*>(p.cache_v + dst) = vx;
            }
        }
    } else {
        // ------------------------------------------------------------- softmax
        const int r = (warp - 4) * 32 + lane;  // query row of the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)((warp - 4) * 32) << 16;
        const float sl2 = p.scale_log2;
        uint32_t t = 0;
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
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < u.ntiles; ++j, ++t) {
                const uint32_t b = t & 1;
                if (!warp_wait(&ctl->s_full[b], (t >> 1) & 1, ctl, hdr)) { ok = false; break; }
                tc_fence_after();
                float sv[kBlockN];
                {
                    uint32_t r0[32], r1[32], r2[32], r3[32];
                    const uint32_t sa = tmem + lane_off + (b ? kColS1 : kColS0);
                    tmem_ld32(sa, r0);
                    tmem_ld32(sa + 32, r1);
                    tmem_ld32(sa + 64, r2);
                    tmem_ld32(sa + 96, r3);
                    tmem_wait_ld();
                    reg_fence(r0);
                    reg_fence(r1);
                    reg_fence(r2);
                    reg_fence(r3);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        sv[i] = __uint_as_float(r0[i]);
                        sv[32 + i] = __uint_as_float(r1[i]);
                        sv[64 + i] = __uint_as_float(r2[i]);
                        sv[96 + i] = __uint_as_float(r3[i]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->s_empty[b]);

                const int kb = tile_key_base(j, s.P, np);
                if (kb < 0 || kb + kBlockN > unit_hi) {
                    const int lo = -kb, hi = row_hi - kb;
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c)
                        if (c < lo || c >= hi) sv[c] = -INFINITY;
                }
                float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
                for (int c = 4; c < kBlockN; c += 4) {
                    mx0 = fmaxf(mx0, sv[c]);
                    mx1 = fmaxf(mx1, sv[c + 1]);
                    mx2 = fmaxf(mx2, sv[c + 2]);
                    mx3 = fmaxf(mx3, sv[c + 3]);
                }
                const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
                const float m_new = fmaxf(m, m_tile);
                float alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m = m_new;
                } else {
                    const bool need = m_new > m + 8.f;
                    rescale = __any_sync(0xffffffffu, need);
                    if (need) {
                        alpha = ex2(m - m_new);
                        m = m_new;
                    }
                }
                const float m_use = m == -INFINITY ? 0.f : m;
                uint32_t pk[kBlockN / 2];
                float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
                for (int c = 0; c < kBlockN; c += 2) {
                    const float p0 = ex2(fmaf(sv[c], sl2, -m_use));
                    const float p1 = ex2(fmaf(sv[c + 1], sl2, -m_use));
                    sum0 += p0;
                    sum1 += p1;
                    pk[c / 2] = pack_bf16(p0, p1);
                }
                l = l * alpha + (sum0 + sum1);
                // P buffer b was last read by the PV MMA of tile t-2
                if (j >= 2 && !warp_wait(&ctl->pv_done[b], ((t >> 1) & 1) ^ 1, ctl, hdr)) { ok = false; break; }
                {
                    const uint32_t pcol = tmem + lane_off + (b ? kColP1 : kColP0);
                    uint32_t w32[32];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) w32[i] = pk[h2 * 32 + i];
                        tmem_st32(pcol + h2 * 32, w32);
                    }
                    tmem_wait_st();
                }
                if (rescale) {
                    // O must hold the PV of tile t-1 before it is scaled
                    if (!warp_wait(&ctl->pv_done[b ^ 1], ((t - 1) >> 1) & 1, ctl, hdr)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_off + kColO + c, o);
                        tmem_wait_ld();
                        reg_fence(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tmem + lane_off + kColO + c, o);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->p_full[b]);
            }
            if (!ok) break;
            // epilogue: O of the unit is final once the PV of its last tile is done
            const uint32_t tl = t - 1;
            if (!warp_wait(&ctl->pv_done[tl & 1], (tl >> 1) & 1, ctl, hdr)) break;
            tc_fence_after();
            const float inv_l = 1.f / l;
            const size_t row = (size_t)(s.q_start + tok) * p.n_heads + h;
            uint4* dst = reinterpret_cast<uint4*>(p.out + row * D);
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + kColO + c, o);
                tmem_wait_ld();
                reg_fence(o);
                if (valid) {
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(o[v4 * 8 + 0]) * inv_l, __uint_as_float(o[v4 * 8 + 1]) * inv_l);
                        w.y = pack_bf16(__uint_as_float(o[v4 * 8 + 2]) * inv_l, __uint_as_float(o[v4 * 8 + 3]) * inv_l);
                        w.z = pack_bf16(__uint_as_float(o[v4 * 8 + 4]) * inv_l, __uint_as_float(o[v4 * 8 + 5]) * inv_l);
                        w.w = pack_bf16(__uint_as_float(o[v4 * 8 + 6]) * inv_l, __uint_as_float(o[v4 * 8 + 7]) * inv_l);
                        dst[c / 8 + v4] = w;
                    }
                }
            }
            if (valid && p.lse) p.lse[row] = (m + lg2(l)) * 0.69314718055994530942f;
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
