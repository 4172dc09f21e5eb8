// attn_fwd.cu -- warp-specialised causal varlen prefill attention for sm_103a.
//
// Computes out = softmax(Q K^T * scale) V per work unit -- two 128-row Q tiles
// ("slots") of one sequence and one KV head, GQA query heads packed into the
// rows -- over the unit's KV tiles (the cached prefix read from the KV cache,
// then the sequence's own new keys), and writes the new K/V into the cache.
// Both slots consume every K/V tile, so each tile loaded from L2 feeds 256
// query rows.
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
// GB300 mapping (one persistent CTA per SM, 384 threads, all 512 TMEM columns:
// slot s owns S_s at [256 s, 256 s + 128) and O_s at [256 s + 128, 256 s + 256);
// P_s is written as bf16 over the first 64 columns of S_s):
//   warp 0, lane 0  fetches units from the longest-first list, loads both Q
//                   tiles once per unit and the K tiles into a ring;
//   warp 0, lane 1  loads the V tiles into a ring of its own;
//   warp 1          tcgen05 issuer, ping-pong over the slots:
//                   PV_0(t), S_0(t+1), PV_1(t), S_1(t+1), ... (S in the SS
//                   form, PV with P read from TMEM and V MN-major in SMEM);
//   warps 2, 3      cache writers (V, K): copy the unit's own new rows out of
//                   the staged tiles in shared memory into the cache; second
//                   releaser of every ring stage;
//   warps 4-7, 8-11 softmax of slot 0 and slot 1: one query row per thread
//                   (its TMEM lane), fp32 running max/sum in registers, exp2
//                   on the MUFU, lazy O rescale, epilogue out = O / l (bf16)
//                   and LSE.
// Variants (template arguments): a paged cache (block table; warp 0's two
// lane halves load K and V, V one tile behind, one TMA box per cache block),
// an int8 cache (codes expanded in shared memory), and the tile-splitting
// schedule, in which a unit whose rows fit one Q tile gives its even KV tiles
// to slot 0 and its odd ones to slot 1 and merges the two partial results
// (decode rows, short launches of one-tile units); there the softmax is
// column-split: the two warps of a sub-partition take half of every row's
// columns for both slots.
// Every wait is bounded in time; on timeout the CTA records PA_DEVERR_TIMEOUT,
// drains its in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <climits>
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
constexpr int kThreads = 384;                   // 4 control warps + 8 softmax warps
constexpr uint32_t kColSlot = 256;              // TMEM columns per slot: S then O
constexpr uint32_t kColO = 128;                 // O offset within a slot

template <int D>
struct Cfg {
    static constexpr int kChunkCols = D >= 64 ? 64 : 32;  // columns per swizzle atom row
    static constexpr int kChunks = D / kChunkCols;
    static constexpr int kRowBytes = kChunkCols * 2;
    static constexpr int kChunkBytes = kBlockM * kRowBytes;
    static constexpr int kTileBytes = kChunks * kChunkBytes;  // 128 rows x D bf16
    static constexpr SmemSwizzle kSw = D >= 64 ? kSwizzle128B : kSwizzle64B;
    static constexpr int kSbo = 8 * kRowBytes;  // byte distance between 8-row groups
    // Paged bf16 cache with two column chunks (d = 128): a prefix tile is
    // staged as [8-row group][chunk][8 rows] -- one TMA box per cache block
    // fills whole groups of both chunks -- so 8-row groups sit kGrpSbo apart
    // and the chunks of a group kSbo apart.
    static constexpr int kGrpSbo = kChunks * kSbo;
    static constexpr int kStagesK = D == 128 ? 2 : 4;
    static constexpr int kStagesV = D == 128 ? 3 : 4;
    static constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
    static constexpr uint32_t kIdescO = idesc_bf16_f32(kBlockM, D, 0, 1);
};

struct UnitSlot {
    Unit u;
    SeqInfo s;
};

struct __align__(16) Ctrl {
    uint64_t q_full, q_empty;
    uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
    uint64_t v_fix[4];  // paged cache: last prefix V tile with the rows past P zeroed
    uint64_t k_conv[4], v_conv[4];  // int8 cache: prefix tile expanded to bf16
    uint64_t ks_full[4];            // int8 cache: row scales of K tile t in kscale[t % 4]
    uint64_t never;                 // test hook: a barrier nothing completes
    uint64_t s_full[kSlots], p_full[kSlots], pv_done[kSlots], o_empty[kSlots];
    uint64_t mma_drain;
    uint64_t unit_full[2], unit_empty[2];
    UnitSlot slot[2];
    uint32_t tmem_base;
    int abort;
    union {
        // int8 cache: the row scales of K tile t (CTA tile counter) in slot t % 4,
        // folded into the scores by the softmax warps (the K tile holds the codes)
        alignas(16) float kscale[4][kBlockN];
        // tile-splitting variant: the column-split softmax's pair exchange,
        // per sub-partition [phase parity][warp half][lane]
        alignas(16) float xsplit[4][2 * 2 * 32];
    };
    uint64_t xs_full[4];  // column-split softmax: both warps of sub-partition sp wrote their value
};

// Tiles first (the dynamic shared window starts 1024-byte aligned, which the
// kernel checks), control block after them.  At least 120 KB so that a second
// CTA never lands on an SM (each CTA holds all 512 TMEM columns).
template <int D>
constexpr int smem_bytes() {
    using C = Cfg<D>;
    return (C::kTileBytes * (kSlots + C::kStagesK + C::kStagesV) + (int)sizeof(Ctrl)) > 120 * 1024
               ? C::kTileBytes * (kSlots + C::kStagesK + C::kStagesV) + (int)sizeof(Ctrl)
               : 120 * 1024;
}

__device__ __forceinline__ bool aborted(const Ctrl* c) { return *reinterpret_cast<const volatile int*>(&c->abort) != 0; }

// Slow path of a bounded wait; gives up when the CTA has aborted or after
// kTimeoutNs, in which case it flags the CTA and the device error word.
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, Ctrl* c, WorkspaceHeader* hdr) {
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

// Bounded wait: one inline probe, then the out-of-line polling loop.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Ctrl* c, WorkspaceHeader* hdr) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, c, hdr);
}

__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "elect.sync _|P1, 0xffffffff;\n\t"
        "selp.b32 %0, 1, 0, P1;\n\t}"
        : "+r"(pred));
    return pred != 0;
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

// 32-byte store (sm_100+); p 32-byte aligned
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// max of three (one instruction on sm_100+)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
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
// sequence has P cached tokens split into np = ceil(P / 128) prefix tiles
// (ending at P, or starting at 0 for a paged cache).
template <bool kPaged>
__device__ __forceinline__ int tile_key_base(int j, int P, int np) {
    if (j >= np) return P + kBlockN * (j - np);
    return kPaged ? kBlockN * j : P - kBlockN * (np - j);
}

// Paged cache: the last prefix tile when P is not a multiple of 128 -- its
// rows from P on hold no prefix key (other tokens' entries, or stale data).
__device__ __forceinline__ bool paged_tail_tile(int j, int P, int np) {
    return j == np - 1 && (P & (kBlockN - 1)) != 0;
}

// The KV tiles a unit streams, [lo, lo + ntiles) in the sequence's tile
// numbering, and the sub-range [a[s], b[s]) of that stream each slot visits
// (a = b = 0 when the slot has no tokens).  With a sliding window the later
// slot may start after the earlier one; the two ranges always touch.
// kAlt (the variant for decode-heavy or small launches): units hold
// unit_slots Q tiles (1 or 2, FwdParams::unit_slots); a unit whose rows fit
// ONE Q tile (a decode row, the last block of a prompt, every unit when
// unit_slots = 1) and that visits at least two KV tiles is "alt": both slots
// work on its rows, slot 0 on the even tiles of the stream and slot 1 on the
// odd ones, so that the two still ping-pong on the tensor pipe, and the two
// partial results are merged in the epilogue.
struct UnitGeo {
    int lo, ntiles, np;
    int a[kSlots], b[kSlots];
    bool alt;
};

template <bool kPaged, bool kAlt>
__device__ __forceinline__ UnitGeo unit_geo(const Unit& u, const SeqInfo& s, int tps, int causal, int window,
                                            int unit_slots) {
    const int nslots = kAlt ? unit_slots : kSlots;  // Q tiles of a unit
    UnitGeo g;
    g.np = prefix_tiles(s.P);
    const TileSpan all = query_tiles(s.n, s.P, u.q0, min(u.q0 + nslots * tps, s.n), causal, window, kPaged);
    g.lo = all.lo;
    g.ntiles = all.hi - all.lo;
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
        const int qs = u.q0 + i * tps;
        g.a[i] = g.b[i] = 0;
        if (i < nslots && qs < s.n) {
            const TileSpan t = query_tiles(s.n, s.P, qs, min(qs + tps, s.n), causal, window, kPaged);
            g.a[i] = t.lo - g.lo;
            g.b[i] = t.hi - g.lo;
        }
    }
    g.alt = kAlt && u.q0 + tps >= min(u.q0 + nslots * tps, s.n) && g.ntiles >= 2;
    return g;
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
    constexpr int kGran = D / 8;  // 16-byte granules per row
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

// Paged cache: copies rows [lo_row, lo_row + nrows) of a staged tile to the
// cache rows of positions pos0, pos0 + 1, ... of one sequence, each through the
// sequence's block table (pool [num_blocks][Hk][block_size][D]).  The
// scheduler has already rejected sequences naming a block outside the pool;
// the range check here only keeps a stray id from turning into a stray store.
template <int D>
__device__ __noinline__ void copy_tile_rows_paged(const uint8_t* tile, __nv_bfloat16* pool, const int32_t* table,
                                                     int block_log2, int num_blocks, int n_kv_heads, int kvh,
                                                     int pos0, int lo_row, int nrows, int lane) {
    using C = Cfg<D>;
    constexpr int kGran = D / 8;
    constexpr int kChunkGran = C::kChunkCols / 8;
    const int total = nrows * kGran;
    const int bmask = (1 << block_log2) - 1;
#pragma unroll 4
    for (int idx = lane; idx < total; idx += 32) {
        const int ri = idx / kGran, g = idx % kGran;
        const int r = lo_row + ri, pos = pos0 + ri;
        const int c = g / kChunkGran, gg = g % kChunkGran;
        const int phys = D >= 64 ? (gg ^ (r & 7)) : (gg ^ ((r >> 1) & 3));
        const uint4 x = *reinterpret_cast<const uint4*>(tile + c * C::kChunkBytes + r * C::kRowBytes + phys * 16);
        const int blk = __ldg(table + (pos >> block_log2));
        if ((unsigned)blk >= (unsigned)num_blocks) continue;
        const size_t row = (((size_t)blk * n_kv_heads + kvh) << block_log2) + (size_t)(pos & bmask);
        *reinterpret_cast<uint4*>(pool + row * D + g * 8) = x;
    }
}

// Zeroes rows [row0, 128) of a staged tile (whole rows, so the swizzle does
// not matter); kGrp: the tile is staged block by block (Cfg::kGrpSbo).
template <int D, bool kGrp>
__device__ __noinline__ void zero_tile_rows(uint8_t* tile, int row0, int lane) {
    using C = Cfg<D>;
    constexpr int kGran = D / 8;
    constexpr int kChunkGran = C::kChunkCols / 8;
    const int total = (kBlockN - row0) * kGran;
    for (int idx = lane; idx < total; idx += 32) {
        const int r = row0 + idx / kGran, g = idx % kGran, c = g / kChunkGran;
        const int off = kGrp ? (r >> 3) * C::kGrpSbo + c * C::kSbo + (r & 7) * C::kRowBytes
                             : c * C::kChunkBytes + r * C::kRowBytes;
        *reinterpret_cast<uint4*>(tile + off + (g % kChunkGran) * 16) = make_uint4(0, 0, 0, 0);
    }
}

// int8 cache, prefix tile: the TMA box of codes (row r = D bytes) lands in the
// upper half of a bf16 stage; this expands it in place into the swizzled bf16
// tile the MMA reads (one warp): value = code * scale[row] rounded to bf16 when
// kScale (sc[q] holds the scale of row 32 q + lane), else the code itself
// (exact in bf16).  Rows go in increasing order, kGroup batches of rows at a
// time, each group read before it is written: the bf16 image of row r ends
// within the codes of rows <= r, so no code is overwritten unread.
template <int D, bool kScale>
__device__ __noinline__ void dequant_tile(uint8_t* stage, const float (&sc)[4], int lane) {
    using C = Cfg<D>;
    constexpr int kGran = D / 8;       // 8-column granules per row
    constexpr int kRows = 32 / kGran;  // rows per batch (one granule per lane)
    constexpr int kGroup = 4;          // batches loaded before any is written
    constexpr int kChunkGran = C::kChunkCols / 8;
    const uint8_t* codes = stage + C::kTileBytes / 2;
    const int g = lane % kGran;
    const int c = g / kChunkGran, gg = g % kChunkGran;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll 1
        for (int r0 = 32 * q; r0 < 32 * q + 32; r0 += kRows * kGroup) {
            uint2 w[kGroup];
            float s[kGroup];
#pragma unroll
            for (int b = 0; b < kGroup; ++b) {
                const int r = r0 + b * kRows + lane / kGran;
                w[b] = *reinterpret_cast<const uint2*>(codes + r * D + g * 8);
                s[b] = kScale ? __shfl_sync(0xffffffffu, sc[q], r & 31) : 1.f;
            }
            __syncwarp();
#pragma unroll
            for (int b = 0; b < kGroup; ++b) {
                const int r = r0 + b * kRows + lane / kGran;
                // code + 128 as the low mantissa byte of 2^23, minus 2^23 + 128: exact
                // (pairs of columns on packed fp32 ops)
                const uint32_t x = w[b].x ^ 0x80808080u, y = w[b].y ^ 0x80808080u;
                const float2 off = make_float2(-8388736.0f, -8388736.0f);
                float2 f[4];  // columns (0,1), (2,3) of x, then of y
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    f[e] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540u + 2 * e)),
                                                  __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7541u + 2 * e))),
                                      off);
                    f[e + 2] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(y, 0x4B000000u, 0x7540u + 2 * e)),
                                                      __uint_as_float(__byte_perm(y, 0x4B000000u, 0x7541u + 2 * e))),
                                          off);
                    if (kScale) {
                        f[e] = __fmul2_rn(f[e], make_float2(s[b], s[b]));
                        f[e + 2] = __fmul2_rn(f[e + 2], make_float2(s[b], s[b]));
                    }
                }
                const int phys = D >= 64 ? (gg ^ (r & 7)) : (gg ^ ((r >> 1) & 3));
                *reinterpret_cast<uint4*>(stage + c * C::kChunkBytes + r * C::kRowBytes + phys * 16) =
                    make_uint4(pack_bf16(f[0].x, f[0].y), pack_bf16(f[1].x, f[1].y), pack_bf16(f[2].x, f[2].y),
                               pack_bf16(f[3].x, f[3].y));
            }
        }
    }
}

// int8 cache write: rows [lo_row, lo_row + nrows) of a staged bf16 tile as
// int8 codes at codes + row * D and their scales at scales[row], row =
// row_index(i) (~0: skip).  Per row, in fp32: scale = max|x| / 127, code = nearest integer (ties
// to even) of x / scale, clamped to +-127; a zero row is scale 0, codes 0.
template <int D, class RowIndex>
__device__ __noinline__ void quant_tile_rows(const uint8_t* tile, int8_t* codes, float* scales, RowIndex row_index,
                                             int lo_row, int nrows, int lane) {
    using C = Cfg<D>;
    constexpr int kGran = D / 8;  // lanes per row
    constexpr int kRows = 32 / kGran;
    constexpr int kChunkGran = C::kChunkCols / 8;
    const int g = lane % kGran;
    const int c = g / kChunkGran, gg = g % kChunkGran;
    for (int i0 = 0; i0 < nrows; i0 += kRows) {
        const int i = i0 + lane / kGran;
        const bool valid = i < nrows;
        const int r = lo_row + (valid ? i : 0);
        const int phys = D >= 64 ? (gg ^ (r & 7)) : (gg ^ ((r >> 1) & 3));
        const uint4 x = *reinterpret_cast<const uint4*>(tile + c * C::kChunkBytes + r * C::kRowBytes + phys * 16);
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
        float v[8];
        float am = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[2 * e] = __uint_as_float(xw[e] << 16);
            v[2 * e + 1] = __uint_as_float(xw[e] & 0xffff0000u);
            am = fmaxf(am, fmaxf(fabsf(v[2 * e]), fabsf(v[2 * e + 1])));
        }
#pragma unroll
        for (int o = 1; o < kGran; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        const float sc = __fdiv_rn(am, 127.0f);
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            int qv = 0;
            if (sc > 0.f) qv = max(-127, min(127, __float2int_rn(__fdiv_rn(v[e], sc))));
            packed[e >> 2] |= (uint32_t)(qv & 0xff) << (8 * (e & 3));
        }
        if (valid) {
            const size_t row = row_index(i);  // cache row of the staged row lo_row + i
            if (row != ~size_t(0)) {
                *reinterpret_cast<uint2*>(codes + row * D + g * 8) = make_uint2(packed[0], packed[1]);
                if (g == 0) scales[row] = sc;
            }
        }
    }
}

// Contiguous cache, one KV ring (K or V): waits for the stage, then
// TMA-loads tile j (index in the sequence) of unit u from the cache (prefix
// tiles) or from the new tokens' k/v.  Out of line: the K and the V loader
// share one copy of this code, which keeps the kernel's hot code within the
// instruction caches.
template <int D, bool kQuant>
__device__ __forceinline__ bool load_kv_tile(const FwdParams& p, Ctrl* ctl, WorkspaceHeader* hdr, uint8_t* ring,
                                          int stages, uint64_t* full, uint64_t* empty, const CUtensorMap* tm_cache,
                                          const CUtensorMap* tm_new, int* last_parity, uint32_t t, int j,
                                          const Unit& u, const SeqInfo& s, int np) {
    using C = Cfg<D>;
    const int st = t % stages;
    const uint32_t ph = (t / stages) & 1;
    const int kb = tile_key_base<false>(j, s.P, np);
    if (!wait_bar(&empty[st], ph ^ 1, ctl, hdr)) return false;
    if (kQuant && j < np) {
        // int8 codes of the prefix tile into the stage's upper half (one box of
        // 128 rows x D bytes), expanded to bf16 by the cache writer
        mbar_arrive_expect_tx(&full[st], kBlockN * D);
        tma_load_3d(ring + st * C::kTileBytes + C::kTileBytes / 2, tm_cache, &full[st], 0, kb,
                    u.b * p.n_kv_heads + u.kvh);
        last_parity[st] = (int)ph;
        return true;
    }
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
}

template <int D, bool kPaged, bool kQuant, bool kAlt = false, bool kHook = false>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = Cfg<D>;
    static_assert(!(kAlt && kQuant), "the merge exchange shares storage with the int8 scale ring");
    // K stages in use.  With an int8 cache the K writer publishes each tile's row
    // scales in a 4-deep ring (Ctrl::kscale) that the softmax warps read after
    // S; it writes the scales of tile t + 4 only once that tile has landed, i.e.
    // once its stage was released by the S of tile t + 4 - kStK, which the MMA
    // warp issues after the PV of tile t + 3 - kStK of every slot.  With at most
    // 3 stages that PV follows every slot's softmax of tile t: the ring slot is
    // free.  (bf16 caches use no scale ring.)
    constexpr int kStK = kQuant && C::kStagesK > 3 ? 3 : C::kStagesK;
    // paged bf16 cache, two column chunks: prefix tiles staged block by block
    constexpr bool kGrp = kPaged && !kQuant && C::kChunks == 2;
    const int unit_slots = kAlt ? p.unit_slots : kSlots;  // Q tiles of a unit
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // swizzled TMA/UMMA tiles need 1024-byte alignment (reported below)
    const bool misaligned = (smem_u32(smem_raw) & 1023u) != 0;
    uint8_t* q_smem = smem_raw;                              // [kSlots] tiles
    uint8_t* k_smem = q_smem + kSlots * C::kTileBytes;       // [kStagesK] tiles
    uint8_t* v_smem = k_smem + C::kStagesK * C::kTileBytes;  // [kStagesV] tiles
    Ctrl* ctl = reinterpret_cast<Ctrl*>(v_smem + C::kStagesV * C::kTileBytes);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    WorkspaceHeader* hdr = p.hdr;
    const int G = p.group;
    const int tps = kBlockM / G;  // query tokens per slot

    // The prologue (barriers, TMEM, tensor-map prefetch) reads nothing the
    // previous kernels of the call write, so it runs before the wait below and
    // overlaps their tail (programmatic stream serialisation).
    if (!misaligned && threadIdx.x == 0) {
        mbar_init(&ctl->q_full, 1);
        mbar_init(&ctl->q_empty, 1);
        for (int s = 0; s < kStK; ++s) {
            mbar_init(&ctl->k_full[s], 1);
            mbar_init(&ctl->k_empty[s], 2);  // MMA commit + cache writer
        }
        for (int s = 0; s < C::kStagesV; ++s) {
            mbar_init(&ctl->v_full[s], 1);
            mbar_init(&ctl->v_empty[s], 2);
            mbar_init(&ctl->v_fix[s], 1);  // V cache writer
            mbar_init(&ctl->v_conv[s], 1);
        }
        for (int s = 0; s < kStK; ++s) mbar_init(&ctl->k_conv[s], 1);  // K cache writer
        for (int s = 0; s < 4; ++s) mbar_init(&ctl->ks_full[s], 1);          // K cache writer
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&ctl->s_full[i], 1);
            mbar_init(&ctl->p_full[i], kAlt ? 8 : 4);  // the slot's 4 softmax warps (all 8: column split)
            mbar_init(&ctl->pv_done[i], 1);
            mbar_init(&ctl->o_empty[i], kAlt ? 8 : 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->unit_full[b], 1);
            mbar_init(&ctl->unit_empty[b], 12);  // MMA + V loader + 2 cache writers + 8 softmax warps
        }
        mbar_init(&ctl->mma_drain, 1);
        for (int s = 0; s < 4; ++s) mbar_init(&ctl->xs_full[s], 64);  // every lane of the pair
        mbar_init(&ctl->never, 1);
        ctl->abort = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tm_q);
        prefetch_tmap(&p.tm_k);
        prefetch_tmap(&p.tm_v);
        prefetch_tmap(&p.tm_ck);
        prefetch_tmap(&p.tm_cv);
    }
    if (!misaligned && warp == 1) {
        tmem_alloc(&ctl->tmem_base, 512);
        tmem_relinquish();
    }
    // wait for the scheduler (and rotary) kernels of this call before reading
    // or writing anything of theirs or of the caller's
    griddep_wait();
    if (misaligned) {
        if (threadIdx.x == 0) atomicOr(&p.hdr->error, PA_DEVERR_SMEM_ALIGN);
        return;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    // On abort, let every copy a producer thread started land before the CTA exits.
    auto drain = [&](uint64_t* bars, const int* last_parity, int n) {
        const uint64_t t0 = globaltimer_ns();
        for (int i = 0; i < n; ++i) {
            if (last_parity[i] < 0) continue;
            while (!mbar_try_wait(&bars[i], (uint32_t)last_parity[i]) && globaltimer_ns() - t0 < kTimeoutNs) {
            }
        }
    };

    // Test hook (a kernel of its own, so that the product kernels' code is not
    // touched by it): the first CTA's producer thread waits on a barrier
    // nothing completes, so that the timeout path (error word, abort, drains,
    // TMEM release in every role) runs on a healthy GPU.
    if (kHook && blockIdx.x == 0 && threadIdx.x == 0) wait_bar(&ctl->never, 0, ctl, hdr);

    if (kPaged && warp == 0) {
        // ------------------------------------- paged cache: unit fetch, Q, K and V loads
        // Lanes 0-15 load K (lane 0 also fetches units and loads Q), lanes
        // 16-31 load V, as one code path: each pass of the loop loads one K
        // tile and one V tile, the V group one tile behind the K group (its
        // first pass is idle).  K tile t waits for the stage that S(t - 2)
        // frees and V tile t - 1 for the one PV(t - 4) frees, which the tensor
        // pipe finishes first, so a pass waits on K alone, as a K loader of
        // its own would; V tile t beside K tile t would hold every K load back
        // until PV(t - 3).  A prefix tile is one TMA box per cache block (both
        // column chunks at d = 128; int8: all D columns) or per (block,
        // 64-column chunk): lane l of a group issues boxes l and l + 16 and
        // loads the block ids of its boxes one tile ahead.
        const bool is_v = lane >= 16;
        const int gl = lane & 15;
        const unsigned gmask = is_v ? 0xFFFF0000u : 0x0000FFFFu;
        const int src = lane & 16;  // the group's leader lane
        const bool gleader = gl == 0;
        uint8_t* ring = is_v ? v_smem : k_smem;
        const int stages = is_v ? C::kStagesV : kStK;
        uint64_t* full = is_v ? ctl->v_full : ctl->k_full;
        uint64_t* empty = is_v ? ctl->v_empty : ctl->k_empty;
        const CUtensorMap* tm_cache = is_v ? &p.tm_cv : &p.tm_ck;
        const CUtensorMap* tm_new = is_v ? &p.tm_v : &p.tm_k;
        const int num_units = hdr->num_units;
        const int br = p.box_rows;
        const int br_log2 = min(p.block_log2, 7);  // box_rows = 1 << br_log2
        const int bmask = (1 << p.block_log2) - 1;
        // ring position of the group's next tile, and per stage whether a copy
        // was started on it (bit of lp_set) with which parity (bit of lp_par)
        int st = 0;
        uint32_t ph = 0, lp_set = 0, lp_par = 0;
        int last_q_parity = -1;
        int u_it = 0;            // units this group has taken so far
        Unit u{};                // the group's current unit ...
        SeqInfo s{};
        UnitGeo ug{};
        const int32_t* tab = p.block_table;
        int j = 0, ntl = 0;      // ... its next tile and its tile count
        bool done = false;       // end of the unit list met (or a wait failed)
        // this lane's boxes of tile jj: box (pair / kChunks), chunk (pair % kChunks)
        // for pair = gl and gl + 16; returns the block id of each (prefix tiles)
        auto fetch_ids = [&](int jj, int& i0, int& i1) {
            i0 = i1 = 0;
            if (jj < ug.np) {
                const int kb = kBlockN * jj;
                const int boxes = (min(kBlockN, s.P - kb) + br - 1) >> br_log2;
                // one box per block (int8: all D columns; bf16 at d = 128: both
                // chunks), else one per (block, chunk)
                const int b0 = kQuant || kGrp ? gl : gl / C::kChunks;
                const int b1 = kQuant || kGrp ? gl + 16 : (gl + 16) / C::kChunks;
                if (b0 < boxes) i0 = __ldg(tab + ((kb + b0 * br) >> p.block_log2));
                if (b1 < boxes) i1 = __ldg(tab + ((kb + b1 * br) >> p.block_log2));
            }
        };
        int id0 = 0, id1 = 0, nid0 = 0, nid1 = 0;
        for (int pass = 0;; ++pass) {
            if (!done && !(is_v && pass == 0)) {
                // the next unit, once the current one has no tile left
                while (!done && j == ntl) {
                    const int sl = u_it & 1;
                    bool ok = true;
                    if (!is_v) {
                        if (gleader) {
                            ok = wait_bar(&ctl->unit_empty[sl], ((u_it >> 1) & 1) ^ 1, ctl, hdr);
                            if (ok) {
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
                            }
                        }
                        ok = __shfl_sync(gmask, ok, src);
                    } else {
                        ok = gleader ? wait_bar(&ctl->unit_full[sl], (u_it >> 1) & 1, ctl, hdr) : true;
                        ok = __shfl_sync(gmask, ok, src);
                    }
                    if (!ok) {
                        done = true;
                        break;
                    }
                    __syncwarp(gmask);  // the slot written by lane 0 (K) / acquired by lane 16 (V) is visible
                    u = ctl->slot[sl].u;
                    s = ctl->slot[sl].s;
                    __syncwarp(gmask);
                    if (is_v && gleader) mbar_arrive(&ctl->unit_empty[sl]);
                    if (u.b < 0) {
                        done = true;
                        break;
                    }
                    if (!is_v && gleader) {
                        // the unit's Q tiles (one or two): rows (token, head-in-group) of each slot
                        ok = wait_bar(&ctl->q_empty, (u_it & 1) ^ 1, ctl, hdr);
                        if (ok) {
                            const int nq = unit_slots == 2 && u.q0 + tps < s.n ? 2 : 1;
                            mbar_arrive_expect_tx(&ctl->q_full, nq * G * tps * C::kRowBytes * C::kChunks);
                            for (int i = 0; i < nq; ++i)
                                for (int c = 0; c < C::kChunks; ++c)
                                    tma_load_3d(q_smem + i * C::kTileBytes + c * C::kChunkBytes, &p.tm_q,
                                                &ctl->q_full, c * C::kChunkCols, u.kvh * G,
                                                s.q_start + u.q0 + i * tps);
                            last_q_parity = u_it & 1;
                        }
                    }
                    if (!is_v && !__shfl_sync(gmask, ok, src)) {
                        done = true;
                        break;
                    }
                    ++u_it;
                    ug = unit_geo<true, kAlt>(u, s, tps, p.causal, p.window, unit_slots);
                    tab = p.block_table + (size_t)u.b * p.max_blocks;
                    j = 0;
                    ntl = ug.ntiles;
                    if (ntl > 0) fetch_ids(ug.lo, id0, id1);
                }
                if (!done) {
                    const int jj = ug.lo + j;
                    if (j + 1 < ntl) fetch_ids(jj + 1, nid0, nid1);  // in flight during this tile
                    const bool ok = gleader ? wait_bar(&empty[st], ph ^ 1, ctl, hdr) : true;
                    if (!__shfl_sync(gmask, ok, src)) {
                        done = true;
                    } else {
                        const int kb = tile_key_base<true>(jj, s.P, ug.np);
                        uint8_t* stage = ring + st * C::kTileBytes;
                        if (kQuant && jj < ug.np) {
                            // int8 codes, one box of br rows x D bytes per block, into the
                            // stage's upper half (expanded to bf16 by the cache writer)
                            const int boxes = (min(kBlockN, s.P - kb) + br - 1) >> br_log2;
                            if (gleader) mbar_arrive_expect_tx(&full[st], boxes * br * D);
                            __syncwarp(gmask);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int box = gl + 16 * h;
                                if (box < boxes)
                                    tma_load_3d(stage + C::kTileBytes / 2 + box * br * D, tm_cache, &full[st], 0,
                                                (kb + box * br) & bmask, (h ? id1 : id0) * p.n_kv_heads + u.kvh);
                            }
                        } else if (kGrp && jj < ug.np) {
                            // one box per block: br rows x both chunks as whole 8-row
                            // groups (at most 16 boxes, one per lane)
                            const int boxes = (min(kBlockN, s.P - kb) + br - 1) >> br_log2;
                            if (gleader) mbar_arrive_expect_tx(&full[st], boxes * br * C::kRowBytes * C::kChunks);
                            __syncwarp(gmask);
                            if (gl < boxes)
                                tma_load_5d(stage + gl * br * C::kRowBytes * C::kChunks, tm_cache, &full[st], 0, 0, 0,
                                            ((kb + gl * br) & bmask) >> 3, id0 * p.n_kv_heads + u.kvh);
                        } else if (jj < ug.np) {
                            const int boxes = (min(kBlockN, s.P - kb) + br - 1) >> br_log2;
                            if (gleader) mbar_arrive_expect_tx(&full[st], boxes * br * C::kRowBytes * C::kChunks);
                            __syncwarp(gmask);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int pair = gl + 16 * h;
                                const int box = pair / C::kChunks, c = pair % C::kChunks;
                                if (box < boxes)
                                    tma_load_3d(stage + c * C::kChunkBytes + box * br * C::kRowBytes, tm_cache,
                                                &full[st], c * C::kChunkCols, (kb + box * br) & bmask,
                                                (h ? id1 : id0) * p.n_kv_heads + u.kvh);
                            }
                        } else {
                            if (gleader) mbar_arrive_expect_tx(&full[st], C::kTileBytes);
                            __syncwarp(gmask);
                            if (gl < C::kChunks)
                                tma_load_3d(stage + gl * C::kChunkBytes, tm_new, &full[st], gl * C::kChunkCols, u.kvh,
                                            s.q_start + kb - s.P);
                        }
                        lp_set |= 1u << st;
                        lp_par = (lp_par & ~(1u << st)) | (ph << st);
                        id0 = nid0;
                        id1 = nid1;
                        ++j;
                        if (++st == stages) {
                            st = 0;
                            ph ^= 1;
                        }
                    }
                }
            }
            if (__all_sync(0xFFFFFFFFu, done)) break;
        }
        if (gleader && aborted(ctl)) {
            int last_parity[4];
            for (int i = 0; i < 4; ++i) last_parity[i] = (lp_set >> i) & 1 ? (int)((lp_par >> i) & 1) : -1;
            if (!is_v) drain(&ctl->q_full, &last_q_parity, 1);
            drain(full, last_parity, stages);
        }
    } else if (warp == 0) {
        if (lane == 0) {
            // ----------------------------------------- unit fetch, Q and K loads
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
                // the unit's Q tiles (one or two): rows (token, head-in-group) of each slot
                if (!wait_bar(&ctl->q_empty, (u_it & 1) ^ 1, ctl, hdr)) break;
                const int nq = unit_slots == 2 && u.q0 + tps < s.n ? 2 : 1;
                mbar_arrive_expect_tx(&ctl->q_full, nq * G * tps * C::kRowBytes * C::kChunks);
                for (int i = 0; i < nq; ++i)
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(q_smem + i * C::kTileBytes + c * C::kChunkBytes, &p.tm_q, &ctl->q_full,
                                    c * C::kChunkCols, u.kvh * G, s.q_start + u.q0 + i * tps);
                last_q_parity[0] = u_it & 1;
                const UnitGeo ug = unit_geo<kPaged, kAlt>(u, s, tps, p.causal, p.window, unit_slots);
                bool ok = true;
                for (int j = 0; j < ug.ntiles && ok; ++j, ++t)
                    ok = load_kv_tile<D, kQuant>(p, ctl, hdr, k_smem, kStK, ctl->k_full, ctl->k_empty, &p.tm_ck,
                                                 &p.tm_k, last_k_parity, t, ug.lo + j, u, s, ug.np);
                if (!ok) break;
            }
            if (aborted(ctl)) {
                drain(&ctl->q_full, last_q_parity, 1);
                drain(ctl->k_full, last_k_parity, kStK);
            }
        } else if (lane == 1) {
            // ------------------------------------------------------- V loads
            // A ring of its own, so K tiles run ahead of S while V tiles wait for PV.
            uint32_t t = 0;
            int last_v_parity[4] = {-1, -1, -1, -1};
            for (int u_it = 0;; ++u_it) {
                const int sl = u_it & 1;
                if (!wait_bar(&ctl->unit_full[sl], (u_it >> 1) & 1, ctl, hdr)) break;
                const UnitSlot us = ctl->slot[sl];
                mbar_arrive(&ctl->unit_empty[sl]);
                if (us.u.b < 0) break;
                const UnitGeo ug = unit_geo<kPaged, kAlt>(us.u, us.s, tps, p.causal, p.window, unit_slots);
                bool ok = true;
                for (int j = 0; j < ug.ntiles && ok; ++j, ++t)
                    ok = load_kv_tile<D, kQuant>(p, ctl, hdr, v_smem, C::kStagesV, ctl->v_full, ctl->v_empty, &p.tm_cv,
                                                 &p.tm_v, last_v_parity, t, ug.lo + j, us.u, us.s, ug.np);
                if (!ok) break;
            }
            if (aborted(ctl)) drain(ctl->v_full, last_v_parity, C::kStagesV);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        // The whole warp runs the loop (waits and descriptors stay warp-uniform);
        // one elected lane issues the MMAs and commits.
        const bool leader = elect_one();
        const uint32_t q_addr = smem_u32(q_smem);
        const uint32_t k_addr = smem_u32(k_smem);
        const uint32_t v_addr = smem_u32(v_smem);
        // descriptor templates; the start-address field (bits 0-13, 16-byte
        // units) is advanced by adding (byte offset >> 4)
        const uint64_t q_desc = smem_desc(q_addr, 16, C::kSbo, C::kSw);
        const uint64_t k_desc = smem_desc(k_addr, 16, C::kSbo, C::kSw);
        const uint64_t v_desc = smem_desc(v_addr, C::kChunkBytes, C::kSbo, C::kSw);
        // block-by-block staging of paged prefix tiles (kGrp)
        const uint64_t k_desc_g = smem_desc(k_addr, 16, C::kGrpSbo, C::kSw);
        const uint64_t v_desc_g = smem_desc(v_addr, C::kSbo, C::kGrpSbo, C::kSw);
        uint32_t t = 0;                // KV tiles of this CTA so far
        uint32_t ns[kSlots] = {0, 0};  // tiles processed per slot so far
        uint32_t no[kSlots] = {0, 0};  // units with the slot active so far
        uint32_t fixpar = 0;           // paged: parity bit per V stage of v_fix
        uint32_t kcpar = 0, vcpar = 0; // int8 cache: parity bit per stage of k_conv / v_conv
        // K tile tt (index jt in the sequence) ready for S: a prefix tile of an
        // int8 cache once the K writer has expanded it, else once TMA landed
        auto wait_k = [&](uint32_t tt, int jt, int np) -> bool {
            const int kst = tt % kStK;
            if (kQuant && jt < np) {
                const bool got = warp_wait(&ctl->k_conv[kst], (kcpar >> kst) & 1, ctl, hdr);
                kcpar ^= 1u << kst;
                return got;
            }
            return warp_wait(&ctl->k_full[kst], (tt / kStK) & 1, ctl, hdr);
        };
        bool ok = true;
        // S of slot i from Q tile qi and K tile tt (grp: a block-staged prefix tile)
        auto issue_s = [&](int i, uint32_t tt, int qi, bool grp) {
            if (leader) {
                const uint32_t koff = (tt % kStK) * C::kTileBytes;
                const uint32_t qoff = qi * C::kTileBytes;
                // K operand: descriptor template and chunk stride of the tile's staging
                const bool g = kGrp && grp;
                const uint64_t kd = g ? k_desc_g : k_desc;
                const uint32_t kcs = g ? C::kSbo : C::kChunkBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk * 16) / C::kChunkCols) * C::kChunkBytes + ((kk * 16) % C::kChunkCols) * 2;
                    const uint32_t koff_kk = ((kk * 16) / C::kChunkCols) * kcs + ((kk * 16) % C::kChunkCols) * 2;
                    mma_ss(tmem + i * kColSlot, q_desc + ((qoff + off) >> 4), kd + ((koff + koff_kk) >> 4),
                           C::kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit(&ctl->s_full[i]);
            }
            __syncwarp();
        };
        auto issue_pv = [&](int i, uint32_t tt, bool first, bool grp) {
            if (leader) {
                const uint32_t voff = (tt % C::kStagesV) * C::kTileBytes;
                // V operand: descriptor template and 16-key step of the tile's staging
                const bool g = kGrp && grp;
                const uint64_t vd = g ? v_desc_g : v_desc;
                const uint32_t vstep = g ? 2 * C::kGrpSbo : 2 * C::kSbo;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_ts(tmem + i * kColSlot + kColO, tmem + i * kColSlot + kk * 8,
                           vd + ((voff + kk * vstep) >> 4), C::kIdescO, (!first || kk > 0) ? 1u : 0u);
                mma_commit(&ctl->pv_done[i]);
            }
            __syncwarp();
        };
        auto commit = [&](uint64_t* bar) {
            if (leader) mma_commit(bar);
            __syncwarp();
        };
        for (int u_it = 0; ok; ++u_it) {
            const int sl = u_it & 1;
            if (!warp_wait(&ctl->unit_full[sl], (u_it >> 1) & 1, ctl, hdr)) break;
            const Unit u = ctl->slot[sl].u;
            const SeqInfo s = ctl->slot[sl].s;
            __syncwarp();
            if (leader) mbar_arrive(&ctl->unit_empty[sl]);
            if (u.b < 0) break;
            const UnitGeo ug = unit_geo<kPaged, kAlt>(u, s, tps, p.causal, p.window, unit_slots);
            const int ntiles = ug.ntiles;
            if (!warp_wait(&ctl->q_full, u_it & 1, ctl, hdr)) break;
            if constexpr (kAlt) if (ug.alt) {
                // (bf16 cache only) V tile tj, index jt in the sequence, ready for PV
                auto wait_v = [&](uint32_t tj, int jt) -> bool {
                    const int vst = tj % C::kStagesV;
                    if (kPaged && paged_tail_tile(jt, s.P, ug.np)) {
                        const bool got = warp_wait(&ctl->v_fix[vst], (fixpar >> vst) & 1, ctl, hdr);
                        fixpar ^= 1u << vst;
                        return got;
                    }
                    return warp_wait(&ctl->v_full[vst], (tj / C::kStagesV) & 1, ctl, hdr);
                };
                // slot i takes the tiles j with j % 2 == i, both from Q tile 0:
                // S_0(0), S_1(1), then per tile j: PV_i(j), S_i(j + 2)
                if (!wait_k(t, ug.lo, ug.np)) break;
                tc_fence_after();
                issue_s(0, t, 0, ug.lo < ug.np);
                commit(&ctl->k_empty[t % kStK]);
                if (!wait_k(t + 1, ug.lo + 1, ug.np)) break;
                tc_fence_after();
                issue_s(1, t + 1, 0, ug.lo + 1 < ug.np);
                commit(&ctl->k_empty[(t + 1) % kStK]);
                if (ntiles == 2) commit(&ctl->q_empty);
                for (int j = 0; j < ntiles && ok; ++j) {
                    const uint32_t tj = t + j;
                    const int i = j & 1, kth = j >> 1;
                    if (!warp_wait(&ctl->p_full[i], (ns[i] + kth) & 1, ctl, hdr)) { ok = false; break; }
                    if (kth == 0 && !warp_wait(&ctl->o_empty[i], (no[i] & 1) ^ 1, ctl, hdr)) { ok = false; break; }
                    if (!wait_v(tj, ug.lo + j)) { ok = false; break; }
                    tc_fence_after();
                    issue_pv(i, tj, kth == 0, ug.lo + j < ug.np);
                    if (j + 2 < ntiles) {
                        if (!wait_k(tj + 2, ug.lo + j + 2, ug.np)) { ok = false; break; }
                        tc_fence_after();
                        issue_s(i, tj + 2, 0, ug.lo + j + 2 < ug.np);
                        commit(&ctl->k_empty[(tj + 2) % kStK]);
                        if (j + 3 == ntiles) commit(&ctl->q_empty);
                    }
                    commit(&ctl->v_empty[tj % C::kStagesV]);
                }
                ns[0] += (ntiles + 1) / 2;
                ns[1] += ntiles / 2;
                no[0] += 1;
                no[1] += 1;
                t += ntiles;
                continue;
            }
            // prologue: S of tile 0 for the slots that start there
            if (!wait_k(t, ug.lo, ug.np)) break;
            tc_fence_after();
            for (int i = 0; i < kSlots; ++i)
                if (ug.a[i] == 0 && ug.b[i] > 0) issue_s(i, t, i, ug.lo < ug.np);
            commit(&ctl->k_empty[t % kStK]);
            if (ntiles == 1) commit(&ctl->q_empty);
            for (int j = 0; j < ntiles && ok; ++j) {
                const uint32_t tj = t + j;
                bool v_ready = false, k_ready = false;
                for (int i = 0; i < kSlots; ++i) {
                    if (j >= ug.a[i] && j < ug.b[i]) {
                        // PV_i(j): P_i(j) written and O_i free (first tile of the slot)
                        if (!warp_wait(&ctl->p_full[i], (ns[i] + j - ug.a[i]) & 1, ctl, hdr)) { ok = false; break; }
                        if (j == ug.a[i] && !warp_wait(&ctl->o_empty[i], (no[i] & 1) ^ 1, ctl, hdr)) { ok = false; break; }
                        if (!v_ready) {
                            const int vst = tj % C::kStagesV;
                            bool got;
                            if (kQuant && ug.lo + j < ug.np) {
                                // int8 prefix tile (a paged tail included: its rows past P
                                // get scale 0 in the expansion)
                                got = warp_wait(&ctl->v_conv[vst], (vcpar >> vst) & 1, ctl, hdr);
                                vcpar ^= 1u << vst;
                            } else if (kPaged && paged_tail_tile(ug.lo + j, s.P, ug.np)) {
                                got = warp_wait(&ctl->v_fix[vst], (fixpar >> vst) & 1, ctl, hdr);
                                fixpar ^= 1u << vst;
                            } else {
                                got = warp_wait(&ctl->v_full[vst], (tj / C::kStagesV) & 1, ctl, hdr);
                            }
                            if (!got) {
                                ok = false;
                                break;
                            }
                            v_ready = true;
                        }
                        tc_fence_after();
                        issue_pv(i, tj, j == ug.a[i], ug.lo + j < ug.np);
                    }
                    if (j + 1 >= ug.a[i] && j + 1 < ug.b[i]) {
                        // S_i(j+1) overwrites P_i(j): issued after PV_i(j) on the in-order tensor pipe
                        if (!k_ready) {
                            if (!wait_k(tj + 1, ug.lo + j + 1, ug.np)) {
                                ok = false;
                                break;
                            }
                            k_ready = true;
                            tc_fence_after();
                        }
                        issue_s(i, tj + 1, i, ug.lo + j + 1 < ug.np);
                    }
                }
                if (!ok) break;
                if (j + 1 < ntiles) {
                    commit(&ctl->k_empty[(tj + 1) % kStK]);
                    if (j + 2 == ntiles) commit(&ctl->q_empty);
                }
                commit(&ctl->v_empty[tj % C::kStagesV]);
            }
            for (int i = 0; i < kSlots; ++i) {
                ns[i] += ug.b[i] - ug.a[i];
                no[i] += ug.b[i] > ug.a[i] ? 1 : 0;
            }
            t += ntiles;
        }
        // every MMA this warp issued has finished before TMEM is released
        if (leader) {
            mma_commit(&ctl->mma_drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&ctl->mma_drain, 0) && globaltimer_ns() - t0 < kTimeoutNs) {
            }
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // -------------------------------------------------------- cache writers
        // Warp 3 writes K, warp 2 writes V.  Each walks every tile of its ring
        // in order and is the second releaser of every stage (with the MMA
        // commit), so it never waits on a barrier phase more than one ahead or
        // behind; on the tiles holding the unit's own tokens it first copies
        // those rows from shared memory into the cache.
        const bool is_k = warp == 3;
        const int stages = is_k ? kStK : C::kStagesV;
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
            const UnitGeo ug = unit_geo<kPaged, kAlt>(us.u, us.s, tps, p.causal, p.window, unit_slots);
            const int np = ug.np;
            const int q_end = min(us.u.q0 + unit_slots * tps, us.s.n);
            bool ok = true;
            for (int jr = 0; jr < ug.ntiles; ++jr, ++t) {
                const int j = ug.lo + jr;  // tile index in the sequence
                const int st = t % stages;
                if (kQuant && j < np) {
                    // int8 prefix tile: expand the codes for the MMA.  V rows
                    // become code * scale; K rows stay the (exact) codes and
                    // their scales go to the scale ring, folded into the scores.
                    const int kb = tile_key_base<kPaged>(j, us.s.P, np);
                    const float* scales = is_k ? p.scale_k : p.scale_v;
                    float sc[4];
                    if (kPaged) {
                        // row scales through the block table; rows from P on (rest of the
                        // last block, stale rows) get scale 0 and so expand to zeros
                        const int32_t* tab = p.block_table + (size_t)us.u.b * p.max_blocks;
                        const int bmask = (1 << p.block_log2) - 1;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int pos = kb + 32 * q + lane;
                            sc[q] = 0.f;
                            if (pos < us.s.P) {
                                const int blk = __ldg(tab + (pos >> p.block_log2));
                                if ((unsigned)blk < (unsigned)p.num_blocks)
                                    sc[q] = __ldg(scales + ((((size_t)blk * p.n_kv_heads + us.u.kvh) << p.block_log2) +
                                                            (pos & bmask)));
                            }
                        }
                    } else {
                        const float* srow = scales + ((size_t)us.u.b * p.n_kv_heads + us.u.kvh) * p.max_cache_len;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int row = kb + 32 * q + lane;  // rows below 0 are zero-filled codes
                            sc[q] = row >= 0 ? __ldg(srow + row) : 0.f;
                        }
                    }
                    if (!warp_wait(&full[st], (t / stages) & 1, ctl, hdr)) { ok = false; break; }
                    if (is_k) {
                        dequant_tile<D, false>(ring + st * C::kTileBytes, sc, lane);
#pragma unroll
                        for (int q = 0; q < 4; ++q) ctl->kscale[t & 3][32 * q + lane] = sc[q];
                    } else {
                        dequant_tile<D, true>(ring + st * C::kTileBytes, sc, lane);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(is_k ? &ctl->k_conv[st] : &ctl->v_conv[st]);
                        if (is_k) mbar_arrive(&ctl->ks_full[t & 3]);
                        mbar_arrive(&empty[st]);
                    }
                    continue;
                }
                if (!warp_wait(&full[st], (t / stages) & 1, ctl, hdr)) { ok = false; break; }
                int lo_row, nrows;
                if (own_rows(j, np, us.u.q0, q_end, lo_row, nrows)) {
                    const int first_tok = (j - np) * kBlockN + lo_row;  // token index within the sequence
                    if (kQuant && kPaged) {
                        const int32_t* tab = p.block_table + (size_t)us.u.b * p.max_blocks;
                        const int pos0 = us.s.P + first_tok, lg = p.block_log2, Hk = p.n_kv_heads, kvh = us.u.kvh;
                        const int nb = p.num_blocks;
                        quant_tile_rows<D>(ring + st * C::kTileBytes, reinterpret_cast<int8_t*>(cache),
                                           is_k ? p.scale_k : p.scale_v,
                                           [=](int i) -> size_t {
                                               const int pos = pos0 + i;
                                               const int blk = __ldg(tab + (pos >> lg));
                                               if ((unsigned)blk >= (unsigned)nb) return ~size_t(0);
                                               return (((size_t)blk * Hk + kvh) << lg) + (pos & ((1 << lg) - 1));
                                           },
                                           lo_row, nrows, lane);
                    } else if (kQuant) {
                        const size_t row0 = ((size_t)us.u.b * p.n_kv_heads + us.u.kvh) * p.max_cache_len +
                                            us.s.P + first_tok;
                        quant_tile_rows<D>(ring + st * C::kTileBytes, reinterpret_cast<int8_t*>(cache),
                                           is_k ? p.scale_k : p.scale_v, [=](int i) -> size_t { return row0 + i; },
                                           lo_row, nrows, lane);
                    } else if (kPaged) {
                        copy_tile_rows_paged<D>(ring + st * C::kTileBytes, cache,
                                                p.block_table + (size_t)us.u.b * p.max_blocks, p.block_log2,
                                                p.num_blocks, p.n_kv_heads, us.u.kvh, us.s.P + first_tok, lo_row, nrows, lane);
                    } else {
                        __nv_bfloat16* dst = cache + (((size_t)us.u.b * p.n_kv_heads + us.u.kvh) * p.max_cache_len +
                                                      us.s.P + first_tok) * D;
                        copy_tile_rows<D>(ring + st * C::kTileBytes, dst, lo_row, nrows, lane);
                    }
                } else if (kPaged && !is_k && paged_tail_tile(j, us.s.P, np)) {
                    // rows from P on may hold anything (NaN included): zero them
                    // so that P = 0 there contributes exactly 0 to O
                    zero_tile_rows<D, kGrp>(ring + st * C::kTileBytes, us.s.P - kBlockN * j, lane);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->v_fix[st]);
                }
                __syncwarp();
                if (lane == 0) {
                    // int8 cache: one ks_full phase per K tile (none for this one's
                    // scales), only after the tile landed, so that the ring never
                    // runs two phases ahead of a softmax warp
                    if (kQuant && is_k) mbar_arrive(&ctl->ks_full[t & 3]);
                    mbar_arrive(&empty[st]);
                }
            }
            if (!ok) break;
        }
    } else if constexpr (kAlt) {
        // ------------------------------------------------- softmax, column split
        // The two warps of sub-partition sp (warps 4 + sp and 8 + sp) share the
        // TMEM lanes (= query rows) [32 sp, 32 sp + 32) of BOTH slots: warp half
        // h takes the score columns [64 h, 64 h + 64) of every tile and the O
        // columns [h D/2, (h + 1) D/2).  Per tile the pair combines its row
        // maxima through shared memory (so both use the same running max, and
        // half 1 writes P over S columns 32-63 only after half 0 has read them);
        // each warp keeps the sum of its own columns, combined at the end of the
        // unit.  Both slots' tiles go through the same warps in the MMA warp's
        // order (slot 0's tile j, then slot 1's), so a tile's exponentials take
        // half the time of a one-warp-per-row softmax and the two slots'
        // softmaxes no longer share a sub-partition at the same time.
        constexpr int kHalfCols = kBlockN / 2;  // score columns per warp
        constexpr int kHalfD = D / 2;           // O columns per warp
        const int half = (warp - 4) >> 2;
        const int sp = warp & 3;
        const int r = sp * 32 + lane;  // query row of the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
        const float sl2 = p.scale_log2;
        uint32_t ns[kSlots] = {0, 0};  // tiles each slot has processed (s_full / pv_done phases)
        uint32_t nx = 0;               // pair exchanges so far (xs_full phase, buffer parity)
        float* xbuf = ctl->xsplit[sp];
        // write this warp's value, wait for the partner's, read it (bounded wait)
        auto exchange = [&](float v, float& other) -> bool {
            const int par = nx & 1;
            xbuf[(par * 2 + half) * 32 + lane] = v;
            tc_fence_before();  // this warp's TMEM loads are ordered before the partner's stores
            mbar_arrive(&ctl->xs_full[sp]);
            const bool got = warp_wait(&ctl->xs_full[sp], par, ctl, hdr);
            tc_fence_after();
            other = xbuf[(par * 2 + (half ^ 1)) * 32 + lane];
            ++nx;
            return got;
        };
        // the warp's O columns of slot i: 32 at a time (16 at d = 32)
        auto o_cols = [&](int i) -> uint32_t { return tmem + lane_off + i * kColSlot + kColO + half * kHalfD; };
        for (int u_it = 0;; ++u_it) {
            const int sl = u_it & 1;
            if (!warp_wait(&ctl->unit_full[sl], (u_it >> 1) & 1, ctl, hdr)) break;
            const UnitSlot us = ctl->slot[sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->unit_empty[sl]);
            if (us.u.b < 0) break;
            const Unit u = us.u;
            const SeqInfo s = us.s;
            const UnitGeo ug = unit_geo<kPaged, kAlt>(u, s, tps, p.causal, p.window, unit_slots);
            bool alt = false;
            if constexpr (kAlt) alt = ug.alt;
            const int np = ug.np;
            const int Lk = s.P + s.n;
            // rows of each slot (alt: both slots hold slot 0's rows)
            int tok[kSlots], row_hi[kSlots], slot_hi[kSlots], row_lo[kSlots], slot_lo[kSlots];
            bool valid[kSlots];
#pragma unroll
            for (int i = 0; i < kSlots; ++i) {
                const int qs = u.q0 + (alt ? 0 : i) * tps;
                const int qe = min(qs + tps, s.n);
                tok[i] = qs + r / G;
                valid[i] = r < tps * G && tok[i] < s.n;
                row_hi[i] = p.causal ? min(s.P + tok[i] + 1, Lk) : Lk;  // keys [0, row_hi) visible
                slot_hi[i] = p.causal ? min(s.P + qs + 1, Lk) : Lk;    // smallest row_hi of the slot
                // sliding window: keys [row_lo, row_hi); slot_lo = largest row_lo of the slot
                row_lo[i] = (p.causal && p.window > 0) ? s.P + tok[i] - p.window + 1 : INT_MIN / 2;
                slot_lo[i] = (p.causal && p.window > 0) ? s.P + qe - p.window : INT_MIN / 2;
            }
            const int hrow = u.kvh * G + r % G;
            float m[kSlots] = {-INFINITY, -INFINITY}, l[kSlots] = {0.f, 0.f};
            int cnt[kSlots] = {0, 0};  // this unit's tiles per slot
            bool ok = true;
            for (int j = 0; j < ug.ntiles && ok; ++j) {
#pragma unroll
                for (int i = 0; i < kSlots; ++i) {
                    const bool in = alt ? (j & 1) == i : (j >= ug.a[i] && j < ug.b[i]);
                    if (!in) continue;
                    if (!warp_wait(&ctl->s_full[i], ns[i] & 1, ctl, hdr)) { ok = false; break; }
                    tc_fence_after();
                    // S_i(j) is complete, and with it every earlier MMA of slot i
                    // (its previous PV included): O may be rescaled below.
                    const uint32_t s_col = tmem + lane_off + i * kColSlot;
                    float sv[kHalfCols];
                    {
                        uint32_t r0[32], r1[32];
                        tmem_ld32(s_col + half * kHalfCols, r0);
                        tmem_ld32(s_col + half * kHalfCols + 32, r1);
                        tmem_wait_ld();
                        reg_fence(r0);
                        reg_fence(r1);
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            sv[c] = __uint_as_float(r0[c]);
                            sv[32 + c] = __uint_as_float(r1[c]);
                        }
                    }
                    const int jt = ug.lo + j;  // tile index in the sequence
                    const int kb = tile_key_base<kPaged>(jt, s.P, np);
                    // paged: the last prefix tile holds prefix keys only below P
                    const bool tail = kPaged && jt < np && kb + kBlockN > s.P;
                    if (kb < 0 || kb + kBlockN > slot_hi[i] || kb < slot_lo[i] || tail) {
                        const int lo = max(-kb, row_lo[i] - kb) - half * kHalfCols;
                        const int hi = (tail ? min(row_hi[i], s.P) : row_hi[i]) - kb - half * kHalfCols;
#pragma unroll
                        for (int c = 0; c < kHalfCols; ++c)
                            if (c < lo || c >= hi) sv[c] = -INFINITY;
                    }
                    // row max of the warp's columns: four chains of three-input maxima
                    float mx0 = fmaxf(sv[0], sv[1]), mx1 = fmaxf(sv[2], sv[3]);
                    float mx2 = fmaxf(sv[4], sv[5]), mx3 = fmaxf(sv[6], sv[7]);
#pragma unroll
                    for (int c = 8; c < kHalfCols; c += 8) {
                        mx0 = fmax3(mx0, sv[c], sv[c + 1]);
                        mx1 = fmax3(mx1, sv[c + 2], sv[c + 3]);
                        mx2 = fmax3(mx2, sv[c + 4], sv[c + 5]);
                        mx3 = fmax3(mx3, sv[c + 6], sv[c + 7]);
                    }
                    const float mh = fmaxf(fmax3(mx0, mx1, mx2), mx3);
                    float mo;
                    if (!exchange(mh, mo)) { ok = false; break; }
                    // the same in both warps: max of (half 0, half 1) in a fixed order
                    const float m_tile = (half == 0 ? fmaxf(mh, mo) : fmaxf(mo, mh)) * sl2;
                    const float m_new = fmaxf(m[i], m_tile);
                    float alpha = 1.f;
                    bool rescale = false;
                    if (cnt[i] == 0) {
                        m[i] = m_new;
                    } else {
                        const bool need = m_new > m[i] + 8.f;
                        rescale = __any_sync(0xffffffffu, need);
                        if (need) {
                            alpha = ex2(m[i] - m_new);
                            m[i] = m_new;
                        }
                    }
                    const float m_use = m[i] == -INFINITY ? 0.f : m[i];
                    // P as bf16 pairs: the warp's 64 scores go to the 32 TMEM
                    // columns at 32 h (over S columns the pair has read)
                    const float2 sl2v = make_float2(sl2, sl2), negm = make_float2(-m_use, -m_use);
                    float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c4 = 0; c4 < 2; ++c4) {
                        uint32_t pk[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const float2 a =
                                __ffma2_rn(make_float2(sv[c4 * 32 + 2 * q], sv[c4 * 32 + 2 * q + 1]), sl2v, negm);
                            const float p0 = ex2(a.x);
                            const float p1 = ex2(a.y);
                            sum2 = __fadd2_rn(sum2, make_float2(p0, p1));
                            pk[q] = pack_bf16(p0, p1);
                        }
                        tmem_st16(s_col + half * (kHalfCols / 2) + c4 * 16, pk);
                    }
                    l[i] = l[i] * alpha + (sum2.x + sum2.y);
                    if (rescale) {
                        if constexpr (kHalfD >= 32) {
#pragma unroll
                            for (int c = 0; c < kHalfD; c += 32) {
                                uint32_t o[32];
                                tmem_ld32(o_cols(i) + c, o);
                                tmem_wait_ld();
                                reg_fence(o);
#pragma unroll
                                for (int q = 0; q < 32; q += 2) {
                                    const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[q]), __uint_as_float(o[q + 1])),
                                                                make_float2(alpha, alpha));
                                    o[q] = __float_as_uint(v.x);
                                    o[q + 1] = __float_as_uint(v.y);
                                }
                                tmem_st32(o_cols(i) + c, o);
                            }
                        } else {
                            uint32_t o[16];
                            tmem_ld16(o_cols(i), o);
                            tmem_wait_ld();
                            reg_fence(o);
#pragma unroll
                            for (int q = 0; q < 16; q += 2) {
                                const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[q]), __uint_as_float(o[q + 1])),
                                                            make_float2(alpha, alpha));
                                o[q] = __float_as_uint(v.x);
                                o[q + 1] = __float_as_uint(v.y);
                            }
                            tmem_st16(o_cols(i), o);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->p_full[i]);
                    ++ns[i];
                    ++cnt[i];
                }
            }
            if (!ok) break;
            // epilogue: a slot's O is final once the PV of its last tile is done.
            // The pair adds its partial sums (in a fixed order, so both get the
            // same l); each warp normalises and writes its half of every row.
            // An alt unit merges the two slots' partial results of the same rows.
            float w[kSlots] = {0.f, 0.f};  // weight of each slot's O in the output row
            bool done = false;
            for (int e = 0; e < kSlots && !done; ++e) {
                // alt: one merged output (e = 0 only); else slot e, if it had tiles
                if (alt ? e > 0 : cnt[e] == 0) continue;
                float lt[kSlots], mm = -INFINITY;
#pragma unroll
                for (int i = 0; i < kSlots; ++i) {
                    lt[i] = 0.f;
                    const bool use = alt ? cnt[i] > 0 : i == e;
                    if (!use) continue;
                    if (!warp_wait(&ctl->pv_done[i], (ns[i] - 1) & 1, ctl, hdr)) { ok = false; break; }
                    float lo_;
                    if (!exchange(l[i], lo_)) { ok = false; break; }
                    lt[i] = half == 0 ? l[i] + lo_ : lo_ + l[i];
                    mm = fmaxf(mm, m[i]);
                }
                if (!ok) break;
                tc_fence_after();
                float lsum = 0.f;
#pragma unroll
                for (int i = 0; i < kSlots; ++i) {
                    const bool use = alt ? cnt[i] > 0 : i == e;
                    w[i] = 0.f;
                    if (!use) continue;
                    const float c = (m[i] == -INFINITY) ? 0.f : ex2(m[i] - mm);  // 1 for a single slot
                    w[i] = c;
                    lsum += lt[i] * c;
                }
                const float inv_l = 1.f / lsum;
                const int orow_slot = alt ? 0 : e;
                const bool v_ok = valid[orow_slot];
                const size_t row = (size_t)(s.q_start + tok[orow_slot]) * p.n_heads + hrow;
                uint4* dst = reinterpret_cast<uint4*>(p.out + row * D + half * kHalfD);
#pragma unroll
                for (int c = 0; c < kHalfD; c += (kHalfD >= 32 ? 32 : 16)) {
                    constexpr int kW = kHalfD >= 32 ? 32 : 16;
                    float o[kW];
#pragma unroll
                    for (int q = 0; q < kW; ++q) o[q] = 0.f;
#pragma unroll
                    for (int i = 0; i < kSlots; ++i) {
                        const bool use = alt ? cnt[i] > 0 : i == e;
                        if (!use) continue;
                        uint32_t ob[kW];
                        if constexpr (kW == 32) tmem_ld32(o_cols(i) + c, ob); else tmem_ld16(o_cols(i) + c, ob);
                        tmem_wait_ld();
                        reg_fence(ob);
                        const float wi = w[i] * inv_l;
#pragma unroll
                        for (int q = 0; q < kW; ++q) o[q] = fmaf(__uint_as_float(ob[q]), wi, o[q]);
                    }
                    if (v_ok) {
#pragma unroll
                        for (int g = 0; g < kW / 16; ++g) {
                            uint32_t pw[8];
#pragma unroll
                            for (int k = 0; k < 8; ++k) pw[k] = pack_bf16(o[g * 16 + 2 * k], o[g * 16 + 2 * k + 1]);
                            if (p.out_align32) {
                                st_global_v8(dst + c / 8 + 2 * g, pw);
                            } else {
                                dst[c / 8 + 2 * g] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                                dst[c / 8 + 2 * g + 1] = make_uint4(pw[4], pw[5], pw[6], pw[7]);
                            }
                        }
                    }
                }
                if (v_ok && half == 0 && p.lse) p.lse[row] = (mm + lg2(lsum)) * 0.69314718055994530942f;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int i = 0; i < kSlots; ++i)
                        if (alt ? cnt[i] > 0 : i == e) mbar_arrive(&ctl->o_empty[i]);
                }
                if (alt) done = true;
            }
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------------- softmax
        // (plain schedule) Warps 4-7 serve slot 0, warps 8-11 slot 1.  Sub-partition sp = warp % 4
        // owns TMEM lanes (= query rows) [32 sp, 32 sp + 32).
        const int slot = (warp - 4) >> 2;
        const int sp = warp & 3;
        const int r = sp * 32 + lane;  // query row of the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
        const uint32_t s_col = tmem + lane_off + slot * kColSlot;
        const uint32_t o_col = s_col + kColO;
        const float sl2 = p.scale_log2;
        uint32_t ns = 0;  // tiles this slot has processed
        uint32_t tg = 0;  // CTA tiles before the current unit (int8 cache: scale ring index)
        for (int u_it = 0;; ++u_it) {
            const int sl = u_it & 1;
            if (!warp_wait(&ctl->unit_full[sl], (u_it >> 1) & 1, ctl, hdr)) break;
            const UnitSlot us = ctl->slot[sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->unit_empty[sl]);
            if (us.u.b < 0) break;
            const Unit u = us.u;
            const SeqInfo s = us.s;
            const UnitGeo ug = unit_geo<kPaged, false>(u, s, tps, p.causal, p.window, unit_slots);
            const int nt = ug.b[slot] - ug.a[slot];  // tiles of this slot: [a, b) of the stream
            const uint32_t tg0 = tg;
            tg += ug.ntiles;
            if (nt == 0) continue;
            const int qs = u.q0 + slot * tps;
            const int qe = min(qs + tps, s.n);
            const int tok = qs + r / G;
            const int h = u.kvh * G + r % G;
            const bool valid = r < tps * G && tok < s.n;
            const int Lk = s.P + s.n;
            const int row_hi = p.causal ? min(s.P + tok + 1, Lk) : Lk;  // keys [0, row_hi) visible
            const int slot_hi = p.causal ? min(s.P + qs + 1, Lk) : Lk;  // smallest row_hi of the slot
            // sliding window: keys [row_lo, row_hi) visible; slot_lo = largest row_lo of the slot
            const int row_lo = (p.causal && p.window > 0) ? s.P + tok - p.window + 1 : INT_MIN / 2;
            const int slot_lo = (p.causal && p.window > 0) ? s.P + qe - p.window : INT_MIN / 2;
            const int np = ug.np;
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < nt; ++j) {
                if (!warp_wait(&ctl->s_full[slot], (ns + j) & 1, ctl, hdr)) { ok = false; break; }
                tc_fence_after();
                // S_slot(j) is complete, and with it every earlier MMA of this
                // slot (the PV of tile j-1 included): O may be rescaled below.
                float sv[kBlockN];
                {
                    uint32_t r0[32], r1[32], r2[32], r3[32];
                    tmem_ld32(s_col, r0);
                    tmem_ld32(s_col + 32, r1);
                    tmem_ld32(s_col + 64, r2);
                    tmem_ld32(s_col + 96, r3);
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
                const int jrel = ug.a[slot] + j;  // tile index in the unit's stream
                const int jt = ug.lo + jrel;  // tile index in the sequence
                if (kQuant && jt < np) {
                    // int8 prefix tile: S holds q . code; scale column c by its row's scale
                    const uint32_t tc = tg0 + jrel;
                    if (!warp_wait(&ctl->ks_full[tc & 3], (tc >> 2) & 1, ctl, hdr)) { ok = false; break; }
                    const float4* ksc = reinterpret_cast<const float4*>(ctl->kscale[tc & 3]);
#pragma unroll
                    for (int c4 = 0; c4 < kBlockN / 4; ++c4) {
                        const float4 f = ksc[c4];
                        const float2 a = __fmul2_rn(make_float2(sv[4 * c4], sv[4 * c4 + 1]), make_float2(f.x, f.y));
                        const float2 b = __fmul2_rn(make_float2(sv[4 * c4 + 2], sv[4 * c4 + 3]), make_float2(f.z, f.w));
                        sv[4 * c4] = a.x;
                        sv[4 * c4 + 1] = a.y;
                        sv[4 * c4 + 2] = b.x;
                        sv[4 * c4 + 3] = b.y;
                    }
                }
                const int kb = tile_key_base<kPaged>(jt, s.P, np);
                // paged: the last prefix tile holds prefix keys only below P
                const bool tail = kPaged && jt < np && kb + kBlockN > s.P;
                if (kb < 0 || kb + kBlockN > slot_hi || kb < slot_lo || tail) {
                    const int lo = max(-kb, row_lo - kb), hi = (tail ? min(row_hi, s.P) : row_hi) - kb;
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c)
                        if (c < lo || c >= hi) sv[c] = -INFINITY;
                }
                // row max: four chains of three-input maxima
                float mx0 = fmaxf(sv[0], sv[1]), mx1 = fmaxf(sv[2], sv[3]);
                float mx2 = fmaxf(sv[4], sv[5]), mx3 = fmaxf(sv[6], sv[7]);
#pragma unroll
                for (int c = 8; c < kBlockN; c += 8) {
                    mx0 = fmax3(mx0, sv[c], sv[c + 1]);
                    mx1 = fmax3(mx1, sv[c + 2], sv[c + 3]);
                    mx2 = fmax3(mx2, sv[c + 4], sv[c + 5]);
                    mx3 = fmax3(mx3, sv[c + 6], sv[c + 7]);
                }
                const float m_tile = fmaxf(fmax3(mx0, mx1, mx2), mx3) * sl2;
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
                // P as bf16 pairs over the first 64 columns of S: chunk c4 of 32
                // scores goes to the 16 columns at 16 c4, all already read above.
                // exponent arguments and the row sum on packed fp32 pairs
                const float2 sl2v = make_float2(sl2, sl2), negm = make_float2(-m_use, -m_use);
                float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 a = __ffma2_rn(make_float2(sv[c4 * 32 + 2 * i], sv[c4 * 32 + 2 * i + 1]), sl2v, negm);
                        const float p0 = ex2(a.x);
                        const float p1 = ex2(a.y);
                        sum2 = __fadd2_rn(sum2, make_float2(p0, p1));
                        pk[i] = pack_bf16(p0, p1);
                    }
                    tmem_st16(s_col + c4 * 16, pk);
                }
                l = l * alpha + (sum2.x + sum2.y);
                if (rescale) {
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(o_col + c, o);
                        tmem_wait_ld();
                        reg_fence(o);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 r = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                                        make_float2(alpha, alpha));
                            o[i] = __float_as_uint(r.x);
                            o[i + 1] = __float_as_uint(r.y);
                        }
                        tmem_st32(o_col + c, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->p_full[slot]);
            }
            if (!ok) break;
            // epilogue: O of the slot is final once the PV of its last tile is done
            if (!warp_wait(&ctl->pv_done[slot], (ns + nt - 1) & 1, ctl, hdr)) break;
            tc_fence_after();
            const float inv_l = 1.f / l;
            const size_t row = (size_t)(s.q_start + tok) * p.n_heads + h;
            uint4* dst = reinterpret_cast<uint4*>(p.out + row * D);
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tmem_ld32(o_col + c, o);
                tmem_wait_ld();
                reg_fence(o);
                if (valid) {
                    // whole 32-byte sectors per store when out allows it: the lanes
                    // of a warp write 32 different rows, so each store is 32 pieces
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t w[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            w[k] = pack_bf16(__uint_as_float(o[h * 16 + 2 * k]) * inv_l,
                                             __uint_as_float(o[h * 16 + 2 * k + 1]) * inv_l);
                        if (p.out_align32) {
                            st_global_v8(dst + c / 8 + 2 * h, w);
                        } else {
                            dst[c / 8 + 2 * h] = make_uint4(w[0], w[1], w[2], w[3]);
                            dst[c / 8 + 2 * h + 1] = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                }
            }
            if (valid && p.lse) p.lse[row] = (m + lg2(l)) * 0.69314718055994530942f;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->o_empty[slot]);
            ns += nt;
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
                     CUtensorMapL2promotion l2, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Paged bf16 pool [num_blocks * Hk][bs][128] as 5-D (64 columns, 8 rows, 2
// chunks, bs / 8 row groups, num_blocks * Hk) with byte strides (256, 128,
// 2048, bs * 256): a box of (64, 8, 2, min(bs, 128) / 8, 1) is one block's rows
// of one KV head, landing in shared memory as [8-row group][chunk][8 rows] of
// 128-byte rows (the staging the MMA descriptors of paged prefix tiles read).
cudaError_t encode_pool_by_block(CUtensorMap* m, const void* ptr, uint64_t bs, uint64_t z, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[5] = {64, 8, 2, bs / 8, z};
    cuuint64_t strides[4] = {256, 128, 2048, bs * 256};
    cuuint32_t box[5] = {64, 8, 2, box_rows / 8, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, bool kPaged, bool kQuant, bool kAlt = false, bool kHook = false>
cudaError_t launch_d(const FwdParams& p, int grid, cudaStream_t st) {
    constexpr int kSmem = smem_bytes<D>();
    static_assert(kSmem <= 232448, "shared memory budget");
    static int configured_for[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured_for[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(attn_fwd_kernel<D, kPaged, kQuant, kAlt, kHook>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmem);
        if (e != cudaSuccess) return e;
        configured_for[dev] = 1;
    }
    // programmatic dependent launch: the prologue may run while the previous
    // kernel of the call finishes (the kernel waits for it before reading its output)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_fwd_kernel<D, kPaged, kQuant, kAlt, kHook>, p);
}

}  // namespace

cudaError_t encode_fwd_maps(FwdParams& p, const void* q, int total_q, int num_seqs, int head_dim, int num_blocks) {
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
    if (p.block_table && p.kv_quant) {
        // int8 pools [num_blocks, Hk, bs, D] viewed (D, bs, num_blocks * Hk), box (D, min(bs, 128), 1)
        const uint64_t bs = 1ull << p.block_log2, Z = (uint64_t)num_blocks * Hk;
        e = encode3d(&p.tm_ck, p.cache_k, D, bs, Z, D, bs * D, (uint32_t)D, p.box_rows, 1, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_DATA_TYPE_UINT8);
        if (e != cudaSuccess) return e;
        return encode3d(&p.tm_cv, p.cache_v, D, bs, Z, D, bs * D, (uint32_t)D, p.box_rows, 1, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_DATA_TYPE_UINT8);
    }
    if (p.block_table && D == 128) {
        // one box per block (both column chunks); the kernel's paged d = 128 loads
        const uint64_t bs = 1ull << p.block_log2, Z = (uint64_t)num_blocks * Hk;
        e = encode_pool_by_block(&p.tm_ck, p.cache_k, bs, Z, (uint32_t)p.box_rows);
        if (e != cudaSuccess) return e;
        return encode_pool_by_block(&p.tm_cv, p.cache_v, bs, Z, (uint32_t)p.box_rows);
    }
    if (p.block_table) {
        // pool [num_blocks, Hk, bs, D] viewed (D, bs, num_blocks * Hk)
        const uint64_t bs = 1ull << p.block_log2, Z = (uint64_t)num_blocks * Hk;
        e = encode3d(&p.tm_ck, p.cache_k, D, bs, Z, D * 2, bs * D * 2, cc, p.box_rows, 1, sw,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (e != cudaSuccess) return e;
        return encode3d(&p.tm_cv, p.cache_v, D, bs, Z, D * 2, bs * D * 2, cc, p.box_rows, 1, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    }
    if (p.kv_quant) {
        // int8 codes [B, Hk, cap, D] viewed (D, cap, B*Hk), box (D, 128, 1), no swizzle
        e = encode3d(&p.tm_ck, p.cache_k, D, cap, (uint64_t)num_seqs * Hk, D, cap * D, (uint32_t)D, kBlockN, 1,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_DATA_TYPE_UINT8);
        if (e != cudaSuccess) return e;
        return encode3d(&p.tm_cv, p.cache_v, D, cap, (uint64_t)num_seqs * Hk, D, cap * D, (uint32_t)D, kBlockN, 1,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_DATA_TYPE_UINT8);
    }
    e = encode3d(&p.tm_ck, p.cache_k, D, cap, (uint64_t)num_seqs * Hk, D * 2, cap * D * 2, cc, kBlockN, 1, sw,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e != cudaSuccess) return e;
    return encode3d(&p.tm_cv, p.cache_v, D, cap, (uint64_t)num_seqs * Hk, D * 2, cap * D * 2, cc, kBlockN, 1, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

template <int D>
cudaError_t launch_dim(const FwdParams& p, int grid, cudaStream_t st) {
    static_assert(D == 32 || D == 64 || D == 128, "head_dim");
    if (p.block_table) {
        if (p.kv_quant) return launch_d<D, true, true>(p, grid, st);
        return p.alt ? launch_d<D, true, false, true>(p, grid, st) : launch_d<D, true, false>(p, grid, st);
    }
    if (p.kv_quant) return launch_d<D, false, true>(p, grid, st);
    return p.alt ? launch_d<D, false, false, true>(p, grid, st) : launch_d<D, false, false>(p, grid, st);
}

cudaError_t launch_attn_fwd(const FwdParams& p, int head_dim, int grid, cudaStream_t st) {
    if (p.wait_timeout_test) {  // the test hook exists for the plain d = 128 kernel only
        if (head_dim != 128 || p.block_table || p.kv_quant) return cudaErrorNotSupported;
        return launch_d<128, false, false, false, true>(p, grid, st);
    }
    switch (head_dim) {
        case 32: return launch_dim<32>(p, grid, st);
        case 64: return launch_dim<64>(p, grid, st);
        case 128: return launch_dim<128>(p, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
