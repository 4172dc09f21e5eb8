// api.cu -- the C ABI (include/prefill_attn.h): argument checks, the
// per-(device, stream) schedule workspace, and the launch sequence.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "prefill_attn.h"

namespace {

thread_local std::string g_last_error;
thread_local int g_last_launches = 0;
thread_local int g_last_schedule = 0;

pa_status fail(pa_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
    int max_units = 0;
    int max_seqs = 0;
    void* rope = nullptr;  // rotated q/k copies (grown on demand)
    size_t rope_bytes = 0;
};

std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// header | SeqInfo[max_seqs] | Unit[max_units] | int[2][max_seqs] (scheduler scratch)
size_t ws_bytes(int max_seqs, int max_units) {
    return align_up(sizeof(pa::WorkspaceHeader), 16) + (size_t)max_seqs * sizeof(pa::SeqInfo) +
           (size_t)max_units * sizeof(pa::Unit) + 2 * (size_t)max_seqs * sizeof(int);
}

pa::SeqInfo* ws_seqs(const Workspace& w) {
    return reinterpret_cast<pa::SeqInfo*>(static_cast<char*>(w.ptr) + align_up(sizeof(pa::WorkspaceHeader), 16));
}

pa::Unit* ws_units(const Workspace& w) { return reinterpret_cast<pa::Unit*>(ws_seqs(w) + w.max_seqs); }

int* ws_seq_scratch(const Workspace& w) { return reinterpret_cast<int*>(ws_units(w) + w.max_units); }

// True while `st` is being captured into a CUDA graph.
bool capturing(cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    return cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive;
}

// Returns the workspace of (device, stream), growing it (stream-ordered) when
// needed.  Under graph capture nothing is allocated: the stream must already
// hold a workspace big enough (from a call outside the capture).
pa_status get_workspace(int dev, cudaStream_t st, int num_seqs, int max_units, Workspace** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace& w = g_ws[std::make_pair(dev, st)];
    if (w.ptr && w.max_seqs >= num_seqs && w.max_units >= max_units) {
        *out = &w;
        return PA_OK;
    }
    if (capturing(st))
        return fail(PA_ERR_UNSUPPORTED,
                    "graph capture: the stream's workspace would have to grow (%d sequences, %d work units); "
                    "run a call of at least these sizes on this stream before capturing",
                    num_seqs, max_units);
    Workspace nw;
    nw.max_seqs = std::max(num_seqs, std::max(w.max_seqs, 64));
    nw.max_units = std::max(max_units, std::max(w.max_units, 4096));
    nw.bytes = ws_bytes(nw.max_seqs, nw.max_units);
    cudaError_t e = cudaMallocAsync(&nw.ptr, nw.bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
    e = cudaMemsetAsync(nw.ptr, 0, sizeof(pa::WorkspaceHeader), st);
    if (e == cudaSuccess && w.ptr)  // keep sticky error bits across a regrow
        e = cudaMemcpyAsync(nw.ptr, w.ptr, sizeof(int), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) {
        cudaFreeAsync(nw.ptr, st);
        return cuda_fail(e, "workspace init");
    }
    if (w.ptr) cudaFreeAsync(w.ptr, st);
    nw.rope = w.rope;  // the rotary scratch is grown on its own
    nw.rope_bytes = w.rope_bytes;
    w = nw;
    *out = &w;
    return PA_OK;
}

// Grows (stream-ordered) the rotated-q/k scratch of a workspace to `bytes`.
pa_status get_rope_scratch(Workspace* w, cudaStream_t st, size_t bytes, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (w->rope_bytes < bytes && capturing(st))
        return fail(PA_ERR_UNSUPPORTED,
                    "graph capture: the stream's rotary scratch would have to grow (%zu bytes); run a call with "
                    "rope_theta of at least these sizes on this stream before capturing",
                    bytes);
    if (w->rope_bytes < bytes) {
        void* nptr = nullptr;
        cudaError_t e = cudaMallocAsync(&nptr, bytes, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(rotary scratch)");
        if (w->rope) cudaFreeAsync(w->rope, st);
        w->rope = nptr;
        w->rope_bytes = bytes;
    }
    *out = w->rope;
    return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pa_status check_args(const void* q, const void* k, const void* v, const int32_t* cu_q, const int32_t* cu_k,
                     const void* cache_k, const void* cache_v, const int32_t* off, const void* out,
                     const float* lse, int num_seqs, int total_q, int max_cache_len, int n_heads,
                     int n_kv_heads, int head_dim, float scale, int causal, bool paged = false) {
    if (num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs must be >= 0 (got %d)", num_seqs);
    if (total_q < 0) return fail(PA_ERR_INVALID_ARG, "total_q must be >= 0 (got %d)", total_q);
    if (max_cache_len < 1) return fail(PA_ERR_INVALID_ARG, "max_cache_len must be >= 1 (got %d)", max_cache_len);
    if (n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "n_heads (%d) must be a positive multiple of n_kv_heads (%d)", n_heads,
                    n_kv_heads);
    if (n_heads / n_kv_heads > pa::kBlockM)
        return fail(PA_ERR_UNSUPPORTED, "n_heads / n_kv_heads = %d exceeds %d", n_heads / n_kv_heads, pa::kBlockM);
    if (head_dim != 32 && head_dim != 64 && head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 32, 64 or 128 (got %d)", head_dim);
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(PA_ERR_INVALID_ARG, "scale must be finite and > 0 (got %g)", (double)scale);
    if (causal != 0 && causal != 1) return fail(PA_ERR_INVALID_ARG, "causal must be 0 or 1 (got %d)", causal);
    if (num_seqs == 0 || total_q == 0) return PA_OK;  // nothing is read or written
    const void* ptrs[] = {q, k, v, cu_q, cu_k, cache_k, cache_v, off, out};
    const char* names[] = {"q", "k", "v", "cu_seqlens_q", "cu_seqlens_k", "cache_k", "cache_v", "cache_offsets", "out"};
    for (int i = 0; i < 9; ++i) {
        if (!ptrs[i]) return fail(PA_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (i != 3 && i != 4 && i != 7 && !aligned16(ptrs[i]))
            return fail(PA_ERR_INVALID_ARG, "%s must be 16-byte aligned", names[i]);
    }
    if ((reinterpret_cast<uintptr_t>(cu_q) | reinterpret_cast<uintptr_t>(cu_k) | reinterpret_cast<uintptr_t>(off)) & 3u)
        return fail(PA_ERR_INVALID_ARG, "metadata arrays must be 4-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(PA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    if (out == q || out == k || out == v) return fail(PA_ERR_INVALID_ARG, "out must not alias q, k or v");
    if (cache_k == k || cache_k == v || cache_v == k || cache_v == v || cache_k == cache_v)
        return fail(PA_ERR_INVALID_ARG, "caches must be distinct and must not alias k or v");
    // Row counts used by 32-bit kernel index arithmetic.
    if ((long long)total_q * n_heads >= (1LL << 31))
        return fail(PA_ERR_UNSUPPORTED, "total_q * n_heads must be < 2^31");
    if (!paged && (long long)num_seqs * n_kv_heads * max_cache_len >= (1LL << 31))
        return fail(PA_ERR_UNSUPPORTED, "num_seqs * n_kv_heads * max_cache_len must be < 2^31");
    return PA_OK;
}

struct Options {
    int window = 0;
    const int32_t* block_table = nullptr;  // paged cache when set
    int block_size = 0, max_blocks = 0, num_blocks = 0;
    float rope_theta = 0.f;                // rotary embedding when > 0
    int kv_quant = 0;                      // 1: int8 cache with fp32 row scales
    float* scale_k = nullptr;
    float* scale_v = nullptr;
    int wait_timeout_test = 0;
    int schedule = 0;  // pa_options.schedule (0: chosen per call)
};

// Reads the caller's options; fields past the caller's struct_size count as zero.
pa_status read_options(const pa_options* opts, int causal, Options* o) {
    *o = Options();
    if (!opts) return PA_OK;
    const size_t have = opts->struct_size;
    if (have < offsetof(pa_options, window) + sizeof(int32_t))
        return fail(PA_ERR_INVALID_ARG, "pa_options.struct_size %u is too small", (unsigned)opts->struct_size);
    o->window = opts->window;
    if (o->window < 0) return fail(PA_ERR_INVALID_ARG, "window must be >= 0 (got %d)", o->window);
    if (o->window > 0 && causal != 1) return fail(PA_ERR_INVALID_ARG, "a sliding window needs causal = 1");
    if (have >= offsetof(pa_options, reserved) + sizeof(int32_t)) {
        if (opts->reserved != 0) return fail(PA_ERR_INVALID_ARG, "pa_options.reserved must be 0");
    }
    if (have >= offsetof(pa_options, num_blocks) + sizeof(int32_t) && opts->block_table) {
        o->block_table = opts->block_table;
        o->block_size = opts->block_size;
        o->max_blocks = opts->max_blocks_per_seq;
        o->num_blocks = opts->num_blocks;
        const int bs = o->block_size;
        if (bs < 8 || bs > 4096 || (bs & (bs - 1)) != 0)
            return fail(PA_ERR_UNSUPPORTED, "block_size must be a power of two in [8, 4096] (got %d)", bs);
        if (o->max_blocks < 1 || o->num_blocks < 1)
            return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq (%d) and num_blocks (%d) must be >= 1", o->max_blocks,
                        o->num_blocks);
        if (reinterpret_cast<uintptr_t>(o->block_table) & 3u)
            return fail(PA_ERR_INVALID_ARG, "block_table must be 4-byte aligned");
    } else if (have >= offsetof(pa_options, block_table) + sizeof(void*) && opts->block_table) {
        return fail(PA_ERR_INVALID_ARG, "pa_options.struct_size %u does not cover the paged-cache fields",
                    (unsigned)opts->struct_size);
    }
    if (have >= offsetof(pa_options, rope_theta) + sizeof(float)) {
        o->rope_theta = opts->rope_theta;
        if (!(o->rope_theta >= 0.f) || !std::isfinite(o->rope_theta))
            return fail(PA_ERR_INVALID_ARG, "rope_theta must be finite and >= 0 (got %g)", (double)o->rope_theta);
    }
    if (have >= offsetof(pa_options, reserved2) + sizeof(int32_t) && opts->reserved2 != 0)
        return fail(PA_ERR_INVALID_ARG, "pa_options.reserved2 must be 0");
    if (have >= offsetof(pa_options, kv_quant) + sizeof(int32_t) && opts->kv_quant != 0) {
        if (have < offsetof(pa_options, cache_v_scale) + sizeof(float*))
            return fail(PA_ERR_INVALID_ARG, "pa_options.struct_size %u does not cover the scale pointers",
                        (unsigned)opts->struct_size);
        if (opts->kv_quant != 1) return fail(PA_ERR_INVALID_ARG, "kv_quant must be 0 or 1 (got %d)", opts->kv_quant);
        if (opts->reserved3 != 0) return fail(PA_ERR_INVALID_ARG, "pa_options.reserved3 must be 0");
        if (!opts->cache_k_scale || !opts->cache_v_scale)
            return fail(PA_ERR_INVALID_ARG, "kv_quant = 1 needs cache_k_scale and cache_v_scale");
        if ((reinterpret_cast<uintptr_t>(opts->cache_k_scale) | reinterpret_cast<uintptr_t>(opts->cache_v_scale)) & 3u)
            return fail(PA_ERR_INVALID_ARG, "cache scales must be 4-byte aligned");
        o->kv_quant = 1;
        o->scale_k = opts->cache_k_scale;
        o->scale_v = opts->cache_v_scale;
    }
    if (have >= offsetof(pa_options, schedule) + sizeof(int32_t)) {
        if (opts->wait_timeout_test != 0 && opts->wait_timeout_test != 1)
            return fail(PA_ERR_INVALID_ARG, "wait_timeout_test must be 0 or 1");
        o->wait_timeout_test = opts->wait_timeout_test;
        if (opts->schedule < 0 || opts->schedule > 3)
            return fail(PA_ERR_INVALID_ARG, "schedule must be 0 .. 3 (got %d)", opts->schedule);
        if ((opts->schedule == 1 || opts->schedule == 3) && (o->kv_quant || o->wait_timeout_test))
            return fail(PA_ERR_INVALID_ARG, "schedule %d needs a bf16 cache and wait_timeout_test = 0",
                        opts->schedule);
        o->schedule = opts->schedule;
    }
    return PA_OK;
}

// Checks that need both the options and the call's sizes.
pa_status check_paged(const Options& o, int max_cache_len, int n_kv_heads) {
    if (!o.block_table) return PA_OK;
    if ((long long)o.max_blocks * o.block_size != max_cache_len)
        return fail(PA_ERR_INVALID_ARG, "max_cache_len (%d) must equal max_blocks_per_seq (%d) * block_size (%d)",
                    max_cache_len, o.max_blocks, o.block_size);
    if ((long long)o.num_blocks * n_kv_heads >= (1LL << 31))
        return fail(PA_ERR_UNSUPPORTED, "num_blocks * n_kv_heads must be < 2^31");
    return PA_OK;
}

// The schedule of a call (pa_options.schedule 1 .. 3).  Two-tile units
// unless the launch is mostly decode rows (new tokens averaging under 64 per
// sequence: a decode unit then splits its KV tiles between both softmax slots
// so that the second does not idle) or is so small that two-tile units would
// not give every SM one (then one-tile units, twice as many, each splitting
// its tiles).  The splitting kernel variant runs other units a few per cent
// slower and one K/V tile then feeds one Q tile instead of two, so it is not
// taken for anything else.  Measured on GB300 (152 SMs), TFLOP/s with
// one-tile / two-tile units: a 512-token chunk over a 4096-token prefix, GQA
// 32/8 (64 two-tile units) 819 / 540; 1024-token prompts (128 units) 315 /
// 296 (MHA) and 318 / 309 (GQA-4); a 1536-token MHA prompt (192 units) 490 /
// 531.  bf16 caches only.
int auto_schedule(int total_q, int num_seqs, int n_heads, int n_kv_heads, bool kv_quant, int sms) {
    if (kv_quant) return 2;
    if ((long long)total_q < 64LL * num_seqs) return 3;
    const int tpu = pa::kSlots * (pa::kBlockM / (n_heads / n_kv_heads));
    const long long full_units = (long long)n_kv_heads * (total_q / tpu);
    return full_units <= sms ? 1 : 2;
}

// Upper bound on the work units of a call (host-side; device metadata unread).
long long unit_bound(int total_q, int num_seqs, int n_heads, int n_kv_heads, int slots) {
    const int group = n_heads / n_kv_heads;
    const int tpu = slots * (pa::kBlockM / group);  // query tokens per work unit
    return (long long)n_kv_heads * ((total_q + tpu - 1) / tpu + num_seqs);
}

int sm_count(int dev, pa_status* s) {
    int sms = 0;
    const cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    *s = e == cudaSuccess ? PA_OK : cuda_fail(e, "cudaDeviceGetAttribute");
    return sms;
}

// Device address of the allocation-free entry point's scratch array in the
// current context, or nullptr if that entry point has not run there yet.
void* noalloc_scratch_if_set_up();

struct Scratch {
    pa::WorkspaceHeader* hdr;
    pa::SeqInfo* seqs;
    pa::Unit* units;
    int max_units;
    int* seq_scratch;      // int[2][num_seqs] for the scheduler
    void* rope = nullptr;  // room for the rotated q and k when the rotary embedding is on
};

// Enqueues the scheduler and the attention kernel (arguments already checked).
pa_status enqueue(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                  const int32_t* cu_seqlens_k, void* cache_k, void* cache_v, const int32_t* cache_offsets, void* out,
                  float* lse, int num_seqs, int total_q, int max_cache_len, int n_heads, int n_kv_heads,
                  int head_dim, float scale, int causal, const Options& o, const Scratch& scr, long long units_bound,
                  int sched, int sms, cudaStream_t stream) {
    const int slots = sched == 1 ? 1 : pa::kSlots;  // Q tiles per unit
    const int group = n_heads / n_kv_heads;
    pa::ScheduleArgs sa;
    sa.cu_seqlens_q = cu_seqlens_q;
    sa.cu_seqlens_k = cu_seqlens_k;
    sa.cache_offsets = cache_offsets;
    sa.hdr = scr.hdr;
    sa.seqs = scr.seqs;
    sa.units = scr.units;
    sa.seq_scratch = scr.seq_scratch;
    sa.seq_group = scr.seq_scratch + num_seqs;
    sa.num_seqs = num_seqs;
    sa.total_q = total_q;
    sa.max_cache_len = max_cache_len;
    sa.n_kv_heads = n_kv_heads;
    sa.head_dim = head_dim;
    sa.group = group;
    sa.causal = causal;
    sa.window = o.window;
    sa.max_units = scr.max_units;
    sa.num_ctas = (int)std::min<long long>(sms, units_bound);
    sa.unit_slots = slots;
    sa.block_table = o.block_table;
    sa.block_size = o.block_size;
    sa.max_blocks = o.max_blocks;
    sa.num_blocks = o.num_blocks;
    cudaError_t e = pa::launch_build_schedule(sa, stream);
    if (e != cudaSuccess) return cuda_fail(e, "schedule launch");

    int launches = 2;
    if (o.rope_theta > 0.f) {
        // rotary prologue: attention then reads the rotated copies
        pa::RopeParams rp;
        rp.q = static_cast<const __nv_bfloat16*>(q);
        rp.k = static_cast<const __nv_bfloat16*>(k);
        rp.q_rot = static_cast<__nv_bfloat16*>(scr.rope);
        rp.k_rot = rp.q_rot + (size_t)total_q * n_heads * head_dim;
        rp.cu_seqlens_q = cu_seqlens_q;
        rp.seqs = scr.seqs;
        rp.total_q = total_q;
        rp.num_seqs = num_seqs;
        rp.n_heads = n_heads;
        rp.n_kv_heads = n_kv_heads;
        rp.head_dim = head_dim;
        for (int i = 0; i < head_dim / 2; ++i)
            rp.inv_freq[i] = 1.0f / std::pow(o.rope_theta, (float)(2 * i) / (float)head_dim);
        e = pa::launch_rope(rp, stream);
        if (e != cudaSuccess) return cuda_fail(e, "rotary prologue launch");
        q = rp.q_rot;
        k = rp.k_rot;
        launches = 3;
    }

    pa::FwdParams p;
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.cache_k = static_cast<__nv_bfloat16*>(cache_k);
    p.cache_v = static_cast<__nv_bfloat16*>(cache_v);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.hdr = scr.hdr;
    p.seqs = scr.seqs;
    p.units = scr.units;
    p.n_heads = n_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = group;
    p.max_cache_len = max_cache_len;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.causal = causal;
    p.window = o.window;
    p.block_table = o.block_table;
    p.block_log2 = 0;
    while (o.block_table && (1 << p.block_log2) < o.block_size) ++p.block_log2;
    p.box_rows = std::min(o.block_size, pa::kBlockN);
    p.max_blocks = o.max_blocks;
    p.num_blocks = o.num_blocks;
    p.kv_quant = o.kv_quant;
    p.wait_timeout_test = o.wait_timeout_test;
    p.alt = sched != 2;
    p.unit_slots = slots;
    p.out_align32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
    p.scale_k = o.scale_k;
    p.scale_v = o.scale_v;
    e = pa::encode_fwd_maps(p, q, total_q, num_seqs, head_dim, o.num_blocks);
    if (e != cudaSuccess) return cuda_fail(e, "tensor map encoding");
    const int grid = (int)std::min<long long>(sms, units_bound);
    e = pa::launch_attn_fwd(p, head_dim, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    g_last_launches = launches;
    g_last_schedule = sched;
    return PA_OK;
}

}  // namespace

extern "C" {


const char* prefill_attn_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_DEVICE_TIMEOUT: return "PA_ERR_DEVICE_TIMEOUT";
        case PA_ERR_DEVICE_METADATA: return "PA_ERR_DEVICE_METADATA";
        case PA_ERR_DEVICE_LAYOUT: return "PA_ERR_DEVICE_LAYOUT";
    }
    return "PA_ERR_UNKNOWN";
}

const char* prefill_attn_last_error(void) { return g_last_error.c_str(); }

int prefill_attn_last_launch_count(void) { return g_last_launches; }

int prefill_attn_last_schedule(void) { return g_last_schedule; }

int prefill_attn_auto_schedule(int total_q, int num_seqs, int n_heads, int n_kv_heads, int kv_quant, int num_sms) {
    if (total_q <= 0 || num_seqs <= 0 || n_heads <= 0 || n_kv_heads <= 0 || num_sms <= 0 ||
        n_heads % n_kv_heads != 0 || n_heads / n_kv_heads > pa::kBlockM)
        return -1;
    return auto_schedule(total_q, num_seqs, n_heads, n_kv_heads, kv_quant != 0, num_sms);
}

pa_status prefill_attn_varlen(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                              const int32_t* cu_seqlens_k, void* cache_k, void* cache_v,
                              const int32_t* cache_offsets, void* out, float* lse, int num_seqs, int total_q,
                              int max_cache_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                              int causal, pa_stream_t stream_) {
    return prefill_attn_varlen_ex(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse,
                                  num_seqs, total_q, max_cache_len, n_heads, n_kv_heads, head_dim, scale, causal,
                                  nullptr, stream_);
}

pa_status prefill_attn_varlen_ex(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                                 const int32_t* cu_seqlens_k, void* cache_k, void* cache_v,
                                 const int32_t* cache_offsets, void* out, float* lse, int num_seqs, int total_q,
                                 int max_cache_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                                 int causal, const pa_options* opts, pa_stream_t stream_) {
    g_last_error.clear();
    g_last_launches = 0;
    g_last_schedule = 0;
    Options o;
    pa_status s = read_options(opts, causal, &o);
    if (s != PA_OK) return s;
    s = check_args(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse, num_seqs,
                   total_q, max_cache_len, n_heads, n_kv_heads, head_dim, scale, causal, o.block_table != nullptr);
    if (s != PA_OK) return s;
    s = check_paged(o, max_cache_len, n_kv_heads);
    if (s != PA_OK) return s;
    if (num_seqs == 0 || total_q == 0) return PA_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const int sms = sm_count(dev, &s);
    if (s != PA_OK) return s;
    const int sched = o.schedule            ? o.schedule
                      : o.wait_timeout_test ? 2  // the hook's kernel
                                            : auto_schedule(total_q, num_seqs, n_heads, n_kv_heads, o.kv_quant != 0, sms);
    const int slots = sched == 1 ? 1 : pa::kSlots;
    const long long max_units_ll = unit_bound(total_q, num_seqs, n_heads, n_kv_heads, slots);
    if (max_units_ll >= (1LL << 31)) return fail(PA_ERR_UNSUPPORTED, "too many work units");
    Workspace* ws = nullptr;
    s = get_workspace(dev, stream, num_seqs, (int)max_units_ll, &ws);
    if (s != PA_OK) return s;
    Scratch scr{static_cast<pa::WorkspaceHeader*>(ws->ptr), ws_seqs(*ws), ws_units(*ws), ws->max_units,
                ws_seq_scratch(*ws)};
    if (o.rope_theta > 0.f) {
        s = get_rope_scratch(ws, stream, (size_t)total_q * (n_heads + n_kv_heads) * head_dim * 2, &scr.rope);
        if (s != PA_OK) return s;
    }
    return enqueue(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse, num_seqs, total_q,
                   max_cache_len, n_heads, n_kv_heads, head_dim, scale, causal, o, scr, max_units_ll, sched, sms,
                   stream);
}

pa_status prefill_attn_varlen_validate(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                                       const int32_t* cu_seqlens_k, void* cache_k, void* cache_v,
                                       const int32_t* cache_offsets, void* out, float* lse, int num_seqs,
                                       int total_q, int max_cache_len, int n_heads, int n_kv_heads, int head_dim,
                                       float scale, int causal, pa_stream_t stream_) {
    g_last_error.clear();
    pa_status s = check_args(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse,
                             num_seqs, total_q, max_cache_len, n_heads, n_kv_heads, head_dim, scale, causal);
    if (s != PA_OK || num_seqs == 0) return s;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    std::vector<int32_t> cq(num_seqs + 1), ck(num_seqs + 1), of(num_seqs);
    cudaError_t e = cudaMemcpyAsync(cq.data(), cu_seqlens_q, cq.size() * 4, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ck.data(), cu_seqlens_k, ck.size() * 4, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(of.data(), cache_offsets, of.size() * 4, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "reading metadata");
    if (cq[0] != 0) return fail(PA_ERR_INVALID_ARG, "cu_seqlens_q[0] = %d, must be 0", cq[0]);
    if (cq[num_seqs] != total_q)
        return fail(PA_ERR_INVALID_ARG, "cu_seqlens_q[num_seqs] = %d but total_q = %d", cq[num_seqs], total_q);
    for (int b = 0; b < num_seqs; ++b) {
        const long long n = (long long)cq[b + 1] - cq[b];
        if (n < 0) return fail(PA_ERR_INVALID_ARG, "cu_seqlens_q decreases at sequence %d", b);
        if (of[b] < 0) return fail(PA_ERR_INVALID_ARG, "cache_offsets[%d] = %d < 0", b, of[b]);
        if ((long long)ck[b + 1] - ck[b] != (long long)of[b] + n)
            return fail(PA_ERR_INVALID_ARG,
                        "sequence %d: cu_seqlens_k gives %lld keys, cache_offsets + seqlen_q = %lld", b,
                        (long long)ck[b + 1] - ck[b], (long long)of[b] + n);
        if ((long long)of[b] + n > max_cache_len)
            return fail(PA_ERR_INVALID_ARG, "sequence %d: %lld tokens exceed max_cache_len %d", b,
                        (long long)of[b] + n, max_cache_len);
    }
    return PA_OK;
}

pa_status prefill_attn_device_status(pa_stream_t stream_, int32_t* flags) {
    g_last_error.clear();
    if (flags) *flags = 0;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    void* words[2] = {nullptr, noalloc_scratch_if_set_up()};  // workspace, allocation-free scratch
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_ws.find(std::make_pair(dev, stream));
        if (it != g_ws.end()) words[0] = it->second.ptr;
    }
    int32_t word = 0;
    for (void* ptr : words) {
        if (!ptr) continue;
        int32_t w = 0, zero = 0;
        e = cudaMemcpy(&w, ptr, sizeof w, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess && w != 0) e = cudaMemcpy(ptr, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
        word |= w;
    }
    if (flags) *flags = word;
    if (word == 0) return PA_OK;
    if (word & PA_DEVERR_TIMEOUT) return fail(PA_ERR_DEVICE_TIMEOUT, "device error word 0x%x", word);
    if (word & PA_DEVERR_SMEM_ALIGN) return fail(PA_ERR_DEVICE_LAYOUT, "device error word 0x%x", word);
    return fail(PA_ERR_DEVICE_METADATA, "device error word 0x%x", word);
}

void prefill_attn_release(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : g_ws) {
        cudaSetDevice(kv.first.first);
        if (kv.second.ptr) cudaFree(kv.second.ptr);
        if (kv.second.rope) cudaFree(kv.second.rope);
    }
    cudaSetDevice(cur);
    g_ws.clear();
}


}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant: the scheduler scratch lives in a fixed device array.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxSeqs = 4096;
constexpr int kNoAllocMaxUnits = 61440;
constexpr size_t kNoAllocHeaderBytes = 16;
constexpr size_t kNoAllocBytes = kNoAllocHeaderBytes + (size_t)kNoAllocMaxSeqs * sizeof(pa::SeqInfo) +
                                 (size_t)kNoAllocMaxUnits * sizeof(pa::Unit) + 2 * (size_t)kNoAllocMaxSeqs * sizeof(int);
static_assert(sizeof(pa::WorkspaceHeader) <= kNoAllocHeaderBytes, "header size");

// In host code this name is only a stand-in for the array; its device address
// comes from cudaGetSymbolAddress, once per device.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// The array's address is looked up once per CUDA context, keyed by the
// context's unique id: a device reset destroys the context (and the loaded
// device code with it), and the next context, even on the same device, gets an
// id of its own and so a fresh lookup.
std::mutex g_noalloc_mu;
std::map<unsigned long long, void*> g_noalloc_addr;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the current context (false if there is none or the driver lacks the call).
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

pa_status noalloc_scratch(void** out) {
    unsigned long long id = 0;
    if (!current_context_id(&id)) return fail(PA_ERR_CUDA, "no current CUDA context");
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    auto it = g_noalloc_addr.find(id);
    if (it != g_noalloc_addr.end()) {
        *out = it->second;
        return PA_OK;
    }
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);  // in the current context
    if (e != cudaSuccess || !ptr) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_noalloc_addr[id] = ptr;
    *out = ptr;
    return PA_OK;
}

}  // namespace

namespace {
void* noalloc_scratch_if_set_up() {
    unsigned long long id = 0;
    if (!current_context_id(&id)) return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    auto it = g_noalloc_addr.find(id);
    return it == g_noalloc_addr.end() ? nullptr : it->second;
}
}  // namespace

extern "C" pa_status prefill_attn_varlen_noalloc(const void* q, const void* k, const void* v,
                                                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                                 void* cache_k, void* cache_v, const int32_t* cache_offsets,
                                                 void* out, float* lse, int num_seqs, int total_q,
                                                 int max_cache_len, int n_heads, int n_kv_heads, int head_dim,
                                                 float scale, int causal, pa_stream_t stream_) {
    g_last_error.clear();
    g_last_launches = 0;
    g_last_schedule = 0;
    pa_status s = check_args(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse,
                             num_seqs, total_q, max_cache_len, n_heads, n_kv_heads, head_dim, scale, causal);
    if (s != PA_OK) return s;
    if (num_seqs == 0 || total_q == 0) return PA_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const int sms = sm_count(dev, &s);
    if (s != PA_OK) return s;
    const int sched = auto_schedule(total_q, num_seqs, n_heads, n_kv_heads, false, sms);
    const long long units = unit_bound(total_q, num_seqs, n_heads, n_kv_heads, sched == 1 ? 1 : pa::kSlots);
    if (num_seqs > kNoAllocMaxSeqs)
        return fail(PA_ERR_UNSUPPORTED, "num_seqs %d exceeds the allocation-free limit %d", num_seqs, kNoAllocMaxSeqs);
    if (units > kNoAllocMaxUnits)
        return fail(PA_ERR_UNSUPPORTED, "up to %lld work units exceed the allocation-free limit %d", units,
                    kNoAllocMaxUnits);
    void* scratch = nullptr;
    s = noalloc_scratch(&scratch);
    if (s != PA_OK) return s;
    // the array keeps the previous call's contents: clear the header (error word, counters)
    e = cudaMemsetAsync(scratch, 0, kNoAllocHeaderBytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the scratch header");
    pa::SeqInfo* seqs = reinterpret_cast<pa::SeqInfo*>(static_cast<unsigned char*>(scratch) + kNoAllocHeaderBytes);
    pa::Unit* units_ws = reinterpret_cast<pa::Unit*>(seqs + kNoAllocMaxSeqs);
    Scratch scr{static_cast<pa::WorkspaceHeader*>(scratch), seqs, units_ws, kNoAllocMaxUnits,
                reinterpret_cast<int*>(units_ws + kNoAllocMaxUnits)};
    return enqueue(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse, num_seqs, total_q,
                   max_cache_len, n_heads, n_kv_heads, head_dim, scale, causal, Options(), scr, units, sched, sms,
                   stream);
}
