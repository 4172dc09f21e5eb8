/*
 * prefill_attn.h -- C ABI of the GB300 (sm_103a) causal varlen prefill-attention
 * library.
 *
 * One call computes, for every sequence b of a flattened varlen batch,
 *     out = softmax(Q K^T * scale) V
 * under a causal mask, where the keys/values of b are its P_b = cache_offsets[b]
 * cached tokens followed by its own n_b new tokens, and writes each new
 * token's K and V once into the per-sequence KV cache.
 *
 * Passages this interface follows (page title, section):
 *   - flattened [Total_Tokens, ...] stream with cumulative offsets cu_seqlens
 *     (e.g. [0, 5, 7, 10] for prompts of 5, 2 and 3 tokens); the kernel reads
 *     cu_seqlens and attends only within one request:
 *     "大模型 Prompt Prefill 阶段的高效 Batching 与算子排布" (nxmr.cn), §2.
 *   - chunked prefill: a chunk attends to its cached prefix plus itself, packed
 *     with one-token decode rows in the same batch: same page §3;
 *     "大模型推理优化：Prefill、Decode与KV Cache的工程实践" (zskr.cn), §2.2.
 *   - attention softmax(QK^T/sqrt(d_k))V and the (num_heads, seq_len, head_dim)
 *     cache layout: "大语言模型推理核心：Prefill与Decode原理及工程优化"
 *     (yfxerp.com), §2.1-§2.2 and §3.2.
 *   - causal lower-triangular mask with the masked upper triangle skipped;
 *     GQA (query heads sharing fewer KV heads): untitled page on prefill/decode
 *     compute accounting (zwxr.cn), §3.3 and §2.4.
 *   - prefill as the producer of the KV cache: "Prefill不是热身：大模型推理的真正
 *     瓶颈与优化核心" (mhpn.cn), §1 and §4.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers on the current CUDA device, dense
 *     and row-major in the layout stated; bf16 means IEEE bfloat16 (2 bytes).
 *     Every pointer must be 16-byte aligned.  The caller owns every buffer and
 *     the stream; the library keeps only a small per-(device, stream) schedule
 *     workspace, freed by prefill_attn_release().
 *   - Functions return a pa_status and never throw.  Arguments checkable on the
 *     host are checked before anything is launched; on PA_ERR_* nothing was
 *     launched.  prefill_attn_last_error() gives a one-line reason.
 *   - Device metadata (cu_seqlens_*, cache_offsets) is read only on the device
 *     by prefill_attn_varlen.  It is trusted for speed but clamped: a sequence
 *     whose metadata is inconsistent is skipped (nothing of it is written) and
 *     the device error word records it (prefill_attn_device_status).
 *   - out must not alias q, k or v; the caches must not alias k or v.
 *   - Inputs are assumed finite.  Cache entries outside [0, P_b) of each slot are
 *     never read, so an uninitialised cache is fine.
 *   - CUDA graphs: prefill_attn_varlen / _ex calls enqueue only kernels and
 *     device copies, so they may be captured into a graph, on a stream that
 *     already ran a call (outside the capture) with at least the same
 *     num_seqs and work units (and the same rotary sizes when rope_theta > 0):
 *     under capture nothing is allocated, and a call whose workspace would have
 *     to grow returns PA_ERR_UNSUPPORTED.  A replay reruns the call with the
 *     sizes and pointers of the capture; the device metadata (cu_seqlens_*,
 *     cache_offsets) and the data in the buffers are read at replay time, so
 *     they may change between replays within those sizes.
 *     prefill_attn_varlen_noalloc allocates nothing at all.
 */
#ifndef PREFILL_ATTN_H
#define PREFILL_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 means the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,     /* a host-checkable argument is wrong */
    PA_ERR_UNSUPPORTED = 2,     /* valid, but outside what this build implements */
    PA_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed */
    PA_ERR_DEVICE_TIMEOUT = 4,  /* a kernel gave up waiting (bounded wait) */
    PA_ERR_DEVICE_METADATA = 5, /* device metadata was inconsistent; sequences skipped */
    PA_ERR_DEVICE_LAYOUT = 6    /* a kernel found its shared-memory window misaligned; it computed nothing */
} pa_status;

/* Bits of the device error word (prefill_attn_device_status). */
#define PA_DEVERR_METADATA 0x1  /* a sequence's cu_seqlens/cache_offsets were inconsistent */
#define PA_DEVERR_TIMEOUT 0x2   /* an mbarrier wait ran out of its iteration budget */
#define PA_DEVERR_OVERFLOW 0x4  /* more work units than the workspace holds */
#define PA_DEVERR_SMEM_ALIGN 0x8 /* the attention kernel's dynamic shared memory was not 1024-byte aligned
                                  * (the swizzled TMA/MMA tiles need it); its CTAs returned at once */

/*
 * prefill_attn_varlen -- causal varlen prefill attention with the KV-cache write.
 *
 *   q             [total_q, n_heads, head_dim] bf16: queries of the new tokens,
 *                 sequences packed head to tail (token-major).
 *   k, v          [total_q, n_kv_heads, head_dim] bf16: keys/values of the NEW
 *                 tokens only, same packing.
 *   cu_seqlens_q  [num_seqs + 1] int32: cu_seqlens_q[0] = 0, non-decreasing,
 *                 cu_seqlens_q[num_seqs] = total_q; sequence b owns rows
 *                 cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1.  Empty sequences allowed.
 *   cu_seqlens_k  [num_seqs + 1] int32: cumulative key counts; key count of b is
 *                 cache_offsets[b] + n_b (prefix + new).
 *   cache_k/v     [num_seqs, n_kv_heads, max_cache_len, head_dim] bf16: slot b is
 *                 sequence b.  Positions [0, P_b) are read as the prefix;
 *                 positions [P_b, P_b + n_b) receive the new k/v (bit copies);
 *                 nothing else is read or written.
 *   cache_offsets [num_seqs] int32: P_b, tokens already cached for b, which is
 *                 also where b's first new token is written.  Requires
 *                 P_b + n_b <= max_cache_len.
 *   out           [total_q, n_heads, head_dim] bf16: attention output, rounded to
 *                 nearest even from fp32.
 *   lse           [total_q, n_heads] fp32 or NULL: natural log of
 *                 sum_j exp(scale * q . k_j) over the visible keys.
 *   num_seqs      batch size (>= 0; 0 is a no-op).
 *   total_q       rows of q/k/v/out (= cu_seqlens_q[num_seqs]; the tensor maps need it).
 *   max_cache_len slot capacity of the caches (>= 1).
 *   n_heads, n_kv_heads  n_heads % n_kv_heads == 0; query head h reads KV head
 *                 h / (n_heads / n_kv_heads).  n_heads / n_kv_heads <= 128.
 *   head_dim      32, 64 or 128.
 *   scale         finite, > 0; usually 1/sqrt(head_dim).
 *   causal        1: query i of b sits at absolute position P_b + i and sees keys
 *                 0 .. P_b + i; 0: every query of b sees all P_b + n_b keys.
 *   stream        the CUDA stream everything is enqueued on.
 *
 * Asynchronous: PA_OK means the work was enqueued on `stream`, not that it has
 * finished.  The call allocates (stream-ordered) only when the schedule
 * workspace for this (device, stream) must grow.
 */
pa_status prefill_attn_varlen(
    const void *q, const void *k, const void *v,
    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
    void *cache_k, void *cache_v, const int32_t *cache_offsets,
    void *out, float *lse,
    int num_seqs, int total_q, int max_cache_len,
    int n_heads, int n_kv_heads, int head_dim,
    float scale, int causal, pa_stream_t stream);

/*
 * Options of prefill_attn_varlen_ex.  Zero-initialise the struct and set
 * struct_size = sizeof(pa_options); a field past the struct_size the caller
 * passes is taken as zero, so older callers keep working as fields are added.
 */
typedef struct pa_options {
    uint32_t struct_size;
    /* Sliding window ("attend over the last W tokens", sliding_window = 4096 in
     * "大语言模型推理核心：Prefill与Decode原理及工程优化" (yfxerp.com), §4.3):
     * 0 = none; W > 0 (requires causal = 1): the query at absolute position p
     * sees keys p - W + 1 .. p only.  KV tiles wholly outside every window of a
     * work unit are not read.  The cache still receives every new token. */
    int32_t window;
    /* Paged KV cache (PagedAttention's block pool and per-request block table:
     * "大模型推理优化：Prefill、Decode与KV Cache的工程实践" (zskr.cn) §4.2,
     * "大语言模型推理核心：Prefill与Decode原理及工程优化" (yfxerp.com) §4.1, and
     * the untitled compute-accounting page (zwxr.cn) §3.4).  block_table = NULL: the
     * contiguous per-sequence cache described under prefill_attn_varlen.
     * Otherwise cache_k and cache_v are pools of num_blocks blocks, each
     * [n_kv_heads][block_size][head_dim] bf16 (the pool is [num_blocks,
     * n_kv_heads, block_size, head_dim], row-major, 16-byte aligned), and
     * block_table is a device array of int32 [num_seqs][max_blocks_per_seq]:
     * position p of sequence b (prefix or new token) lives in row
     * p % block_size of block block_table[b * max_blocks_per_seq + p / block_size].
     * block_size is a power of two, 8 .. 4096; max_cache_len must equal
     * max_blocks_per_seq * block_size; num_blocks * n_kv_heads < 2^31.  Blocks
     * may be shared between sequences (a common prefix) as long as no two
     * sequences of a call write the same row.  Only the entries for positions
     * [0, cache_offsets[b] + seqlen_q[b]) are read; a sequence whose entry
     * there is outside [0, num_blocks) is rejected on the device like other
     * inconsistent metadata (PA_DEVERR_METADATA, nothing of it read or
     * written).  The call may read the rows of a sequence's last prefix block
     * past its prefix (their values never reach the result: any bit pattern,
     * NaN included, is fine there). */
    const int32_t *block_table;
    int32_t block_size;
    int32_t max_blocks_per_seq;
    int32_t num_blocks;
    int32_t reserved;  /* must be 0 */
    /* Rotary position embedding ("Prefill不是热身：大模型推理的真正瓶颈与优化核心"
     * (mhpn.cn) §5.1: the token at position m has its Q/K rotated by the angles
     * m * inv_freq[i], inv_freq[i] = 1 / rope_theta^(2i / head_dim)).
     * 0 = none (q and k are used as given).  rope_theta > 0: every new query
     * and key is rotated to its absolute position cache_offsets[b] + i before
     * attention, pairing dimension i with i + head_dim/2 (the Llama
     * "rotate-half" layout), and the cache receives the rotated key; cached
     * prefix keys are used as stored, i.e. already rotated.  inv_freq is
     * computed on the host in fp32 as 1.0f / powf(rope_theta, 2i / head_dim),
     * the angle is one fp32 multiply, and the rotation is fp32 rounded to bf16.
     * q and k are not modified: the rotated copies live in the library's
     * per-stream workspace (total_q * (n_heads + n_kv_heads) * head_dim * 2
     * bytes more).  The call then runs three kernels instead of two. */
    float rope_theta;
    int32_t reserved2;  /* must be 0 */
    /* Quantised KV cache ("大模型推理优化：Prefill、Decode与KV Cache的工程实践"
     * (zskr.cn) §4.3: INT8 keys and values, queries at full precision,
     * per-token granularity).  0 = bf16 cache.  1 = int8: cache_k and cache_v
     * are int8 [num_seqs, n_kv_heads, max_cache_len, head_dim] codes and
     * cache_k_scale / cache_v_scale fp32 [num_seqs, n_kv_heads, max_cache_len]
     * (4-byte aligned) hold one scale per cached (token, KV head) row; the row
     * stands for code * scale.  Each new row x (the rotated key when RoPE is on,
     * rounded to bf16) is written as scale = max|x| / 127 and code = the
     * nearest integer, ties to even, of x / scale (fp32 division), clamped to
     * +-127; an all-zero row is scale 0, codes 0.  The cached prefix is read
     * dequantised (code * scale, rounded to bf16 for the tensor cores); the
     * chunk's own keys and values are used at full precision.  With a
     * block_table the code and scale pools are [num_blocks, n_kv_heads,
     * block_size, head_dim] int8 and [num_blocks, n_kv_heads, block_size]
     * fp32, addressed through the table like the bf16 pools. */
    int32_t kv_quant;
    int32_t reserved3;  /* must be 0 */
    float *cache_k_scale;
    float *cache_v_scale;
    /* Test hook, 0 in normal use; head_dim 128, contiguous bf16 cache only
     * (PA_ERR_CUDA otherwise).  1: in the first CTA the producer thread first
     * waits on a barrier that nothing completes.  The wait gives up
     * after its bound (2 s), the CTA records PA_DEVERR_TIMEOUT in the device
     * error word, drains its copies, frees its tensor memory and exits; the
     * other CTAs finish their work units, and the rows of the units the first
     * CTA had taken are left unwritten.  It lets a test run the timeout path on
     * a healthy GPU: the call returns normally, prefill_attn_device_status
     * reports PA_ERR_DEVICE_TIMEOUT, and the context stays usable. */
    int32_t wait_timeout_test;
    /* Work schedule.  A work unit is a block of query tokens of one sequence
     * against one KV head, in Q tiles of 128 rows (128 / G tokens x the G
     * query heads of that KV head); the kernel runs two Q tiles ("slots")
     * against each K/V tile it loads.
     * 0 = chosen by the library per call:
     * 2 = units of two Q tiles sharing every K/V tile (quantised caches and
     *     launches with many units);
     * 3 = the same, but a unit whose rows fit one Q tile (a decode row, the
     *     last block of a prompt) splits its KV tiles between the two slots
     *     (even / odd tiles, partial results merged at the end), so that the
     *     second slot does not idle (launches where the new tokens average
     *     under 64 per sequence);
     * 1 = units of one Q tile, each splitting its KV tiles that way (launches
     *     with at most one two-tile unit per SM: twice the units).
     * 1 and 3 need a bf16 cache and wait_timeout_test = 0 (else
     * PA_ERR_INVALID_ARG).  Results agree within the stated tolerances
     * whatever the schedule (not bitwise: the summation order differs); the
     * cache contents are the same bits. */
    int32_t schedule;
} pa_options;

/*
 * prefill_attn_varlen_ex -- prefill_attn_varlen with options (NULL = none).
 * Same arguments, layouts, ownership and errors as prefill_attn_varlen, plus
 * PA_ERR_INVALID_ARG for a bad option (reason in prefill_attn_last_error()).
 */
pa_status prefill_attn_varlen_ex(
    const void *q, const void *k, const void *v,
    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
    void *cache_k, void *cache_v, const int32_t *cache_offsets,
    void *out, float *lse,
    int num_seqs, int total_q, int max_cache_len,
    int n_heads, int n_kv_heads, int head_dim,
    float scale, int causal, const pa_options *opts, pa_stream_t stream);

/*
 * prefill_attn_varlen_noalloc -- prefill_attn_varlen that allocates nothing.
 * The pages have no counterpart to this call; it exists for integration.
 *
 * Some callers cannot allocate device memory when they call in: serving
 * engines that hand nearly all of HBM to their own KV-cache arena at start-up
 * (a cudaMalloc would then fail, or carve into memory the arena counts on),
 * and runtimes that forbid allocation on the request path because an
 * allocation can synchronise the device and stall every stream.  This entry
 * point takes the same arguments as prefill_attn_varlen and computes the same
 * result, but the scheduler's scratch (the sanitised per-sequence metadata and
 * the sorted work list) lives in one fixed array of about 1 MiB compiled into
 * this library, instead of a workspace the library allocates.  That array is
 * resident on every device that loads the library until the process exits.
 *
 * Limits: num_seqs <= 4096 and at most 61440 work units, where the host bounds
 * the units as n_kv_heads * (ceil(total_q / (2 * (128 / G))) + num_seqs) with
 * G = n_heads / n_kv_heads.  A larger call returns PA_ERR_UNSUPPORTED with the
 * reason in prefill_attn_last_error() and launches nothing.
 *
 * The first call on each device looks up the array's device address on the
 * host (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call uses the same array: each call first clears its header (the work
 * counter and the device error word), so calls whose work overlaps on the GPU
 * -- on different streams, or on different host threads -- race on it and must
 * be serialised by the caller.  The error word of the array (the last call's
 * PA_DEVERR_* bits: metadata rejected, a wait timed out, too many units) is
 * read and cleared by prefill_attn_device_status, like a workspace's.  The
 * address lookup is kept per CUDA context, so a device reset (which unloads
 * the library's device code and reloads it elsewhere) is followed by a new
 * lookup on the next call.
 */
pa_status prefill_attn_varlen_noalloc(
    const void *q, const void *k, const void *v,
    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
    void *cache_k, void *cache_v, const int32_t *cache_offsets,
    void *out, float *lse,
    int num_seqs, int total_q, int max_cache_len,
    int n_heads, int n_kv_heads, int head_dim,
    float scale, int causal, pa_stream_t stream);

/*
 * prefill_attn_varlen_validate -- strict host-side check of the same arguments.
 * Copies the three metadata arrays to the host (synchronises `stream`) and
 * checks every rule stated above: PA_OK or PA_ERR_INVALID_ARG with the reason
 * in prefill_attn_last_error().  Launches nothing.  Meant for tests and debug
 * builds of callers; the fast path does not call it.
 */
pa_status prefill_attn_varlen_validate(
    const void *q, const void *k, const void *v,
    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
    void *cache_k, void *cache_v, const int32_t *cache_offsets,
    void *out, float *lse,
    int num_seqs, int total_q, int max_cache_len,
    int n_heads, int n_kv_heads, int head_dim,
    float scale, int causal, pa_stream_t stream);

/*
 * prefill_attn_device_status -- synchronise `stream`, then read and clear the
 * device error word of the current device's (device, stream) workspace, and,
 * once prefill_attn_varlen_noalloc has run on the current device, the error
 * word of its fixed scratch too (which holds the bits of the last such call:
 * each call clears it; synchronise that call's stream first if it is another
 * one).  *flags receives the union of the PA_DEVERR_* bits (may be NULL).
 * Returns PA_OK when the words were zero; else PA_ERR_DEVICE_TIMEOUT if the
 * timeout bit was set, PA_ERR_DEVICE_LAYOUT if the shared-memory alignment bit
 * was, else PA_ERR_DEVICE_METADATA.
 */
pa_status prefill_attn_device_status(pa_stream_t stream, int32_t *flags);

/* Free every workspace this library allocated (all devices, all streams).
 * The caller must make sure no launch that uses them is still running. */
void prefill_attn_release(void);

/* Static string naming a status code. */
const char *prefill_attn_status_string(pa_status s);

/* Reason for the last PA_ERR_* returned on this thread ("" if none). */
const char *prefill_attn_last_error(void);

/* Number of kernel launches the last successful prefill_attn_varlen call on
 * this thread enqueued (0 for an empty batch). */
int prefill_attn_last_launch_count(void);

/* The work schedule (pa_options.schedule: 1, 2 or 3) that the last
 * successful call on this thread ran (0 if it launched nothing). */
int prefill_attn_last_schedule(void);

/* The schedule the library picks when pa_options.schedule is 0, for a call
 * with these sizes on a GPU with num_sms SMs (kv_quant as in pa_options):
 * 2 for int8 caches; else 3 when total_q < 64 * num_seqs (decode rows); else
 * 1 when n_kv_heads * (total_q / (256 / G)) two-tile units, G = n_heads /
 * n_kv_heads, would not exceed the SMs; else 2.  Host-only (no CUDA
 * call); -1 for sizes a call rejects (a non-positive size or n_heads not a
 * multiple of n_kv_heads). */
int prefill_attn_auto_schedule(int total_q, int num_seqs, int n_heads, int n_kv_heads, int kv_quant, int num_sms);

#ifdef __cplusplus
}
#endif

#endif /* PREFILL_ATTN_H */
