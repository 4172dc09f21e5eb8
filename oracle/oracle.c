/*
 * oracle.c -- plain fp64 CPU definition of causal varlen prefill attention
 * with the KV-cache write.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may call,
 * link or load this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header or constant
 * with the CUDA path.
 *
 * Pages cited (title, site), by short name:
 *   [mhpn]   "Prefill不是热身：大模型推理的真正瓶颈与优化核心" (mhpn.cn)
 *   [zskr]   "大模型推理优化：Prefill、Decode与KV Cache的工程实践" (zskr.cn)
 *   [nxmr]   "大模型 Prompt Prefill 阶段的高效 Batching 与算子排布" (nxmr.cn)
 *   [yfxerp] "大语言模型推理核心：Prefill与Decode原理及工程优化" (yfxerp.com)
 *   [zwxr]   the untitled page on prefill/decode compute accounting (zwxr.cn)
 *
 * What it computes, written out as its definition (no tiling, no online
 * softmax, no reordering beyond the plain loops below):
 *
 *  - Scaled dot-product attention softmax(Q K^T * scale) V, one query row at a
 *    time ([yfxerp] §2.2; [mhpn] §3).  The softmax denominator runs over the
 *    whole visible row ([yfxerp] §2.2: leaving out any key changes every
 *    weight of the row).
 *  - Varlen packing: sequence b owns query rows cu_seqlens_q[b] ..
 *    cu_seqlens_q[b+1]-1 of the flattened stream and attends only inside
 *    itself ([nxmr] §2, cu_seqlens = [0, 5, 7, 10]).
 *  - Causal lower-triangular mask: a position sees itself and the positions
 *    before it ([zwxr] §3.3).
 *  - Chunked prefill: a chunk of n new tokens of sequence b follows
 *    P = cache_offsets[b] tokens already in the cache; its keys are the P cached
 *    keys followed by its own n keys, and new query i sits at absolute position
 *    P + i ([zskr] §2.2; [nxmr] §3).  A decode row is the chunk n = 1: it sees
 *    the cache plus itself ([zwxr] §1.2: the new token attends to all 301
 *    positions after its K/V are appended).
 *  - GQA: query head h reads KV head h / (n_heads / n_kv_heads)
 *    ([zwxr] §2.4: 32 query heads over 8 KV heads; contiguous groups).
 *  - Sliding window (optional, causal only): with a window of W tokens the
 *    query at absolute position p sees only keys p - W + 1 .. p, the W most
 *    recent positions including itself ([yfxerp] §4.3: attend over the last
 *    4096 tokens).
 *  - KV-cache production: cache[b][kvh][P + i][:] = k[cu_q[b] + i][kvh][:] (and
 *    the same for v), a bit copy into the (kv_heads, seq, head_dim) layout of
 *    [yfxerp] §2.1 / §3.2; every other cache entry is left as it was.
 *  - Paged cache (optional; [zskr] §4.2, [yfxerp] §4.1, [zwxr] §3.4): the cache
 *    is a pool of fixed-size blocks, [num_blocks][kv_heads][block_size][head_dim],
 *    and position p of sequence b lives in row p % block_size of block
 *    block_table[b][p / block_size].  Reads of the prefix and writes of the new
 *    tokens both go through the table; blocks may be shared between sequences.
 *  - Rotary position embedding (optional, rope_theta > 0; [mhpn] §5.1): the new
 *    query and key at absolute position m are rotated by the angles
 *    m * inv_freq[i], inv_freq[i] = 1 / theta^(2i / head_dim), i < head_dim/2,
 *    in the rotate-half pairing of the Llama models the page names (dimension i
 *    pairs with i + head_dim/2).  inv_freq and the angles are fp32, as the
 *    page's formula computes them; cos/sin and the rotation are fp64.  The
 *    rotated query and key are model-dtype tensors (the page discusses RoPE for
 *    FP16/BF16 models): both are rounded to bf16 (nearest, ties to even), and
 *    that rotated key is what attention uses and what the cache receives.
 *    Cached prefix keys are used as stored (they were rotated when written).
 *  - Quantised cache (optional, kv_quant = 1; [zskr] §4.3: INT8 keys and values,
 *    queries at full precision, per-token granularity among the page's
 *    options): each cached (token, KV head) row is int8 codes plus one fp32
 *    scale; the value it stands for is code * scale.  A new row x (its bf16
 *    values; the rotated key rounded to bf16 when RoPE is on) is stored as
 *    scale = max|x| / 127 and code = nearest integer (ties to even) of x / scale,
 *    all in fp32 (the precision the codes are decided in on the GPU too); a
 *    zero row is stored as scale 0, codes 0.  The prefix is read dequantised;
 *    the chunk's own keys and values are used at full precision.
 *
 * Inputs q, k, v and the caches are bf16 bit patterns (uint16); each value is
 * widened exactly to fp64 before any arithmetic.  Outputs are fp64:
 *   out[t][h][e]  = sum_j w_j V_j[e],  w_j = exp(s_j - m) / Z over visible j
 *   lse[t][h]     = m + ln Z            (natural log of sum_j exp(s_j))
 * with s_j = scale * <q, K_j>, m = max_j s_j, Z = sum_j exp(s_j - m).
 * Subtracting m is a mathematical identity that keeps exp() finite.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: it is the top half of an IEEE fp32. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;            /* [T][H][d], [T][Hk][d], [T][Hk][d] */
    const void *cache_k, *cache_v;         /* [B][Hk][cap][d] bf16 (or int8 codes), read for the prefix */
    const int32_t *cu_q, *off;
    double *out, *lse;
    int num_seqs, cap, n_heads, n_kv_heads, d;
    double scale;
    int causal;
    int window; /* 0: none */
    const int32_t *block_table; /* paged cache: [num_seqs][max_blocks]; NULL: contiguous slots */
    int block_size, max_blocks, num_blocks;
    const double *rope_cos, *rope_sin; /* [max_cache_len][d/2]; NULL: no rotary embedding */
    int kv_quant;                      /* 1: int8 codes + fp32 per-row scales */
    const float *scale_k, *scale_v;    /* [B][Hk][cap] (or the pool's rows) */
} problem;

/* The rotation of a head vector x (fp64, length d) to absolute position pos. */
static void rope_rotate(const problem *pb, int pos, double *x)
{
    const int half = pb->d / 2;
    const double *c = pb->rope_cos + (size_t)pos * half;
    const double *sn = pb->rope_sin + (size_t)pos * half;
    for (int i = 0; i < half; ++i) {
        const double a = x[i], b = x[i + half];
        x[i] = a * c[i] - b * sn[i];
        x[i + half] = b * c[i] + a * sn[i];
    }
}

static uint16_t double_to_bf16(double x);

/* The rotated head vector as the model-dtype (bf16) tensor it is. */
static void rope_rotate_bf16(const problem *pb, int pos, double *x)
{
    rope_rotate(pb, pos, x);
    for (int e = 0; e < pb->d; ++e)
        x[e] = bf16_to_double(double_to_bf16(x[e]));
}

/* Nearest bf16 (ties to even) of a finite double, as a bit pattern. */
static uint16_t double_to_bf16(double x)
{
    if (x == 0.0)
        return signbit(x) ? 0x8000 : 0;
    int e;
    frexp(x, &e);            /* |x| = f * 2^e, f in [0.5, 1) */
    if (e < -125)
        e = -125;            /* bf16 subnormal spacing 2^-133 */
    const double q = ldexp(1.0, e - 8); /* spacing of 8-significant-bit values near x */
    const double r = nearbyint(x / q) * q; /* default rounding mode: ties to even */
    const float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Row of the cache holding position `pos` of sequence b, KV head kvh. */
static size_t cache_row(const problem *pb, int b, int kvh, int pos)
{
    if (pb->block_table) {
        const int blk = pb->block_table[(size_t)b * pb->max_blocks + pos / pb->block_size];
        return ((size_t)blk * pb->n_kv_heads + kvh) * pb->block_size + (size_t)(pos % pb->block_size);
    }
    return ((size_t)b * pb->n_kv_heads + kvh) * pb->cap + (size_t)pos;
}

/* Key (which = 0) or value (which = 1) j of sequence b, KV head kvh, widened
 * to fp64 in `dst`: the cached prefix (dequantised when the cache is int8),
 * then the new tokens (rotated to their position when RoPE is on and
 * `rotate` is set). */
static void load_key(const problem *pb, int which, int b, int kvh, int j, int rotate, double *dst)
{
    const int d = pb->d;
    const int P = pb->off[b];
    if (j < P) {
        const size_t row = cache_row(pb, b, kvh, j);
        if (pb->kv_quant) {
            const int8_t *codes = (const int8_t *)(which ? pb->cache_v : pb->cache_k) + row * d;
            const double sc = (double)(which ? pb->scale_v : pb->scale_k)[row];
            for (int e = 0; e < d; ++e)
                dst[e] = (double)codes[e] * sc;
        } else {
            const uint16_t *r = (const uint16_t *)(which ? pb->cache_v : pb->cache_k) + row * d;
            for (int e = 0; e < d; ++e)
                dst[e] = bf16_to_double(r[e]);
        }
        return;
    }
    const uint16_t *r = (which ? pb->v : pb->k) + ((size_t)(pb->cu_q[b] + (j - P)) * pb->n_kv_heads + kvh) * d;
    for (int e = 0; e < d; ++e)
        dst[e] = bf16_to_double(r[e]);
    if (rotate && pb->rope_cos)
        rope_rotate_bf16(pb, j, dst);
}

/* One query row (sequence b, new token i, head h).  `s` has room for P+n
 * doubles, `qv` and `kv` for head_dim each. */
static void attend_row(const problem *pb, int b, int i, int h, double *s, double *qv, double *kv)
{
    const int d = pb->d;
    const int P = pb->off[b];
    const int n = pb->cu_q[b + 1] - pb->cu_q[b];
    const int Lk = P + n;
    const int kvh = h / (pb->n_heads / pb->n_kv_heads);
    const size_t t = (size_t)pb->cu_q[b] + (size_t)i;
    const uint16_t *qrow = pb->q + (t * pb->n_heads + h) * d;
    /* visible keys: first .. last (inclusive) */
    const int last = pb->causal ? P + i : Lk - 1;
    const int first = (pb->causal && pb->window > 0 && P + i - pb->window + 1 > 0) ? P + i - pb->window + 1 : 0;

    for (int e = 0; e < d; ++e)
        qv[e] = bf16_to_double(qrow[e]);
    if (pb->rope_cos)
        rope_rotate_bf16(pb, P + i, qv);
    double m = -INFINITY;
    for (int j = first; j <= last; ++j) {
        load_key(pb, 0, b, kvh, j, 1, kv);
        double dot = 0.0;
        for (int e = 0; e < d; ++e)
            dot += qv[e] * kv[e];
        s[j] = pb->scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    double Z = 0.0;
    for (int j = first; j <= last; ++j)
        Z += exp(s[j] - m);

    double *orow = pb->out + (t * pb->n_heads + h) * d;
    for (int e = 0; e < d; ++e)
        orow[e] = 0.0;
    for (int j = first; j <= last; ++j) {
        const double w = exp(s[j] - m) / Z;
        load_key(pb, 1, b, kvh, j, 0, kv);
        for (int e = 0; e < d; ++e)
            orow[e] += w * kv[e];
    }
    if (pb->lse)
        pb->lse[t * pb->n_heads + h] = m + log(Z);
}

/* Sequence that owns flattened token t (cu_q is non-decreasing). */
static int owner(const int32_t *cu_q, int num_seqs, int64_t t)
{
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (cu_q[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo; /* the last sequence starting at or before t owns it */
}

/* cos and sin of every position's rotary angles, [n_pos][d/2] each (cos
 * first, then sin): inv_freq[i] = 1 / theta^(2i / d) and the angle
 * pos * inv_freq[i] in fp32, as the page's formula computes them
 * ([mhpn] §5.1), then cos/sin in fp64.  NULL when out of memory. */
static double *rope_table(double rope_theta, int head_dim, int n_pos)
{
    const int half = head_dim / 2;
    const size_t n_tab = (size_t)(n_pos > 0 ? n_pos : 1) * half;
    double *tab = (double *)malloc(2 * n_tab * sizeof(double));
    if (!tab)
        return NULL;
    for (int i = 0; i < half; ++i) {
        const float inv_freq = 1.0f / powf((float)rope_theta, (float)(2 * i) / (float)head_dim);
        for (int pos = 0; pos < n_pos; ++pos) {
            const float angle = (float)pos * inv_freq;
            tab[(size_t)pos * half + i] = cos((double)angle);
            tab[n_tab + (size_t)pos * half + i] = sin((double)angle);
        }
    }
    return tab;
}

/* The rotation alone, before the bf16 rounding that the attention above
 * applies: head vectors x (bf16 bit patterns, [n_vec][head_dim]) rotated to
 * the positions pos[n_vec] (each in [0, max_pos)), widened exactly and
 * written to out ([n_vec][head_dim], fp64).  Returns 0, -1 on bad sizes, -6
 * when out of memory. */
int oracle_rope_rotate(const uint16_t *x, int64_t n_vec, int head_dim, const int32_t *pos, int max_pos,
                       double rope_theta, double *out)
{
    if (n_vec < 0 || head_dim <= 0 || head_dim % 2 != 0 || max_pos <= 0 || !(rope_theta > 0))
        return -1;
    for (int64_t r = 0; r < n_vec; ++r)
        if (pos[r] < 0 || pos[r] >= max_pos)
            return -1;
    double *tab = rope_table(rope_theta, head_dim, max_pos);
    if (!tab)
        return -6;
    problem pb;
    memset(&pb, 0, sizeof pb);
    pb.d = head_dim;
    pb.rope_cos = tab;
    pb.rope_sin = tab + (size_t)max_pos * (head_dim / 2);
    for (int64_t r = 0; r < n_vec; ++r) {
        double *o = out + (size_t)r * head_dim;
        for (int e = 0; e < head_dim; ++e)
            o[e] = bf16_to_double(x[(size_t)r * head_dim + e]);
        rope_rotate(&pb, pos[r], o);
    }
    free(tab);
    return 0;
}

/*
 * Returns 0 on success, a negative code for inconsistent metadata:
 *  -1 bad sizes, -2 cu_seqlens_q not starting at 0 or decreasing,
 *  -3 cu_seqlens_k inconsistent with cache_offsets + seqlen_q,
 *  -4 a sequence does not fit its cache slot, -5 a selected row out of range,
 *  -6 out of memory, -7 a window without the causal mask, -8 a bad block table.
 *
 * Paged cache: block_table != NULL, the caches are [num_blocks][Hk][block_size]
 * [head_dim] pools and max_cache_len must be max_blocks * block_size.
 *
 * rope_theta > 0 turns the rotary embedding on (head_dim must be even).
 *
 * kv_quant = 1: the caches are int8 codes and scale_k/scale_v (fp32, one per
 * cache row) their scales; scale_k_out/scale_v_out receive the scales of the
 * cache image (may be NULL when the cache images are).
 *
 * rows: optional list of (t * n_heads + h) query rows to compute; NULL = all.
 * Only the selected rows of out/lse are written.  The cache image
 * (cache_k_out/cache_v_out, may be NULL) is written in full: a copy of the
 * input cache with every new token's K/V stored at its slot position.
 */
int oracle_prefill_attention(
    const uint16_t *q, const uint16_t *k, const uint16_t *v,
    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, const int32_t *cache_offsets,
    const void *cache_k, const void *cache_v,
    void *cache_k_out, void *cache_v_out,
    double *out, double *lse,
    int num_seqs, int max_cache_len, int n_heads, int n_kv_heads, int head_dim,
    double scale, int causal, int window,
    const int32_t *block_table, int block_size, int max_blocks, int num_blocks,
    double rope_theta,
    int kv_quant, const float *scale_k, const float *scale_v, float *scale_k_out, float *scale_v_out,
    const int64_t *rows, int64_t n_rows, int n_threads)
{
    if (window < 0 || (window > 0 && !causal))
        return -7;
    if (num_seqs < 0 || max_cache_len < 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 ||
        n_heads % n_kv_heads != 0 || rope_theta < 0 || (rope_theta > 0 && head_dim % 2 != 0) ||
        kv_quant < 0 || kv_quant > 1 || (kv_quant && (!scale_k || !scale_v)))
        return -1;
    if (num_seqs > 0 && cu_seqlens_q[0] != 0)
        return -2;
    for (int b = 0; b < num_seqs; ++b) {
        int n = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        if (n < 0)
            return -2;
        if (cu_seqlens_k[b + 1] - cu_seqlens_k[b] != cache_offsets[b] + n)
            return -3;
        if (cache_offsets[b] < 0 || cache_offsets[b] + n > max_cache_len)
            return -4;
        if (block_table) {
            if (block_size <= 0 || max_blocks * block_size != max_cache_len)
                return -8;
            const int used = (cache_offsets[b] + n + block_size - 1) / block_size;
            for (int L = 0; L < used; ++L)
                if (block_table[(size_t)b * max_blocks + L] < 0 || block_table[(size_t)b * max_blocks + L] >= num_blocks)
                    return -8;
        }
    }
    const int64_t total_q = num_seqs > 0 ? cu_seqlens_q[num_seqs] : 0;

    problem pb = {q, k, v, cache_k, cache_v, cu_seqlens_q, cache_offsets, out, lse,
                  num_seqs, max_cache_len, n_heads, n_kv_heads, head_dim, scale, causal, window,
                  block_table, block_size, max_blocks, num_blocks, NULL, NULL, kv_quant, scale_k, scale_v};

    double *rope_tab = NULL;
    if (rope_theta > 0) {
        rope_tab = rope_table(rope_theta, head_dim, max_cache_len);
        if (!rope_tab)
            return -6;
        pb.rope_cos = rope_tab;
        pb.rope_sin = rope_tab + (size_t)(max_cache_len > 0 ? max_cache_len : 1) * (head_dim / 2);
    }

    const int64_t n_all = total_q * n_heads;
    const int64_t n_work = rows ? n_rows : n_all;
    if (rows) {
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= n_all) {
                free(rope_tab);
                return -5;
            }
    }
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * ((size_t)(max_cache_len > 0 ? max_cache_len : 1) +
                                                       2 * (size_t)head_dim));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t w = 0; w < n_work; ++w) {
            if (!s)
                continue;
            const int64_t r = rows ? rows[w] : w;
            const int64_t t = r / n_heads;
            const int h = (int)(r % n_heads);
            const int b = owner(cu_seqlens_q, num_seqs, t);
            attend_row(&pb, b, (int)(t - cu_seqlens_q[b]), h, s + 2 * (size_t)head_dim, s, s + head_dim);
        }
        free(s);
    }
    if (failed) {
        free(rope_tab);
        return -6;
    }

    /* The cache image: everything as it was, plus the new tokens at P + i. */
    const size_t cache_rows = block_table ? (size_t)num_blocks * n_kv_heads * block_size
                                          : (size_t)num_seqs * n_kv_heads * max_cache_len;
    const size_t elem = kv_quant ? sizeof(int8_t) : sizeof(uint16_t);
    for (int c = 0; c < 2; ++c) {
        uint8_t *dst = (uint8_t *)(c == 0 ? cache_k_out : cache_v_out);
        const uint8_t *src = (const uint8_t *)(c == 0 ? cache_k : cache_v);
        float *sdst = c == 0 ? scale_k_out : scale_v_out;
        const float *ssrc = c == 0 ? scale_k : scale_v;
        const uint16_t *fresh = c == 0 ? k : v;
        if (!dst)
            continue;
        if (dst != src)
            memcpy(dst, src, cache_rows * head_dim * elem);
        if (kv_quant && sdst && sdst != ssrc)
            memcpy(sdst, ssrc, cache_rows * sizeof(float));
        for (int b = 0; b < num_seqs; ++b) {
            const int P = cache_offsets[b];
            const int n = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
            for (int kvh = 0; kvh < n_kv_heads; ++kvh)
                for (int i = 0; i < n; ++i) {
                    const size_t row = cache_row(&pb, b, kvh, P + i);
                    const uint16_t *in = fresh + ((size_t)(cu_seqlens_q[b] + i) * n_kv_heads + kvh) * head_dim;
                    uint16_t x[head_dim]; /* the row as bf16: rotated and rounded when RoPE is on */
                    if (c == 0 && pb.rope_cos) {
                        double xr[head_dim];
                        for (int e = 0; e < head_dim; ++e)
                            xr[e] = bf16_to_double(in[e]);
                        rope_rotate(&pb, P + i, xr);
                        for (int e = 0; e < head_dim; ++e)
                            x[e] = double_to_bf16(xr[e]);
                    } else {
                        memcpy(x, in, (size_t)head_dim * sizeof(uint16_t));
                    }
                    if (!kv_quant) {
                        memcpy(dst + row * head_dim * elem, x, (size_t)head_dim * sizeof(uint16_t));
                        continue;
                    }
                    /* int8 codes with one fp32 scale per row, decided in fp32 */
                    float amax = 0.0f;
                    for (int e = 0; e < head_dim; ++e) {
                        const float a = fabsf((float)bf16_to_double(x[e]));
                        if (a > amax)
                            amax = a;
                    }
                    const float sc = amax / 127.0f;
                    int8_t *codes = (int8_t *)dst + row * head_dim;
                    for (int e = 0; e < head_dim; ++e) {
                        float qv = 0.0f;
                        if (sc > 0.0f) {
                            qv = rintf((float)bf16_to_double(x[e]) / sc);
                            if (qv > 127.0f)
                                qv = 127.0f;
                            if (qv < -127.0f)
                                qv = -127.0f;
                        }
                        codes[e] = (int8_t)qv;
                    }
                    if (sdst)
                        sdst[row] = sc;
                }
        }
    }
    free(rope_tab);
    return 0;
}
