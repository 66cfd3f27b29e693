/*
 * oracle.c -- plain fp64 CPU oracle for paged grouped-query decode / verify
 * attention, the KV append that precedes it, greedy prefix acceptance,
 * stochastic acceptance (speculative sampling), greedy acceptance over a draft
 * tree and the cache compaction that follows it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the package's smoke check and the bench's CPU
 * baseline leg do.  It shares no code, header or table with the CUDA kernels.
 *
 * Sources (web pages; cited by page title and section):
 *   [CS336-RU]  "CS336, лекции 10 и 12: инференс и оценка моделей"
 *   [KV-AR]     "جعل inference رخيصًا: KV cache وbatching والتكميم"
 *   [SONAR-KK]  "Болжау арқылы Sonar модельдерін жылдамдату"
 *   [CS336-ZH]  "Stanford CS336 Day 13 - Inference"
 *
 * Everything is written from the plain definitions, in fp64, one output element
 * at a time; there is no tiling, no online softmax and no split of the context.
 * Input elements (IEEE binary16 or bfloat16) are widened to double exactly.
 *
 * Notation follows [CS336-RU] §"Напоминание: трансформер": B sequences, T new
 * query tokens per sequence, N query heads, K key/value heads, G = N/K, head
 * size H.  Paged layout follows [CS336-RU] §"PagedAttention" (fixed-size blocks
 * of tokens plus a per-sequence block table):
 *   q            [B][T][N][H]
 *   k/v cache    [num_blocks][block_size][K][H]
 *   block_tables [B][max_blocks]   logical block i of sequence b -> physical id
 *   context_lens [B]               tokens held for b, INCLUDING the T new ones
 * (the last reading is ours: the pages define no such array.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Per-sequence error codes written to seq_err (0 = fine).  Same meaning as the
 * library's status codes of the same names, restated here on purpose. */
#define ORACLE_ERR_CONTEXT 7  /* context length < T, <= 0 or beyond the table */
#define ORACLE_ERR_BLOCK_ID 8 /* a needed block-table entry is not a valid block */

/* ---- element widening (IEEE 754 binary16; bfloat16 = top half of binary32) ---- */

double oracle_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25); /* (1.m) * 2^(e-15) */
    return sign ? -v : v;
}

double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double widen(uint16_t x, int dtype) {
    return dtype == 0 ? oracle_f16_to_f64(x) : oracle_bf16_to_f64(x);
}

/* ---- KV append ------------------------------------------------------------
 * [KV-AR], KV-cache section: each new token's key and value vectors are stored
 * once and reused by every later step.  [CS336-RU] §"PagedAttention": logical
 * position j of sequence b lives in physical block block_tables[b][j / bs] at
 * row j % bs.  Token t of the T new ones sits at position ctx_b - T + t.
 * A byte copy: the result must be bit-identical. */
int oracle_kv_append(int B, int T, int K, int H, int block_size, int num_blocks,
                     int max_blocks, const uint16_t *k_new, const uint16_t *v_new,
                     uint16_t *k_cache, uint16_t *v_cache,
                     const int32_t *block_tables, const int32_t *context_lens,
                     int32_t *seq_err) {
    int any = 0;
    size_t row = (size_t)K * H; /* one token's K heads x H elements */
    for (int b = 0; b < B; ++b) {
        int ctx = context_lens[b];
        if (seq_err) seq_err[b] = 0;
        if (ctx < T || ctx > (long long)max_blocks * block_size) {
            if (seq_err) seq_err[b] = ORACLE_ERR_CONTEXT;
            any = 1;
            continue;
        }
        for (int t = 0; t < T; ++t) {
            int pos = ctx - T + t;
            int blk = block_tables[(size_t)b * max_blocks + pos / block_size];
            if (blk < 0 || blk >= num_blocks) {
                if (seq_err && !seq_err[b]) seq_err[b] = ORACLE_ERR_BLOCK_ID;
                any = 1;
                continue;
            }
            size_t dst = ((size_t)blk * block_size + pos % block_size) * row;
            size_t src = ((size_t)b * T + t) * row;
            memcpy(k_cache + dst, k_new + src, row * sizeof(uint16_t));
            memcpy(v_cache + dst, v_new + src, row * sizeof(uint16_t));
        }
    }
    return any;
}

/* ---- quantized KV cache ----------------------------------------------------
 * [KV-AR], quantization section: symmetric absolute-maximum quantization --
 * qmax = 2^(bits-1) - 1, scale = max|W| / qmax, codes round(W / scale) clamped
 * to [-qmax-1, qmax], reconstruction codes * scale -- and fewer bytes per
 * element make every memory-bound decode step faster.  [CS336-RU]
 * §"Квантование": fp8 (e4m3) and int8 are the one-byte formats.
 *
 * Readings:
 *   - The rule is applied to every cached vector (one key or value row of one
 *     KV head, H elements), its fp32 scale stored per block as
 *     scale[block][kv head][row]: the append writes one token at a time, and a
 *     scale over a whole block would change as the block fills.
 *   - int8: qmax = 127.  e4m3 (OCP FP8 E4M3, finite max 448 -- the page's
 *     "[-240, 240]" is the range of another e4m3 variant): scale = max|W| / 448
 *     and the code is x / scale rounded to the nearest e4m3 value, ties to
 *     even, saturating at +-448.
 *   - The codes are integers decided in floating point, so they are computed in
 *     fp32 as the kernel does: max|W| of the widened elements, then scale =
 *     max / qmax and x / scale as IEEE fp32 divisions, ties to even.  A row of
 *     zeros has scale 0 and all codes 0. */
#define ORACLE_KV_INT8 1
#define ORACLE_KV_E4M3 2

/* e4m3 code (sign | 4-bit exponent, bias 7 | 3-bit mantissa) nearest to x,
 * ties to even, saturating at +-448 (no infinities; 0x7f / 0xff are NaN). */
static uint8_t e4m3_encode(float xf) {
    double x = (double)xf;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x)) return 0x7f;
    double v = fabs(x);
    if (v >= 448.0) return sign | 0x7e; /* saturate (448 itself is 0x7e) */
    if (v == 0.0) return sign;
    int e;
    (void)frexp(v, &e); /* v = f * 2^e, f in [0.5, 1) */
    int E = e - 1;      /* v in [2^E, 2^(E+1)) */
    if (E < -6) E = -6; /* subnormals: spacing 2^-9, like the lowest binade */
    double m = ldexp(v, 3 - E); /* v / 2^(E-3), exact */
    int mi = (int)nearbyint(m); /* ties to even under the default rounding */
    if (mi >= 16) {             /* rounded up into the next binade */
        mi = 8;
        E += 1;
    }
    if (mi < 8) return sign | (uint8_t)mi; /* subnormal (E == -6) */
    int field = E + 7;
    if (field > 15 || (field == 15 && mi - 8 > 6)) return sign | 0x7e;
    return sign | (uint8_t)(field << 3) | (uint8_t)(mi - 8);
}

/* value of an e4m3 code (NaN for 0x7f / 0xff) */
double oracle_e4m3_to_f64(uint8_t c) {
    int field = (c >> 3) & 15, m = c & 7;
    double s = (c & 0x80) ? -1.0 : 1.0;
    if (field == 15 && m == 7) return NAN;
    if (field == 0) return s * ldexp((double)m, -9);
    return s * ldexp(8.0 + m, field - 10);
}

uint8_t oracle_e4m3_from_float(float x) { return e4m3_encode(x); }

/* Quantize one row of n elements (fp16/bf16 bits) to one-byte codes. */
void oracle_quantize_row(const uint16_t *x, int n, int dtype, int kind, uint8_t *codes,
                         float *scale_out) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf((float)widen(x[i], dtype));
        if (a > amax) amax = a;
    }
    const float qmax = kind == ORACLE_KV_INT8 ? 127.0f : 448.0f;
    volatile float scale = amax / qmax; /* one fp32 division */
    *scale_out = scale;
    for (int i = 0; i < n; ++i) {
        if (scale == 0.0f) {
            codes[i] = 0;
            continue;
        }
        volatile float y = (float)widen(x[i], dtype) / scale; /* one fp32 division */
        if (kind == ORACLE_KV_INT8) {
            if (y != y) { /* a NaN element: code 0 */
                codes[i] = 0;
                continue;
            }
            float r = nearbyintf(y);
            if (r > 127.0f) r = 127.0f;
            if (r < -128.0f) r = -128.0f;
            codes[i] = (uint8_t)(int8_t)(int)r;
        } else {
            codes[i] = e4m3_encode(y);
        }
    }
}

/* Every row of an array [nrows][n] (a whole cache, for tests). */
void oracle_quantize_rows(const uint16_t *x, int nrows, int n, int dtype, int kind,
                          uint8_t *codes, float *scales) {
    for (int r = 0; r < nrows; ++r)
        oracle_quantize_row(x + (size_t)r * n, n, dtype, kind, codes + (size_t)r * n, &scales[r]);
}

static double code_value(uint8_t c, int kind) {
    return kind == ORACLE_KV_INT8 ? (double)(int8_t)c : oracle_e4m3_to_f64(c);
}

/* Quantized append: as oracle_kv_append, but each new key / value row of each
 * KV head is quantized on its way into the one-byte caches [NB][bs][K][H]; its
 * scale goes to k_scale / v_scale [NB][K][bs]. */
int oracle_kv_append_quant(int B, int T, int K, int H, int block_size, int num_blocks,
                           int max_blocks, int dtype, int kind, const uint16_t *k_new,
                           const uint16_t *v_new, uint8_t *k_cache, uint8_t *v_cache,
                           float *k_scale, float *v_scale, const int32_t *block_tables,
                           const int32_t *context_lens, int32_t *seq_err) {
    int any = 0;
    for (int b = 0; b < B; ++b) {
        int ctx = context_lens[b];
        if (seq_err) seq_err[b] = 0;
        if (ctx < T || ctx > (long long)max_blocks * block_size) {
            if (seq_err) seq_err[b] = ORACLE_ERR_CONTEXT;
            any = 1;
            continue;
        }
        for (int t = 0; t < T; ++t) {
            int pos = ctx - T + t;
            int blk = block_tables[(size_t)b * max_blocks + pos / block_size];
            if (blk < 0 || blk >= num_blocks) {
                if (seq_err && !seq_err[b]) seq_err[b] = ORACLE_ERR_BLOCK_ID;
                any = 1;
                continue;
            }
            int row = pos % block_size;
            for (int k = 0; k < K; ++k) {
                size_t src = (((size_t)b * T + t) * K + k) * H;
                size_t dst = (((size_t)blk * block_size + row) * K + k) * H;
                size_t sc = ((size_t)blk * K + k) * block_size + row;
                oracle_quantize_row(k_new + src, H, dtype, kind, k_cache + dst, &k_scale[sc]);
                oracle_quantize_row(v_new + src, H, dtype, kind, v_cache + dst, &v_scale[sc]);
            }
        }
    }
    return any;
}

/* ---- attention -------------------------------------------------------------
 * [CS336-RU] §"Арифметическая интенсивность инференса" (attention layer: scores
 * A = Q K^T, Y = softmax(A) V) and §"Уменьшаем KV-кэш" (GQA: N query heads, K
 * key/value heads, each KV head serves N/K query heads).  Readings: query head
 * n uses KV head n / G (contiguous groups); scores are multiplied by `scale`
 * (1/sqrt(H) unless given); query token t of the T new ones sees every cached
 * position j <= ctx - T + t (full prefix, causal among the new tokens).
 *
 * Local (sliding-window) attention, [CS336-RU] §"Уменьшаем KV-кэш" (local
 * attention: attend only to a recent stretch of the context, the KV cache no
 * longer grows with the sequence) and [CS336-ZH] §"Local Attention" (only
 * the last k tokens are attended; tokens that leave the window can be dropped
 * from the cache): with window > 0, query token t sees only positions
 * last-window < j <= last, last = ctx - T + t --
 * our reading of "the last k tokens" is the window tokens ending at the query
 * itself.  window == 0 is full attention.  Only the blocks holding a visible
 * position are looked up (blocks wholly below every window may be freed).
 *
 * Tree verification, [SONAR-KK] §"EAGLE": drafts form a tree (Top-K candidates
 * at each node), and verifying the tree in the target model needs a custom
 * attention mask.  With tree_mask != NULL, new token t (t < T) sees the whole
 * prefix (positions < ctx - T), itself, and new token j < t iff bit j of
 * tree_mask[b][t] is set: for a tree laid out in topological order (every
 * node after its parent), its ancestors.  Bits j >= t are ignored.
 * tree_mask == NULL is the chain (token t sees new tokens 0..t).  Window and
 * tree mask are not combined (the call rejects both at once).
 *
 * For each listed sequence b = b_list[i] (all b when b_list is NULL) writes
 * out[i][t][n][h] in fp64.  A sequence with a bad context length or a bad
 * block id gets an all-zero output and a nonzero seq_err[i]. */
int oracle_attention(int B, int T, int N, int K, int H, int block_size,
                     int num_blocks, int max_blocks, int dtype, double scale,
                     int window, const uint64_t *tree_mask, int kv_kind,
                     const float *k_scale, const float *v_scale, const uint16_t *q,
                     const void *k_cache, const void *v_cache, const int32_t *block_tables,
                     const int32_t *context_lens, const int32_t *b_list, int nb,
                     double *out, int32_t *seq_err, int nthreads) {
    if (K <= 0 || N % K != 0 || window < 0 || (window > 0 && tree_mask)) return -1;
    if (tree_mask && T > 64) return -1;
    int G = N / K;
    if (!b_list) nb = B;
    if (scale <= 0) scale = 1.0 / sqrt((double)H);
    int any = 0;

    /* validate each listed sequence first (plain loop) */
    int32_t *bad = (int32_t *)calloc((size_t)(nb > 0 ? nb : 1), sizeof(int32_t));
    for (int i = 0; i < nb; ++i) {
        int b = b_list ? b_list[i] : i;
        int ctx = context_lens[b];
        if (ctx < T || ctx <= 0 || ctx > (long long)max_blocks * block_size) {
            bad[i] = ORACLE_ERR_CONTEXT;
        } else {
            int nblk = (ctx + block_size - 1) / block_size;
            int lo = window > 0 ? ctx - T - window + 1 : 0; /* first visible position */
            if (lo < 0) lo = 0;
            for (int j = lo / block_size; j < nblk; ++j) {
                int blk = block_tables[(size_t)b * max_blocks + j];
                if (blk < 0 || blk >= num_blocks) {
                    bad[i] = ORACLE_ERR_BLOCK_ID;
                    break;
                }
            }
        }
        if (seq_err) seq_err[i] = bad[i];
        if (bad[i]) any = 1;
    }

    long long work = (long long)nb * T * N;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long long w = 0; w < work; ++w) {
        int i = (int)(w / ((long long)T * N));
        int t = (int)((w / N) % T);
        int n = (int)(w % N);
        int b = b_list ? b_list[i] : i;
        double *o = out + (((size_t)i * T + t) * N + n) * H;
        if (bad[i]) {
            for (int h = 0; h < H; ++h) o[h] = 0.0;
            continue;
        }
        int ctx = context_lens[b];
        int last = ctx - T + t; /* last visible position for query token t */
        int first = 0;          /* first visible position */
        if (window > 0 && last - window + 1 > 0) first = last - window + 1;
        int kh = n / G;
        const uint16_t *qv = q + (((size_t)b * T + t) * N + n) * H;
        double *s = (double *)malloc(sizeof(double) * (size_t)(last + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)H);
        for (int h = 0; h < H; ++h) qd[h] = widen(qv[h], dtype);
        /* scores s_j = scale * <q, k_j> */
        /* visible(j): in the band first..last and, with a tree, a prefix
         * position, the token itself or a new token its mask row selects */
        const int first_new = ctx - T;
        const uint64_t mrow = tree_mask ? tree_mask[(size_t)b * T + t] : 0;
#define VISIBLE(j)                                                                   \
    (!tree_mask || (j) < first_new || (j) - first_new == t ||                       \
     (((j) - first_new) < 64 && ((mrow >> ((j) - first_new)) & 1u)))
        double smax = -INFINITY;
        for (int j = first; j <= last; ++j) {
            if (!VISIBLE(j)) continue;
            int blk = block_tables[(size_t)b * max_blocks + j / block_size];
            const size_t off = (((size_t)blk * block_size + j % block_size) * K + kh) * H;
            double acc = 0.0;
            if (kv_kind) { /* one-byte codes times the row's scale */
                const uint8_t *kr = (const uint8_t *)k_cache + off;
                const double sc = k_scale[((size_t)blk * K + kh) * block_size + j % block_size];
                for (int h = 0; h < H; ++h) acc += qd[h] * (code_value(kr[h], kv_kind) * sc);
            } else {
                const uint16_t *kr = (const uint16_t *)k_cache + off;
                for (int h = 0; h < H; ++h) acc += qd[h] * widen(kr[h], dtype);
            }
            s[j] = scale * acc;
            if (s[j] > smax) smax = s[j];
        }
        /* softmax weights p_j = exp(s_j - max) / sum, then out = sum_j p_j v_j */
        double denom = 0.0;
        for (int j = first; j <= last; ++j) {
            if (!VISIBLE(j)) continue;
            s[j] = exp(s[j] - smax);
            denom += s[j];
        }
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int j = first; j <= last; ++j) {
            if (!VISIBLE(j)) continue;
            int blk = block_tables[(size_t)b * max_blocks + j / block_size];
            const size_t off = (((size_t)blk * block_size + j % block_size) * K + kh) * H;
            double p = s[j] / denom;
            if (kv_kind) {
                const uint8_t *vr = (const uint8_t *)v_cache + off;
                const double sc = v_scale[((size_t)blk * K + kh) * block_size + j % block_size];
                for (int h = 0; h < H; ++h) o[h] += p * (code_value(vr[h], kv_kind) * sc);
            } else {
                const uint16_t *vr = (const uint16_t *)v_cache + off;
                for (int h = 0; h < H; ++h) o[h] += p * widen(vr[h], dtype);
            }
        }
        free(qd);
        free(s);
    }
    free(bad);
    return any;
}

/* ---- greedy prefix acceptance ----------------------------------------------
 * [KV-AR], speculative-decoding section: with greedy decoding a drafted token is
 * kept only if the target model would have produced it.  [SONAR-KK]
 * §"Спекулятивті кодтан шығару": the longest accepted prefix is found, and the
 * target's logits at the first mismatch (or after the last draft) give one more
 * token, so n drafts yield between 1 and n+1 tokens.
 *
 * logits [B][T][V] fp32; draft [B][T-1]: draft[b][i] is the token fed at input
 * position i+1, checked against the target's choice g_i = argmax logits[b][i].
 * accepted[b] = a, the largest i <= T-1 with draft[b][j] == g_j for all j < i;
 * next_token[b] = g_a.  If ctx_inout is given, ctx_inout[b] -= (T-1-a): the
 * KV entries of the rejected drafts are dropped.
 *
 * argmax reading: the first index of the largest value wins ties; a NaN counts
 * as larger than every number and the first NaN wins (torch/numpy behaviour). */
static int argmax_row(const float *x, int V) {
    int best = 0;
    for (int v = 1; v < V; ++v) {
        if (isnan(x[best])) break; /* nothing beats the first NaN */
        if (isnan(x[v]) || x[v] > x[best]) best = v;
    }
    return best;
}

void oracle_accept_prefix(int B, int T, int V, const float *logits,
                          const int32_t *draft, int32_t *accepted,
                          int32_t *next_token, int32_t *ctx_inout) {
    for (int b = 0; b < B; ++b) {
        int a = 0;
        while (a < T - 1) {
            int g = argmax_row(logits + ((size_t)b * T + a) * V, V);
            if (draft[(size_t)b * (T - 1) + a] != g) break;
            ++a;
        }
        accepted[b] = a;
        next_token[b] = argmax_row(logits + ((size_t)b * T + a) * V, V);
        if (ctx_inout) ctx_inout[b] -= (T - 1 - a);
    }
}

/* argmax of one row, exposed so tests can pin the tie / NaN reading directly. */
int oracle_argmax(const float *x, int V) { return argmax_row(x, V); }

/* ---- speculative sampling: stochastic acceptance ---------------------------
 * [CS336-RU] §"Спекулятивное сэмплирование": the draft model p proposes tokens,
 * the target model q scores them in one pass, and a modified rejection sampler
 * decides.  Draft token x (drawn from p) is kept with probability
 * min(1, q(x)/p(x)); at the first rejection one token is drawn from the
 * residual max(q - p, 0), renormalised, and the run stops; if every draft is
 * kept, one more token is drawn from the target's next distribution.  The
 * page's two-token example shows the emitted token is an exact sample of q.
 *
 * q [B][T][V] fp32 (q[b][t] is the target's distribution after the prefix and
 * drafts 0..t-1); p [B][T-1][V] fp32 (the draft's distribution that draft[b][t]
 * was drawn from); u [B][T] fp64 uniforms in [0,1): u[b][t], t < T-1, decides
 * draft t, u[b][T-1] draws the final token.
 *
 * Our readings where the page leaves the arithmetic open:
 *   - "kept with probability min(1, q/p)" is the test u * p(x) < q(x) with u,
 *     p(x), q(x) widened to double (the product is then exact; p(x) = 0 keeps x
 *     iff q(x) > 0).  A draft id outside [0, V) is rejected.
 *   - A categorical draw from weights w_v is the inverse CDF on the weights
 *     rounded down to multiples of 2^-40: W_v = floor(w_v * 2^40), S = sum W_v
 *     (exact integers), r = floor(u * S) (double product, clamped to S-1), and
 *     the token is the least v with W_0 + ... + W_v > r.  The rounding moves at
 *     most V * 2^-40 of probability mass.
 *   - The residual weight is max(q(v) - p(v), 0) with the difference rounded
 *     once to fp32.  A residual of total weight zero (q == p up to rounding)
 *     falls back to q itself.
 *   - An entry that is not a probability (NaN, < 0, > 1) is taken as 0, and a
 *     uniform outside [0, 1) as 0; either sets seq_err[b] = ORACLE_ERR_PROBS.
 *     A row with no weight at all gives token 0 and ORACLE_ERR_PROBS.
 *   - ctx_inout[b] -= (T-1-a) as in greedy acceptance; a result below zero
 *     leaves it unchanged and sets ORACLE_ERR_CONTEXT.
 * Requires 1 <= T <= 64. */
#define ORACLE_ERR_PROBS 10 /* an input is not a probability or a uniform in [0,1) */

static float clean_prob(float x, int *bad) {
    if (x >= 0.0f && x <= 1.0f) return x;
    *bad = 1;
    return 0.0f;
}

/* floor(w * 2^40) for w in [0, 1] */
static uint64_t fixed40(float w) { return (uint64_t)((double)w * 1099511627776.0); }

/* weight of token v: residual max(q - p, 0) when p is given, else q */
static uint64_t draw_weight(const float *qrow, const float *prow, int v, int *bad) {
    float w = clean_prob(qrow[v], bad);
    if (prow) {
        float d = w - clean_prob(prow[v], bad);
        w = d > 0.0f ? d : 0.0f;
    }
    return fixed40(w);
}

static int draw_token(const float *qrow, const float *prow, int V, double u, int *bad) {
    uint64_t S = 0;
    for (int v = 0; v < V; ++v) S += draw_weight(qrow, prow, v, bad);
    if (S == 0) return -1;
    uint64_t r = (uint64_t)(u * (double)S);
    if (r > S - 1) r = S - 1;
    uint64_t c = 0;
    for (int v = 0; v < V; ++v) {
        c += draw_weight(qrow, prow, v, bad);
        if (c > r) return v;
    }
    return V - 1; /* not reached: c ends at S > r */
}

void oracle_accept_sampled(int B, int T, int V, const float *q, const float *p,
                           const int32_t *draft, const double *u, int32_t *accepted,
                           int32_t *next_token, int32_t *ctx_inout, int32_t *seq_err) {
    for (int b = 0; b < B; ++b) {
        int bad = 0;
        const double *ub = u + (size_t)b * T;
        double uu[64];
        for (int t = 0; t < T && t < 64; ++t) {
            uu[t] = ub[t];
            if (!(uu[t] >= 0.0 && uu[t] < 1.0)) {
                uu[t] = 0.0;
                bad = 1;
            }
        }
        int a = 0;
        while (a < T - 1) {
            const int x = draft[(size_t)b * (T - 1) + a];
            if (x < 0 || x >= V) break;
            const double qx = clean_prob(q[((size_t)b * T + a) * V + x], &bad);
            const double px = clean_prob(p[((size_t)b * (T - 1) + a) * V + x], &bad);
            if (!(uu[a] * px < qx)) break;
            ++a;
        }
        const float *qrow = q + ((size_t)b * T + a) * V;
        const float *prow = (a < T - 1) ? p + ((size_t)b * (T - 1) + a) * V : NULL;
        int tok = draw_token(qrow, prow, V, uu[T - 1], &bad);
        if (tok < 0 && prow) tok = draw_token(qrow, NULL, V, uu[T - 1], &bad);
        if (tok < 0) {
            tok = 0;
            bad = 1;
        }
        accepted[b] = a;
        next_token[b] = tok;
        seq_err[b] = bad ? ORACLE_ERR_PROBS : 0;
        if (ctx_inout) {
            const int nc = ctx_inout[b] - (T - 1 - a);
            if (nc < 0) {
                if (!seq_err[b]) seq_err[b] = ORACLE_ERR_CONTEXT;
            } else {
                ctx_inout[b] = nc;
            }
        }
    }
}

/* ---- greedy acceptance over a draft tree ------------------------------------
 * [SONAR-KK] §"EAGLE": instead of one chain the draft explores a tree (the top
 * candidates at each node, to a fixed depth); the target scores every node in
 * one pass, each node attending only to its ancestors (a custom attention
 * mask), and the longest candidate sequence is kept for continuation, together
 * with one more token from the target.  §"Спекулятивті кодтан шығару" gives the
 * chain case of the same rule (longest accepted prefix, then one target token).
 *
 * Nodes 0..T-1 are the T new positions of sequence b.  Node 0 is the root (the
 * token that follows the committed prefix; parents[b][0] is -1); node i >= 1
 * has parent parents[b][i] < i and carries the drafted token draft[b][i-1].
 * logits[b][i] is the target's prediction after the root-to-i path, and
 * g_i = argmax logits[b][i] (argmax_row's reading).
 *
 * Readings (the page gives the rule in words only):
 *   - with greedy decoding a node is acceptable iff the target would have
 *     produced every token on its path: for every edge p -> c on the path from
 *     the root to node i, draft[b][c-1] == g_p.  The root always is.
 *   - "the longest" is the acceptable node of greatest depth (depth = edges
 *     from the root); among several of the same depth (only possible when
 *     siblings carry the same token) the lowest node index.
 *   - outputs: accepted[b] = a = depth of that node m; path[b][0..a-1] = the
 *     nodes of the root-to-m path below the root, by depth, and -1 in the
 *     other T-1-a entries; next_token[b] = g_m; ctx_inout[b] -= T-1-a (the
 *     cache keeps the root and the a accepted tokens once they are compacted,
 *     see oracle_kv_compact).
 *   - a malformed tree (parents[b][0] != -1, or parents[b][i] outside [0, i))
 *     sets seq_err[b] = ORACLE_ERR_TREE; a node whose path to the root meets a
 *     bad entry is not acceptable; everything else is decided as above.
 *   - a context length that would drop below zero is left unchanged
 *     (ORACLE_ERR_CONTEXT, unless the tree error was set first).
 * With parents[b][i] = i-1 for every i this is exactly the chain rule of
 * oracle_accept_prefix. */
#define ORACLE_ERR_TREE 11 /* a draft tree's parent entry is out of range */

/* Nodes of the path from the root to node i, root excluded, deepest first;
 * returns their count (the depth of i), or -1 if the walk meets a parent entry
 * outside [0, node). */
static int tree_path_up(const int32_t *par, int i, int *nodes) {
    int d = 0;
    while (i != 0) {
        const int p = par[i];
        if (p < 0 || p >= i) return -1;
        nodes[d++] = i;
        i = p;
    }
    return d;
}

void oracle_accept_tree(int B, int T, int V, const float *logits, const int32_t *draft,
                        const int32_t *parents, int32_t *accepted, int32_t *next_token,
                        int32_t *path, int32_t *ctx_inout, int32_t *seq_err) {
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parents + (size_t)b * T;
        const int32_t *dr = draft + (size_t)b * (T > 1 ? T - 1 : 0);
        const float *lg = logits + (size_t)b * T * V;
        int err = par[0] == -1 ? 0 : ORACLE_ERR_TREE;
        for (int i = 1; i < T; ++i)
            if (par[i] < 0 || par[i] >= i) err = ORACLE_ERR_TREE;
        int best = 0, best_depth = 0;
        int up[64];
        for (int i = 1; i < T; ++i) {
            const int d = tree_path_up(par, i, up);
            if (d < 0) continue;
            int ok = 1;
            for (int e = 0; e < d && ok; ++e) {
                const int c = up[e], p = par[c];
                if (dr[c - 1] != argmax_row(lg + (size_t)p * V, V)) ok = 0;
            }
            if (ok && d > best_depth) { /* strict: the lower index keeps a tie */
                best = i;
                best_depth = d;
            }
        }
        const int a = tree_path_up(par, best, up);
        for (int j = 0; j < T - 1; ++j) path[(size_t)b * (T - 1) + j] = j < a ? up[a - 1 - j] : -1;
        accepted[b] = a;
        next_token[b] = argmax_row(lg + (size_t)best * V, V);
        if (ctx_inout) {
            const int nc = ctx_inout[b] - (T - 1 - a);
            if (nc < 0) {
                if (!err) err = ORACLE_ERR_CONTEXT;
            } else {
                ctx_inout[b] = nc;
            }
        }
        seq_err[b] = err;
    }
}

/* ---- cache compaction after tree acceptance ---------------------------------
 * [SONAR-KK] §"EAGLE" keeps the accepted branch of the tree and continues from
 * it; [CS336-RU] §"PagedAttention" stores a sequence's tokens in its blocks in
 * order.  The T tree nodes were appended at positions base .. base+T-1 (node i
 * at base+i); after acceptance the sequence must read as the prefix, the root
 * and the a accepted tokens in order, so position base+j (j = 1..a) takes the
 * cached K and V rows (every KV head) of node path[b][j-1].
 * context_lens[b] is the length AFTER acceptance (oracle_accept_tree's
 * ctx_inout): base = context_lens[b] - 1 - a.
 * Rows are moved as raw bytes (esize bytes per element: 2 for a cache in q's
 * dtype, 1 for one-byte codes); with k_scale / v_scale ([NB][K][bs] fp32, the
 * one-byte caches' row scales) the scales move with their rows.
 * Checks (the sequence is left untouched and seq_err[b] set): a outside
 * [0, T-1] or a path that is not strictly increasing within [1, T)
 * (ORACLE_ERR_TREE); base < 0, or base+T-1 beyond the bs*max_blocks rows
 * the table addresses (ORACLE_ERR_CONTEXT); a block holding one of the
 * positions base .. base+T-1 whose id is outside [0, NB) (ORACLE_ERR_BLOCK_ID).
 * Every source row is read before any destination row is written. */
int oracle_kv_compact(int B, int T, int K, int H, int bs, int NB, int max_blocks, int esize,
                      uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale,
                      const int32_t *block_tables, const int32_t *context_lens,
                      const int32_t *path, const int32_t *accepted, int32_t *seq_err) {
    const size_t row = (size_t)H * esize;
    uint8_t *tmp = (uint8_t *)malloc((size_t)(T > 1 ? T : 1) * K * row * 2 + 1);
    float *tsc = (float *)malloc((size_t)(T > 1 ? T : 1) * K * 2 * sizeof(float) + 4);
    if (!tmp || !tsc) {
        free(tmp);
        free(tsc);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        const int a = accepted[b];
        const int32_t *pt = path + (size_t)b * (T > 1 ? T - 1 : 0);
        const int32_t *tab = block_tables + (size_t)b * max_blocks;
        seq_err[b] = 0;
        int ok = a >= 0 && a <= T - 1;
        for (int j = 0; ok && j < a; ++j)
            if (pt[j] < 1 || pt[j] >= T || (j > 0 && pt[j] <= pt[j - 1])) ok = 0;
        if (!ok) {
            seq_err[b] = ORACLE_ERR_TREE;
            continue;
        }
        const long long base = (long long)context_lens[b] - 1 - a;
        if (base < 0 || base + T > (long long)bs * max_blocks) {
            seq_err[b] = ORACLE_ERR_CONTEXT;
            continue;
        }
        for (long long pos = base; pos < base + T; ++pos) {
            const int id = tab[pos / bs];
            if (id < 0 || id >= NB) ok = 0;
        }
        if (!ok) {
            seq_err[b] = ORACLE_ERR_BLOCK_ID;
            continue;
        }
        /* gather every source row first ... */
        for (int j = 0; j < a; ++j) {
            const long long pos = base + pt[j];
            const size_t blk = (size_t)tab[pos / bs], r = (size_t)(pos % bs);
            for (int k = 0; k < K; ++k) {
                const size_t src = ((blk * bs + r) * K + k) * row;
                memcpy(tmp + (((size_t)j * K + k) * 2 + 0) * row, k_cache + src, row);
                memcpy(tmp + (((size_t)j * K + k) * 2 + 1) * row, v_cache + src, row);
                if (k_scale) {
                    tsc[((size_t)j * K + k) * 2 + 0] = k_scale[(blk * K + k) * bs + r];
                    tsc[((size_t)j * K + k) * 2 + 1] = v_scale[(blk * K + k) * bs + r];
                }
            }
        }
        /* ... then write position base+1+j for the (j+1)-th accepted node */
        for (int j = 0; j < a; ++j) {
            const long long pos = base + 1 + j;
            const size_t blk = (size_t)tab[pos / bs], r = (size_t)(pos % bs);
            for (int k = 0; k < K; ++k) {
                const size_t dst = ((blk * bs + r) * K + k) * row;
                memcpy(k_cache + dst, tmp + (((size_t)j * K + k) * 2 + 0) * row, row);
                memcpy(v_cache + dst, tmp + (((size_t)j * K + k) * 2 + 1) * row, row);
                if (k_scale) {
                    k_scale[(blk * K + k) * bs + r] = tsc[((size_t)j * K + k) * 2 + 0];
                    v_scale[(blk * K + k) * bs + r] = tsc[((size_t)j * K + k) * 2 + 1];
                }
            }
        }
    }
    free(tmp);
    free(tsc);
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
