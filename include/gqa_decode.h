/*
 * gqa_decode.h -- C ABI of the paged grouped-query decode-attention library
 * (hand-written CUDA for sm_103a / GB300).
 *
 * Operations on a paged KV cache, all asynchronous on the caller's stream:
 *   gqa_kv_append        write the T newest tokens' keys and values into the cache
 *   gqa_decode_attention attention of one new query token per sequence (T == 1)
 *   gqa_verify_attention the same for T >= 1 new tokens, causal among them
 *   gqa_tree_verify_attention  the same with a tree mask among the new tokens
 *   gqa_accept_prefix    greedy longest-prefix acceptance of draft tokens
 *   gqa_kv_append_quant  the append into a one-byte (int8 / e4m3) cache, and
 *   gqa_decode_attention_quant / gqa_verify_attention_quant  attention over it
 *   gqa_append_decode_attention_quant / gqa_append_verify_attention_quant  both
 *                        in one call; gqa_tree_verify_attention_quant
 *   gqa_accept_sampled   stochastic acceptance of draft tokens (speculative
 *                        sampling: modified rejection sampling)
 *   gqa_accept_tree      greedy acceptance over a draft tree, and
 *   gqa_kv_compact       the kept branch's cached rows moved behind its root
 *
 * Sources (web pages, cited by title and section):
 *   "CS336, лекции 10 и 12: инференс и оценка моделей" (CS336 lectures 10/12,
 *     Russian translation): §"Напоминание: трансформер" (notation B,T,N,K,G,H),
 *     §"Арифметическая интенсивность инференса" (KV cache; attention of the new
 *     token over the cache; decode is memory-bound), §"Уменьшаем KV-кэш" (GQA),
 *     §"Спекулятивное сэмплирование" (verify several drafted tokens in one pass),
 *     §"PagedAttention" (fixed-size blocks + per-sequence block table; fused
 *     block-read + attention kernel; FlashDecoding).
 *   "جعل inference رخيصًا: KV cache وbatching والتكميم" (KV cache, batching and
 *     quantization): the KV-cache section (cache == recompute; bytes per token)
 *     and the speculative-decoding section (greedy acceptance).
 *   "Болжау арқылы Sonar модельдерін жылдамдату" (Accelerating Sonar through
 *     speculation): §"Спекулятивті кодтан шығару" (longest accepted prefix plus
 *     one target token), §"Спекулятивті кодтан шығару арқылы инференс"
 *     (appending accepted tokens on the GPU, avoiding a GPU->CPU sync) and
 *     §"EAGLE" (draft trees verified under a custom attention mask; the
 *     longest agreeing branch kept).
 *
 * Conventions for every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except the
 *     `const gqa_shape*`, which is a host pointer read during the call only.
 *     The library allocates no device memory and keeps no pointer after return.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All work is
 *     enqueued on it; the call returns without synchronising.
 *   - The return value reports host-side validation only (arguments, shapes,
 *     alignment, launch errors).  Problems found in device data (a context
 *     length out of range, a bad block id) are reported through the optional
 *     device int32 `dev_status`: the first nonzero gqa_status code written
 *     wins, later ones are dropped; the library never clears it.  The affected
 *     sequence's outputs are written as zeros (attention) or left untouched
 *     (append).  No kernel ever traps or waits without a time limit.
 *   - Layouts are dense row-major with the last dimension contiguous:
 *       q, out        [B][T][N][H]      (dtype of the shape)
 *       k_new, v_new  [B][T][K][H]
 *       k/v cache     [num_blocks][block_size][K][H]
 *       block_tables  int32 [B][max_blocks_per_seq]: logical block i of
 *                     sequence b -> physical block id
 *       context_lens  int32 [B]: tokens held for sequence b INCLUDING the T new
 *                     ones; new token t sits at position context_lens[b]-T+t.
 *     q, out, k/v caches, k_new, v_new must be 16-byte aligned.
 *   - Query head n reads KV head n / G, G = N / K (contiguous groups).
 */
#ifndef GQA_DECODE_H
#define GQA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GQA_OK = 0,
    GQA_ERR_NULL = 1,      /* a required pointer is NULL */
    GQA_ERR_SHAPE = 2,     /* unsupported or inconsistent sizes (see each call) */
    GQA_ERR_DTYPE = 3,     /* dtype not GQA_F16 / GQA_BF16 */
    GQA_ERR_ALIGN = 4,     /* a tensor pointer is not 16-byte aligned */
    GQA_ERR_WORKSPACE = 5, /* workspace NULL or smaller than the size query */
    GQA_ERR_CUDA = 6,      /* a CUDA runtime / driver call failed */
    GQA_ERR_CONTEXT = 7,   /* device: context_lens[b] < T, < 1 or > capacity */
    GQA_ERR_BLOCK_ID = 8,  /* device: a block-table entry in use not in [0,num_blocks) */
    GQA_ERR_TIMEOUT = 9,   /* device: a bounded wait inside a kernel gave up */
    GQA_ERR_PROBS = 10,    /* device: an entry read is not a probability in [0,1], a
                              uniform is not in [0,1), or a row has no weight */
    GQA_ERR_TREE = 11      /* device: a draft tree's parent entry, or an accepted
                              branch passed to gqa_kv_compact, is out of range */
} gqa_status;

typedef enum { GQA_F16 = 0, GQA_BF16 = 1 } gqa_dtype;

/* Element type of the KV cache: the dtype of q (2 bytes), or one-byte codes
 * with an fp32 scale per cached row (see gqa_kv_append_quant). */
typedef enum { GQA_KV_SAME = 0, GQA_KV_INT8 = 1, GQA_KV_E4M3 = 2 } gqa_kv_dtype;

/* Problem sizes, in the pages' notation (CS336 lecture 10, §"Напоминание:
 * трансформер"): B sequences, T new query tokens per sequence, N query heads,
 * K key/value heads (G = N/K), head size H. */
typedef struct {
    int B;
    int T;
    int N;
    int K;
    int H;                  /* 64 or 128 */
    int block_size;         /* tokens per cache block; must be 16 */
    int num_blocks;         /* physical blocks in each cache tensor */
    int max_blocks_per_seq; /* columns of block_tables */
    gqa_dtype dtype;        /* element type of q, out, caches, k_new, v_new */
    float scale;            /* score scale; <= 0 selects 1/sqrt(H) */
    unsigned int flags;     /* GQA_FLAG_* bits, 0 for plain stream order */
    int window;             /* local attention: > 0 limits each query to the last
                               `window` positions up to itself; 0 = all */
    int kv_dtype;           /* gqa_kv_dtype of the caches; GQA_KV_SAME except for
                               the _quant calls */
} gqa_shape;

/* Local (sliding-window) attention, for the attention calls: CS336 lecture 10
 * §"Уменьшаем KV-кэш" (attend only to a recent stretch of context; the cache no
 * longer grows with the sequence; hybrid schedules interleave local and global
 * layers) and "Stanford CS336 Day 13 - Inference" §"Local Attention" (only the
 * last k tokens are attended; older tokens may be dropped from the cache).
 * With window = W > 0, new token t (position i = context_lens[b] - T + t) sees
 * positions i-W+1 .. i only.  Blocks wholly below position
 * context_lens[b] - T - W + 1 are never read, so their table entries may hold
 * anything (freed blocks); only the blocks of the window are checked. */

/* Launch with programmatic dependent launch: the kernel may be scheduled while
 * the previous kernel on the stream is still finishing, and waits for it (with
 * griddepcontrol.wait) before its first access to device memory, so the
 * results are exactly those of plain stream order; only launch latency and
 * set-up are overlapped. */
#define GQA_FLAG_PDL 1u
/* Attention only, implies GQA_FLAG_PDL.  The caller promises that the work
 * still running from earlier on the stream writes neither block_tables,
 * context_lens nor any cache position below context_lens[b] - T.  The kernel
 * then starts streaming those cache blocks before the previous kernel has
 * finished; q, the T newest positions, the workspace and `out` are still
 * touched only after it has. */
#define GQA_FLAG_EARLY_KV 2u
/* Attention only: which kernel computes the call.  By default the library
 * picks by shape: the tensor-memory kernel (tcgen05.mma, accumulators in
 * tensor memory, 128 query rows of one KV head per tile) where a KV head has
 * many query rows (T * N / K >= 32, a cache in q's dtype, with or without a
 * window); for small calls -- a cache in q's dtype,
 * T * N / K <= 8, no window, no tree mask, B * K <= 304 and max_blocks_per_seq
 * <= 64 (H = 64) or 48 (H = 128) -- the direct warp-level kernel (one CTA per
 * (sequence, KV head), every warp loading its own cache blocks, no split of a
 * context over CTAs); the persistent warp-level mma.sync kernel (contexts split
 * evenly over all SMs, pieces merged through the workspace) otherwise.
 * GQA_FLAG_WARP_MMA forces the persistent warp-level kernel;
 * GQA_FLAG_TENSOR_MEMORY forces the tensor-memory one, which serves a cache
 * in q's dtype; GQA_FLAG_DIRECT forces the direct
 * one, which serves a cache in q's dtype with T * N / K <= 8, no window and no
 * tree mask, at any context length (GQA_ERR_SHAPE where the forced kernel
 * cannot serve the call, or with more than one of the flags).  All compute the
 * same function; results differ only by rounding order.  The workspace size
 * does not depend on the kernel. */
#define GQA_FLAG_WARP_MMA 4u
#define GQA_FLAG_TENSOR_MEMORY 8u
#define GQA_FLAG_DIRECT 16u

/* Which attention kernel serves a call with this shape and these flags (host
 * logic only; no device work), for a call without a tree mask (a tree mask
 * rules the direct kernel out): GQA_ENGINE_WARP_MMA (persistent warp-level),
 * GQA_ENGINE_TENSOR_MEMORY, GQA_ENGINE_DIRECT, or 0 if the shape fails the
 * common checks or a forced kernel cannot serve it.  The call itself may still
 * reject the shape for a reason of its own (H = 64 with a one-byte cache, a
 * tree mask with T > 64). */
#define GQA_ENGINE_WARP_MMA 1
#define GQA_ENGINE_TENSOR_MEMORY 2
#define GQA_ENGINE_DIRECT 3
int gqa_attention_engine(const gqa_shape *shape);

/* Library version (major*10000 + minor*100 + patch). */
int gqa_version(void);

/* Static description of a status code (never NULL). */
const char *gqa_status_string(int status);

/* KV append.  KV-cache section of "جعل inference رخيصًا: KV cache وbatching
 * والتكميم" (each new token's key/value vectors are stored once) with the block
 * addressing of CS336 lecture 10 §"PagedAttention": for b < B, t < T, position
 * pos = context_lens[b] - T + t goes to block block_tables[b][pos / 16], row
 * pos % 16.  k_new[b][t] (K*H elements) is copied there bit for bit; same for
 * v_new.  Requires T >= 1, K >= 1, H in {64,128}.  Device errors: a sequence
 * with context_lens[b] < T or > 16*max_blocks_per_seq is skipped
 * (GQA_ERR_CONTEXT); a token whose block id is out of range is skipped
 * (GQA_ERR_BLOCK_ID). */
gqa_status gqa_kv_append(const gqa_shape *shape, const void *k_new, const void *v_new,
                         void *k_cache, void *v_cache, const int32_t *block_tables,
                         const int32_t *context_lens, int32_t *dev_status,
                         void *stream);

/* Bytes of device workspace gqa_decode_attention / gqa_verify_attention need
 * for this shape on the CURRENT device: a fixed 256 KiB region of int32
 * publication flags (one per thread block and warp of query rows) followed by
 * the split-context partial results of whichever kernel may serve the shape
 * (see GQA_FLAG_TENSOR_MEMORY).  Returns 0 if the shape is invalid.
 * The workspace must be zero-filled before its first use (for example with
 * gqa_workspace_clear); every call whose kernels finish without
 * GQA_ERR_TIMEOUT leaves the flag region zero-filled again (the
 * partial-result region is scratch and never needs clearing), so one buffer
 * can be reused by later calls of any shape that fits.  Calls that share a
 * workspace must not overlap on the GPU (use one stream, or one workspace per
 * stream).  After GQA_ERR_TIMEOUT, clear the workspace again before reusing
 * it. */
size_t gqa_attention_workspace_size(const gqa_shape *shape);

/* Zero-fill `bytes` of workspace on `stream` (a cudaMemsetAsync). */
gqa_status gqa_workspace_clear(void *workspace, size_t bytes, void *stream);

/* Decode attention, T == 1.  CS336 lecture 10 §"Арифметическая интенсивность
 * инференса" (Y = softmax(Q K^T) V of the new token over the cached keys and
 * values) with GQA from §"Уменьшаем KV-кэш" and paged reads from
 * §"PagedAttention".  For each b, query head n (KV head k = n / G):
 *   s_j = scale * <q[b][0][n], K_b[j][k]>,   j = 0 .. context_lens[b]-1
 *   out[b][0][n] = sum_j softmax(s)_j * V_b[j][k]
 * where K_b[j] is row j % 16 of block block_tables[b][j / 16].  fp32
 * accumulation; `out` gets q's dtype (round to nearest even).  The context is
 * split across thread blocks and the pieces merged with their log-sum-exp
 * weights (FlashDecoding, named in §"PagedAttention"); the result equals the
 * unsplit softmax up to rounding.  Requires: T == 1, N % K == 0, H in {64,128},
 * block_size == 16, N/K <= 8192, a workspace of at least
 * gqa_attention_workspace_size(shape) bytes (zeroed, see above).  Device
 * errors: a sequence whose context length is < 1, < T or above
 * 16*max_blocks_per_seq (GQA_ERR_CONTEXT) or whose table holds a block id
 * outside [0, num_blocks) among its first ceil(len/16) entries
 * (GQA_ERR_BLOCK_ID) gets an all-zero output. */
gqa_status gqa_decode_attention(const gqa_shape *shape, const void *q,
                                const void *k_cache, const void *v_cache,
                                const int32_t *block_tables,
                                const int32_t *context_lens, void *out,
                                void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, void *stream);

/* Decode attention that allocates nothing (no counterpart on the pages: it is
 * a convenience of this library).  For callers that cannot call cudaMalloc --
 * a host program that keeps all device memory in its own pool, a decode loop
 * that must not let cudaMalloc / cudaFree synchronise the device, a plain C
 * caller without an allocator -- this computes exactly what
 * gqa_decode_attention computes, with the same requirements, but takes no
 * workspace: its scratch is a static 8 MiB device array inside the library,
 * held on every GPU that loads the library until the process exits.
 *  - Shapes whose scratch exceeds 8 MiB are rejected with GQA_ERR_WORKSPACE.
 *    The scratch is what the kernel that serves the call needs: the
 *    warp-level kernel's workspace, or the tensor-memory kernel's where the
 *    shape picks that one (T * N / K >= 32).  The latter is 256 KiB
 *    plus 132 KiB of split-context partials per SM, so it exceeds 8 MiB, and
 *    such shapes are rejected, on every GPU with more than 60 SMs (GB300 has
 *    152).  gqa_attention_workspace_size may report more: it also covers a
 *    kernel forced by a flag.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address; make that first call before any stream capture.
 *  - Each call first clears, on `stream`, the part of the array that must
 *    start at zero (one cudaMemsetAsync; nothing is allocated or freed).
 *    That memset sits between the previous kernel on the stream and the
 *    attention launch, so GQA_FLAG_PDL / GQA_FLAG_EARLY_KV give no launch
 *    overlap through this entry point (the results are the same).
 *  - All calls share the one array: calls whose work overlaps on the GPU (on
 *    different streams or from different host threads) race on it. */
gqa_status gqa_decode_attention_noalloc(const gqa_shape *shape, const void *q,
                                        const void *k_cache, const void *v_cache,
                                        const int32_t *block_tables,
                                        const int32_t *context_lens, void *out,
                                        int32_t *dev_status, void *stream);

/* Verify attention, T >= 1 new tokens per sequence (speculative verification:
 * CS336 lecture 10 §"Спекулятивное сэмплирование" -- the target model scores
 * several drafted tokens in one pass).  As gqa_decode_attention, except that
 * new token t (t < T) sees cached positions j <= context_lens[b] - T + t: the
 * whole prefix plus the new tokens up to itself.  Requires T * (N/K) <= 8192.
 * The T*(N/K) query rows of a KV head are processed in chunks of at most 48
 * rows (one per consumer warp and 8 rows); beyond 48 rows every chunk reads
 * the KV head's blocks again, from L2 when they are still there. */
gqa_status gqa_verify_attention(const gqa_shape *shape, const void *q,
                                const void *k_cache, const void *v_cache,
                                const int32_t *block_tables,
                                const int32_t *context_lens, void *out,
                                void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, void *stream);

/* KV append fused into attention: the same results (cache bytes and
 * attention output) as gqa_kv_append followed by gqa_decode_attention /
 * gqa_verify_attention on the same stream, in one launch.  The kernel takes the
 * T newest positions' keys and values from k_new / v_new [B][T][K][H] (16-byte
 * aligned) instead of the cache and writes them into the caches, as the
 * pages' speculative-decoding blog does on the GPU ("Болжау арқылы Sonar
 * модельдерін жылдамдату" §"Спекулятивті кодтан шығару арқылы инференс").
 * With GQA_FLAG_EARLY_KV the kernel can then stream every older cache block
 * before the previous kernel on the stream finishes (q, k_new, v_new, the
 * workspace and out stay ordered after it).  Requirements and device errors as
 * for the unfused calls; a sequence whose blocks include an invalid id gets a
 * zero output and its new tokens may not be written. */
gqa_status gqa_append_decode_attention(const gqa_shape *shape, const void *q,
                                       const void *k_new, const void *v_new, void *k_cache,
                                       void *v_cache, const int32_t *block_tables,
                                       const int32_t *context_lens, void *out, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status,
                                       void *stream);
gqa_status gqa_append_verify_attention(const gqa_shape *shape, const void *q,
                                       const void *k_new, const void *v_new, void *k_cache,
                                       void *v_cache, const int32_t *block_tables,
                                       const int32_t *context_lens, void *out, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status,
                                       void *stream);

/* Tree verification: verify_attention with a custom mask among the T new
 * tokens.  "Болжау арқылы Sonar модельдерін жылдамдату" §"EAGLE": drafts form a
 * tree (Top-K candidates at each node) and the target model verifies the
 * tree's sequences with a custom attention mask (which, applied to the whole
 * sequence, the page reports slowing attention by up to 50 %).  Here the mask
 * only concerns the new tokens:
 *   tree_mask  uint64 [B][T], 8-byte aligned: new token t sees the whole
 *              prefix (positions < context_lens[b] - T), itself, and new token
 *              j < t iff bit j of tree_mask[b][t] is set -- for a tree laid out
 *              in topological order, its ancestors.  Bits j >= t are ignored;
 *              the chain mask (bits 0..t-1 set) gives gqa_verify_attention.
 * Requirements, layouts, workspace and device errors as gqa_verify_attention;
 * shape->window must be 0 and T <= 64.  The _append_ form fuses gqa_kv_append as
 * gqa_append_verify_attention does. */
gqa_status gqa_tree_verify_attention(const gqa_shape *shape, const void *q,
                                     const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables,
                                     const int32_t *context_lens, const uint64_t *tree_mask,
                                     void *out, void *workspace, size_t workspace_bytes,
                                     int32_t *dev_status, void *stream);
gqa_status gqa_append_tree_verify_attention(const gqa_shape *shape, const void *q,
                                            const void *k_new, const void *v_new,
                                            void *k_cache, void *v_cache,
                                            const int32_t *block_tables,
                                            const int32_t *context_lens,
                                            const uint64_t *tree_mask, void *out,
                                            void *workspace, size_t workspace_bytes,
                                            int32_t *dev_status, void *stream);

/* One-byte KV cache.  Quantization section of "جعل inference رخيصًا: KV cache
 * وbatching والتكميم" (symmetric absolute-maximum quantization: scale =
 * max|x| / qmax, codes round(x / scale) clamped; decode being bandwidth bound,
 * fewer bytes per element make each step faster) and CS336 lecture 10
 * §"Квантование" (fp8 e4m3 and int8 as one-byte formats).
 *   caches    int8 or e4m3 codes [num_blocks][16][K][H] (shape->kv_dtype)
 *   k_scale, v_scale  fp32 [num_blocks][K][16]: the scale of each cached row
 * Every appended key / value row of one KV head (H elements) is quantized on
 * its own: scale = max|x| / qmax (qmax = 127 for int8, 448 -- the largest
 * finite e4m3 value -- for e4m3) and code = x / scale rounded to nearest even
 * (int8: clamped to [-128, 127]; e4m3: saturating), both divisions in IEEE
 * fp32.  A row of zeros gets scale 0 and codes 0.  Attention reads
 * code * scale.  The append needs k_new / v_new in the dtype of the shape,
 * H in {64, 128}; other requirements and device errors as gqa_kv_append. */
gqa_status gqa_kv_append_quant(const gqa_shape *shape, const void *k_new, const void *v_new,
                               void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                               const int32_t *block_tables, const int32_t *context_lens,
                               int32_t *dev_status, void *stream);

/* Decode / verify attention over a one-byte cache written by
 * gqa_kv_append_quant: as gqa_decode_attention / gqa_verify_attention, with
 * K_b[j] = code * k_scale[block][k][row] (likewise V).  shape->kv_dtype is
 * GQA_KV_INT8 or GQA_KV_E4M3; requires H == 128 (GQA_ERR_SHAPE otherwise);
 * k_scale / v_scale 16-byte aligned.  shape->window works as for the other
 * attention calls (rows and scales below every new token's window are never
 * used), and more than 48 query rows per KV head run in row chunks, each
 * reading the KV head's blocks once.  Served by the warp-level kernel
 * (GQA_FLAG_TENSOR_MEMORY: GQA_ERR_SHAPE).  The products run on f16 tensor-core operands: q is
 * rounded to f16 (exact for |q| in f16's normal range), the codes convert
 * exactly; fp32 accumulation. */
gqa_status gqa_decode_attention_quant(const gqa_shape *shape, const void *q,
                                      const void *k_cache, const void *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_tables,
                                      const int32_t *context_lens, void *out, void *workspace,
                                      size_t workspace_bytes, int32_t *dev_status,
                                      void *stream);
gqa_status gqa_verify_attention_quant(const gqa_shape *shape, const void *q,
                                      const void *k_cache, const void *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_tables,
                                      const int32_t *context_lens, void *out, void *workspace,
                                      size_t workspace_bytes, int32_t *dev_status,
                                      void *stream);

/* Tree verification over a one-byte cache: gqa_tree_verify_attention with the
 * caches and row scales of gqa_verify_attention_quant (tree_mask as there:
 * uint64 [B][T], T <= 64; no window). */
gqa_status gqa_tree_verify_attention_quant(const gqa_shape *shape, const void *q,
                                          const void *k_cache, const void *v_cache,
                                          const float *k_scale, const float *v_scale,
                                          const int32_t *block_tables,
                                          const int32_t *context_lens,
                                          const uint64_t *tree_mask, void *out, void *workspace,
                                          size_t workspace_bytes, int32_t *dev_status,
                                          void *stream);

/* The append and the one-byte attention in one call: gqa_kv_append_quant
 * followed by gqa_decode_attention_quant / gqa_verify_attention_quant on the
 * same stream, as two launches (the attention launch chained to the append by
 * programmatic dependent launch when the flags ask for it).  k_new / v_new
 * [B][T][K][H] in the dtype of the shape.  (A one-launch form, with the new
 * rows quantized inside the attention kernel, measured slower than the two
 * launches on a 256-sequence int8 batch: that kernel is bound by its producer
 * warp's issue rate and its consumer warps' registers.)  Requirements, flags
 * and device errors as the two calls. */
gqa_status gqa_append_decode_attention_quant(const gqa_shape *shape, const void *q,
                                             const void *k_new, const void *v_new,
                                             void *k_cache, void *v_cache, float *k_scale,
                                             float *v_scale, const int32_t *block_tables,
                                             const int32_t *context_lens, void *out,
                                             void *workspace, size_t workspace_bytes,
                                             int32_t *dev_status, void *stream);
gqa_status gqa_append_verify_attention_quant(const gqa_shape *shape, const void *q,
                                             const void *k_new, const void *v_new,
                                             void *k_cache, void *v_cache, float *k_scale,
                                             float *v_scale, const int32_t *block_tables,
                                             const int32_t *context_lens, void *out,
                                             void *workspace, size_t workspace_bytes,
                                             int32_t *dev_status, void *stream);

/* Greedy prefix acceptance.  Speculative-decoding section of "جعل inference
 * رخيصًا" (a drafted token is kept only if the target would produce it) and
 * "Болжау арқылы Sonar модельдерін жылдамдату" §"Спекулятивті кодтан шығару"
 * (longest accepted prefix, then one token from the target's logits).
 *   target_logits fp32 [B][T][V]; draft_ids int32 [B][T-1]
 *   g_t = argmax_v target_logits[b][t][v]   (first index wins ties; NaN is
 *         larger than any number and the first NaN wins)
 *   accepted[b]   = largest a <= T-1 with draft_ids[b][j] == g_j for all j < a
 *   next_token[b] = g_a
 *   context_lens_inout[b] -= T-1-a  (if not NULL: drops the KV entries of the
 *                                    rejected drafts, on the device)
 * Requires B >= 0, 1 <= T <= 64, V >= 1.  target_logits must be 16-byte
 * aligned.  Device errors: a context length that would drop below zero is
 * left unchanged (GQA_ERR_CONTEXT).
 * workspace: device memory of at least gqa_accept_workspace_size(B, T) bytes,
 * 16-byte aligned and zero-filled before its first use; every call leaves it
 * zero-filled again, so one buffer serves later calls of any size that fits.
 * With it, each sequence's columns are split over many thread blocks (about
 * four per SM over the batch) that store their per-row maxima in the
 * workspace; the block that finishes last (an atomic ticket) combines them
 * and walks the drafts.  No block waits for another.  Calls that share a workspace must not
 * overlap on the GPU.  workspace == NULL (workspace_bytes ignored) runs one
 * thread-block cluster of up to 8 blocks per sequence instead (B <= 65535),
 * which needs no scratch but fills the GPU only for large batches.  Both give
 * the same results. */
size_t gqa_accept_workspace_size(int B, int T);
gqa_status gqa_accept_prefix(int B, int T, int V, const float *target_logits,
                             const int32_t *draft_ids, int32_t *accepted,
                             int32_t *next_token, int32_t *context_lens_inout,
                             void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, void *stream);

/* Greedy acceptance over a draft tree.  "Болжау арқылы Sonar модельдерін
 * жылдамдату" §"EAGLE": the draft explores a tree of candidates, the target
 * scores every node in one pass (gqa_tree_verify_attention), and the longest
 * branch the target agrees with is kept, plus one token from the target.
 * Nodes 0..T-1 are the T new positions of a sequence; node 0 is the root (the
 * token after the committed prefix).
 *   target_logits fp32 [B][T][V]   row i: the target's prediction after the
 *                                  root-to-node-i branch; g_i = its argmax
 *                                  (ties and NaN as in gqa_accept_prefix)
 *   draft_ids     int32 [B][T-1]   draft_ids[b][i-1]: node i's token
 *   parents       int32 [B][T]     parents[b][0] = -1; parents[b][i] < i
 *   Node i >= 1 is kept iff its parent is kept and draft_ids[b][i-1] equals
 *   g of its parent (the root is always kept).  The kept node m of greatest
 *   depth ends the accepted branch; among nodes of equal depth (siblings with
 *   the same token) the lowest index wins.
 *   accepted[b]   = a = depth of m (edges from the root)
 *   path[b][0..a-1] = the branch's nodes below the root, by depth; -1 in the
 *                     other T-1-a entries
 *   next_token[b] = g_m
 *   context_lens_inout[b] -= T-1-a  (if not NULL); then gqa_kv_compact moves
 *                     the branch's cached rows behind the root
 * A chain (parents[b][i] = i-1) gives exactly gqa_accept_prefix's results.
 * Requirements, workspace and the two kernels as gqa_accept_prefix;
 * draft_ids and path may be NULL when T == 1.  Device errors: a parent entry
 * outside [0, i) (or a root entry other than -1) is reported (GQA_ERR_TREE)
 * and that node and its descendants are never kept; a context length that
 * would drop below zero is left unchanged (GQA_ERR_CONTEXT). */
gqa_status gqa_accept_tree(int B, int T, int V, const float *target_logits,
                           const int32_t *draft_ids, const int32_t *parents,
                           int32_t *accepted, int32_t *next_token, int32_t *path,
                           int32_t *context_lens_inout, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status, void *stream);

/* Cache compaction after tree acceptance.  §"EAGLE" (same page): decoding
 * continues from the kept branch, and CS336 lecture 10 §"PagedAttention"
 * stores a sequence's tokens in its blocks in order.  The T tree nodes were
 * appended at positions base .. base+T-1 (node i at base+i, as
 * gqa_append_verify_attention writes them); afterwards position base+j
 * (j = 1..a) holds the K and V rows, every KV head, of node path[b][j-1],
 * with base = context_lens[b] - 1 - a.
 *   shape          T = tree nodes (<= 64), K, H, block_size, num_blocks,
 *                  max_blocks_per_seq, kv_dtype (N, dtype as for the cache's
 *                  attention calls; q-side fields are not used)
 *   context_lens   int32 [B], the lengths AFTER acceptance (gqa_accept_tree's
 *                  context_lens_inout)
 *   path, accepted gqa_accept_tree's outputs ([B][T-1], [B])
 *   k_scale, v_scale  fp32 [num_blocks][K][block_size] row scales of a
 *                  one-byte cache (kv_dtype GQA_KV_INT8 / GQA_KV_E4M3; moved
 *                  with their rows); NULL for a cache in q's dtype
 * Rows move as raw bytes: the result is bit for bit the branch's rows.
 * Caches 16-byte aligned.  The blocks holding positions base .. base+T-1
 * must not be shared with another sequence.  Device errors (the sequence is
 * left untouched): a outside [0, T-1] or a branch that is not strictly
 * increasing within [1, T) (GQA_ERR_TREE); base < 0 or base+T beyond
 * 16*max_blocks_per_seq (GQA_ERR_CONTEXT); a block holding one of positions
 * base .. base+T-1 outside [0, num_blocks) (GQA_ERR_BLOCK_ID).
 * GQA_FLAG_PDL in shape->flags chains the launch to the acceptance kernel. */
gqa_status gqa_kv_compact(const gqa_shape *shape, void *k_cache, void *v_cache,
                          float *k_scale, float *v_scale, const int32_t *block_tables,
                          const int32_t *context_lens, const int32_t *path,
                          const int32_t *accepted, int32_t *dev_status, void *stream);

/* Stochastic acceptance (speculative sampling).  CS336 lecture 10
 * §"Спекулятивное сэмплирование": modified rejection sampling with the draft
 * model p as proposal and the target model q as target; draft token x is kept
 * with probability min(1, q(x)/p(x)), the first rejection is replaced by a draw
 * from max(q - p, 0) renormalised, and when every draft is kept one more token
 * is drawn from the target's last distribution.  The emitted tokens are then
 * exact samples of q (the page's two-token proof).
 *   target_probs  fp32 [B][T][V]   q_t: target's distribution for the token
 *                                  after the prefix and drafts 0..t-1
 *   draft_probs   fp32 [B][T-1][V] p_t: the distribution draft_ids[b][t] was
 *                                  drawn from (NULL allowed when T == 1)
 *   draft_ids     int32 [B][T-1]   (NULL allowed when T == 1)
 *   uniforms      fp64 [B][T] in [0,1): uniforms[b][t], t < T-1, decides draft
 *                 t; uniforms[b][T-1] draws the final token.  The caller draws
 *                 them (any generator); the call itself is deterministic.
 *   accepted[b]   = a, the number of drafts kept (a run from the start)
 *   next_token[b] = the token drawn at position a
 *   context_lens_inout[b] -= T-1-a  (if not NULL, as in gqa_accept_prefix)
 * Arithmetic, identical on every device and in any thread order:
 *   - draft t is kept iff u * p_t(x) < q_t(x), u and both probabilities widened
 *     to double (the product is exact); an id outside [0, V) is rejected;
 *   - a draw from weights w_v is the inverse CDF on W_v = floor(w_v * 2^40)
 *     (integers): S = sum_v W_v, r = min(floor(u * S), S-1) in double, token =
 *     least v with W_0 + ... + W_v > r; the residual weight is max(q - p, 0)
 *     with the difference rounded once to fp32; a residual with S == 0 falls
 *     back to q itself.
 * Requires 0 <= B <= 2^28, 1 <= T <= 64, V >= 1; no alignment (16-byte aligned
 * rows with V % 4 == 0 are read with 16-byte loads).  Device errors: an entry read
 * that is NaN, < 0 or > 1 counts as 0, and a uniform outside [0,1) as 0
 * (GQA_ERR_PROBS); a row with no weight gives token 0 (GQA_ERR_PROBS); a
 * context length that would drop below zero is left unchanged
 * (GQA_ERR_CONTEXT). */
gqa_status gqa_accept_sampled(int B, int T, int V, const float *target_probs,
                              const float *draft_probs, const int32_t *draft_ids,
                              const double *uniforms, int32_t *accepted,
                              int32_t *next_token, int32_t *context_lens_inout,
                              int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* GQA_DECODE_H */
