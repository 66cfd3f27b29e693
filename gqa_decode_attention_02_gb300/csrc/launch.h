// launch.h -- host-side launchers shared between the kernel files and api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gqa_decode.h"

namespace gqa {

// Launch plan of the attention kernel for one shape on the current device.
struct AttnPlan {
    int grid;            // persistent CTAs
    int consumer_warps;  // row warps per group (8 * tiles_per_warp query rows each)
    int threads;
    size_t smem;         // dynamic shared memory per CTA
    int stages;          // depth of the shared-memory ring
    int groups;          // stage-parallel consumer groups
    int tiles_per_warp;  // 8-row query tiles per consumer warp (1 or 2)
    bool general;        // the kernel variant with window, tree mask and row chunks
    int chunks;          // row chunks per KV head (T*G rows, at most 48 per chunk)
    int rows_per_chunk;
    size_t flags_bytes;             // fixed region of publication flags
    size_t partial_floats_per_cta;
    size_t workspace;    // total bytes
    // The direct kernel serves the call instead (one CTA per segment, no
    // workspace use; grid, threads and smem above are then its own).
    bool direct;
};

// Fills `plan`; `masked`: a tree mask will be passed.  The plan picks the plain
// kernel or the general one (window, tree mask, row chunks).  Returns GQA_OK
// or a validation error.
gqa_status attention_plan(const gqa_shape& s, bool masked, AttnPlan* plan);

// k_new / v_new == nullptr: attention over the cache as it is; otherwise the
// T newest tokens are appended from them by the same launch (the caches are
// then written).
gqa_status launch_attention(const gqa_shape& s, const AttnPlan& plan, const void* q,
                            const void* k_new, const void* v_new, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables,
                            const int32_t* context_lens, const uint64_t* tree_mask,
                            const float* k_scale, const float* v_scale, void* out,
                            void* workspace, int32_t* dev_status, cudaStream_t stream);

gqa_status launch_kv_append(const gqa_shape& s, const void* k_new, const void* v_new,
                            void* k_cache, void* v_cache, const int32_t* block_tables,
                            const int32_t* context_lens, int32_t* dev_status,
                            cudaStream_t stream);

// workspace == nullptr: one thread-block cluster per sequence; otherwise many
// blocks per sequence whose keys meet in the workspace (accept_workspace_bytes).
// parents == nullptr: prefix acceptance of a chain of drafts; otherwise
// acceptance over the draft tree parents [B][T], the accepted branch's nodes
// written to path [B][T-1].
size_t accept_workspace_bytes(int B, int T);
gqa_status launch_accept_prefix(int B, int T, int V, const float* logits,
                                const int32_t* draft, const int32_t* parents,
                                int32_t* accepted, int32_t* next_token, int32_t* path,
                                int32_t* ctx_io, void* workspace, int32_t* dev_status,
                                cudaStream_t stream);

// Moves the cached rows of an accepted tree branch behind its root (see
// gqa_kv_compact); k_scale / v_scale non-null for one-byte caches.
gqa_status launch_kv_compact(const gqa_shape& s, void* k_cache, void* v_cache, float* k_scale,
                             float* v_scale, const int32_t* block_tables,
                             const int32_t* context_lens, const int32_t* path,
                             const int32_t* accepted, int32_t* dev_status, cudaStream_t stream);

gqa_status launch_accept_sampled(int B, int T, int V, const float* q, const float* p,
                                 const int32_t* draft, const double* u, int32_t* accepted,
                                 int32_t* next_token, int32_t* ctx_io, int32_t* dev_status,
                                 cudaStream_t stream);

gqa_status launch_kv_append_quant(const gqa_shape& s, const void* k_new, const void* v_new,
                                  void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  int32_t* dev_status, cudaStream_t stream);

// TMA view (h, kv head, block*16 + row) of a cache, 128-byte boxes of 16 rows.
bool make_cache_map(CUtensorMap* m, const void* base, const gqa_shape& s);
// 5-D TMA view (dim, query head within its group, KV head, new token,
// sequence) of a [B][T][N][H = 128] tensor of q's dtype (q or out); one box =
// 64 dims x hpc heads x tpc tokens of one KV head, 128-byte swizzled.
// Elements outside the tensor read as zero and are not written.
bool make_rows_map(CUtensorMap* m, const void* base, const gqa_shape& s, int hpc, int tpc);

// The direct warp-level kernel (one CTA per (sequence, KV head)): which
// shapes it can serve, and which it serves by default.  Host logic only.
bool direct_attention_supported(const gqa_shape& s, bool masked);
bool direct_attention_preferred(const gqa_shape& s, bool masked);

// Tensor-memory attention (tcgen05): decode / verify / tree verify and local
// attention with H = 64 or 128 over a cache in q's dtype, no fused append (the caller
// appends first).  `preferred`: the shapes where it is the faster kernel.  The
// workspace holds the publication flags (flags_bytes, as the warp-level
// kernel's plan lays them out) and then the partial results of split segments.
bool tc_attention_supported(const gqa_shape& s);
bool tc_attention_preferred(const gqa_shape& s);
size_t tc_workspace_bytes(const gqa_shape& s, size_t flags_bytes);
gqa_status launch_tc_attention(const gqa_shape& s, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               const int32_t* context_lens, const uint64_t* tree_mask, void* out,
                               void* workspace, size_t flags_bytes, int32_t* dev_status,
                               cudaStream_t stream);

// Cached per-device SM count (0 on failure).
int device_sm_count();

}  // namespace gqa
