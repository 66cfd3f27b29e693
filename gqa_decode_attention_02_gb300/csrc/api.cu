// api.cu -- the extern "C" entry points declared in include/gqa_decode.h:
// host-side argument validation, then one launch per operation.
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gqa_status check_common(const gqa_shape* s) {
    if (!s) return GQA_ERR_NULL;
    if (s->dtype != GQA_F16 && s->dtype != GQA_BF16) return GQA_ERR_DTYPE;
    if (s->B < 0 || s->T < 1 || s->N < 1 || s->K < 1 || s->N % s->K != 0) return GQA_ERR_SHAPE;
    if (s->H != 64 && s->H != 128) return GQA_ERR_SHAPE;
    if (s->block_size != 16 || s->num_blocks < 1 || s->max_blocks_per_seq < 1)
        return GQA_ERR_SHAPE;
    if ((long long)s->num_blocks * 16 > (1ll << 31) - 1) return GQA_ERR_SHAPE;
    if ((long long)s->max_blocks_per_seq * 16 > (1ll << 30)) return GQA_ERR_SHAPE;
    if ((long long)s->B * s->K * s->max_blocks_per_seq > (1ll << 31) - 1) return GQA_ERR_SHAPE;
    if (s->window < 0) return GQA_ERR_SHAPE;
    if (s->kv_dtype < GQA_KV_SAME || s->kv_dtype > GQA_KV_E4M3) return GQA_ERR_DTYPE;
    return GQA_OK;
}

gqa_status attention_entry(const gqa_shape* s, bool decode_only, bool fused, const void* q,
                           const void* k_new, const void* v_new, const void* k_cache,
                           const void* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, const uint64_t* tree_mask, void* out,
                           void* workspace, size_t ws_bytes, int32_t* dev_status,
                           void* stream, const float* k_scale = nullptr,
                           const float* v_scale = nullptr) {
    gqa_status st = check_common(s);
    if (st != GQA_OK) return st;
    if (decode_only && s->T != 1) return GQA_ERR_SHAPE;
    // one-byte caches come with their row scales (the _quant calls), others without
    if ((s->kv_dtype != GQA_KV_SAME) != (k_scale != nullptr)) return GQA_ERR_DTYPE;
    if (k_scale && !v_scale) return GQA_ERR_NULL;
    if (k_scale && (!aligned16(k_scale) || !aligned16(v_scale))) return GQA_ERR_ALIGN;
    if (s->B == 0) return GQA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return GQA_ERR_NULL;
    if (fused && (!k_new || !v_new)) return GQA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return GQA_ERR_ALIGN;
    if (fused && (!aligned16(k_new) || !aligned16(v_new))) return GQA_ERR_ALIGN;
    if (tree_mask && s->window > 0) return GQA_ERR_SHAPE;  // not combined
    if (tree_mask && s->T > 64) return GQA_ERR_SHAPE;      // one 64-bit row per new token
    if (tree_mask && (reinterpret_cast<uintptr_t>(tree_mask) & 7u) != 0) return GQA_ERR_ALIGN;
    const bool force_warp = (s->flags & GQA_FLAG_WARP_MMA) != 0;
    const bool force_tc = (s->flags & GQA_FLAG_TENSOR_MEMORY) != 0;
    const bool force_direct = (s->flags & GQA_FLAG_DIRECT) != 0;
    if ((int)force_warp + (int)force_tc + (int)force_direct > 1) return GQA_ERR_SHAPE;
    if (force_tc && !gqa::tc_attention_supported(*s)) return GQA_ERR_SHAPE;
    gqa::AttnPlan plan;
    st = gqa::attention_plan(*s, tree_mask != nullptr, &plan);
    if (st != GQA_OK) return st;
    if (!workspace || ws_bytes < plan.workspace) return GQA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GQA_ERR_ALIGN;
    if (force_tc || (!force_warp && !force_direct && gqa::tc_attention_preferred(*s))) {
        if (ws_bytes < gqa::tc_workspace_bytes(*s, plan.flags_bytes)) return GQA_ERR_WORKSPACE;
        cudaStream_t cs = static_cast<cudaStream_t>(stream);
        if (fused) {
            st = gqa::launch_kv_append(*s, k_new, v_new, const_cast<void*>(k_cache),
                                       const_cast<void*>(v_cache), block_tables, context_lens,
                                       dev_status, cs);
            if (st != GQA_OK) return st;
        }
        return gqa::launch_tc_attention(*s, q, k_cache, v_cache, block_tables, context_lens,
                                        tree_mask, out, workspace, plan.flags_bytes, dev_status,
                                        cs);
    }
    if (fused && k_scale) {
        // One-byte cache: the append is a launch of its own just before the
        // attention launch.  (Both one-launch forms measured slower on the
        // 256-sequence int8 batch, whose attention kernel is bound by its
        // producer warp's issue rate and its consumers' registers: the rows
        // quantized by the consumers 467 us, by the producer 417 us, against
        // 360 + 9 us for the two launches.)
        cudaStream_t cs = static_cast<cudaStream_t>(stream);
        st = gqa::launch_kv_append_quant(*s, k_new, v_new, const_cast<void*>(k_cache),
                                         const_cast<void*>(v_cache),
                                         const_cast<float*>(k_scale),
                                         const_cast<float*>(v_scale), block_tables,
                                         context_lens, dev_status, cs);
        if (st != GQA_OK) return st;
        return gqa::launch_attention(*s, plan, q, nullptr, nullptr, k_cache, v_cache,
                                     block_tables, context_lens, tree_mask, k_scale, v_scale,
                                     out, workspace, dev_status, cs);
    }
    return gqa::launch_attention(*s, plan, q, fused ? k_new : nullptr, fused ? v_new : nullptr,
                                 k_cache, v_cache, block_tables, context_lens, tree_mask,
                                 k_scale, v_scale, out, workspace, dev_status,
                                 static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int gqa_version(void) { return 200; }

const char* gqa_status_string(int status) {
    switch (status) {
        case GQA_OK: return "ok";
        case GQA_ERR_NULL: return "a required pointer is NULL";
        case GQA_ERR_SHAPE: return "unsupported or inconsistent sizes";
        case GQA_ERR_DTYPE: return "unsupported dtype";
        case GQA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case GQA_ERR_WORKSPACE: return "workspace missing or too small";
        case GQA_ERR_CUDA: return "CUDA call failed";
        case GQA_ERR_CONTEXT: return "context length out of range";
        case GQA_ERR_BLOCK_ID: return "block id out of range";
        case GQA_ERR_TIMEOUT: return "bounded wait inside a kernel timed out";
        case GQA_ERR_PROBS: return "invalid probability, uniform or empty distribution";
        case GQA_ERR_TREE: return "draft tree parent or accepted path out of range";
        default: return "unknown status";
    }
}

gqa_status gqa_kv_append(const gqa_shape* shape, const void* k_new, const void* v_new,
                         void* k_cache, void* v_cache, const int32_t* block_tables,
                         const int32_t* context_lens, int32_t* dev_status, void* stream) {
    gqa_status st = check_common(shape);
    if (st != GQA_OK) return st;
    if (shape->kv_dtype != GQA_KV_SAME) return GQA_ERR_DTYPE;  // use gqa_kv_append_quant
    if (shape->B == 0) return GQA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !block_tables || !context_lens)
        return GQA_ERR_NULL;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return GQA_ERR_ALIGN;
    return gqa::launch_kv_append(*shape, k_new, v_new, k_cache, v_cache, block_tables,
                                 context_lens, dev_status, static_cast<cudaStream_t>(stream));
}

gqa_status gqa_kv_append_quant(const gqa_shape* shape, const void* k_new, const void* v_new,
                               void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                               const int32_t* block_tables, const int32_t* context_lens,
                               int32_t* dev_status, void* stream) {
    gqa_status st = check_common(shape);
    if (st != GQA_OK) return st;
    if (shape->kv_dtype != GQA_KV_INT8 && shape->kv_dtype != GQA_KV_E4M3) return GQA_ERR_DTYPE;
    if (shape->B == 0) return GQA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !k_scale || !v_scale || !block_tables ||
        !context_lens)
        return GQA_ERR_NULL;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(k_scale) || !aligned16(v_scale))
        return GQA_ERR_ALIGN;
    return gqa::launch_kv_append_quant(*shape, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                                       block_tables, context_lens, dev_status,
                                       static_cast<cudaStream_t>(stream));
}

int gqa_attention_engine(const gqa_shape* shape) {
    if (check_common(shape) != GQA_OK) return 0;
    const bool force_warp = (shape->flags & GQA_FLAG_WARP_MMA) != 0;
    const bool force_tc = (shape->flags & GQA_FLAG_TENSOR_MEMORY) != 0;
    const bool force_direct = (shape->flags & GQA_FLAG_DIRECT) != 0;
    if ((int)force_warp + (int)force_tc + (int)force_direct > 1) return 0;
    if (force_tc) return gqa::tc_attention_supported(*shape) ? GQA_ENGINE_TENSOR_MEMORY : 0;
    if (force_direct) return gqa::direct_attention_supported(*shape, false) ? GQA_ENGINE_DIRECT : 0;
    if (force_warp) return GQA_ENGINE_WARP_MMA;
    if (gqa::tc_attention_preferred(*shape)) return GQA_ENGINE_TENSOR_MEMORY;
    return gqa::direct_attention_preferred(*shape, false) ? GQA_ENGINE_DIRECT
                                                          : GQA_ENGINE_WARP_MMA;
}

size_t gqa_attention_workspace_size(const gqa_shape* shape) {
    if (check_common(shape) != GQA_OK) return 0;
    // the largest need of the kernels that may serve the shape (the direct
    // kernel uses none, so its flag does not change the size)
    gqa_shape sh = *shape;
    sh.flags &= ~GQA_FLAG_DIRECT;
    gqa::AttnPlan plain, general;
    if (gqa::attention_plan(sh, false, &plain) != GQA_OK) return 0;
    if (gqa::attention_plan(sh, true, &general) != GQA_OK) return 0;
    size_t w = plain.workspace > general.workspace ? plain.workspace : general.workspace;
    const size_t tc = gqa::tc_workspace_bytes(*shape, plain.flags_bytes);  // 0: not served
    return tc > w ? tc : w;
}

gqa_status gqa_workspace_clear(void* workspace, size_t bytes, void* stream) {
    if (bytes == 0) return GQA_OK;
    if (!workspace) return GQA_ERR_NULL;
    return cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GQA_OK
               : GQA_ERR_CUDA;
}

gqa_status gqa_decode_attention(const gqa_shape* shape, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                const int32_t* context_lens, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
    return attention_entry(shape, true, false, q, nullptr, nullptr, k_cache, v_cache,
                           block_tables, context_lens, nullptr, out, workspace,
                           workspace_bytes, dev_status, stream);
}

gqa_status gqa_verify_attention(const gqa_shape* shape, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                const int32_t* context_lens, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
    return attention_entry(shape, false, false, q, nullptr, nullptr, k_cache, v_cache,
                           block_tables, context_lens, nullptr, out, workspace,
                           workspace_bytes, dev_status, stream);
}

gqa_status gqa_append_decode_attention(const gqa_shape* shape, const void* q,
                                       const void* k_new, const void* v_new, void* k_cache,
                                       void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, void* out, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status,
                                       void* stream) {
    return attention_entry(shape, true, true, q, k_new, v_new, k_cache, v_cache, block_tables,
                           context_lens, nullptr, out, workspace, workspace_bytes, dev_status,
                           stream);
}

gqa_status gqa_append_verify_attention(const gqa_shape* shape, const void* q,
                                       const void* k_new, const void* v_new, void* k_cache,
                                       void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, void* out, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status,
                                       void* stream) {
    return attention_entry(shape, false, true, q, k_new, v_new, k_cache, v_cache, block_tables,
                           context_lens, nullptr, out, workspace, workspace_bytes, dev_status,
                           stream);
}

gqa_status gqa_tree_verify_attention(const gqa_shape* shape, const void* q,
                                     const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     const uint64_t* tree_mask, void* out, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (!tree_mask) return GQA_ERR_NULL;
    return attention_entry(shape, false, false, q, nullptr, nullptr, k_cache, v_cache,
                           block_tables, context_lens, tree_mask, out, workspace,
                           workspace_bytes, dev_status, stream);
}

gqa_status gqa_append_tree_verify_attention(const gqa_shape* shape, const void* q,
                                            const void* k_new, const void* v_new,
                                            void* k_cache, void* v_cache,
                                            const int32_t* block_tables,
                                            const int32_t* context_lens,
                                            const uint64_t* tree_mask, void* out,
                                            void* workspace, size_t workspace_bytes,
                                            int32_t* dev_status, void* stream) {
    if (!tree_mask) return GQA_ERR_NULL;
    return attention_entry(shape, false, true, q, k_new, v_new, k_cache, v_cache, block_tables,
                           context_lens, tree_mask, out, workspace, workspace_bytes, dev_status,
                           stream);
}

gqa_status gqa_decode_attention_quant(const gqa_shape* shape, const void* q,
                                      const void* k_cache, const void* v_cache,
                                      const float* k_scale, const float* v_scale,
                                      const int32_t* block_tables,
                                      const int32_t* context_lens, void* out, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status,
                                      void* stream) {
    if (!k_scale || !v_scale) return GQA_ERR_NULL;
    return attention_entry(shape, true, false, q, nullptr, nullptr, k_cache, v_cache,
                           block_tables, context_lens, nullptr, out, workspace,
                           workspace_bytes, dev_status, stream, k_scale, v_scale);
}

gqa_status gqa_verify_attention_quant(const gqa_shape* shape, const void* q,
                                      const void* k_cache, const void* v_cache,
                                      const float* k_scale, const float* v_scale,
                                      const int32_t* block_tables,
                                      const int32_t* context_lens, void* out, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status,
                                      void* stream) {
    if (!k_scale || !v_scale) return GQA_ERR_NULL;
    return attention_entry(shape, false, false, q, nullptr, nullptr, k_cache, v_cache,
                           block_tables, context_lens, nullptr, out, workspace,
                           workspace_bytes, dev_status, stream, k_scale, v_scale);
}

gqa_status gqa_tree_verify_attention_quant(const gqa_shape* shape, const void* q,
                                          const void* k_cache, const void* v_cache,
                                          const float* k_scale, const float* v_scale,
                                          const int32_t* block_tables,
                                          const int32_t* context_lens,
                                          const uint64_t* tree_mask, void* out, void* workspace,
                                          size_t workspace_bytes, int32_t* dev_status,
                                          void* stream) {
    if (!k_scale || !v_scale || !tree_mask) return GQA_ERR_NULL;
    return attention_entry(shape, false, false, q, nullptr, nullptr, k_cache, v_cache,
                           block_tables, context_lens, tree_mask, out, workspace,
                           workspace_bytes, dev_status, stream, k_scale, v_scale);
}

gqa_status gqa_append_decode_attention_quant(const gqa_shape* shape, const void* q,
                                             const void* k_new, const void* v_new,
                                             void* k_cache, void* v_cache, float* k_scale,
                                             float* v_scale, const int32_t* block_tables,
                                             const int32_t* context_lens, void* out,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* dev_status, void* stream) {
    if (!k_scale || !v_scale) return GQA_ERR_NULL;
    return attention_entry(shape, true, true, q, k_new, v_new, k_cache, v_cache, block_tables,
                           context_lens, nullptr, out, workspace, workspace_bytes, dev_status,
                           stream, k_scale, v_scale);
}

gqa_status gqa_append_verify_attention_quant(const gqa_shape* shape, const void* q,
                                             const void* k_new, const void* v_new,
                                             void* k_cache, void* v_cache, float* k_scale,
                                             float* v_scale, const int32_t* block_tables,
                                             const int32_t* context_lens, void* out,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* dev_status, void* stream) {
    if (!k_scale || !v_scale) return GQA_ERR_NULL;
    return attention_entry(shape, false, true, q, k_new, v_new, k_cache, v_cache, block_tables,
                           context_lens, nullptr, out, workspace, workspace_bytes, dev_status,
                           stream, k_scale, v_scale);
}

size_t gqa_accept_workspace_size(int B, int T) { return gqa::accept_workspace_bytes(B, T); }

gqa_status gqa_accept_prefix(int B, int T, int V, const float* target_logits,
                             const int32_t* draft_ids, int32_t* accepted, int32_t* next_token,
                             int32_t* context_lens_inout, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (B < 0 || T < 1 || T > 64 || V < 1) return GQA_ERR_SHAPE;
    if (!workspace && B > 65535) return GQA_ERR_SHAPE;  // one cluster per sequence (grid y)
    if (B == 0) return GQA_OK;
    if (!target_logits || !accepted || !next_token || (T > 1 && !draft_ids))
        return GQA_ERR_NULL;
    if (!aligned16(target_logits)) return GQA_ERR_ALIGN;
    if ((long long)T * V > (1ll << 31) - 1) return GQA_ERR_SHAPE;
    if (workspace) {
        if (workspace_bytes < gqa::accept_workspace_bytes(B, T)) return GQA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return GQA_ERR_ALIGN;
    }
    return gqa::launch_accept_prefix(B, T, V, target_logits, draft_ids, nullptr, accepted,
                                     next_token, nullptr, context_lens_inout, workspace,
                                     dev_status, static_cast<cudaStream_t>(stream));
}

gqa_status gqa_accept_tree(int B, int T, int V, const float* target_logits,
                           const int32_t* draft_ids, const int32_t* parents, int32_t* accepted,
                           int32_t* next_token, int32_t* path, int32_t* context_lens_inout,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream) {
    if (B < 0 || T < 1 || T > 64 || V < 1) return GQA_ERR_SHAPE;
    if (!workspace && B > 65535) return GQA_ERR_SHAPE;  // one cluster per sequence (grid y)
    if (B == 0) return GQA_OK;
    if (!target_logits || !parents || !accepted || !next_token ||
        (T > 1 && (!draft_ids || !path)))
        return GQA_ERR_NULL;
    if (!aligned16(target_logits)) return GQA_ERR_ALIGN;
    if ((long long)T * V > (1ll << 31) - 1) return GQA_ERR_SHAPE;
    if (workspace) {
        if (workspace_bytes < gqa::accept_workspace_bytes(B, T)) return GQA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return GQA_ERR_ALIGN;
    }
    return gqa::launch_accept_prefix(B, T, V, target_logits, draft_ids, parents, accepted,
                                     next_token, path, context_lens_inout, workspace,
                                     dev_status, static_cast<cudaStream_t>(stream));
}

gqa_status gqa_kv_compact(const gqa_shape* shape, void* k_cache, void* v_cache, float* k_scale,
                          float* v_scale, const int32_t* block_tables,
                          const int32_t* context_lens, const int32_t* path,
                          const int32_t* accepted, int32_t* dev_status, void* stream) {
    gqa_status st = check_common(shape);
    if (st != GQA_OK) return st;
    if (shape->T > 64) return GQA_ERR_SHAPE;
    const bool one_byte = shape->kv_dtype != GQA_KV_SAME;
    if (!one_byte && (k_scale || v_scale)) return GQA_ERR_DTYPE;  // scales: one-byte caches only
    if (one_byte && (!k_scale || !v_scale)) return GQA_ERR_NULL;
    if (shape->B == 0 || shape->T == 1) return GQA_OK;  // nothing can move
    if (!k_cache || !v_cache || !block_tables || !context_lens || !path || !accepted)
        return GQA_ERR_NULL;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return GQA_ERR_ALIGN;
    return gqa::launch_kv_compact(*shape, k_cache, v_cache, k_scale, v_scale, block_tables,
                                  context_lens, path, accepted, dev_status,
                                  static_cast<cudaStream_t>(stream));
}

gqa_status gqa_accept_sampled(int B, int T, int V, const float* target_probs,
                              const float* draft_probs, const int32_t* draft_ids,
                              const double* uniforms, int32_t* accepted, int32_t* next_token,
                              int32_t* context_lens_inout, int32_t* dev_status, void* stream) {
    if (B < 0 || T < 1 || T > 64 || V < 1 || B > (1 << 28)) return GQA_ERR_SHAPE;
    if (B == 0) return GQA_OK;
    if (!target_probs || !uniforms || !accepted || !next_token) return GQA_ERR_NULL;
    if (T > 1 && (!draft_probs || !draft_ids)) return GQA_ERR_NULL;
    return gqa::launch_accept_sampled(B, T, V, target_probs, T > 1 ? draft_probs : nullptr,
                                      T > 1 ? draft_ids : nullptr, uniforms, accepted,
                                      next_token, context_lens_inout, dev_status,
                                      static_cast<cudaStream_t>(stream));
}

}  // extern "C"
