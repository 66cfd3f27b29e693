// kv_compact.cu -- after greedy acceptance over a draft tree, move the cached
// rows of the accepted branch so the sequence reads in order again.
//
// "Болжау арқылы Sonar модельдерін жылдамдату" §"EAGLE": the target scores
// every node of the draft tree in one pass and the longest agreeing branch is
// kept for continuation.  The T nodes were appended at positions base ..
// base+T-1 (node i at base+i, CS336 lecture 10 §"PagedAttention" block
// addressing); the kept branch root, p_1, .. p_a must end up at base,
// base+1, .. base+a, so position base+j takes node p_j's K and V rows.
//
// One thread block per (sequence, KV head).  The branch's nodes have
// increasing indices (every parent precedes its children), so a destination
// may be another step's source: the block reads all of its rows into shared
// memory first and writes them after a barrier.  Different blocks touch
// disjoint bytes (another KV head's slice of the same rows, or another
// sequence's blocks).
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxT = 64;
constexpr int kMaxRowVec = 16;  // 16-byte chunks of one cached row (H = 128, 2-byte elements)

__global__ void __launch_bounds__(kThreads)
    kv_compact_kernel(uint4* k_cache, uint4* v_cache, float* k_scale, float* v_scale,
                      const int32_t* __restrict__ block_tables,
                      const int32_t* __restrict__ context_lens, const int32_t* __restrict__ path,
                      const int32_t* __restrict__ accepted, int32_t* status, int T, int K,
                      int row_vec, int max_blocks, int num_blocks) {
    __shared__ uint4 stage[2 * (kMaxT - 1) * kMaxRowVec];
    __shared__ float sscale[2 * (kMaxT - 1)];
    __shared__ int spath[kMaxT];
    griddep_launch_dependents();
    griddep_wait();  // accepted, path and context_lens follow the acceptance kernel
    const int b = blockIdx.x, k = blockIdx.y, tid = threadIdx.x;
    const bool reporter = tid == 0 && k == 0;  // one report per sequence
    const int a = accepted[b];
    // the branch: a in [0, T-1], nodes strictly increasing within [1, T)
    int bad = !(a >= 0 && a <= T - 1);
    if (!bad && tid < a) {
        const int32_t* pb = path + (size_t)b * (T - 1);
        const int p = pb[tid];
        const int prev = tid ? pb[tid - 1] : 0;
        bad = p < 1 || p >= T || p <= prev;
        spath[tid] = p;
    }
    if (__syncthreads_or(bad)) {
        if (reporter) report(status, GQA_ERR_TREE);
        return;
    }
    // the T positions from base on lie inside the table
    const long long base = (long long)context_lens[b] - 1 - a;
    if (base < 0 || base + T > 16ll * max_blocks) {
        if (reporter) report(status, GQA_ERR_CONTEXT);
        return;
    }
    const int32_t* table = block_tables + (size_t)b * max_blocks;
    const int blk_lo = (int)(base >> 4), nblk = (int)((base + T - 1) >> 4) - blk_lo + 1;
    int bad_id = 0;
    if (tid < nblk) {
        const int id = table[blk_lo + tid];
        bad_id = id < 0 || id >= num_blocks;
    }
    if (__syncthreads_or(bad_id)) {
        if (reporter) report(status, GQA_ERR_BLOCK_ID);
        return;
    }
    if (a == 0) return;
    // every source row (K then V chunks of node p_j's row) into shared memory ...
    const int per_node = 2 * row_vec;
    const int items = a * per_node;
    for (int it = tid; it < items; it += kThreads) {
        const int j = it / per_node, r = it - j * per_node;
        const int v = r >= row_vec, c = r - v * row_vec;
        const long long pos = base + spath[j];
        const size_t off = (((size_t)table[pos >> 4] * 16 + (pos & 15)) * K + k) * row_vec + c;
        stage[it] = (v ? v_cache : k_cache)[off];
    }
    if (k_scale && tid < 2 * a) {
        const int j = tid >> 1, v = tid & 1;
        const long long pos = base + spath[j];
        sscale[tid] = (v ? v_scale : k_scale)[((size_t)table[pos >> 4] * K + k) * 16 + (pos & 15)];
    }
    __syncthreads();
    // ... then position base+1+j takes the (j+1)-th node's row
    for (int it = tid; it < items; it += kThreads) {
        const int j = it / per_node, r = it - j * per_node;
        const int v = r >= row_vec, c = r - v * row_vec;
        const long long pos = base + 1 + j;
        const size_t off = (((size_t)table[pos >> 4] * 16 + (pos & 15)) * K + k) * row_vec + c;
        (v ? v_cache : k_cache)[off] = stage[it];
    }
    if (k_scale && tid < 2 * a) {
        const int j = tid >> 1, v = tid & 1;
        const long long pos = base + 1 + j;
        (v ? v_scale : k_scale)[((size_t)table[pos >> 4] * K + k) * 16 + (pos & 15)] = sscale[tid];
    }
}

}  // namespace

gqa_status launch_kv_compact(const gqa_shape& s, void* k_cache, void* v_cache, float* k_scale,
                             float* v_scale, const int32_t* block_tables,
                             const int32_t* context_lens, const int32_t* path,
                             const int32_t* accepted, int32_t* dev_status, cudaStream_t stream) {
    if (s.B == 0 || s.T <= 1) return GQA_OK;
    if (s.T > kMaxT || s.K > 65535) return GQA_ERR_SHAPE;
    const int esize = s.kv_dtype == GQA_KV_SAME ? 2 : 1;
    const int row_vec = s.H * esize / 16;
    if (row_vec < 1 || row_vec > kMaxRowVec) return GQA_ERR_SHAPE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)s.B, (unsigned)s.K, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (s.flags & (GQA_FLAG_PDL | GQA_FLAG_EARLY_KV)) ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, kv_compact_kernel, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
        k_scale, v_scale, block_tables, context_lens, path, accepted, dev_status, s.T, s.K,
        row_vec, s.max_blocks_per_seq, s.num_blocks);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
