// kv_append.cu -- write the T newest tokens' keys and values into the paged cache.
//
// KV-cache section of "جعل inference رخيصًا: KV cache وbatching والتكميم": the
// keys and values of a position never change once computed, so each new token's
// K/V vectors are stored once and every later step attends over them.  The
// addressing is the block table of CS336 lecture 10 §"PagedAttention": position
// pos of sequence b lives in block block_tables[b][pos/16], row pos%16.
//
// A pure copy: one warp per (b, t) moves K*H 2-byte elements (a contiguous
// row of the [blocks][16][K][H] cache) with 16-byte loads and stores.
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace gqa {
namespace {

__global__ void __launch_bounds__(128)
    kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                     const int32_t* __restrict__ block_tables,
                     const int32_t* __restrict__ context_lens, int32_t* status, int B, int T,
                     int row_vec, int max_blocks, int num_blocks) {
    griddep_launch_dependents();
    griddep_wait();  // k_new / v_new and the cache follow the previous kernels
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const long long pairs = (long long)B * T;
    for (long long wi = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); wi < pairs;
         wi += (long long)gridDim.x * wpb) {
        const int b = (int)(wi / T), t = (int)(wi % T);
        const int ctx = context_lens[b];
        if (ctx < T || ctx > max_blocks * 16) {
            if (lane == 0 && t == 0) report(status, GQA_ERR_CONTEXT);
            continue;
        }
        const int pos = ctx - T + t;
        const int blk = block_tables[(size_t)b * max_blocks + (pos >> 4)];
        if (blk < 0 || blk >= num_blocks) {
            if (lane == 0) report(status, GQA_ERR_BLOCK_ID);
            continue;
        }
        const size_t dst = ((size_t)blk * 16 + (pos & 15)) * row_vec;
        const size_t src = (size_t)wi * row_vec;
        for (int v = lane; v < row_vec; v += 32) {
            k_cache[dst + v] = __ldg(k_new + src + v);
            v_cache[dst + v] = __ldg(v_new + src + v);
        }
    }
}

}  // namespace

gqa_status launch_kv_append(const gqa_shape& s, const void* k_new, const void* v_new,
                            void* k_cache, void* v_cache, const int32_t* block_tables,
                            const int32_t* context_lens, int32_t* dev_status,
                            cudaStream_t stream) {
    const long long pairs = (long long)s.B * s.T;
    if (pairs == 0) return GQA_OK;
    const int row_vec = s.K * s.H * 2 / 16;
    const int wpb = 4;
    long long blocks = (pairs + wpb - 1) / wpb;
    const int sms = device_sm_count();
    const long long cap = (long long)(sms > 0 ? sms : 148) * 16;
    if (blocks > cap) blocks = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(32 * wpb);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (s.flags & (GQA_FLAG_PDL | GQA_FLAG_EARLY_KV)) ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, kv_append_kernel, static_cast<const uint4*>(k_new),
        static_cast<const uint4*>(v_new), static_cast<uint4*>(k_cache),
        static_cast<uint4*>(v_cache), block_tables, context_lens, dev_status, s.B, s.T, row_vec,
        s.max_blocks_per_seq, s.num_blocks);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
