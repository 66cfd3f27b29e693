// kv_quant.cu -- append the T newest tokens' keys and values to a one-byte
// (int8 or e4m3) paged cache.
//
// Quantization section of "جعل inference رخيصًا: KV cache وbatching والتكميم":
// symmetric absolute-maximum quantization -- scale = max|x| / qmax, codes
// round(x / scale) clamped -- and, the decode step being bandwidth bound,
// fewer bytes per cached element make every step faster.  CS336 lecture 10
// §"Квантование" names fp8 (e4m3) and int8 as the one-byte formats.  Each
// cached key or value row of one KV head (H elements) gets its own fp32 scale,
// stored per block as scale[block][kv head][row]; qmax is 127 for int8 and the
// largest finite e4m3 value, 448, for e4m3 (codes rounded to nearest even,
// saturating).
//
// One warp per (token, KV head): each lane widens H/32 elements, a warp max
// gives max|x|, then scale and every x / scale are IEEE fp32 divisions.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace gqa {
namespace {

template <bool BF16>
__device__ __forceinline__ float widen16(uint16_t b) {
    if (BF16) return __uint_as_float((uint32_t)b << 16);
    return __half2float(__ushort_as_half(b));
}

// One row of H elements -> H one-byte codes and a scale (whole warp).
template <bool BF16, int KIND, int H>
__device__ __forceinline__ void quantize_row(const uint16_t* __restrict__ src, uint8_t* dst,
                                             float* scale_dst, int lane) {
    constexpr int EPL = H / 32;  // elements per lane: 4 (H = 128) or 2 (H = 64)
    float x[EPL];
    if (EPL == 4) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(src) + lane);
        x[0] = widen16<BF16>((uint16_t)(w.x & 0xffffu));
        x[1] = widen16<BF16>((uint16_t)(w.x >> 16));
        x[2] = widen16<BF16>((uint16_t)(w.y & 0xffffu));
        x[3] = widen16<BF16>((uint16_t)(w.y >> 16));
    } else {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(src) + lane);
        x[0] = widen16<BF16>((uint16_t)(w & 0xffffu));
        x[1] = widen16<BF16>((uint16_t)(w >> 16));
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(amax, KIND == GQA_KV_INT8 ? 127.f : 448.f);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        uint32_t code = 0;
        if (scale != 0.f) {
            const float y = __fdiv_rn(x[e], scale);
            if (KIND == GQA_KV_INT8) {
                int r = (y != y) ? 0 : __float2int_rn(y);
                r = min(127, max(-128, r));
                code = (uint32_t)(r & 0xff);
            } else {
                code = (uint32_t)__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
            }
        }
        packed |= code << (8 * e);
    }
    if (EPL == 4)
        reinterpret_cast<uint32_t*>(dst)[lane] = packed;
    else
        reinterpret_cast<uint16_t*>(dst)[lane] = (uint16_t)packed;
    if (lane == 0) *scale_dst = scale;
}

template <bool BF16, int KIND, int H>
__global__ void __launch_bounds__(128)
    kv_append_quant_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                           uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                           const int32_t* __restrict__ block_tables,
                           const int32_t* __restrict__ context_lens, int32_t* status, int B,
                           int T, int K, int max_blocks, int num_blocks) {
    griddep_launch_dependents();
    griddep_wait();  // k_new / v_new and the cache follow the previous kernels
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const long long rows = (long long)B * T * K;
    for (long long wi = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); wi < rows;
         wi += (long long)gridDim.x * wpb) {
        const int k = (int)(wi % K);
        const long long bt = wi / K;
        const int b = (int)(bt / T), t = (int)(bt % T);
        const int ctx = context_lens[b];
        if (ctx < T || ctx > max_blocks * 16) {
            if (lane == 0 && t == 0 && k == 0) report(status, GQA_ERR_CONTEXT);
            continue;
        }
        const int pos = ctx - T + t;
        const int blk = block_tables[(size_t)b * max_blocks + (pos >> 4)];
        if (blk < 0 || blk >= num_blocks) {
            if (lane == 0 && k == 0) report(status, GQA_ERR_BLOCK_ID);
            continue;
        }
        const int row = pos & 15;
        const size_t src = (size_t)wi * H;
        const size_t dst = (((size_t)blk * 16 + row) * K + k) * H;
        const size_t sc = ((size_t)blk * K + k) * 16 + row;
        quantize_row<BF16, KIND, H>(k_new + src, k_cache + dst, k_scale + sc, lane);
        quantize_row<BF16, KIND, H>(v_new + src, v_cache + dst, v_scale + sc, lane);
    }
}

template <bool BF16, int KIND, int H>
const void* append_kernel() {
    return reinterpret_cast<const void*>(&kv_append_quant_kernel<BF16, KIND, H>);
}

const void* pick_append(bool bf16, int kind, int H) {
    if (kind == GQA_KV_INT8) {
        if (H == 128) return bf16 ? append_kernel<true, GQA_KV_INT8, 128>()
                                  : append_kernel<false, GQA_KV_INT8, 128>();
        return bf16 ? append_kernel<true, GQA_KV_INT8, 64>()
                    : append_kernel<false, GQA_KV_INT8, 64>();
    }
    if (H == 128) return bf16 ? append_kernel<true, GQA_KV_E4M3, 128>()
                              : append_kernel<false, GQA_KV_E4M3, 128>();
    return bf16 ? append_kernel<true, GQA_KV_E4M3, 64>() : append_kernel<false, GQA_KV_E4M3, 64>();
}

}  // namespace

gqa_status launch_kv_append_quant(const gqa_shape& s, const void* k_new, const void* v_new,
                                  void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  int32_t* dev_status, cudaStream_t stream) {
    const long long rows = (long long)s.B * s.T * s.K;
    if (rows == 0) return GQA_OK;
    const int wpb = 4;
    long long blocks = (rows + wpb - 1) / wpb;
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
    const uint16_t* kn = static_cast<const uint16_t*>(k_new);
    const uint16_t* vn = static_cast<const uint16_t*>(v_new);
    uint8_t* kc = static_cast<uint8_t*>(k_cache);
    uint8_t* vc = static_cast<uint8_t*>(v_cache);
    int B = s.B, T = s.T, K = s.K, mb = s.max_blocks_per_seq, nb = s.num_blocks;
    void* args[] = {&kn, &vn, &kc, &vc, &k_scale, &v_scale, (void*)&block_tables,
                    (void*)&context_lens, &dev_status, &B, &T, &K, &mb, &nb};
    const cudaError_t e = cudaLaunchKernelExC(
        &cfg, pick_append(s.dtype == GQA_BF16, s.kv_dtype, s.H), args);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
