// noalloc.cu -- decode attention that allocates nothing, for callers that
// cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: a host program that
// reserved (nearly) all device memory for its own pool at start-up, where a
// further allocation would fail or fragment that pool; code on a
// latency-critical decode path, where cudaMalloc / cudaFree can synchronise
// the device; or a plain C caller with no allocator of its own at hand.  For
// them gqa_decode_attention_noalloc runs the same split-context decode kernel
// as gqa_decode_attention, but with its scratch (split-segment tickets and
// partial results) in a file-scope device array of fixed size, so the caller passes
// only inputs and outputs.
//
// The array costs every GPU that loads the library kScratchBytes of device
// memory until the process exits.  Its device address is looked up once per
// device, by the first call made with that device current.  Every call uses
// the same array and finds the previous call's contents in it: the region
// that must start at zero is cleared on the caller's stream before each
// launch.  Calls whose work overlaps on the GPU (other streams, or other host
// threads) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"

namespace {

constexpr size_t kScratchBytes = 8u << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (in host code the name
// g_scratch is only a host-side stand-in, never a device address).
gqa_status scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return GQA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GQA_OK;
}

}  // namespace

extern "C" gqa_status gqa_decode_attention_noalloc(const gqa_shape* shape, const void* q,
                                                   const void* k_cache, const void* v_cache,
                                                   const int32_t* block_tables,
                                                   const int32_t* context_lens, void* out,
                                                   int32_t* dev_status, void* stream) {
    if (!shape) return GQA_ERR_NULL;
    if (shape->T != 1) return GQA_ERR_SHAPE;  // decode: one new token per sequence
    gqa::AttnPlan plan;
    const gqa_status st = gqa::attention_plan(*shape, false, &plan);
    if (st != GQA_OK) return st;
    // the scratch of the kernel that serves the call (no engine is forced here)
    const bool tc = (shape->flags & GQA_FLAG_WARP_MMA) == 0 &&
                    ((shape->flags & GQA_FLAG_TENSOR_MEMORY) != 0 ||
                     gqa::tc_attention_preferred(*shape));
    const size_t need = tc ? gqa::tc_workspace_bytes(*shape, plan.flags_bytes) : plan.workspace;
    if (need == 0) return GQA_ERR_SHAPE;
    if (need > kScratchBytes) return GQA_ERR_WORKSPACE;  // beyond the fixed 8 MiB
    void* scratch = nullptr;
    const gqa_status ss = scratch_on_current_device(&scratch);
    if (ss != GQA_OK) return ss;
    // The tickets must read zero when the kernel starts.  A call that ended
    // normally left them zero, but one that timed out may not have.
    if (cudaMemsetAsync(scratch, 0, plan.flags_bytes, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return GQA_ERR_CUDA;
    return gqa_decode_attention(shape, q, k_cache, v_cache, block_tables, context_lens, out,
                                scratch, kScratchBytes, dev_status, stream);
}
