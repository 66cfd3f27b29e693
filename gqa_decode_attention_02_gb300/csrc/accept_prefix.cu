// accept_prefix.cu -- greedy longest-prefix acceptance of drafted tokens.
//
// Speculative-decoding section of "جعل inference رخيصًا: KV cache وbatching
// والتكميم": with greedy decoding a drafted token is accepted only if the target
// model would have produced it.  "Болжау арқылы Sonar модельдерін жылдамдату"
// §"Спекулятивті кодтан шығару": the longest accepted run is found, and the
// target's logits at the first mismatch (or after the last draft) supply one
// more token; §"Спекулятивті кодтан шығару арқылы инференс": doing this
// bookkeeping on the GPU avoids a GPU->CPU synchronisation, so the sequence
// length is updated here, on the device.
//
// One thread-block cluster per sequence.  The cluster's CS blocks split the
// vocabulary into CS column slices; each block reduces its slice of every row
// (several rows' 16-byte loads in flight at once) to a 64-bit argmax key
//     (order-preserving image of the value) << 32 | (~index)
// so that a plain max over keys picks the largest value and, among equal
// values, the smallest index; NaN maps above +inf (first NaN wins) and -0 is
// folded into +0.  Block r writes its key for row t into block 0's shared
// memory (distributed shared memory); after one cluster barrier block 0 takes
// the max over ranks, walks the drafts and writes the results.
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kMaxT = 64;
constexpr int kMaxCluster = 8;
constexpr int kThreads = 512;
constexpr int kRowsPerPass = 8;  // rows whose loads are in flight together

__device__ __forceinline__ unsigned long long argmax_key(float x, uint32_t idx) {
    uint32_t u = __float_as_uint(x);
    uint32_t o;
    if (x != x) {
        o = 0xffffffffu;
    } else {
        if (u == 0x80000000u) u = 0u;  // -0 == +0
        o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    return ((unsigned long long)o << 32) | (unsigned long long)(0xffffffffu - idx);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void st_remote_u64(const void* local, uint32_t rank,
                                              unsigned long long v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(remote), "l"(v) : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Cluster rank r reduces columns [r*S, min(V, (r+1)*S)) of every row of its
// sequence (S a multiple of 4): the T slices are loaded a few rows at a time
// with 16-byte loads (vec) or scalar loads, all of a pass in flight together.
template <bool kVec>
__global__ void __launch_bounds__(kThreads)
    accept_kernel(const float* __restrict__ logits, const int32_t* __restrict__ draft,
                  int32_t* accepted, int32_t* next_token, int32_t* ctx_io, int32_t* status,
                  int T, int V, int cs) {
    __shared__ unsigned long long table[kMaxT * kMaxCluster];  // used in rank 0
    __shared__ unsigned long long red[kThreads / 32][kRowsPerPass];
    __shared__ int sdraft[kMaxT];  // the drafts, fetched while the logits stream
    griddep_launch_dependents();
    griddep_wait();  // logits and lengths follow the previous kernels
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = (((V + cs - 1) / cs) + 3) & ~3;
    const int c_lo = min(V, (int)rank * S), c_hi = min(V, c_lo + S);
    const float* row0 = logits + (size_t)b * T * V;
    if (rank == 0 && tid < T - 1) sdraft[tid] = __ldg(draft + (size_t)b * (T - 1) + tid);
    // Block 0's shared memory may be written only once block 0 is running:
    // arrive now, wait before the first remote store.
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    for (int t0 = 0; t0 < T; t0 += kRowsPerPass) {
        unsigned long long key[kRowsPerPass];
#pragma unroll
        for (int i = 0; i < kRowsPerPass; ++i) key[i] = 0ull;  // below every real key
        if (kVec) {
            // columns c_lo + 4*(tid + k*kThreads), all rows of the pass; the
            // next column chunk's loads are issued before this one is reduced,
            // so two chunks are in flight (one DRAM round trip for two)
            const int step = 4 * kThreads;
            int c = c_lo + 4 * tid;
            float4 cur[kRowsPerPass], nxt[kRowsPerPass];
#pragma unroll
            for (int i = 0; i < kRowsPerPass; ++i)
                if (t0 + i < T && c < c_hi)
                    cur[i] = __ldg(reinterpret_cast<const float4*>(row0 + (size_t)(t0 + i) * V + c));
            for (; c < c_hi; c += step) {
                const int cn = c + step;
#pragma unroll
                for (int i = 0; i < kRowsPerPass; ++i)
                    if (t0 + i < T && cn < c_hi)
                        nxt[i] = __ldg(reinterpret_cast<const float4*>(row0 + (size_t)(t0 + i) * V + cn));
#pragma unroll
                for (int i = 0; i < kRowsPerPass; ++i) {
                    if (t0 + i < T) {
                        key[i] = umax64(key[i], argmax_key(cur[i].x, (uint32_t)c));
                        key[i] = umax64(key[i], argmax_key(cur[i].y, (uint32_t)c + 1));
                        key[i] = umax64(key[i], argmax_key(cur[i].z, (uint32_t)c + 2));
                        key[i] = umax64(key[i], argmax_key(cur[i].w, (uint32_t)c + 3));
                    }
                }
#pragma unroll
                for (int i = 0; i < kRowsPerPass; ++i) cur[i] = nxt[i];
            }
        } else {
            for (int c = c_lo + tid; c < c_hi; c += kThreads) {
#pragma unroll
                for (int i = 0; i < kRowsPerPass; ++i)
                    if (t0 + i < T)
                        key[i] = umax64(key[i],
                                        argmax_key(__ldg(row0 + (size_t)(t0 + i) * V + c),
                                                   (uint32_t)c));
            }
        }
#pragma unroll
        for (int i = 0; i < kRowsPerPass; ++i) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                key[i] = umax64(key[i], __shfl_xor_sync(0xffffffffu, key[i], o));
        }
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < kRowsPerPass; ++i) red[warp][i] = key[i];
        }
        if (t0 == 0) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        __syncthreads();
        if (tid < kRowsPerPass && t0 + tid < T) {
            unsigned long long k = 0ull;
            for (int wi = 0; wi < kThreads / 32; ++wi) k = umax64(k, red[wi][tid]);
            st_remote_u64(&table[(t0 + tid) * kMaxCluster + rank], 0, k);
        }
        __syncthreads();
    }
    cluster_sync_all();
    if (rank != 0 || tid != 0) return;
    int g[kMaxT];
    for (int t = 0; t < T; ++t) {
        unsigned long long k = 0ull;
        for (int r = 0; r < cs; ++r) k = umax64(k, table[t * kMaxCluster + r]);
        g[t] = (int)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
    }
    int a = 0;
    while (a < T - 1 && sdraft[a] == g[a]) ++a;
    accepted[b] = a;
    next_token[b] = g[a];
    if (ctx_io) {
        const int nc = ctx_io[b] - (T - 1 - a);
        if (nc < 0)
            report(status, GQA_ERR_CONTEXT);
        else
            ctx_io[b] = nc;
    }
}

}  // namespace

gqa_status launch_accept_prefix(int B, int T, int V, const float* logits, const int32_t* draft,
                                int32_t* accepted, int32_t* next_token, int32_t* ctx_io,
                                int32_t* dev_status, cudaStream_t stream) {
    if (B == 0) return GQA_OK;
    // one cluster of up to 8 blocks per sequence; each block takes V/cs columns
    int cs = (int)((V + 1023) / 1024);
    if (cs > kMaxCluster) cs = kMaxCluster;
    if (cs < 1) cs = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, B, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // 16-byte loads need every row to start on a 16-byte boundary
    const bool vec = (V % 4) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
    const cudaError_t e =
        vec ? cudaLaunchKernelEx(&cfg, accept_kernel<true>, logits, draft, accepted, next_token,
                                 ctx_io, dev_status, T, V, cs)
            : cudaLaunchKernelEx(&cfg, accept_kernel<false>, logits, draft, accepted, next_token,
                                 ctx_io, dev_status, T, V, cs);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
