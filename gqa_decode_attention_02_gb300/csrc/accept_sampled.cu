// accept_sampled.cu -- stochastic acceptance of drafted tokens (speculative
// sampling).
//
// "CS336, лекции 10 и 12: инференс и оценка моделей" §"Спекулятивное
// сэмплирование": rejection sampling with the draft model p as proposal and the
// target model q as target, modified to always emit a token.  Draft token x is
// kept with probability min(1, q(x)/p(x)); the first rejected position draws
// its replacement from max(q - p, 0); if every draft is kept, one more token is
// drawn from the target's last distribution.  The emitted tokens are exact
// samples of q.
//
// One thread-block cluster of CS <= 8 blocks per sequence; block k owns column
// slice k of the vocabulary and each of its threads a contiguous run of it:
//   1. every block evaluates the draft tests (u * p(x) < q(x) in double, an
//      exact product; a handful of loads) and takes the first rejection a;
//   2. each thread sums the integer weights W_v = floor(w_v * 2^40) of its run
//      of the row to draw from; the block reduces them to its slice total and
//      writes it into every block of the cluster (distributed shared memory);
//   3. after one cluster barrier every block knows S = sum of the slice totals,
//      r = floor(u * S) and the slice holding the crossing; that block scans
//      its thread sums and the thread whose run holds it finds the least v
//      with W_0 + ... + W_v > r.
// The weights are exact integers, so the sums do not depend on their order and
// the drawn index is the same whatever the thread layout.
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxT = 64;
constexpr int kMaxCluster = 8;
constexpr int kVecInFlight = 4;  // 16-byte loads of a run issued together

// floor(w * 2^40) for w in [0, 1], from the bits (exact; w <= 0 gives 0)
__device__ __forceinline__ unsigned long long fixed40(float w) {
    if (!(w > 0.f)) return 0ull;
    const uint32_t u = __float_as_uint(w);
    const int e = (int)(u >> 23);  // biased exponent, 0 for subnormals
    if (e == 0) return 0ull;       // below 2^-126: far below 2^-40
    const unsigned long long m = (unsigned long long)((u & 0x7fffffu) | 0x800000u);
    // w = m * 2^(e - 150)  ->  w * 2^40 = m * 2^(e - 110)
    const int sh = e - 110;
    if (sh >= 0) return m << sh;
    return (-sh >= 64) ? 0ull : (m >> -sh);
}

__device__ __forceinline__ float clean_prob(float x, bool& bad) {
    if (x >= 0.f && x <= 1.f) return x;
    bad = true;
    return 0.f;
}

// Weight of one column: the residual max(q - p, 0) (difference rounded once
// to fp32) when the draft row is used, else q itself.
__device__ __forceinline__ unsigned long long weight(float qv, float pv, bool resid, bool& bad) {
    float w = clean_prob(qv, bad);
    if (resid) {
        const float d = __fsub_rn(w, clean_prob(pv, bad));
        w = d > 0.f ? d : 0.f;
    }
    return fixed40(w);
}

__device__ __forceinline__ unsigned long long warp_incl_scan(unsigned long long x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void st_cluster_u64(const void* local, uint32_t rank,
                                               unsigned long long v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(remote), "l"(v) : "memory");
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Sum of the weights of columns [c, e) (e - c <= run length).  With kVec, c
// and e are multiples of 4 and the rows 16-byte aligned.
template <bool kVec>
__device__ __forceinline__ unsigned long long run_sum(const float* qrow, const float* prow,
                                                      bool resid, int c, int e, bool& bad) {
    unsigned long long s = 0ull;
    if (kVec) {
        for (; c < e; c += 4 * kVecInFlight) {
            float4 qv[kVecInFlight], pv[kVecInFlight];
#pragma unroll
            for (int i = 0; i < kVecInFlight; ++i) {
                qv[i] = pv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (c + 4 * i < e) {
                    qv[i] = __ldg(reinterpret_cast<const float4*>(qrow + c + 4 * i));
                    if (resid) pv[i] = __ldg(reinterpret_cast<const float4*>(prow + c + 4 * i));
                }
            }
#pragma unroll
            for (int i = 0; i < kVecInFlight; ++i) {
                if (c + 4 * i < e) {
                    s += weight(qv[i].x, pv[i].x, resid, bad);
                    s += weight(qv[i].y, pv[i].y, resid, bad);
                    s += weight(qv[i].z, pv[i].z, resid, bad);
                    s += weight(qv[i].w, pv[i].w, resid, bad);
                }
            }
        }
    } else {
        for (; c < e; ++c)
            s += weight(__ldg(qrow + c), resid ? __ldg(prow + c) : 0.f, resid, bad);
    }
    return s;
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads)
    accept_sampled_kernel(const float* __restrict__ q, const float* __restrict__ p,
                          const int32_t* __restrict__ draft, const double* __restrict__ u,
                          int32_t* accepted, int32_t* next_token, int32_t* ctx_io,
                          int32_t* status, int T, int V, int cs) {
    // slice totals of every block of the cluster, one table per draw attempt
    __shared__ unsigned long long s_tot[2][kMaxCluster];
    __shared__ unsigned long long s_warp[kWarps];
    __shared__ int s_first;
    __shared__ int s_bad;
    __shared__ unsigned char s_tbad[kMaxT];
    __shared__ double s_ufin;

    griddep_launch_dependents();
    griddep_wait();  // the probabilities come from the previous kernels
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.x / cs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Remote stores into a block may start only once it runs: arrive now, wait
    // before the first one.
    cluster_arrive();
    if (tid == 0) {
        s_first = T - 1;
        s_bad = 0;
    }
    __syncthreads();

    // ---- 1. every draft test at once; the first rejection wins ------------
    if (tid < T) {
        bool bad_u = false, bad_t = false;
        double ut = u[(size_t)b * T + tid];
        if (!(ut >= 0.0 && ut < 1.0)) {
            ut = 0.0;
            bad_u = true;
        }
        if (tid < T - 1) {
            const int x = draft[(size_t)b * (T - 1) + tid];
            bool keep = false;
            if (x >= 0 && x < V) {
                const double qx = clean_prob(q[((size_t)b * T + tid) * V + x], bad_t);
                const double px = clean_prob(p[((size_t)b * (T - 1) + tid) * V + x], bad_t);
                keep = __dmul_rn(ut, px) < qx;
            }
            if (!keep) atomicMin(&s_first, tid);
        } else {
            s_ufin = ut;
        }
        s_tbad[tid] = bad_t ? 1 : 0;  // counts only if this test was reached
        if (bad_u && rank == 0) s_bad = 1;
    }
    __syncthreads();
    const int a = s_first;
    if (tid == 0 && rank == 0)
        for (int t = 0; t <= a && t < T - 1; ++t)
            if (s_tbad[t]) s_bad = 1;

    // ---- 2./3. draw from the residual (or q), falling back to q once -----
    const float* qrow = q + ((size_t)b * T + a) * V;
    const float* prow = (a < T - 1) ? p + ((size_t)b * (T - 1) + a) * V : nullptr;
    const int slice = ((((V + cs - 1) / cs) + 3) / 4) * 4;
    const int c_lo = min(V, (int)rank * slice), c_hi = min(V, c_lo + slice);
    int run = (c_hi - c_lo + kThreads - 1) / kThreads;
    if (kVec) run = ((run + 3) / 4) * 4;
    const int r_lo = min(c_hi, c_lo + tid * run), r_hi = min(c_hi, r_lo + run);
    bool resid = prow != nullptr;
    bool empty = false;
    for (int attempt = 0; attempt < 2; ++attempt) {  // block- and cluster-uniform
        bool bad = false;
        const unsigned long long mine = run_sum<kVec>(qrow, prow, resid, r_lo, r_hi, bad);
        if (bad) s_bad = 1;
        // block scan of the thread sums (thread order is column order)
        const unsigned long long incl = warp_incl_scan(mine, lane);
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        unsigned long long slice_tot = 0ull;
        if (warp == 0) {
            const unsigned long long x = lane < kWarps ? s_warp[lane] : 0ull;
            const unsigned long long wi = warp_incl_scan(x, lane);
            slice_tot = __shfl_sync(0xffffffffu, wi, kWarps - 1);
            if (lane < kWarps) s_warp[lane] = wi - x;  // exclusive prefix of each warp
        }
        if (attempt == 0) cluster_wait();  // every block of the cluster is running
        if (warp == 0 && lane < cs) st_cluster_u64(&s_tot[attempt][rank], lane, slice_tot);
        cluster_arrive();
        cluster_wait();  // every slice total is in every block
        unsigned long long S = 0ull;
        for (int k = 0; k < cs; ++k) S += s_tot[attempt][k];
        if (S == 0ull) {
            if (resid) {  // vanishing residual: draw from q instead
                resid = false;
                continue;
            }
            empty = true;  // nothing to draw from at all
            break;
        }
        unsigned long long r = __double2ull_rz(__dmul_rn(s_ufin, __ull2double_rn(S)));
        if (r > S - 1ull) r = S - 1ull;
        unsigned long long base = 0ull;
        int kstar = cs - 1;
        for (int k = 0; k < cs; ++k) {
            const unsigned long long t = s_tot[attempt][k];
            if (base + t > r) {
                kstar = k;
                break;
            }
            base += t;
        }
        if ((int)rank == kstar) {
            const unsigned long long rr = r - base;  // offset inside this slice
            const unsigned long long ex = s_warp[warp] + (incl - mine);
            if (mine > 0ull && ex <= rr && rr < ex + mine) {  // exactly one thread
                unsigned long long cum = ex;
                int tok = r_hi - 1;
                bool dummy = false;
                for (int c = r_lo; c < r_hi; ++c) {
                    cum += weight(__ldg(qrow + c), resid ? __ldg(prow + c) : 0.f, resid, dummy);
                    if (cum > rr) {
                        tok = c;
                        break;
                    }
                }
                next_token[b] = tok;
            }
        }
        break;
    }

    __syncthreads();
    if (tid == 0) {
        bool bad = s_bad != 0;
        if (rank == 0) {
            if (empty) {
                next_token[b] = 0;
                bad = true;
            }
            accepted[b] = a;
            if (ctx_io) {
                const int nc = ctx_io[b] - (T - 1 - a);
                if (nc < 0)
                    report(status, GQA_ERR_CONTEXT);
                else
                    ctx_io[b] = nc;
            }
        }
        if (bad) report(status, GQA_ERR_PROBS);
    }
}

}  // namespace

gqa_status launch_accept_sampled(int B, int T, int V, const float* q, const float* p,
                                 const int32_t* draft, const double* u, int32_t* accepted,
                                 int32_t* next_token, int32_t* ctx_io, int32_t* dev_status,
                                 cudaStream_t stream) {
    // 16-byte loads need every row of q and p to start on a 16-byte boundary
    const bool vec = (V % 4) == 0 && (reinterpret_cast<uintptr_t>(q) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
    // one cluster of up to 8 blocks per sequence, about 8 columns per thread
    int cs = (int)((V + kThreads * 8 - 1) / (kThreads * 8));
    if (cs > kMaxCluster) cs = kMaxCluster;
    if (cs < 1) cs = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cs * B), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e =
        vec ? cudaLaunchKernelEx(&cfg, accept_sampled_kernel<true>, q, p, draft, u, accepted,
                                 next_token, ctx_io, dev_status, T, V, cs)
            : cudaLaunchKernelEx(&cfg, accept_sampled_kernel<false>, q, p, draft, u, accepted,
                                 next_token, ctx_io, dev_status, T, V, cs);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
