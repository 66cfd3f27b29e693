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
// One block of 1024 threads per sequence:
//   1. threads t < T evaluate every draft test at once (u * p(x) < q(x) in
//      double, an exact product) and the block takes the first rejection a;
//   2. each warp sums the integer weights W_v = floor(w_v * 2^40) of its
//      contiguous column segment of the row to draw from (16-byte loads when
//      rows are 16-byte aligned);
//   3. warp 0 scans the 32 segment sums, picks r = floor(u * S) and the
//      segment that holds the crossing; that warp re-reads its segment (now in
//      cache) and finds the least v with W_0 + ... + W_v > r.
// The weights are exact integers, so the sums do not depend on their order and
// the drawn index is the same whatever the thread layout.
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxT = 64;
constexpr int kGroup = 4;  // chunks of one warp whose loads are in flight together

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
// to fp32) when the draft row is given, else q itself.
template <bool kResid>
__device__ __forceinline__ unsigned long long weight(float qv, float pv, bool& bad) {
    float w = clean_prob(qv, bad);
    if (kResid) {
        const float d = __fsub_rn(w, clean_prob(pv, bad));
        w = d > 0.f ? d : 0.f;
    }
    return fixed40(w);
}

__device__ __forceinline__ unsigned long long warp_sum(unsigned long long x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ unsigned long long warp_incl_scan(unsigned long long x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Column layout of one warp's segment [lo, hi): chunk k covers kW*32 columns
// starting at lo + k*kW*32; lane l takes kW consecutive columns of the chunk.
// kW = 4 with 16-byte loads, 1 with scalar loads.
template <bool kVec>
struct Seg {
    static constexpr int kW = kVec ? 4 : 1;
    static constexpr int kChunk = 32 * kW;

    // lane's kW values of chunk starting at c (columns >= hi read as 0 weight)
    template <bool kResid>
    __device__ static void weights(const float* qrow, const float* prow, int c, int hi,
                                   unsigned long long (&w)[kW], bool& bad) {
        if (kVec) {
            float4 qv = make_float4(0.f, 0.f, 0.f, 0.f), pv = qv;
            if (c < hi) {  // hi is a multiple of 4 here
                qv = __ldg(reinterpret_cast<const float4*>(qrow + c));
                if (kResid) pv = __ldg(reinterpret_cast<const float4*>(prow + c));
            }
            const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
            const float pa[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
            for (int e = 0; e < kW; ++e)
                w[e] = (c < hi) ? weight<kResid>(qa[e], pa[e], bad) : 0ull;
        } else {
            w[0] = 0ull;
            if (c < hi) w[0] = weight<kResid>(__ldg(qrow + c), kResid ? __ldg(prow + c) : 0.f, bad);
        }
    }

    // Sum of the segment's weights (every lane gets it).
    template <bool kResid>
    __device__ static unsigned long long sum(const float* qrow, const float* prow, int lo,
                                             int hi, int lane, bool& bad) {
        unsigned long long s = 0ull;
        for (int c0 = lo; c0 < hi; c0 += kGroup * kChunk) {
            unsigned long long w[kGroup][kW];
#pragma unroll
            for (int g = 0; g < kGroup; ++g)
                weights<kResid>(qrow, prow, c0 + g * kChunk + lane * kW, hi, w[g], bad);
#pragma unroll
            for (int g = 0; g < kGroup; ++g)
#pragma unroll
                for (int e = 0; e < kW; ++e) s += w[g][e];
        }
        return warp_sum(s);
    }

    // Least column v of the segment with base + W_lo + ... + W_v > r (the
    // caller guarantees that the segment holds it).  Returns -1 if not found.
    template <bool kResid>
    __device__ static int find(const float* qrow, const float* prow, int lo, int hi, int lane,
                               unsigned long long base, unsigned long long r) {
        bool bad = false;  // already recorded by the sum pass
        for (int c = lo; c < hi; c += kChunk) {
            unsigned long long w[kW];
            weights<kResid>(qrow, prow, c + lane * kW, hi, w, bad);
            unsigned long long ls = 0ull;
#pragma unroll
            for (int e = 0; e < kW; ++e) ls += w[e];
            const unsigned long long incl = warp_incl_scan(ls, lane);
            const unsigned long long tot = __shfl_sync(0xffffffffu, incl, 31);
            const unsigned hit = __ballot_sync(0xffffffffu, base + incl > r);
            if (hit) {
                const int l = __ffs(hit) - 1;
                int v = -1;
                if (lane == l) {
                    unsigned long long cum = base + incl - ls;
#pragma unroll
                    for (int e = 0; e < kW; ++e) {
                        cum += w[e];
                        if (v < 0 && cum > r) v = c + lane * kW + e;
                    }
                }
                return __shfl_sync(0xffffffffu, v, l);
            }
            base += tot;
        }
        return -1;
    }
};

template <bool kVec>
__global__ void __launch_bounds__(kThreads)
    accept_sampled_kernel(const float* __restrict__ q, const float* __restrict__ p,
                          const int32_t* __restrict__ draft, const double* __restrict__ u,
                          int32_t* accepted, int32_t* next_token, int32_t* ctx_io,
                          int32_t* status, int T, int V) {
    using S = Seg<kVec>;
    __shared__ int s_first;
    __shared__ int s_bad;
    __shared__ unsigned char s_tbad[kMaxT];
    __shared__ double s_ufin;
    __shared__ unsigned long long s_wsum[kWarps];
    __shared__ int s_wstar, s_resid, s_tok;
    __shared__ unsigned long long s_base, s_r;

    griddep_launch_dependents();
    griddep_wait();  // the probabilities come from the previous kernels
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
        if (bad_u) s_bad = 1;
    }
    __syncthreads();
    const int a = s_first;
    if (tid == 0) {
        for (int t = 0; t <= a && t < T - 1; ++t)
            if (s_tbad[t]) s_bad = 1;
        s_resid = (a < T - 1) ? 1 : 0;
    }
    __syncthreads();

    // ---- 2./3. draw from the residual (or q), falling back to q once -----
    const float* qrow = q + ((size_t)b * T + a) * V;
    const float* prow = (a < T - 1) ? p + ((size_t)b * (T - 1) + a) * V : nullptr;
    const int seg = ((((V + kWarps - 1) / kWarps) + 3) / 4) * 4;
    const int lo = min(V, warp * seg), hi = min(V, lo + seg);
    int tok = -1;
    for (int attempt = 0; attempt < 2; ++attempt) {
        const bool resid = s_resid != 0;  // block-uniform
        bool bad = false;
        const unsigned long long ws = resid ? S::template sum<true>(qrow, prow, lo, hi, lane, bad)
                                            : S::template sum<false>(qrow, prow, lo, hi, lane, bad);
        if (lane == 0) s_wsum[warp] = ws;
        if (bad) s_bad = 1;
        __syncthreads();
        if (warp == 0) {
            const unsigned long long x = s_wsum[lane];
            const unsigned long long incl = warp_incl_scan(x, lane);
            const unsigned long long tot = __shfl_sync(0xffffffffu, incl, 31);
            if (tot == 0ull) {
                if (lane == 0) {
                    s_wstar = -1;
                    if (resid)
                        s_resid = 0;  // vanishing residual: draw from q instead
                    else
                        s_bad = 1;    // nothing to draw from at all
                }
            } else {
                unsigned long long r = (unsigned long long)__double2ull_rz(
                    __dmul_rn(s_ufin, __ull2double_rn(tot)));
                if (r > tot - 1ull) r = tot - 1ull;
                const unsigned hit = __ballot_sync(0xffffffffu, incl > r);
                const int l = __ffs(hit) - 1;
                if (lane == l) {
                    s_wstar = l;
                    s_base = incl - x;
                    s_r = r;
                }
            }
        }
        __syncthreads();
        const int wstar = s_wstar;
        if (wstar >= 0) {
            if (warp == wstar) {
                const int v = resid ? S::template find<true>(qrow, prow, lo, hi, lane, s_base, s_r)
                                    : S::template find<false>(qrow, prow, lo, hi, lane, s_base, s_r);
                if (lane == 0) s_tok = v;
            }
            __syncthreads();
            tok = s_tok;
            break;
        }
        if (!resid || s_resid != 0) break;  // nothing left to try
        __syncthreads();  // every thread has read s_resid before the next round
    }

    if (tid == 0) {
        int bad = s_bad;
        if (tok < 0) {
            tok = 0;
            bad = 1;
        }
        accepted[b] = a;
        next_token[b] = tok;
        if (bad) report(status, GQA_ERR_PROBS);
        if (ctx_io) {
            const int nc = ctx_io[b] - (T - 1 - a);
            if (nc < 0)
                report(status, GQA_ERR_CONTEXT);
            else
                ctx_io[b] = nc;
        }
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e =
        vec ? cudaLaunchKernelEx(&cfg, accept_sampled_kernel<true>, q, p, draft, u, accepted,
                                 next_token, ctx_io, dev_status, T, V)
            : cudaLaunchKernelEx(&cfg, accept_sampled_kernel<false>, q, p, draft, u, accepted,
                                 next_token, ctx_io, dev_status, T, V);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
