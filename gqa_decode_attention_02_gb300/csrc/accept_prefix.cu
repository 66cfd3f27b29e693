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
// Every row's argmax is a max over 64-bit keys
//     (order-preserving image of the value) << 32 | (~index)
// so that one max picks the largest value and, among equal values, the
// smallest index; NaN maps above +inf (first NaN wins) and -0 is folded into
// +0.  A max over keys does not depend on the order it is taken in, so any
// split of the columns gives the same result.
//
// Greedy acceptance over a draft tree ("Болжау арқылы Sonar модельдерін
// жылдамдату" §"EAGLE": the longest branch of candidates the target agrees
// with is kept, plus one token from the target) shares the argmax pass and
// differs only in the last step (finish_acceptance).
//
// Two kernels compute the same thing:
//  * accept_grid_kernel (with a workspace): S thread blocks per sequence, S
//    chosen so that the whole batch is ~4 blocks per SM; block r reduces
//    columns [r*W, (r+1)*W) of all T rows of its sequence with every load of
//    the slice in flight at once, stores its T keys in its own workspace
//    slots and takes a ticket (an acq_rel atomicAdd on the sequence's
//    counter); the block that draws the last ticket takes the max of the S
//    blocks' keys (zeroing their slots), walks the drafts, writes the results
//    and resets the counter.  No block ever waits for another.
//  * accept_kernel (no workspace): one thread-block cluster of up to 8 blocks
//    per sequence; block r writes its keys into block 0's shared memory
//    (distributed shared memory) and, after one cluster barrier, block 0
//    takes the max over ranks and walks the drafts.
#include <cuda_runtime.h>

#include <algorithm>

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

// The last step, by one thread once every row's argmax is known (g_of(t));
// depth: shared scratch of kMaxT ints.
// Chain (tree == false): a = the longest run of drafts equal to the target's
// choices, next = g_a.  Tree: node i >= 1 (parent spar[i] < i, token
// sdraft[i-1]) is kept iff its parent is kept and its token is the target's
// choice at the parent; a node with a parent entry outside [0, i) is never
// kept (GQA_ERR_TREE, also for a root entry other than -1).  The kept node m
// of greatest depth, the lowest index among equals, ends the accepted
// branch: a = depth(m), path = the branch's nodes below the root by depth
// (then -1), next = g_m.  Both: context_lens[b] -= T-1-a unless that drops
// below zero (GQA_ERR_CONTEXT, the length unchanged).
template <typename GOf>
__device__ void finish_acceptance(int b, int T, bool tree, const int* sdraft, const int* spar,
                                  int* depth, GOf g_of, int32_t* accepted, int32_t* next_token,
                                  int32_t* path, int32_t* ctx_io, int32_t* status) {
    int a = 0, m = 0;
    if (!tree) {
        while (a < T - 1 && sdraft[a] == g_of(a)) ++a;
        m = a;
    } else {
        unsigned long long kept = 1ull;  // bit i: node i kept (the root always)
        bool bad = spar[0] != -1;
        depth[0] = 0;
        for (int i = 1; i < T; ++i) {
            const int p = spar[i];
            depth[i] = 0;
            if (p < 0 || p >= i) {
                bad = true;
                continue;
            }
            depth[i] = depth[p] + 1;
            if (((kept >> p) & 1ull) && sdraft[i - 1] == g_of(p)) {
                kept |= 1ull << i;
                if (depth[i] > a) {  // strict: the lower index keeps a tie
                    a = depth[i];
                    m = i;
                }
            }
        }
        if (bad) report(status, GQA_ERR_TREE);
        int32_t* pb = path + (size_t)b * (T - 1);
        int cur = m;
        for (int j = a - 1; j >= 0; --j) {
            pb[j] = cur;
            cur = spar[cur];
        }
        for (int j = a; j < T - 1; ++j) pb[j] = -1;
    }
    accepted[b] = a;
    next_token[b] = g_of(m);
    if (ctx_io) {
        const int nc = ctx_io[b] - (T - 1 - a);
        if (nc < 0)
            report(status, GQA_ERR_CONTEXT);
        else
            ctx_io[b] = nc;
    }
}

// Cluster rank r reduces columns [r*S, min(V, (r+1)*S)) of every row of its
// sequence (S a multiple of 4): the T slices are loaded a few rows at a time
// with 16-byte loads (vec) or scalar loads, all of a pass in flight together.
template <bool kVec>
__global__ void __launch_bounds__(kThreads)
    accept_kernel(const float* __restrict__ logits, const int32_t* __restrict__ draft,
                  const int32_t* __restrict__ parents, int32_t* accepted, int32_t* next_token,
                  int32_t* path, int32_t* ctx_io, int32_t* status, int T, int V, int cs) {
    __shared__ unsigned long long table[kMaxT * kMaxCluster];  // used in rank 0
    __shared__ unsigned long long red[kThreads / 32][kRowsPerPass];
    __shared__ int sdraft[kMaxT];  // the drafts, fetched while the logits stream
    __shared__ int spar[kMaxT];    // the tree's parent entries (tree acceptance)
    __shared__ int sdepth[kMaxT];  // node depths (tree acceptance, thread 0 of rank 0)
    griddep_launch_dependents();
    griddep_wait();  // logits and lengths follow the previous kernels
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = (((V + cs - 1) / cs) + 3) & ~3;
    const int c_lo = min(V, (int)rank * S), c_hi = min(V, c_lo + S);
    const float* row0 = logits + (size_t)b * T * V;
    if (rank == 0 && tid < T - 1) sdraft[tid] = __ldg(draft + (size_t)b * (T - 1) + tid);
    if (parents && rank == 0 && tid < T) spar[tid] = __ldg(parents + (size_t)b * T + tid);
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
    auto g_of = [&](int t) {
        unsigned long long k = 0ull;
        for (int r = 0; r < cs; ++r) k = umax64(k, table[t * kMaxCluster + r]);
        return (int)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
    };
    finish_acceptance(b, T, parents != nullptr, sdraft, spar, sdepth, g_of, accepted, next_token,
                      path, ctx_io, status);
}


// ---- many blocks per sequence, keys meeting in the workspace ----------------------
constexpr int kGridThreads = 256;
constexpr int kLoadsInFlight = 8;  // loads of one thread issued before any is reduced
constexpr int kBlocksPerSm = 4;    // blocks of the whole launch per SM (the register file holds 4)
constexpr int kSplitSms = 256;     // SMs counted at most (keeps the workspace size device-free)

// The most blocks per sequence (sizes the workspace, whatever the device).
long long accept_max_split(int B) {
    return std::max<long long>(1, ((long long)kBlocksPerSm * kSplitSms + B - 1) / B);
}
// Blocks per sequence for B sequences of V columns on `sms` SMs, and the
// columns each takes (a multiple of 4, at least 256 unless V is smaller).
void accept_split(int B, int V, int sms, int* S_out, int* W_out) {
    const long long n = (long long)kBlocksPerSm * std::min(sms, kSplitSms);
    long long S = std::max<long long>(1, (n + B - 1) / B);
    S = std::min<long long>(S, std::max(1, V / 256));
    int W = (int)((V + S - 1) / S);
    W = (W + 3) & ~3;
    *S_out = (V + W - 1) / W;
    *W_out = W;
}

// Ticket of a sequence (GPU scope, acq_rel): the block's key stores precede
// it (ordered by __syncthreads before thread 0 takes it); the block that
// draws the last ticket has acquired every other block's stores.
__device__ __forceinline__ unsigned seq_ticket(unsigned* t) {
    unsigned v;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(v) : "l"(t) : "memory");
    return v;
}

// Block (b, r) = blockIdx.x / S, blockIdx.x % S reduces columns
// [r*W, min(V, (r+1)*W)) of rows 0..T-1 of sequence b to T keys, stores them
// in its own slots parts[b][r][0..T-1] and takes a ticket; the block that
// draws the last ticket of b folds the S blocks' keys and walks the drafts.
// The workspace (tickets [B], then parts [B][S][T]) is zero when the kernel
// starts and zero again when it ends.
template <bool kVec>
__global__ void __launch_bounds__(kGridThreads)
    accept_grid_kernel(const float* __restrict__ logits, const int32_t* __restrict__ draft,
                       const int32_t* __restrict__ parents, int32_t* accepted,
                       int32_t* next_token, int32_t* path, int32_t* ctx_io, int32_t* status,
                       unsigned* tickets, unsigned long long* parts, int T, int V, int S, int W) {
    __shared__ unsigned long long red[kGridThreads / 32][kMaxT];
    __shared__ unsigned long long skey[kMaxT];
    __shared__ int sdraft[kMaxT];
    __shared__ int spar[kMaxT];
    __shared__ int sdepth[kMaxT];
    __shared__ int s_last;
    griddep_launch_dependents();
    griddep_wait();  // logits and lengths follow the previous kernels
    const int b = blockIdx.x / S, r = blockIdx.x - b * S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kCols = kVec ? 4 : 1;          // columns per load
    constexpr int kSpan = kCols * kGridThreads;  // columns per chunk of a row
    const int c_lo = r * W, c_hi = min(V, c_lo + W);
    const int nch = (c_hi - c_lo + kSpan - 1) / kSpan;  // chunks per row (>= 1)
    const int items = T * nch;                          // (row, chunk) pairs, row-major
    const float* row0 = logits + (size_t)b * T * V;
    // this thread's draft id (for the last block's walk), in flight with the logits
    const int my_draft = (tid < T - 1) ? __ldg(draft + (size_t)b * (T - 1) + tid) : 0;
    const int my_parent = (parents && tid < T) ? __ldg(parents + (size_t)b * T + tid) : 0;
    // Per row, this thread's running argmax over its columns, which it visits
    // in increasing order: (bv, bi) is replaced by (x, c) iff bv is not NaN and
    // !(x <= bv) -- x larger, or x NaN -- so the first NaN wins, then the
    // largest value, and among equal values (-0 == +0) the first index.
    float bv = 0.f;
    uint32_t bi = 0xffffffffu;  // no column yet
    int t = 0, ch = 0;          // (row, chunk) of the next item; block-uniform
    auto visit = [&](float x, uint32_t c) {
        if (bi == 0xffffffffu || (bv == bv && !(x <= bv))) {
            bv = x;
            bi = c;
        }
    };
    // End of a row: the warp's argmax (the largest ordered value, then the
    // smallest index holding it), as a 64-bit key, into red[warp][row].
    auto flush = [&](int row) {
        uint32_t o = 0u;  // below every ordered value: a thread with no column
        if (bi != 0xffffffffu) {
            uint32_t u = __float_as_uint(bv);
            if (bv != bv) u = 0x7fffffffu;           // every NaN above +inf
            if (u == 0x80000000u) u = 0u;             // -0 == +0
            o = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);  // order-preserving
        }
        const uint32_t wo = __reduce_max_sync(0xffffffffu, o);
        const uint32_t wi = __reduce_min_sync(0xffffffffu, o == wo ? bi : 0xffffffffu);
        if (lane == 0) red[warp][row] = ((unsigned long long)wo << 32) | (0xffffffffu - wi);
        bi = 0xffffffffu;
    };
    for (int i0 = 0; i0 < items; i0 += kLoadsInFlight) {
        float4 v[kLoadsInFlight];
        {
            int tt = t, cc = ch;
#pragma unroll
            for (int j = 0; j < kLoadsInFlight; ++j) {
                const int c = c_lo + kCols * tid + cc * kSpan;
                if (i0 + j < items && c < c_hi) {
                    const float* src = row0 + (size_t)tt * V + c;
                    if (kVec)
                        v[j] = __ldg(reinterpret_cast<const float4*>(src));
                    else
                        v[j].x = __ldg(src);
                }
                if (++cc == nch) {
                    cc = 0;
                    ++tt;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kLoadsInFlight; ++j) {
            if (i0 + j < items) {
                const int c = c_lo + kCols * tid + ch * kSpan;
                if (c < c_hi) {
                    visit(v[j].x, (uint32_t)c);
                    if (kVec) {
                        visit(v[j].y, (uint32_t)c + 1);
                        visit(v[j].z, (uint32_t)c + 2);
                        visit(v[j].w, (uint32_t)c + 3);
                    }
                }
                if (++ch == nch) {  // the row is done
                    flush(t);
                    ch = 0;
                    ++t;
                }
            }
        }
    }
    if (tid < T - 1) sdraft[tid] = my_draft;
    if (tid < T) spar[tid] = my_parent;
    __syncthreads();
    // this block's key of each row into its own slot
    for (int t = tid; t < T; t += kGridThreads) {
        unsigned long long k = 0ull;
#pragma unroll
        for (int wi = 0; wi < kGridThreads / 32; ++wi) k = umax64(k, red[wi][t]);
        parts[((size_t)b * S + r) * T + t] = k;
    }
    __syncthreads();
    if (tid == 0) s_last = seq_ticket(tickets + b) == (unsigned)(S - 1);
    __syncthreads();
    if (!s_last) return;
    // The last block of sequence b: every block's keys are in (thread 0's
    // acquire, then the barrier, order these loads after them).  Warp w folds
    // rows w, w + 8, ...; the slots are zeroed behind the reads, so every call
    // leaves the whole workspace zero-filled and calls of other sizes can
    // share it.
    unsigned long long* pb = parts + (size_t)b * S * T;
    for (int row = warp; row < T; row += kGridThreads / 32) {
        unsigned long long k = 0ull;
        for (int r0 = 0; r0 < S; r0 += 64) {  // two loads in flight per lane
            const int ra = r0 + lane, rb = r0 + 32 + lane;
            const unsigned long long ka = ra < S ? __ldcg(pb + (size_t)ra * T + row) : 0ull;
            const unsigned long long kb = rb < S ? __ldcg(pb + (size_t)rb * T + row) : 0ull;
            if (ra < S) pb[(size_t)ra * T + row] = 0ull;
            if (rb < S) pb[(size_t)rb * T + row] = 0ull;
            k = umax64(k, umax64(ka, kb));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) k = umax64(k, __shfl_xor_sync(0xffffffffu, k, o));
        if (lane == 0) skey[row] = k;
    }
    __syncthreads();
    if (tid != 0) return;
    tickets[b] = 0u;  // ready for the next call
    auto g_of = [&](int t) { return (int)(0xffffffffu - (uint32_t)(skey[t] & 0xffffffffull)); };
    finish_acceptance(b, T, parents != nullptr, sdraft, spar, sdepth, g_of, accepted, next_token,
                      path, ctx_io, status);
}

}  // namespace

size_t accept_workspace_bytes(int B, int T) {
    if (B < 0 || T < 1 || T > kMaxT) return 0;
    const size_t tickets = ((size_t)B * 4 + 15) / 16 * 16;
    const size_t parts = 8 * (size_t)T * B * (size_t)accept_max_split(B);
    return std::max<size_t>(16, tickets + parts);
}

gqa_status launch_accept_prefix(int B, int T, int V, const float* logits, const int32_t* draft,
                                const int32_t* parents, int32_t* accepted, int32_t* next_token,
                                int32_t* path, int32_t* ctx_io, void* workspace,
                                int32_t* dev_status, cudaStream_t stream) {
    if (B == 0) return GQA_OK;
    // 16-byte loads need every row to start on a 16-byte boundary
    const bool vec = (V % 4) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
    if (workspace) {
        const int sms = device_sm_count();
        if (sms < 1) return GQA_ERR_CUDA;
        int S = 1, W = V;
        accept_split(B, V, sms, &S, &W);
        if ((long long)B * S > 0x7fffffffll) return GQA_ERR_SHAPE;
        unsigned* tickets = static_cast<unsigned*>(workspace);
        unsigned long long* parts = reinterpret_cast<unsigned long long*>(
            static_cast<uint8_t*>(workspace) + ((size_t)B * 4 + 15) / 16 * 16);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(B * S), 1, 1);
        cfg.blockDim = dim3(kGridThreads, 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cfg.attrs = nullptr;
        cfg.numAttrs = 0;
        const cudaError_t e =
            vec ? cudaLaunchKernelEx(&cfg, accept_grid_kernel<true>, logits, draft, parents,
                                     accepted, next_token, path, ctx_io, dev_status, tickets,
                                     parts, T, V, S, W)
                : cudaLaunchKernelEx(&cfg, accept_grid_kernel<false>, logits, draft, parents,
                                     accepted, next_token, path, ctx_io, dev_status, tickets,
                                     parts, T, V, S, W);
        return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
    }
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
    const cudaError_t e =
        vec ? cudaLaunchKernelEx(&cfg, accept_kernel<true>, logits, draft, parents, accepted,
                                 next_token, path, ctx_io, dev_status, T, V, cs)
            : cudaLaunchKernelEx(&cfg, accept_kernel<false>, logits, draft, parents, accepted,
                                 next_token, path, ctx_io, dev_status, T, V, cs);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
