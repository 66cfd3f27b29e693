// attention.cu -- paged grouped-query decode / verify attention for sm_103a.
//
// What it computes (CS336 lecture 10, Russian translation, §"Арифметическая
// интенсивность инференса" and §"Уменьшаем KV-кэш"; paged reads from
// §"PagedAttention"): for sequence b, new token t < T and query head n, with KV
// head k = n / G,
//     s_j = scale * <q[b,t,n,:], K_b[j,k,:]>   for j <= ctx_b - T + t
//     out[b,t,n,:] = sum_j softmax(s)_j V_b[j,k,:]
// where K_b[j] / V_b[j] is row j % 16 of physical block block_tables[b][j/16].
//
// Why it is shaped this way.  The same section derives that decode attention
// reads every cached key and value once and does only ~1 flop per byte per
// query row, so HBM bandwidth bounds it whatever the batch; with GQA the G
// query heads of one KV head (times the T new tokens) share each K/V byte, so
// all T*G rows of a KV head are processed together and every KV byte crosses
// HBM once.
//
// Structure of one CTA (persistent; grid = SMs x resident CTAs):
//  * Work order.  The tiles of the whole batch are laid out as segments
//    (b, k) in b-major order, each segment being a few start-up units and
//    then ceil(ctx_b/16) tiles of 16 tokens (one cache block of one KV head).
//    CTA c takes the contiguous range [c*quota, (c+1)*quota) of those units,
//    so every CTA streams about the same bytes and pays about the same
//    per-segment costs however ragged the context lengths are.  A segment cut by
//    a range boundary is finished by merging its pieces with log-sum-exp
//    weights -- the context split of FlashDecoding (named in §"PagedAttention"),
//    balanced over the whole batch.  Every CTA derives the plan from
//    context_lens itself (one warp scan), so the host never reads device data.
//  * One producer warp walks the range in stages of up to four consecutive
//    tiles of one segment, reads block ids 32 at a time and issues TMA tiled
//    loads (3-D view [blocks*16 rows][K][H], box 16 rows x 64 elements,
//    128-byte swizzle) of the K and V tiles into a ring of stages.  Each stage
//    has a metadata barrier, armed as soon as the stage's description is
//    written (so consumers can fetch q for a new segment while the tiles are
//    in flight), and a data barrier completed by the TMA transaction count.
//  * Consumer warp w owns query rows 8w..8w+7 (rows r = t*G + g).  Per stage
//    it computes S^T[16 tokens x 8 rows] = K_tile . Q^T for every tile with
//    mma.sync m16n8k16 (tokens on M, so no tensor-core rows are wasted on a
//    small G; the tiles give independent mma chains), keeps a running max /
//    sum in the log2 domain (rescaling the accumulator only when the max grows
//    by more than 2^8, which leaves the result unchanged up to rounding),
//    transposes P in registers with movmatrix and accumulates
//    O^T[H x 8 rows] += V_tile^T . P^T, again on mma.sync.
//  * Stage-parallel consumer groups: group g computes the stages whose index
//    is g modulo the group count; at a segment boundary the groups' states
//    meet in shared memory and group 0 finishes the segment.
//  * A finished segment is written directly when the CTA owns all of it.  Of
//    a split segment, every piece's row warp publishes its partial result and
//    takes a ticket (an acq_rel atomicAdd on the segment's counter); the warp
//    that draws the last ticket folds all pieces in piece order (the same
//    arithmetic whichever CTA it runs in: a deterministic result), stores the
//    rows and resets the counter.  No CTA ever waits for another, so the
//    result does not depend on which CTAs are resident at the same time.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "launch.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kMaxRowWarps = 6;            // query rows per chunk <= 48
constexpr long long kMaxRows = 8192;       // T*G: above 48 the rows go in chunks
constexpr int kGroups = 2;                 // stage-parallel consumer groups (default)
constexpr int kMaxThreads = 32 * (kGroups * kMaxRowWarps + 1);
constexpr int kEnd = 1, kBad = 2;
constexpr int kTilesPerStage = 4;          // cache blocks per pipeline stage (2-byte cache)
constexpr int kMaxTilesPerStage = 8;       // ... and over one-byte codes
constexpr int kQuotaMin = 2 * kTilesPerStage;  // units per CTA at least: fewer split pieces
// Start-up cost of a segment in the work partition, in tiles: a segment
// occupies kSegUnits units and then its tiles, so a CTA that starts many
// (short) segments -- each with its q rows, new rows and epilogue -- streams
// fewer tiles.
constexpr int kSegUnits = 6;
constexpr float kRescaleGap = 8.0f;        // log2-domain slack before rescaling
constexpr long long kMaxFlags = 65536;     // CTAs * row warps per launch

struct AttnParams {
    const void* q;
    void* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* partials;
    int32_t* flags;  // tickets: per (CTA holding a split segment's first piece, row warp)
    int32_t* status;
    int B, T, N, K, G, R, nt;  // nt: row warps per consumer group
    // Row chunks: the R = T*G query rows of a KV head are split into C chunks
    // of Rc rows; the pair (KV head k, chunk c) is the virtual head k*C + c,
    // KC = K*C of them, each its own segment over the same cache blocks.
    int C, Rc, KC;
    int max_blocks, num_blocks;
    float scale_log2;
    int stages;    // depth of the shared-memory ring
    int groups;    // stage-parallel consumer groups
    int early_kv;  // GQA_FLAG_EARLY_KV: stream old cache blocks before the wait
    int window;    // local attention: each query sees its last `window` positions (0: all)
    // Tree verification: new token t sees new token j < t only if bit j of
    // tree_mask[b * T + t] is set (nullptr: the chain, all j < t).
    const uint64_t* tree_mask;
    // One-byte caches: fp32 scale of every cached row, [num_blocks][K][16].
    const float* k_scale;
    const float* v_scale;
    // Fused append (k_new != nullptr): the T newest positions are taken from
    // k_new / v_new [B][T][K][H] and written into the caches by this kernel.
    const void* k_new;
    const void* v_new;
    void* k_cache;
    void* v_cache;
};

// Description of one pipeline stage, written by the producer.
template <int NT>
struct StageMetaT {
    int b, k, blk_i, ntiles;  // segment (b, k); its tiles blk_i .. blk_i+ntiles-1
    int ctx, seg_start, nblk, quota;  // seg_start: partition unit of the segment's first tile
    int cta_start, flags, pad0, pad1;
    int blk[NT];  // physical block of each tile
};

// KVQ: cache element kind -- 0: the dtype of q (2 bytes), GQA_KV_INT8 /
// GQA_KV_E4M3: one-byte codes with an fp32 scale per cached row.
template <int H, int KVQ = 0>
struct Cfg {
    static constexpr int kElemBytes = KVQ ? 1 : 2;
    static constexpr int kTileBytes = 16 * H * kElemBytes;  // 16 tokens x H elements
    static constexpr int kScaleBytes = KVQ ? 16 * 4 : 0;      // the tile's row scales
    // tiles per stage (one-byte stages with eight tiles were measured slower:
    // twice the shared memory per CTA)
    static constexpr int kTiles = kTilesPerStage;
    // K tiles, V tiles (then K scales, V scales), rounded to the 1 KB alignment
    // of a 128-byte-swizzled TMA destination
    static constexpr int kStageBytes =
        (2 * kTiles * (kTileBytes + kScaleBytes) + 1023) / 1024 * 1024;
    // Ring depth: two CTAs per SM fit at H = 128; at H = 64 four stages let
    // three fit (the 24-layer batch of short contexts ran 272 us per step,
    // against 283 with six stages and two CTAs).  One-byte caches: the deepest
    // ring tried (the launch takes the depth that fits the most CTAs per SM).
    static constexpr int kStages = KVQ ? 4 : (H == 128) ? 3 : 4;
    static constexpr int kHalves = KVQ ? 1 : H / 64;  // 128-byte swizzle spans per row
    static constexpr int kSteps = H / 16;  // k16 steps of QK^T == m16 tiles of PV
    static constexpr int kAccFloats = H / 4;  // accumulator floats per lane
    static constexpr int kHeaderFloats = 32;  // m[8], l[8], flag, pad
    static constexpr int kSectionFloats = kHeaderFloats + 32 * kAccFloats;
    // stages, barriers (full/meta/empty per stage + combine), stage
    // descriptions, abort flag; the combine scratch is added per launch
    using Meta = StageMetaT<kTiles>;  // one stage's description
    static constexpr size_t kStageOverhead = 24 + sizeof(Meta);  // barriers + meta
    static constexpr size_t kFixed = 1024 + 8 + 64;  // alignment, combine barrier, flag
    static constexpr size_t kScratchBytesPerRowWarp =
        2 * 32 * (4 + kAccFloats) * sizeof(float);  // per row warp of each extra group
};

// First logical block a segment reads: the one holding the earliest position
// any of the T new tokens sees (0 without a window).
__device__ __forceinline__ int first_block(int ctx, int T, int window) {
    return window > 0 ? max(0, ctx - T - window + 1) >> 4 : 0;
}

// Tiles (cache blocks) of one (b, k) segment; 0 for an invalid context length.
__device__ __forceinline__ int seq_blocks(int ctx, int T, int max_blocks, int window) {
    return (ctx >= T && ctx >= 1 && ctx <= max_blocks * 16)
               ? ((ctx + 15) >> 4) - first_block(ctx, T, window)
               : 0;
}
// Partition units of a segment of nblk tiles: its start-up units, then its tiles.
__device__ __forceinline__ int seg_units(int nblk) { return nblk > 0 ? nblk + kSegUnits : 0; }

// Zero the outputs of one sequence (T x N x H elements of 2 bytes).
template <int H>
__device__ void zero_sequence(const AttnParams& p, int b) {
    const size_t n16 = (size_t)p.T * p.N * H * 2 / 16;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + (size_t)b * n16 * 16);
    for (size_t i = 0; i < n16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
}

// Tickets of split segments (GPU scope): every piece's warp stores its
// partial result, then (after __syncwarp, which orders its lanes' stores
// before lane 0) takes a ticket with an acq_rel atomic; the warp that draws
// the last ticket has acquired every earlier piece's stores.
__device__ __forceinline__ unsigned ticket_acq_rel(int32_t* t) {
    unsigned v;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(v)
                 : "l"(t)
                 : "memory");
    return v;
}
// Tickets drawn so far (acquire: the pieces that drew them are visible).
__device__ __forceinline__ unsigned ticket_seen(const int32_t* t) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(t) : "memory");
    return v;
}

// Barriers of one CTA.
struct Bars {
    uint64_t* full;   // data landed (TMA transaction count)
    uint64_t* meta;   // stage description written
    uint64_t* empty;  // every consumer warp is done with the stage
    uint64_t* cbar;   // consumer groups' states written to the combine scratch
};

// L2 prefetch of the q rows segment (b, k) will read: for each new token t,
// the G query heads of KV head k are contiguous (G*H elements).
template <int H>
__device__ __forceinline__ void prefetch_q(const AttnParams& p, int b, int k) {
    const uint16_t* base = static_cast<const uint16_t*>(p.q);
    for (int t = 0; t < p.T; ++t)
        prefetch_l2(base + (((size_t)b * p.T + t) * p.N + (size_t)k * p.G) * H,
                    (uint32_t)(p.G * H * 2));
}

// ---------------------------------------------------------------------------
template <int H, bool GENERAL, int KVQ>
__device__ void producer(const CUtensorMap* tmk, const CUtensorMap* tmv, const AttnParams& p,
                         uint8_t* stages, const Bars& bar, typename Cfg<H, KVQ>::Meta* meta,
                         volatile int* abort_flag) {
    using C = Cfg<H, KVQ>;
    const int win = GENERAL ? p.window : 0;  // compile-time 0 for the plain kernel
    const int nC = GENERAL ? p.C : 1;        // row chunks (1 in the plain kernel)
    const int nKC = GENERAL ? p.KC : p.K;    // virtual heads
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        tma_prefetch_desc(tmk);
        tma_prefetch_desc(tmv);
    }
    // Without the early-KV promise every global access waits for the grids
    // this launch depends on; with it, context_lens, block_tables and the
    // cache below position ctx - T may be read first, and the wait happens
    // before the first stage that holds one of the T newest positions and
    // before any write.
    bool waited = false;
    if (!p.early_kv) {
        griddep_wait();
        waited = true;
    }
    // 1. Partition units per sequence and their prefix sum (lane l owns a run of b).
    const int per = (p.B + 31) / 32;
    const int lo = min(p.B, lane * per), hi = min(p.B, lo + per);
    int local = 0;
    bool invalid = false;
    for (int b = lo; b < hi; ++b) {
        const int n = seq_blocks(p.context_lens[b], p.T, p.max_blocks, win);
        local += seg_units(n);
        invalid |= (n == 0);
    }
    if (blockIdx.x == 0 && __any_sync(FULL, invalid)) {
        if (!waited) {
            griddep_wait();
            waited = true;
        }
        for (int b = lo; b < hi; ++b) {
            if (seq_blocks(p.context_lens[b], p.T, p.max_blocks, win) == 0) {
                report(p.status, GQA_ERR_CONTEXT);
                zero_sequence<H>(p, b);
            }
        }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += v;
    }
    const int excl = incl - local;
    const long long total = (long long)nKC * __shfl_sync(FULL, incl, 31);
    const int quota = max((int)((total + gridDim.x - 1) / gridDim.x), kQuotaMin);
    const long long c0 = (long long)blockIdx.x * quota;
    const long long c1 = min(total, c0 + quota);
    // Chunked rows read every block once per chunk: keep them in L2 then.
    const uint64_t pol = nC > 1 ? policy_evict_normal() : policy_evict_first();

    int it = 0;  // stages issued
    bool aborted = false;
    if (c0 < c1) {
        // 2. Locate unit c0: the lane whose run of sequences contains it.
        const bool mine = (long long)nKC * excl <= c0 && c0 < (long long)nKC * incl;
        const unsigned owners = __ballot_sync(FULL, mine);
        const int owner = __ffs(owners) - 1;
        int fb = 0;
        long long fbase = 0;
        if (lane == owner) {
            long long acc = (long long)nKC * excl;
            for (int b = lo; b < hi; ++b) {
                const long long n = (long long)nKC *
                                    seg_units(seq_blocks(p.context_lens[b], p.T, p.max_blocks, win));
                if (c0 < acc + n) {
                    fb = b;
                    fbase = acc;
                    break;
                }
                acc += n;
            }
        }
        int b = __shfl_sync(FULL, fb, owner);
        long long base = __shfl_sync(FULL, fbase, owner);  // first unit of segment (b, 0)
        // Lane-distributed look-ahead windows: context lengths of sequences
        // b .. b+31, and the first 32 block ids of sequence b+1, fetched before
        // they are needed so that moving to the next sequence costs no
        // dependent global load.
        int cbase = b;
        int ctxw = (b + lane < p.B) ? __ldg(p.context_lens + b + lane) : 0;
        int ctx = __shfl_sync(FULL, ctxw, 0);
        int nblk = seq_blocks(ctx, p.T, p.max_blocks, win);
        int f0 = first_block(ctx, p.T, win);  // tile i is logical block f0 + i
        // the range starts in segment k, at unit u of it (its first tile is
        // unit kSegUnits): the first tile of the range is i
        const int rel = (int)(c0 - base);
        int k = rel / seg_units(nblk);
        int i = max(0, rel - k * seg_units(nblk) - kSegUnits);
        // KV head of virtual head k, kept incrementally (the issue path of
        // this warp is on the critical path: no division per stage)
        int kv = k / nC, kc = k - kv * nC;
        int ids = 0, ids_base = -(1 << 30);
        // Block ids held besides the current window: the first window of
        // sequence ids0_b (every head's segment of a sequence starts there) and
        // the window at pf_base of sequence pf_b, loaded eight stages before
        // its first use -- a load on the issue path stalls every stage behind it.
        int ids0 = 0, ids0_b = -1, ids_pf = 0, pf_base = -1, pf_b = -1;
        auto load_ids = [&](int from) {
            return (from + lane < nblk)
                       ? __ldg(p.block_tables + (size_t)b * p.max_blocks + f0 + from + lane)
                       : 0;
        };
        auto next_ids = [&](int bn) {
            const int cn = (bn < p.B) ? __shfl_sync(FULL, ctxw, min(bn - cbase, 31)) : 0;
            const int nn =
                (bn < p.B && bn - cbase < 32) ? seq_blocks(cn, p.T, p.max_blocks, win) : 0;
            const int fn = first_block(cn, p.T, win);
            return (lane < nn) ? __ldg(p.block_tables + (size_t)bn * p.max_blocks + fn + lane) : 0;
        };
        int ids_next = next_ids(b + 1);
        if (lane == 0) prefetch_q<H>(p, b, GENERAL ? kv : k);
        bool next_ok = (b + 1 < p.B) && (b + 1 - cbase < 32);  // ids_next is b+1's

        // 3. Stream the range, one stage (up to four tiles of a segment) at a time.
        long long x = base + (long long)k * seg_units(nblk) + kSegUnits + i;  // unit of tile i
        while (x < c1) {
            const int run = (int)min((long long)min(C::kTiles, nblk - i), c1 - x);
            if (i < ids_base || i + run > ids_base + 32) {  // warp-uniform refill
                ids = (i == pf_base && b == pf_b) ? ids_pf
                      : (i == 0 && b == ids0_b)   ? ids0
                                                  : load_ids(i);
                ids_base = i;
                if (i == 0) {
                    ids0 = ids;
                    ids0_b = b;
                }
                pf_base = i + 32;
                pf_b = b;
                ids_pf = load_ids(pf_base);
            }
            int blk[C::kTiles];
            bool bad = false;
#pragma unroll
            for (int j = 0; j < C::kTiles; ++j) {
                blk[j] = __shfl_sync(FULL, ids, min(i - ids_base + j, 31));
                if (j < run) bad |= (blk[j] < 0 || blk[j] >= p.num_blocks);
            }
            // (with the append fused in, the new positions come from k_new /
            // v_new after the consumers' wait, so only an error waits here)
            if (!waited && ((!p.k_new && (f0 + i + run - 1) * 16 + 15 >= ctx - p.T) || bad)) {
                griddep_wait();  // the stage holds new positions (or reports an error)
                waited = true;
            }
            if (lane == 0) {
                const int s = it % p.stages;
                bool ok = true;
                if (it >= p.stages)
                    ok = mbar_wait(smem_addr(&bar.empty[s]), ((it / p.stages) - 1) & 1);
                if (!ok) report(p.status, GQA_ERR_TIMEOUT);
                if (!ok || *abort_flag) {
                    *abort_flag = 1;
                    aborted = true;
                } else {
                    auto& m = meta[s];
                    m.b = b;
                    m.k = k;
                    m.blk_i = f0 + i;  // logical block index
                    m.ntiles = run;
                    m.ctx = ctx;
                    m.seg_start = (int)(base + (long long)k * seg_units(nblk) + kSegUnits);
                    m.nblk = nblk;
                    m.quota = quota;
                    m.cta_start = (int)c0;
                    m.flags = bad ? kBad : 0;
#pragma unroll
                    for (int j = 0; j < C::kTiles; ++j) m.blk[j] = blk[j];
                    mbar_arrive(smem_addr(&bar.meta[s]));
                    const uint32_t fb_ = smem_addr(&bar.full[s]);
                    if (bad) {
                        report(p.status, GQA_ERR_BLOCK_ID);
                        mbar_arrive(fb_);
                    } else {
                        mbar_arrive_expect_tx(fb_, (uint32_t)(run * 2 * C::kTileBytes));
                        const uint32_t dst = smem_addr(stages + (size_t)s * C::kStageBytes);
#pragma unroll
                        for (int j = 0; j < C::kTiles; ++j) {
                            if (j < run) {
#pragma unroll
                                for (int hh = 0; hh < C::kHalves; ++hh) {
                                    tma_load_3d(dst + j * C::kTileBytes + hh * 2048, tmk, fb_,
                                                hh * 64, GENERAL ? kv : k, blk[j] * 16, pol);
                                    tma_load_3d(dst + (C::kTiles + j) * C::kTileBytes +
                                                    hh * 2048,
                                                tmv, fb_, hh * 64, GENERAL ? kv : k, blk[j] * 16,
                                                pol);
                                }
                            }
                        }
                    }
                }
            }
            aborted = __shfl_sync(FULL, aborted, 0);
            if (aborted) break;
            if constexpr (KVQ != 0) {
                // The stage's row scales (K and V, 64 B per tile: 512 B) with one
                // 16-byte cp.async per lane -- a bulk copy per tile was measured
                // to cost a quarter of the launch.  Lane 0 has waited for the slot
                // (the warp barrier below orders the other lanes after it); each lane's
                // copy completes as one of the full barrier's 32 extra arrivals.
                static_assert(C::kTiles * 2 * 4 == 32, "one 16-byte piece per lane");
                __syncwarp();  // orders every lane after lane 0's wait for the slot
                const int s = it % p.stages;
                const int j = lane >> 3, part = (lane >> 2) & 1, ch = lane & 3;
                if (!bad && j < run) {
                    const float* src = (part ? p.v_scale : p.k_scale) +
                                       ((size_t)blk[j] * p.K + (GENERAL ? kv : k)) * 16 + ch * 4;
                    cp_async_16(smem_addr(stages + (size_t)s * C::kStageBytes) +
                                    2 * C::kTiles * C::kTileBytes + (part * C::kTiles + j) * 64 +
                                    ch * 16,
                                src);
                }
                cp_async_mbar_arrive_noinc(smem_addr(&bar.full[s]));
            }
            ++it;
            x += run;
            i += run;
            if (i == nblk) {
                i = 0;
                x += kSegUnits;  // the next segment's start-up units
                const bool more = x < c1;
                if (GENERAL && ++kc == nC) {
                    kc = 0;
                    ++kv;
                }
                if (++k == nKC) {
                    k = 0;
                    kv = 0;
                    base += (long long)nKC * seg_units(nblk);
                    ids_base = -(1 << 30);
                    if (x < c1) {
                        const int b_prev = b;
                        do {
                            ++b;
                            if (b >= cbase + 32) {  // warp-uniform window refill
                                cbase = b;
                                ctxw = (b + lane < p.B) ? __ldg(p.context_lens + b + lane) : 0;
                            }
                            ctx = __shfl_sync(FULL, ctxw, b - cbase);
                            nblk = seq_blocks(ctx, p.T, p.max_blocks, win);
                        } while (nblk == 0);
                        f0 = first_block(ctx, p.T, win);
                        if (b == b_prev + 1 && next_ok) {  // prefetched ids are b's
                            ids0 = ids_next;
                            ids0_b = b;
                        }
                        ids_next = next_ids(b + 1);
                        next_ok = (b + 1 < p.B) && (b + 1 - cbase < 32);
                    }
                }
                if (more && lane == 0) prefetch_q<H>(p, b, GENERAL ? kv : k);  // next segment's q
            }
        }
    }
    // 4. End marker (a stage with no data), then, after an abort, let every
    //    copy already issued land before the CTA exits.
    bool end_sent = false;
    if (lane == 0) {
        if (!aborted) {
            const int s = it % p.stages;
            const bool ok = it < p.stages ||
                            mbar_wait(smem_addr(&bar.empty[s]), ((it / p.stages) - 1) & 1);
            if (ok) {
                meta[s].flags = kEnd;
                mbar_arrive(smem_addr(&bar.meta[s]));
                mbar_arrive(smem_addr(&bar.full[s]));
                end_sent = true;
            } else {
                report(p.status, GQA_ERR_TIMEOUT);
                *abort_flag = 1;
                aborted = true;
            }
        }
    }
    if constexpr (KVQ != 0) {  // the full barrier's 32 extra arrivals
        end_sent = __shfl_sync(FULL, end_sent, 0);
        if (end_sent) mbar_arrive(smem_addr(&bar.full[it % p.stages]));
    }
    if (lane == 0) {
        if (aborted) {
            for (int j = max(0, it - p.stages); j < it; ++j)
                mbar_wait(smem_addr(&bar.full[j % p.stages]), (j / p.stages) & 1);
        }
    }
}

// ---------------------------------------------------------------------------
// Consumer warp state.  The warp owns NW tiles of 8 query rows: tile u holds
// rows 8*(w*NW + u) .. +7 (rows r = t*G + g).  Every K / V fragment it reads
// from shared memory feeds NW mma, so more rows per warp means fewer warps
// re-reading the same stage.
template <int H, bool BF16, int NW, bool GENERAL, int KVQ>
struct Consumer {
    using C = Cfg<H, KVQ>;
    using E = Elt<BF16 && !KVQ>;  // the mma type: f16 over one-byte codes
    using EO = Elt<BF16>;         // the output type
    static constexpr unsigned FULL = 0xffffffffu;

    const AttnParams& p;
    const int w, lane, g, q4;
    int t0[NW], t1[NW];  // new-token index of this lane's two C-fragment rows, per tile
    uint32_t qf[NW][C::kSteps][2];
    float acc[NW][C::kSteps][4];
    float m0[NW], m1[NW], l0[NW], l1[NW];
    bool bad;
    int cb, ck, cstart, cnblk, cquota, ccta0;
    unsigned seen;  // lane 0: tickets of the current split segment read before its close
    // Fused append with one new token: this lane's 16-byte chunk of the new
    // key (lanes < H/8) or value (the next H/8 lanes) row, loaded when the
    // segment starts so that it has landed by the stage that holds it.
    uint4 newrow;
    int rbase, rend;  // query rows [rbase, rend) of the current chunk
    // int8 codes enter the QK^T mma as c + 1152 (no subtraction per pair):
    // 1152 * sum_h q_h is taken off every score of query rows 2q4 / 2q4+1
    float qbias0[NW], qbias1[NW];
    // ... and V codes as c + 1152 too: pv* sum the scaled probabilities fed to
    // the PV mma per row; 1152 * pv comes off the accumulator when the segment
    // closes (before any combine or merge, which are linear in it)
    float pv0[NW], pv1[NW];

    __device__ int row0(int u) const { return (GENERAL ? rbase : 0) + 8 * (w * NW + u); }
    __device__ int row_end() const { return GENERAL ? rend : p.R; }

    __device__ void set_row_tokens() {
#pragma unroll
        for (int u = 0; u < NW; ++u) {
            const int r0 = row0(u) + 2 * q4;
            t0[u] = min(r0 / p.G, p.T - 1);
            t1[u] = min((r0 + 1) / p.G, p.T - 1);
        }
    }

    __device__ Consumer(const AttnParams& p_, int w_)
        : p(p_), w(w_), lane(threadIdx.x & 31), g((threadIdx.x & 31) >> 2), q4(threadIdx.x & 3),
          rbase(0), rend(0) {
        if (!GENERAL) set_row_tokens();  // one chunk: the rows never change
    }

    // Start segment (b, k): reset the running state and fetch the B fragments
    // of Q^T (k = head dim, n = query row): row row0(u)+g, dims kk*16 + 2*q4 +
    // {0,1} and the same + 8.  The loads complete while the stage's tiles land.
    // holds_last: this warp will process the segment's last tile (the one that
    // holds the new token of a fused append).
    __device__ void begin(const typename C::Meta& md, bool holds_last) {
        cb = md.b;
        if (GENERAL) {  // md.k is the virtual head (KV head, row chunk)
            ck = md.k / p.C;
            rbase = (md.k - ck * p.C) * p.Rc;
            rend = min(p.R, rbase + p.Rc);
            set_row_tokens();
        } else {
            ck = md.k;
        }
        cstart = md.seg_start;
        cnblk = md.nblk;
        cquota = md.quota;
        ccta0 = md.cta_start;
        bad = false;
        if constexpr (KVQ == 0 && !GENERAL) {
            constexpr int kChunks = H / 8;
            if (p.k_new && p.T == 1 && holds_last && lane < 2 * kChunks) {
                const bool is_v = lane >= kChunks;
                const size_t row = ((size_t)cb * p.K + ck) * kChunks;
                newrow = __ldg(static_cast<const uint4*>(is_v ? p.v_new : p.k_new) + row +
                               (is_v ? lane - kChunks : lane));
            }
        }
#pragma unroll
        for (int u = 0; u < NW; ++u) {
            m0[u] = m1[u] = -INFINITY;
            l0[u] = l1[u] = 0.f;
            pv0[u] = pv1[u] = 0.f;
#pragma unroll
            for (int mt = 0; mt < C::kSteps; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[u][mt][e] = 0.f;
            const int r = row0(u) + g;
            float qsum_row = 0.f;
            if (r < row_end()) {
                const int t = r / p.G, gg = r % p.G;
                const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                    static_cast<const uint16_t*>(p.q) +
                    (((size_t)cb * p.T + t) * p.N + (size_t)ck * p.G + gg) * H);
                if constexpr (KVQ != 0) {
                    // permuted dims: lane q4 takes dims 32*q4 .. +31, four per
                    // k-step (see stage_q); f16 for the mma (bf16 -> f16 is
                    // exact in f16's normal range)
                    const uint4* q16 = reinterpret_cast<const uint4*>(qrow) + 4 * q4;
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 v = __ldg(q16 + i);
                        w[4 * i] = v.x;
                        w[4 * i + 1] = v.y;
                        w[4 * i + 2] = v.z;
                        w[4 * i + 3] = v.w;
                    }
                    float qs = 0.f;  // sum of this lane's 32 dims, as the mma sees them
#pragma unroll
                    for (int kk = 0; kk < C::kSteps; ++kk) {
                        qf[u][kk][0] = to_f16x2(w[2 * kk]);
                        qf[u][kk][1] = to_f16x2(w[2 * kk + 1]);
                        qs += Elt<false>::lo(qf[u][kk][0]) + Elt<false>::hi(qf[u][kk][0]) +
                              Elt<false>::lo(qf[u][kk][1]) + Elt<false>::hi(qf[u][kk][1]);
                    }
                    qsum_row = qs;
                } else {
#pragma unroll
                    for (int kk = 0; kk < C::kSteps; ++kk) {
                        qf[u][kk][0] = __ldg(qrow + kk * 8 + q4);
                        qf[u][kk][1] = __ldg(qrow + kk * 8 + 4 + q4);
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < C::kSteps; ++kk) qf[u][kk][0] = qf[u][kk][1] = 0u;
            }
            if constexpr (KVQ == GQA_KV_INT8) {
                // row g's sum over the four lanes that hold it, then the sums of
                // query rows 2q4 and 2q4+1 (lanes 8*q4 and 8*q4+4 hold them)
                qsum_row += __shfl_xor_sync(FULL, qsum_row, 1);
                qsum_row += __shfl_xor_sync(FULL, qsum_row, 2);
                qbias0[u] = 1152.f * __shfl_sync(FULL, qsum_row, 8 * q4);
                qbias1[u] = 1152.f * __shfl_sync(FULL, qsum_row, 8 * q4 + 4);
            }
        }
    }

    // Fused append: the tiles holding the T newest positions may carry stale
    // rows there (TMA read the cache before this call writes it).  Overwrite
    // those rows of the staged K and V tiles with k_new / v_new, and let row
    // warp 0 write them into the caches (each new position of KV head k lies in
    // exactly one tile, handled by exactly one CTA).  Every row warp of the
    // group patches its own copy of the same bytes before reading them.
    __device__ bool patch_new_rows(uint32_t kbase, const typename C::Meta& md) {
        constexpr int kChunks = H / 8;  // 16-byte chunks per row
        const uint32_t vbase = kbase + C::kTiles * C::kTileBytes;
        const int first_new = md.ctx - p.T;
        bool any = false;
        for (int j = 0; j < md.ntiles; ++j) {  // warp-uniform
            const int tb = (md.blk_i + j) * 16;
            const int lo = max(first_new, tb), hi = min(md.ctx, tb + 16);
            for (int pos = lo; pos < hi; ++pos) {
                any = true;
                const int r = pos - tb, t = pos - first_new;
                if (lane < 2 * kChunks) {
                    const bool is_v = lane >= kChunks;
                    const int c = is_v ? lane - kChunks : lane;
                    const size_t row = (((size_t)cb * p.T + t) * p.K + ck) * kChunks;
                    const uint4 val =
                        (!GENERAL && p.T == 1) ? newrow  // loaded when the segment started
                                 : __ldg(static_cast<const uint4*>(is_v ? p.v_new : p.k_new) +
                                         row + c);
                    const uint32_t dst = (is_v ? vbase : kbase) + j * C::kTileBytes +
                                         (c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
                    st_shared_v4(dst, val);
                    if (w == 0 && (!GENERAL || rbase == 0)) {  // one writer: row chunk 0
                        uint4* cache = static_cast<uint4*>(is_v ? p.v_cache : p.k_cache);
                        cache[(((size_t)md.blk[j] * 16 + r) * p.K + ck) * kChunks + c] = val;
                    }
                }
            }
        }
        if (any) {
            // the generic-proxy writes must precede the next TMA write into this
            // stage buffer (issued after every consumer released it)
            fence_proxy_async_shared();
            __syncwarp();
        }
        return any;
    }

    // Two q elements (the dtype of q) -> f16x2.
    static __device__ __forceinline__ uint32_t to_f16x2(uint32_t x) {
        if constexpr (BF16)
            return Elt<false>::pack(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
        else
            return x;
    }

    // Scores of one stage -> masked (unused tiles, causal bound, window, tree
    // mask, slots past the context) and scaled into the log2 domain by tsc
    // (per tile, for tokens g and g+8); running max with lazy rescale; ref*
    // get the exponent references of the stage.
    // NJ tiles starting at tile j0 of the stage.
    template <int NJ>
    __device__ void mask_and_max(float (&sc)[NW][NJ][4], const typename C::Meta& md, int j0,
                                 const float (&tsc)[NJ][2], float (&ref0)[NW],
                                 float (&ref1)[NW]) {
        const int win = GENERAL ? p.window : 0;
        const int ntl = md.ntiles;
#pragma unroll
        for (int u = 0; u < NW; ++u) {
            float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int tb = (md.blk_i + j0 + j) * 16;
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[u][j][e] *= tsc[j][e >> 1];
                if (j0 + j >= ntl) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[u][j][e] = -INFINITY;
                } else if (tb + 15 > md.ctx - p.T - (GENERAL && p.tree_mask ? 1 : 0) ||
                           (win > 0 && tb < md.ctx - win)) {
                    // some position hidden from some row: above its causal
                    // bound lim, or (local attention) at or below lim - window,
                    // or (tree) a new position -- the first new token too
                    const int lim0 = md.ctx - p.T + t0[u], lim1 = md.ctx - p.T + t1[u];
                    const int pos0 = tb + g, pos8 = pos0 + 8;
                    const int wl = win > 0 ? win : (1 << 30);
                    bool h00 = pos0 > lim0 || pos0 <= lim0 - wl;
                    bool h01 = pos0 > lim1 || pos0 <= lim1 - wl;
                    bool h80 = pos8 > lim0 || pos8 <= lim0 - wl;
                    bool h81 = pos8 > lim1 || pos8 <= lim1 - wl;
                    if (GENERAL && p.tree_mask) {
                        // tree: a new position other than the row's own is
                        // visible only if the row's mask selects it
                        const int fn = md.ctx - p.T;
                        const uint64_t mk0 = __ldg(p.tree_mask + (size_t)cb * p.T + t0[u]);
                        const uint64_t mk1 = __ldg(p.tree_mask + (size_t)cb * p.T + t1[u]);
                        auto off = [&](int pos, int lim, uint64_t mk) {
                            return pos >= fn && pos < lim && !((mk >> (pos - fn)) & 1ull);
                        };
                        h00 |= off(pos0, lim0, mk0);
                        h01 |= off(pos0, lim1, mk1);
                        h80 |= off(pos8, lim0, mk0);
                        h81 |= off(pos8, lim1, mk1);
                    }
                    if (h00) sc[u][j][0] = -INFINITY;
                    if (h01) sc[u][j][1] = -INFINITY;
                    if (h80) sc[u][j][2] = -INFINITY;
                    if (h81) sc[u][j][3] = -INFINITY;
                }
                x0 = fmaxf(x0, fmaxf(sc[u][j][0], sc[u][j][2]));
                x1 = fmaxf(x1, fmaxf(sc[u][j][1], sc[u][j][3]));
            }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                x0 = fmaxf(x0, __shfl_xor_sync(FULL, x0, o));
                x1 = fmaxf(x1, __shfl_xor_sync(FULL, x1, o));
            }
            const bool need0 = x0 > m0[u] + kRescaleGap, need1 = x1 > m1[u] + kRescaleGap;
            if (__any_sync(FULL, need0 || need1)) {
                const float n0 = need0 ? x0 : m0[u], n1 = need1 ? x1 : m1[u];
                const float f0 = need0 ? fast_exp2(m0[u] - n0) : 1.f;
                const float f1 = need1 ? fast_exp2(m1[u] - n1) : 1.f;
                l0[u] *= f0;
                l1[u] *= f1;
                if constexpr (KVQ == GQA_KV_INT8) {
                    pv0[u] *= f0;
                    pv1[u] *= f1;
                }
#pragma unroll
                for (int mt = 0; mt < C::kSteps; ++mt) {
                    acc[u][mt][0] *= f0;
                    acc[u][mt][1] *= f1;
                    acc[u][mt][2] *= f0;
                    acc[u][mt][3] *= f1;
                }
                m0[u] = n0;
                m1[u] = n1;
            }
            ref0[u] = (m0[u] == -INFINITY) ? 0.f : m0[u];
            ref1[u] = (m1[u] == -INFINITY) ? 0.f : m1[u];
        }
    }

    // One stage: md.ntiles tiles of 16 tokens starting at tile md.blk_i.
    // One stage over one-byte codes (H = 128, one 8-row tile per warp).  The
    // head dimension is permuted so that each lane's fragment elements are
    // contiguous bytes of shared memory (the dot products and the output are
    // unchanged by a permutation applied to q, K and V alike):
    //   QK^T, k-step kk: fragment column c <-> dim 32*(c%8/2) + 4*kk + c%2 + 2*(c/8),
    //     so lane q4 reads dims 32*q4 .. +31 of its two token rows (32 bytes each);
    //   PV, m-tile mt: fragment row m <-> dim 16*(m%8) + 2*mt + m/8,
    //     so lane g reads dims 16*g .. +15 of its four tokens (16 bytes each)
    //     and holds output dims 16*g .. +15 of its two query rows.
    // Codes become f16 with integer ops only, exactly: int8 codes as c + 1152 on
    // the K side (1152 * sum(q) is taken off each score) and as c on the V
    // side; e4m3 codes as their values times 2^-8 (the row scales carry the
    // 256).  The K row scales multiply the scores, the V row scales the
    // probabilities.  The row sums add the fp32 probabilities: the PV operand
    // (probability x scale, rounded to f16) has no unscaled counterpart, so
    // rounding the sums as well would only add a second error of 2^-12 relative.
    __device__ void stage_q(uint32_t kbase, const typename C::Meta& md) {
        static_assert(H == 128 && NW == 1, "one-byte caches: H = 128, one tile per warp");
        // the stage's tiles in runs of four (the online softmax takes any split)
#pragma unroll 1
        for (int j0 = 0; j0 < C::kTiles && j0 < md.ntiles; j0 += 4) stage_q4(kbase, md, j0);
    }

    // The factor between a code's value and the f16 it becomes (e4m3 codes turn
    // into their values times 2^-8).
    static constexpr float kCodeScale = KVQ == GQA_KV_E4M3 ? 256.f : 1.f;

    // Tiles j0 .. j0+3 of a one-byte stage.
    __device__ void stage_q4(uint32_t kbase, const typename C::Meta& md, int j0) {
        constexpr int NJ = 4;
        const uint32_t vbase = kbase + C::kTiles * C::kTileBytes;
        const uint32_t ksb = vbase + C::kTiles * C::kTileBytes;  // K row scales
        const uint32_t vsb = ksb + C::kTiles * 64;                // V row scales
        const int ntl = md.ntiles;
        float sc[NW][NJ][4];
        float tsc[NJ][2];
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) {
            const int j = j0 + jj;
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[0][jj][e] = 0.f;
            const uint32_t kt = kbase + j * C::kTileBytes;
            const uint32_t c0 = (uint32_t)(((2 * q4) ^ g) << 4);
            const uint32_t c1 = (uint32_t)(((2 * q4 + 1) ^ g) << 4);
            const uint4 ra = ld_shared_v4(kt + g * 128 + c0);
            const uint4 rb = ld_shared_v4(kt + g * 128 + c1);
            const uint4 sa = ld_shared_v4(kt + (g + 8) * 128 + c0);
            const uint4 sb = ld_shared_v4(kt + (g + 8) * 128 + c1);
            const uint32_t w0[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
            const uint32_t w1[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
            for (int kk = 0; kk < C::kSteps; ++kk) {
                uint32_t a[4];
                if constexpr (KVQ == GQA_KV_INT8) {  // codes + 1152 (see qbias)
                    const uint32_t x0 = w0[kk] ^ 0x80808080u, x1 = w1[kk] ^ 0x80808080u;
                    a[0] = u8x2_to_f16x2_biased<false>(x0);  // token g, dims +0, +1
                    a[1] = u8x2_to_f16x2_biased<false>(x1);  // token g+8
                    a[2] = u8x2_to_f16x2_biased<true>(x0);   // token g, dims +2, +3
                    a[3] = u8x2_to_f16x2_biased<true>(x1);
                } else {  // e4m3 values times 2^-8 (see kCodeScale)
                    a[0] = e4m3x2_to_f16x2_scaled<false>(w0[kk]);
                    a[1] = e4m3x2_to_f16x2_scaled<false>(w1[kk]);
                    a[2] = e4m3x2_to_f16x2_scaled<true>(w0[kk]);
                    a[3] = e4m3x2_to_f16x2_scaled<true>(w1[kk]);
                }
                E::mma(sc[0][jj], a, qf[0][kk][0], qf[0][kk][1]);
            }
            if constexpr (KVQ == GQA_KV_INT8) {
                sc[0][jj][0] -= qbias0[0];
                sc[0][jj][1] -= qbias1[0];
                sc[0][jj][2] -= qbias0[0];
                sc[0][jj][3] -= qbias1[0];
            }
            tsc[jj][0] = p.scale_log2 * kCodeScale * ld_shared_f32(ksb + j * 64 + g * 4);
            tsc[jj][1] = p.scale_log2 * kCodeScale * ld_shared_f32(ksb + j * 64 + (g + 8) * 4);
        }
        float ref0[NW], ref1[NW];
        mask_and_max(sc, md, j0, tsc, ref0, ref1);
        // ---- O^T += V^T . (P * v_scale)^T, tile by tile -----------------------
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) {
            const int j = j0 + jj;
            if (j >= ntl) break;  // warp-uniform
            const int tb = (md.blk_i + j) * 16;
            // slots past the context, and (local attention) positions below
            // every new token's window, may hold anything, NaN scales included
            const int lo_min = (GENERAL && p.window > 0) ? md.ctx - p.T - p.window + 1 : 0;
            const bool tail = tb + 16 > md.ctx || tb < lo_min;
            float svg = kCodeScale * ld_shared_f32(vsb + j * 64 + g * 4);
            float sv8 = kCodeScale * ld_shared_f32(vsb + j * 64 + (g + 8) * 4);
            if (tail) {
                if (tb + g >= md.ctx || tb + g < lo_min) svg = 0.f;
                if (tb + g + 8 >= md.ctx || tb + g + 8 < lo_min) sv8 = 0.f;
            }
            const float e0 = fast_exp2(sc[0][jj][0] - ref0[0]);
            const float e1 = fast_exp2(sc[0][jj][1] - ref1[0]);
            const float e2 = fast_exp2(sc[0][jj][2] - ref0[0]);
            const float e3 = fast_exp2(sc[0][jj][3] - ref1[0]);
            l0[0] += e0 + e2;
            l1[0] += e1 + e3;
            const float f0 = e0 * svg, f1 = e1 * svg, f2 = e2 * sv8, f3 = e3 * sv8;
            const uint32_t w0p = E::pack(f0, f1), w1p = E::pack(f2, f3);
            if constexpr (KVQ == GQA_KV_INT8) {
                pv0[0] += E::lo(w0p) + E::lo(w1p);
                pv1[0] += E::hi(w0p) + E::hi(w1p);
            }
            const uint32_t pb0 = movm_t(w0p);  // tokens 2q4, +1
            const uint32_t pb1 = movm_t(w1p);  // tokens 2q4+8, +9
            // f16 outputs: each operand's rounding error enters as a second f16
            // term (a half ulp of f16 relative to |V| would take half of the
            // output's own error budget; bf16 outputs round far more coarsely)
            uint32_t lb0 = 0u, lb1 = 0u;
            if constexpr (!BF16) {
                const uint32_t w0l = E::pack(f0 - E::lo(w0p), f1 - E::hi(w0p));
                const uint32_t w1l = E::pack(f2 - E::lo(w1p), f3 - E::hi(w1p));
                if constexpr (KVQ == GQA_KV_INT8) {
                    pv0[0] += E::lo(w0l) + E::lo(w1l);
                    pv1[0] += E::hi(w0l) + E::hi(w1l);
                }
                lb0 = movm_t(w0l);
                lb1 = movm_t(w1l);
            }
            const uint32_t vt = vbase + j * C::kTileBytes;
            const int t0_ = 2 * q4, t1_ = t0_ + 1, t2_ = t0_ + 8, t3_ = t0_ + 9;
            const uint4 x0 = ld_shared_v4(vt + t0_ * 128 + ((g ^ (t0_ & 7)) << 4));
            const uint4 x1 = ld_shared_v4(vt + t1_ * 128 + ((g ^ (t1_ & 7)) << 4));
            const uint4 x2 = ld_shared_v4(vt + t2_ * 128 + ((g ^ (t2_ & 7)) << 4));
            const uint4 x3 = ld_shared_v4(vt + t3_ * 128 + ((g ^ (t3_ & 7)) << 4));
            uint32_t y0[4] = {x0.x, x0.y, x0.z, x0.w}, y1[4] = {x1.x, x1.y, x1.z, x1.w};
            uint32_t y2[4] = {x2.x, x2.y, x2.z, x2.w}, y3[4] = {x3.x, x3.y, x3.z, x3.w};
            if constexpr (KVQ == GQA_KV_INT8) {  // offset the codes by 128 once per word
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    y0[i] ^= 0x80808080u;
                    y1[i] ^= 0x80808080u;
                    y2[i] ^= 0x80808080u;
                    y3[i] ^= 0x80808080u;
                }
            }
#pragma unroll
            for (int mt = 0; mt < C::kSteps; ++mt) {
                // dims 16g + 2mt (+1): byte 2*(mt&1) (+1) of word mt/2; interleave
                // the two tokens of each pair, then two bytes -> f16x2
                const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                const uint32_t p01 = prmt(y0[mt >> 1], y1[mt >> 1], sel);
                const uint32_t p23 = prmt(y2[mt >> 1], y3[mt >> 1], sel);
                uint32_t a[4];
                // (no masking of slots past the context: every code becomes a
                // finite f16, and those slots' probabilities are exactly 0)
                if constexpr (KVQ == GQA_KV_INT8) {  // c + 1152 (see pv0 / pv1)
                    a[0] = u8x2_to_f16x2_biased<false>(p01);  // dim +0, tokens 2q4, +1
                    a[1] = u8x2_to_f16x2_biased<true>(p01);   // dim +1
                    a[2] = u8x2_to_f16x2_biased<false>(p23);  // dim +0, tokens +8, +9
                    a[3] = u8x2_to_f16x2_biased<true>(p23);
                } else {
                    a[0] = e4m3x2_to_f16x2_scaled<false>(p01);
                    a[1] = e4m3x2_to_f16x2_scaled<true>(p01);
                    a[2] = e4m3x2_to_f16x2_scaled<false>(p23);
                    a[3] = e4m3x2_to_f16x2_scaled<true>(p23);
                }
                E::mma(acc[0][mt], a, pb0, pb1);
                if constexpr (!BF16) E::mma(acc[0][mt], a, lb0, lb1);
            }
        }
    }

    __device__ void stage(uint32_t kbase, const typename C::Meta& md) {
        if constexpr (KVQ != 0) {
            stage_q(kbase, md);
            return;
        }
        const int win = GENERAL ? p.window : 0;  // compile-time 0 for the plain kernel
        if (p.k_new && (md.blk_i + md.ntiles) * 16 > md.ctx - p.T) patch_new_rows(kbase, md);
        const uint32_t vbase = kbase + C::kTiles * C::kTileBytes;
        const int ntl = md.ntiles;
        // ---- S^T = K_tile . Q^T for every tile and row tile (independent chains)
        float sc[NW][C::kTiles][4];
#pragma unroll
        for (int u = 0; u < NW; ++u)
#pragma unroll
            for (int j = 0; j < C::kTiles; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[u][j][e] = 0.f;
        {
            const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int chk = lane >> 4;
#pragma unroll
            for (int kk = 0; kk < C::kSteps; ++kk) {
                const int hh = kk >> 2;
                const int chunk = ((kk & 3) << 1) + chk;
                const uint32_t off = hh * 2048 + tok * 128 + ((chunk ^ (tok & 7)) << 4);
#pragma unroll
                for (int j = 0; j < C::kTiles; ++j) {
                    uint32_t a[4];
                    ldsm_x4(kbase + j * C::kTileBytes + off, a);
#pragma unroll
                    for (int u = 0; u < NW; ++u) E::mma(sc[u][j], a, qf[u][kk][0], qf[u][kk][1]);
                }
            }
        }
        float ref0[NW], ref1[NW];
        {
            float tsc[C::kTiles][2];
#pragma unroll
            for (int j = 0; j < C::kTiles; ++j) tsc[j][0] = tsc[j][1] = p.scale_log2;
            mask_and_max(sc, md, 0, tsc, ref0, ref1);
        }
        // ---- O^T += V_tile^T . P^T, tile by tile ------------------------------------
        const int tok = (lane & 7) + (lane >> 4) * 8;
        const int dof = ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int j = 0; j < C::kTiles; ++j) {
            if (j >= ntl) break;  // warp-uniform
            uint32_t pb0[NW], pb1[NW];
#pragma unroll
            for (int u = 0; u < NW; ++u) {
                const uint32_t pt0 = E::pack(fast_exp2(sc[u][j][0] - ref0[u]),
                                             fast_exp2(sc[u][j][1] - ref1[u]));  // token g
                const uint32_t pt1 = E::pack(fast_exp2(sc[u][j][2] - ref0[u]),
                                             fast_exp2(sc[u][j][3] - ref1[u]));  // token g+8
                l0[u] += E::lo(pt0) + E::lo(pt1);
                l1[u] += E::hi(pt0) + E::hi(pt1);
                // P^T as the B operand: tokens 2*q4+{0,1} (+8) of query row g.
                pb0[u] = movm_t(pt0);
                pb1[u] = movm_t(pt1);
            }
            const int tb = (md.blk_i + j) * 16;
            // NaN-safe: zero V elements of slots past the context and, with a
            // window, of positions below every new token's window (a block
            // only partly inside the window may hold anything there)
            const int lo_min = win > 0 ? md.ctx - p.T - win + 1 : 0;
            const bool tail = tb + 16 > md.ctx || tb < lo_min;
            uint32_t v01 = 0xffffffffu, v89 = 0xffffffffu;
            if (tail) {
                const int pb = tb + 2 * q4;
                auto ok = [&](int x) { return x < md.ctx && x >= lo_min; };
                v01 = (ok(pb) ? 0x0000ffffu : 0u) | (ok(pb + 1) ? 0xffff0000u : 0u);
                v89 = (ok(pb + 8) ? 0x0000ffffu : 0u) | (ok(pb + 9) ? 0xffff0000u : 0u);
            }
            const uint32_t vt = vbase + j * C::kTileBytes;
#pragma unroll
            for (int mt = 0; mt < C::kSteps; ++mt) {
                const int d0 = mt * 16 + dof;
                const int hh = d0 >> 6;
                const int chunk = (d0 & 63) >> 3;
                uint32_t a[4];
                ldsm_x4_t(vt + hh * 2048 + tok * 128 + ((chunk ^ (tok & 7)) << 4), a);
                if (tail) {
                    a[0] &= v01;
                    a[1] &= v01;
                    a[2] &= v89;
                    a[3] &= v89;
                }
#pragma unroll
                for (int u = 0; u < NW; ++u) E::mma(acc[u][mt], a, pb0[u], pb1[u]);
            }
        }
    }

    // Normalise and store the rows of tile u of segment (cb, ck).
    // One-byte caches: lane g holds output dims 16g .. +15 of query rows 2q4
    // (acc[mt][0], acc[mt][2]) and 2q4+1 (acc[mt][1], acc[mt][3]).
    __device__ void store_q(int u, float L0, float L1, bool is_bad) {
        const float i0 = (!is_bad && L0 > 0.f) ? 1.f / L0 : 0.f;
        const float i1 = (!is_bad && L1 > 0.f) ? 1.f / L1 : 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = row0(u) + 2 * q4 + half;
            if (r >= row_end()) continue;
            const float iv = half ? i1 : i0;
            const int t = r / p.G, gg = r % p.G;
            uint4* dst = reinterpret_cast<uint4*>(
                static_cast<uint16_t*>(p.out) +
                (((size_t)cb * p.T + t) * p.N + (size_t)ck * p.G + gg) * H + 16 * g);
            uint32_t w[8];
#pragma unroll
            for (int mt = 0; mt < C::kSteps; ++mt)
                w[mt] = is_bad ? 0u : EO::pack(acc[u][mt][half] * iv, acc[u][mt][2 + half] * iv);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
    }

    __device__ void store(int u, float L0, float L1, bool is_bad) {
        if constexpr (KVQ != 0) {
            store_q(u, L0, L1, is_bad);
            return;
        }
        const float i0 = (!is_bad && L0 > 0.f) ? 1.f / L0 : 0.f;
        const float i1 = (!is_bad && L1 > 0.f) ? 1.f / L1 : 0.f;
        const int r = row0(u) + g;
        uint32_t* dst = nullptr;
        if (r < row_end()) {
            const int t = r / p.G, gg = r % p.G;
            dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) +
                                              (((size_t)cb * p.T + t) * p.N +
                                               (size_t)ck * p.G + gg) * H);
        }
#pragma unroll
        for (int mt = 0; mt < C::kSteps; ++mt) {
            uint32_t x = is_bad ? 0u : E::pack(acc[u][mt][0] * i0, acc[u][mt][1] * i1);
            uint32_t y = is_bad ? 0u : E::pack(acc[u][mt][2] * i0, acc[u][mt][3] * i1);
            x = movm_t(x);  // -> row g, dims mt*16 + 2*q4 + {0,1}
            y = movm_t(y);  // -> row g, dims mt*16 + 8 + 2*q4 + {0,1}
            if (dst) {
                dst[mt * 8 + q4] = x;
                dst[mt * 8 + 4 + q4] = y;
            }
        }
    }

    // Partial-result section of tile u in CTA `cta`, slot 0 for the CTA's
    // first segment (a piece other than a segment's first) and slot 1 for its
    // last (the first piece of a segment): a CTA holds at most one of each.
    __device__ float* section(int cta, int slot, int u) const {
        return p.partials +
               ((((size_t)cta * 2 + slot) * p.nt + w) * NW + u) * C::kSectionFloats;
    }
    // Ticket of a split segment for this row warp, indexed by the CTA that
    // holds the segment's first piece.
    __device__ int32_t* ticket(int first_cta) const {
        return p.flags + (size_t)first_cta * p.nt + w;
    }

    // Row sums: each lane holds the sum over its own tokens; add up the 8 lanes
    // that share a row pair.
    __device__ void reduce_l() {
#pragma unroll
        for (int u = 0; u < NW; ++u) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                l0[u] += __shfl_xor_sync(FULL, l0[u], o);
                l1[u] += __shfl_xor_sync(FULL, l1[u], o);
            }
        }
        if constexpr (KVQ == GQA_KV_INT8) {  // remove the V codes' offset
#pragma unroll
            for (int u = 0; u < NW; ++u) {
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    pv0[u] += __shfl_xor_sync(FULL, pv0[u], o);
                    pv1[u] += __shfl_xor_sync(FULL, pv1[u], o);
                }
                const float b0 = 1152.f * pv0[u], b1 = 1152.f * pv1[u];
#pragma unroll
                for (int mt = 0; mt < C::kSteps; ++mt) {
                    acc[u][mt][0] -= b0;
                    acc[u][mt][1] -= b1;
                    acc[u][mt][2] -= b0;
                    acc[u][mt][3] -= b1;
                }
            }
        }
    }

    // Per-lane layout of a group's state in the combine scratch.
    static constexpr int kScratchFloats = NW * (4 + C::kAccFloats);

    __device__ void save_state(float* slot) const {
        float4* d = reinterpret_cast<float4*>(slot);
#pragma unroll
        for (int u = 0; u < NW; ++u) {
            float4* du = d + u * (1 + C::kSteps);
            du[0] = make_float4(m0[u], m1[u], l0[u], l1[u]);
#pragma unroll
            for (int mt = 0; mt < C::kSteps; ++mt)
                du[1 + mt] = make_float4(acc[u][mt][0], acc[u][mt][1], acc[u][mt][2],
                                         acc[u][mt][3]);
        }
    }

    // Fold a (max, sum, accumulator) state of tile u into this one.
    __device__ void fold(int u, float mc0, float mc1, float lc0, float lc1, const float4* v) {
        const float n0 = fmaxf(m0[u], mc0), n1 = fmaxf(m1[u], mc1);
        const float a0 = (m0[u] == -INFINITY) ? 0.f : fast_exp2(m0[u] - n0);
        const float a1 = (m1[u] == -INFINITY) ? 0.f : fast_exp2(m1[u] - n1);
        const float b0 = (mc0 == -INFINITY) ? 0.f : fast_exp2(mc0 - n0);
        const float b1 = (mc1 == -INFINITY) ? 0.f : fast_exp2(mc1 - n1);
        l0[u] = l0[u] * a0 + lc0 * b0;
        l1[u] = l1[u] * a1 + lc1 * b1;
#pragma unroll
        for (int mt = 0; mt < C::kSteps; ++mt) {
            acc[u][mt][0] = acc[u][mt][0] * a0 + v[mt].x * b0;
            acc[u][mt][1] = acc[u][mt][1] * a1 + v[mt].y * b1;
            acc[u][mt][2] = acc[u][mt][2] * a0 + v[mt].z * b0;
            acc[u][mt][3] = acc[u][mt][3] * a1 + v[mt].w * b1;
        }
        m0[u] = n0;
        m1[u] = n1;
    }

    // Fold another group's state (same segment, same rows) into this one.
    __device__ void absorb(const float* slot) {
        const float4* d = reinterpret_cast<const float4*>(slot);
#pragma unroll
        for (int u = 0; u < NW; ++u) {
            const float4* du = d + u * (1 + C::kSteps);
            const float4 h = du[0];
            fold(u, h.x, h.y, h.z, h.w, du + 1);
        }
    }

    // The first piece of a split segment ends its CTA's range, so the other
    // pieces have usually drawn their tickets by then: read the count early
    // (lane 0, before the groups meet), so that finalize can merge at once.
    __device__ void peek_ticket() {
        const int first = cstart / cquota;
        const int last = (cstart + cnblk - 1) / cquota;
        seen = 0u;
        if (lane == 0 && first != last && (int)blockIdx.x == first) seen = ticket_seen(ticket(first));
    }

    // Finish the segment (row sums already reduced).  A split segment's pieces
    // sit in CTAs first..last.  If the others have all drawn tickets when the
    // first piece closes (the usual case: it ends its CTA's range), it folds
    // them into its own state right away.  Otherwise each piece's warp
    // publishes its partial (max, sum, accumulator, invalid-block flag) and
    // takes a ticket, and the warp that draws the last one folds the pieces.
    // Either way the fold runs in CTA order from the first piece's state,
    // exactly as stored -- a deterministic result -- and the merger stores
    // the rows and resets the ticket for the next call.  Nothing waits.
    __device__ void finalize() {
        const int first = cstart / cquota;
        const int last = (cstart + cnblk - 1) / cquota;
        const int me = blockIdx.x;
        if (first == last) {
#pragma unroll
            for (int u = 0; u < NW; ++u) store(u, l0[u], l1[u], bad);
            return;
        }
        if (me == first && __shfl_sync(FULL, seen, 0) == (unsigned)(last - first)) {
            __syncwarp();  // lane 0's acquire before every lane's loads
            merge_others(first, last);
            return;
        }
        auto slot_of = [&](int c) { return c == first ? 1 : 0; };
#pragma unroll
        for (int u = 0; u < NW; ++u) {
            float* sec = section(me, slot_of(me), u);
            if (g == 0) {
                sec[2 * q4] = m0[u];
                sec[2 * q4 + 1] = m1[u];
                sec[8 + 2 * q4] = l0[u];
                sec[8 + 2 * q4 + 1] = l1[u];
            }
            if (lane == 0) sec[16] = bad ? 1.f : 0.f;
            float4* a4 = reinterpret_cast<float4*>(sec + C::kHeaderFloats) + lane * C::kSteps;
#pragma unroll
            for (int mt = 0; mt < C::kSteps; ++mt)
                a4[mt] = make_float4(acc[u][mt][0], acc[u][mt][1], acc[u][mt][2], acc[u][mt][3]);
        }
        __syncwarp();  // orders the lanes' stores before lane 0's ticket
        unsigned drawn = 0;
        if (lane == 0) drawn = ticket_acq_rel(ticket(first));
        drawn = __shfl_sync(FULL, drawn, 0);
        if (drawn != (unsigned)(last - first)) return;  // another piece's warp merges
        __syncwarp();  // orders lane 0's acquire before every lane's loads
        merge_others(first, last);
    }

    // Combine every piece of the split segment, in two passes whose loads are
    // all in flight together: the rows' maxima M over the pieces, then the
    // sums of the pieces' (sum, accumulator) with weights 2^(m_c - M), in CTA
    // order from the first piece (this warp's registers if it holds it).  The
    // result does not depend on which warp merges.  Store the rows and reset
    // the ticket.
    __device__ void merge_others(int first, int last) {
        const int me = blockIdx.x;
        constexpr int kUnroll = (H == 64) ? 4 : 1;  // pieces whose loads are in flight at once
        bool any_bad = false;
#pragma unroll
        for (int u = 0; u < NW; ++u) {
            if (me != first) {  // the first piece's state
                const float* sc = section(first, 1, u);
                m0[u] = __ldcg(sc + 2 * q4);
                m1[u] = __ldcg(sc + 2 * q4 + 1);
                l0[u] = __ldcg(sc + 8 + 2 * q4);
                l1[u] = __ldcg(sc + 8 + 2 * q4 + 1);
                any_bad |= __ldcg(sc + 16) != 0.f;
                const float4* b4 =
                    reinterpret_cast<const float4*>(sc + C::kHeaderFloats) + lane * C::kSteps;
#pragma unroll
                for (int mt = 0; mt < C::kSteps; ++mt) {
                    const float4 v = __ldcg(b4 + mt);
                    acc[u][mt][0] = v.x;
                    acc[u][mt][1] = v.y;
                    acc[u][mt][2] = v.z;
                    acc[u][mt][3] = v.w;
                }
            } else {
                any_bad |= bad;
            }
            // pass 1: the maxima of the two rows this lane holds
            float M0 = m0[u], M1 = m1[u];
#pragma unroll kUnroll
            for (int c = first + 1; c <= last; ++c) {
                const float* sc = section(c, 0, u);
                M0 = fmaxf(M0, __ldcg(sc + 2 * q4));
                M1 = fmaxf(M1, __ldcg(sc + 2 * q4 + 1));
            }
            // pass 2: the first piece scaled, then the others added in order
            {
                const float a0 = (m0[u] == -INFINITY) ? 0.f : fast_exp2(m0[u] - M0);
                const float a1 = (m1[u] == -INFINITY) ? 0.f : fast_exp2(m1[u] - M1);
                l0[u] *= a0;
                l1[u] *= a1;
#pragma unroll
                for (int mt = 0; mt < C::kSteps; ++mt) {
                    acc[u][mt][0] *= a0;
                    acc[u][mt][1] *= a1;
                    acc[u][mt][2] *= a0;
                    acc[u][mt][3] *= a1;
                }
            }
#pragma unroll kUnroll
            for (int c = first + 1; c <= last; ++c) {
                const float* sc = section(c, 0, u);
                const float mc0 = __ldcg(sc + 2 * q4), mc1 = __ldcg(sc + 2 * q4 + 1);
                const float lc0 = __ldcg(sc + 8 + 2 * q4), lc1 = __ldcg(sc + 8 + 2 * q4 + 1);
                any_bad |= __ldcg(sc + 16) != 0.f;
                const float4* b4 =
                    reinterpret_cast<const float4*>(sc + C::kHeaderFloats) + lane * C::kSteps;
                float4 v[C::kSteps];
#pragma unroll
                for (int mt = 0; mt < C::kSteps; ++mt) v[mt] = __ldcg(b4 + mt);
                const float a0 = (mc0 == -INFINITY) ? 0.f : fast_exp2(mc0 - M0);
                const float a1 = (mc1 == -INFINITY) ? 0.f : fast_exp2(mc1 - M1);
                l0[u] += lc0 * a0;
                l1[u] += lc1 * a1;
#pragma unroll
                for (int mt = 0; mt < C::kSteps; ++mt) {
                    acc[u][mt][0] += v[mt].x * a0;
                    acc[u][mt][1] += v[mt].y * a1;
                    acc[u][mt][2] += v[mt].z * a0;
                    acc[u][mt][3] += v[mt].w * a1;
                }
            }
            m0[u] = M0;
            m1[u] = M1;
        }
        if (lane == 0) *ticket(first) = 0;  // ready for the next call
#pragma unroll
        for (int u = 0; u < NW; ++u) store(u, l0[u], l1[u], any_bad);
    }
};

// Consumer warp w belongs to group w / nt (stage-parallel: group g computes
// the stages whose index is g modulo the group count) and owns query rows
// 8*(w % nt) .. +7.  Every warp reads every stage's description, so all groups
// agree on segment boundaries; at each boundary the groups' partial states
// meet in shared memory and group 0 finishes the segment.
template <int H, bool BF16, int NW, bool GENERAL, int KVQ>
__device__ void consumer(const AttnParams& p, uint8_t* stages, const Bars& bar,
                         const typename Cfg<H, KVQ>::Meta* meta, float* scratch,
                         volatile int* abort_flag,
                         int w) {
    using C = Cfg<H, KVQ>;
    using CS = Consumer<H, BF16, NW, GENERAL, KVQ>;
    const int gi = w / p.nt, wr = w % p.nt;
    CS cs(p, wr);
    const int lane = threadIdx.x & 31;
    griddep_wait();  // q, the workspace and out follow the previous kernels
    auto slot = [&](int buf, int gg) {
        return scratch +
               ((((size_t)buf * (p.groups - 1) + (gg - 1)) * p.nt + wr) * 32 + lane) *
                   CS::kScratchFloats;
    };
    int nseg = 0;  // segments closed so far (phase of the combine barrier)
    auto close = [&]() -> bool {
        if (gi == 0) cs.peek_ticket();  // its latency overlaps the groups' meeting
        cs.reduce_l();
        const int buf = nseg & 1;  // double buffer: group 0 may still read the other
        if (gi != 0) cs.save_state(slot(buf, gi));
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(bar.cbar));
        if (!mbar_wait(smem_addr(bar.cbar), nseg & 1)) {
            if (lane == 0) report(p.status, GQA_ERR_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
        if (gi == 0) {
#pragma unroll
            for (int gg = 1; gg < p.groups; ++gg) cs.absorb(slot(buf, gg));
            cs.finalize();
        }
        ++nseg;
        return true;
    };
    int cur = -1;
    for (int it = 0;; ++it) {
        const int s = it % p.stages;
        const uint32_t par = (it / p.stages) & 1;
        if (!mbar_wait(smem_addr(&bar.meta[s]), par)) {
            if (lane == 0) report(p.status, GQA_ERR_TIMEOUT);
            *abort_flag = 1;
            return;
        }
        const auto md = meta[s];
        if (md.flags & kEnd) {
            if (cur >= 0) close();
            return;
        }
        const int seg = md.b * (GENERAL ? p.KC : p.K) + md.k;
        if (seg != cur) {
            if (cur >= 0 && !close()) return;
            // the segment's piece in this CTA holds the new token iff this CTA
            // holds the segment's last tile
            cs.begin(md, (md.seg_start + md.nblk - 1) / md.quota == (int)blockIdx.x);
            cur = seg;
        }
        if (md.flags & kBad) {
            cs.bad = true;
        } else if (it % p.groups == gi) {
            if (!mbar_wait(smem_addr(&bar.full[s]), par)) {
                if (lane == 0) report(p.status, GQA_ERR_TIMEOUT);
                *abort_flag = 1;
                return;
            }
            cs.stage(smem_addr(stages + (size_t)s * C::kStageBytes), md);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bar.empty[s]));
    }
}

// NW = 1: up to 6 row warps per group; NW = 2 (two 8-row tiles per warp, for
// many query rows) up to 3, with the register budget of the smaller CTA.
// GENERAL: local attention, a tree mask or row chunks (all compiled out of the
// plain kernel, which then runs with no window, the chain mask and one chunk).
template <int H, bool BF16, int NW, bool GENERAL, int KVQ>
__global__ void __launch_bounds__(NW == 1 ? kMaxThreads : 32 * (kGroups * kMaxRowWarps / 2 + 1))
    attention_kernel(const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
    using C = Cfg<H, KVQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    Bars bar;
    bar.full = reinterpret_cast<uint64_t*>(smem + (size_t)p.stages * C::kStageBytes);
    bar.meta = bar.full + p.stages;
    bar.empty = bar.meta + p.stages;
    bar.cbar = bar.empty + p.stages;
    auto* meta = reinterpret_cast<typename C::Meta*>(bar.cbar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(meta + p.stages);
    float* scratch = reinterpret_cast<float*>(
        (reinterpret_cast<uintptr_t>(abort_flag + 1) + 15) & ~uintptr_t(15));
    const int consumers = p.groups * p.nt;

    const int warp = threadIdx.x >> 5;
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            // one-byte caches: the producer warp's 32 scale copies arrive too
            mbar_init(smem_addr(&bar.full[s]), KVQ ? 33 : 1);
            mbar_init(smem_addr(&bar.meta[s]), 1);
            mbar_init(smem_addr(&bar.empty[s]), consumers);
        }
        mbar_init(smem_addr(bar.cbar), consumers);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == consumers)
        producer<H, GENERAL, KVQ>(&tmk, &tmv, p, stages, bar, meta, abort_flag);
    else
        consumer<H, BF16, NW, GENERAL, KVQ>(p, stages, bar, meta, scratch, abort_flag, warp);
}

// ---------------------------------------------------------------------------
// Direct kernel, for small problems: one CTA per (b, k) segment and no split.
// Every warp loads its own stages (four tiles each: stages w, w + W, ...) with
// cp.async into a buffer of its own, in the layout the TMA writes (128-byte
// swizzle), and runs the consumer's stage code on it; the warps' states are
// combined in shared memory and warp 0 stores the rows.  The critical path is
// one round trip for the context length and the block ids, one for the tiles
// of every warp at once, the stages, and one combine in shared memory.  (The
// persistent kernel's producer issues the stages one after another, and its
// split segments meet through global memory: round trips that dominate when
// the whole call is a few microseconds of HBM traffic.)
template <int H>
struct Direct {
    static constexpr int kWarps = H == 64 ? 8 : 6;  // one 16 / 32 KB stage buffer each
    static constexpr int kMaxStagesPerWarp = 2;     // longer segments: the persistent kernel
};

// Copy tiles 0 .. run-1 (cache blocks blk[j]) of KV head k into a stage buffer,
// K tiles then V tiles, each row's 16-byte chunk c at chunk c ^ (row & 7) of its
// 128-byte span; one group of cp.async per call.
template <int H>
__device__ void direct_load(uint32_t buf, const AttnParams& p, int k,
                            const int (&blk)[kTilesPerStage], int run, int lane) {
    using C = Cfg<H, 0>;
    constexpr int kChunks = H / 8;          // 16-byte chunks per row
    constexpr int kPerTile = 16 * kChunks;  // chunks per tile
    const uint8_t* kc = static_cast<const uint8_t*>(p.k_cache);
    const uint8_t* vc = static_cast<const uint8_t*>(p.v_cache);
#pragma unroll
    for (int j = 0; j < kTilesPerStage; ++j) {
        if (j < run) {  // warp-uniform
#pragma unroll
            for (int x = lane; x < kPerTile; x += 32) {
                const int r = x / kChunks, c = x % kChunks;
                const size_t src = (((size_t)blk[j] * 16 + r) * p.K + k) * (H * 2) + c * 16;
                const uint32_t off = (c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
                cp_async_16(buf + j * C::kTileBytes + off, kc + src);
                cp_async_16(buf + (C::kTiles + j) * C::kTileBytes + off, vc + src);
            }
        }
    }
    cp_async_commit();
}

template <int H, bool BF16>
__global__ void __launch_bounds__(32 * Direct<H>::kWarps)
    direct_kernel(const AttnParams p) {
    using C = Cfg<H, 0>;
    using CS = Consumer<H, BF16, 1, false, 0>;
    static_assert(C::kTiles == kTilesPerStage, "stage layout of the two-byte cache");
    constexpr int W = Direct<H>::kWarps;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_bad[W];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* scratch = reinterpret_cast<float*>(smem + (size_t)W * C::kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x / p.K, k = blockIdx.x - b * p.K;
    griddep_launch_dependents();
    // Without the early-KV promise every global access waits for the grids
    // this launch depends on; with it, the length, the block ids and the
    // cache below position ctx - T may be read first.
    bool waited = false;
    if (!p.early_kv) {
        griddep_wait();
        waited = true;
    }
    // The block ids of this warp's first two stages, loaded together with the
    // length (entries past the length are read but not used): lanes 0-3 the
    // first stage's, lanes 4-7 the second's.
    const int* bt_row = p.block_tables + (size_t)b * p.max_blocks;
    const int pre_i = lane < 4 ? warp * C::kTiles + lane : (warp + W) * C::kTiles + lane - 4;
    const int pre_id = (lane < 8 && pre_i < p.max_blocks) ? __ldg(bt_row + pre_i) : 0;
    const int ctx = __ldg(p.context_lens + b);
    const int nblk = seq_blocks(ctx, p.T, p.max_blocks, 0);
    if (nblk == 0) {  // invalid length: this KV head's rows are zeros
        griddep_wait();
        if (threadIdx.x == 0) report(p.status, GQA_ERR_CONTEXT);
        constexpr int kRow16 = H * 2 / 16;
        for (int x = threadIdx.x; x < p.T * p.G * kRow16; x += blockDim.x) {
            const int row = x / kRow16, t = row / p.G, gg = row - t * p.G;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                  (((size_t)b * p.T + t) * p.N +
                                                   (size_t)k * p.G + gg) * H);
            dst[x - row * kRow16] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    const int nst = (nblk + C::kTiles - 1) / C::kTiles;  // stages of the segment
    const uint32_t buf = smem_addr(smem + (size_t)warp * C::kStageBytes);
    CS cs(p, 0);  // every warp holds all (at most 8) query rows
    typename C::Meta md;
    md.b = b;
    md.k = k;
    md.ctx = ctx;
    md.nblk = nblk;
    md.seg_start = 0;
    md.quota = 1 << 30;
    md.cta_start = 0;
    md.flags = 0;
    bool bad = false, began = false;
    for (int st = warp, round = 0; st < nst; st += W, ++round) {  // warp-uniform
        const int i = st * C::kTiles;
        const int run = min(C::kTiles, nblk - i);
        const int id = round < 2 ? pre_id
                       : (lane < run) ? __ldg(bt_row + i + lane) : 0;
        const int src = round == 1 ? 4 : 0;  // the lanes holding this stage's ids
        bool sbad = false;
#pragma unroll
        for (int j = 0; j < C::kTiles; ++j) {
            md.blk[j] = __shfl_sync(FULL, id, round < 2 ? src + j : j);
            if (j < run) sbad |= (md.blk[j] < 0 || md.blk[j] >= p.num_blocks);
        }
        md.blk_i = i;
        md.ntiles = run;
        // a stage holding new positions that an earlier kernel wrote waits for it
        if (!waited && (sbad || (!p.k_new && (i + run) * 16 > ctx - p.T))) {
            griddep_wait();
            waited = true;
        }
        if (!sbad) direct_load<H>(buf, p, k, md.blk, run, lane);
        if (!began) {  // q (and k_new / v_new) follow the previous kernels
            if (!waited) {
                griddep_wait();
                waited = true;
            }
            cs.begin(md, (nst - 1) % W == warp);
            began = true;
        }
        if (sbad) {
            if (lane == 0) report(p.status, GQA_ERR_BLOCK_ID);
            bad = true;
            continue;
        }
        cp_async_wait_all();
        __syncwarp();  // every lane's copies landed before any lane reads them
        cs.stage(buf, md);
        __syncwarp();  // every lane done with the buffer before the next copies
    }
    // combine: warps 1 .. active-1 hand their states to warp 0, in warp order
    const int active = min(W, nst);
    if (began) cs.reduce_l();
    if (warp > 0 && warp < active)
        cs.save_state(scratch + ((size_t)(warp - 1) * 32 + lane) * CS::kScratchFloats);
    if (lane == 0) s_bad[warp] = bad ? 1 : 0;
    __syncthreads();
    if (warp == 0) {
        bool any_bad = false;
        for (int w = 0; w < active; ++w) any_bad |= s_bad[w] != 0;
        for (int w = 1; w < active; ++w)
            cs.absorb(scratch + ((size_t)(w - 1) * 32 + lane) * CS::kScratchFloats);
        cs.store(0, cs.l0[0], cs.l1[0], any_bad);
    }
}

// ---------------------------------------------------------------------------
// Host side
// The instantiated variants, for each head size and dtype: (nw, general) in
// {(1, no), (1, yes), (2, no)} over a cache in q's dtype, and for H = 128
// (1, no) and (1, yes) over int8 and e4m3 caches.
template <int H, bool BF16>
const void* kernel_ptr(int nw, bool general, int kvq) {
    if constexpr (H == 128) {
        if (kvq == GQA_KV_INT8)
            return general ? reinterpret_cast<const void*>(
                                 &attention_kernel<H, BF16, 1, true, GQA_KV_INT8>)
                           : reinterpret_cast<const void*>(
                                 &attention_kernel<H, BF16, 1, false, GQA_KV_INT8>);
        if (kvq == GQA_KV_E4M3)
            return general ? reinterpret_cast<const void*>(
                                 &attention_kernel<H, BF16, 1, true, GQA_KV_E4M3>)
                           : reinterpret_cast<const void*>(
                                 &attention_kernel<H, BF16, 1, false, GQA_KV_E4M3>);
    }
    if (nw == 2) return reinterpret_cast<const void*>(&attention_kernel<H, BF16, 2, false, 0>);
    return general ? reinterpret_cast<const void*>(&attention_kernel<H, BF16, 1, true, 0>)
                   : reinterpret_cast<const void*>(&attention_kernel<H, BF16, 1, false, 0>);
}

const void* pick_kernel(int H, bool bf16, int nw, bool general, int kvq) {
    if (H == 64)
        return bf16 ? kernel_ptr<64, true>(nw, general, kvq) : kernel_ptr<64, false>(nw, general, kvq);
    return bf16 ? kernel_ptr<128, true>(nw, general, kvq) : kernel_ptr<128, false>(nw, general, kvq);
}

// Consumer groups for nt row warps: two.  (A third group was measured slower
// on the 40-row verify workload: stages then contend for shared memory; four
// groups for one row warp were measured slower on the 24-layer batch of short
// contexts, 313 vs 285 us per step.  Over a one-byte cache, the 256-sequence
// ragged batch ran 365 us with two groups and two stages -- five CTAs per SM --
// against 423 with three groups and 490 with four groups and four stages: what
// bounds it is each CTA's one-stage-at-a-time producer, so CTAs per SM count
// for more than warps per CTA.)
int groups_for(int, int) { return kGroups; }

// Row warps a group may have with nw 8-row tiles per warp (48 rows at most).
int max_row_warps(int nw) { return nw == 1 ? kMaxRowWarps : kMaxRowWarps / 2; }

// Dynamic shared memory of one CTA: nt row warps (nw tiles each) per consumer
// group and a ring of `stages` stages.
template <int H, int KVQ>
size_t smem_of(int nt, int nw, int stages, int groups) {
    using C = Cfg<H, KVQ>;
    return C::kFixed + (size_t)stages * (C::kStageBytes + C::kStageOverhead) +
           (size_t)(groups - 1) * nt * nw * C::kScratchBytesPerRowWarp;
}
size_t smem_for(int H, int nt, int nw, int stages, int kvq, int groups) {
    if (kvq) return smem_of<128, 1>(nt, nw, stages, groups);  // both one-byte kinds: H = 128
    return H == 64 ? smem_of<64, 0>(nt, nw, stages, groups)
                   : smem_of<128, 0>(nt, nw, stages, groups);
}
int default_stages(int H, int kvq) {
    if (kvq) return Cfg<128, 1>::kStages;
    return H == 64 ? Cfg<64>::kStages : Cfg<128>::kStages;
}
// The largest dynamic shared memory any launch of a variant asks for.
size_t max_smem(int H, int nw, int kvq) {
    size_t m = 0;
    for (int nt = 1; nt <= max_row_warps(nw); ++nt)
        m = std::max(m, smem_for(H, nt, nw, default_stages(H, kvq), kvq, groups_for(nt, kvq)));
    return m;
}

size_t section_floats(int H) {
    return H == 64 ? Cfg<64>::kSectionFloats : Cfg<128>::kSectionFloats;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// 3-D view of a cache [num_blocks][16][K][H]: (h, kv head, block*16 + row);
// one box = 16 rows x 128 bytes of one KV head (64 two-byte elements, or 128
// one-byte codes), 128-byte swizzled.
bool encode_cache_map(CUtensorMap* m, const void* base, const gqa_shape& s) {
    auto fn = encode_fn();
    if (!fn) return false;
    const bool q8 = s.kv_dtype != GQA_KV_SAME;
    const cuuint64_t eb = q8 ? 1 : 2;
    const cuuint64_t dims[3] = {(cuuint64_t)s.H, (cuuint64_t)s.K,
                                (cuuint64_t)s.num_blocks * 16};
    const cuuint64_t strides[2] = {(cuuint64_t)s.H * eb, (cuuint64_t)s.K * s.H * eb};
    const cuuint32_t box[3] = {q8 ? 128u : 64u, 1, 16};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                             : s.dtype == GQA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          // a one-byte row of a KV head is 128 B: promoting to
                          // 256 B would fetch the next head's row as well
                          q8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                             : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// CTAs of one variant resident per SM, queried once per (device, variant,
// shared memory) so
// that later calls -- including calls being captured into a CUDA graph -- make
// no attribute or occupancy API calls.
int resident_ctas(int H, bool bf16, int nt, int nw, bool general, int kvq, int groups,
                  size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_tuple(dev, H, (int)bf16, nt,
                                     ((nw * 2 + (int)general) * 4 + kvq) * 8 + groups, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const void* kern = pick_kernel(H, bf16, nw, general, kvq);
    // The attribute belongs to the kernel, whatever the row-warp count: set it
    // to the largest launch any shape makes.
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)max_smem(H, nw, kvq)) !=
        cudaSuccess)
        return 0;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern,
                                                      32 * (groups * nt + 1),
                                                      smem) !=
        cudaSuccess)
        return 0;
    cache[key] = occ;
    return occ;
}

}  // namespace

bool make_cache_map(CUtensorMap* m, const void* base, const gqa_shape& s) {
    return encode_cache_map(m, base, s);
}

bool make_rows_map(CUtensorMap* m, const void* base, const gqa_shape& s, int hpc, int tpc) {
    auto fn = encode_fn();
    if (!fn || (s.H != 64 && s.H != 128) || hpc < 1 || hpc > 256 || tpc < 1 || tpc > 256)
        return false;
    const cuuint64_t G = (cuuint64_t)(s.N / s.K), H = (cuuint64_t)s.H, e = 2;
    const cuuint64_t dims[5] = {H, G, (cuuint64_t)s.K, (cuuint64_t)s.T, (cuuint64_t)s.B};
    const cuuint64_t strides[4] = {H * e, G * H * e, (cuuint64_t)s.N * H * e,
                                   (cuuint64_t)s.T * s.N * H * e};
    const cuuint32_t box[5] = {64, (cuuint32_t)hpc, 1, (cuuint32_t)tpc, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(m, s.dtype == GQA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          5, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static int cache[64] = {0};
    if (dev < 64 && cache[dev]) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cache[dev] = n;
    return n;
}

namespace {

// Dynamic shared memory of the direct kernel: a stage buffer per warp and the
// combine scratch of every warp but the first.
template <int H>
size_t direct_smem_of() {
    using C = Cfg<H, 0>;
    constexpr int W = Direct<H>::kWarps;
    return 1024 + (size_t)W * C::kStageBytes +
           (size_t)(W - 1) * 32 * (4 + C::kAccFloats) * sizeof(float);
}

const void* direct_ptr(int H, bool bf16) {
    if (H == 64)
        return bf16 ? reinterpret_cast<const void*>(&direct_kernel<64, true>)
                    : reinterpret_cast<const void*>(&direct_kernel<64, false>);
    return bf16 ? reinterpret_cast<const void*>(&direct_kernel<128, true>)
                : reinterpret_cast<const void*>(&direct_kernel<128, false>);
}

// The direct kernel's shared-memory attribute, set once per (device, variant).
bool direct_ready(int H, bool bf16) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, bool> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const auto key = std::make_tuple(dev, H, (int)bf16);
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find(key);
    if (it != done.end()) return it->second;
    const size_t smem = H == 64 ? direct_smem_of<64>() : direct_smem_of<128>();
    const bool ok = cudaFuncSetAttribute(direct_ptr(H, bf16),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem) == cudaSuccess;
    done[key] = ok;
    return ok;
}

// Segments (sequence, KV head) the direct kernel takes by default: two waves
// of one CTA per SM on a GB300 (152 SMs).  (The 24-layer batch of short
// contexts at 128 sequences -- 256 segments -- ran 12.7 us per layer direct
// against 14.6 persistent; at 256 sequences 21.6 against 21.0.)
constexpr long long kDirectMaxSegments = 2 * 152;

}  // namespace

bool direct_attention_supported(const gqa_shape& s, bool masked) {
    return s.kv_dtype == GQA_KV_SAME && !masked && s.window == 0 && s.block_size == 16 &&
           (s.H == 64 || s.H == 128) && s.K >= 1 && s.N % s.K == 0 &&
           (long long)s.T * (s.N / s.K) <= 8;
}

bool direct_attention_preferred(const gqa_shape& s, bool masked) {
    if ((s.flags & (GQA_FLAG_WARP_MMA | GQA_FLAG_TENSOR_MEMORY)) != 0) return false;
    if ((s.flags & GQA_FLAG_DIRECT) != 0) return direct_attention_supported(s, masked);
    const long long max_tiles =
        4LL * (s.H == 64 ? Direct<64>::kWarps * Direct<64>::kMaxStagesPerWarp
                         : Direct<128>::kWarps * Direct<128>::kMaxStagesPerWarp);
    return direct_attention_supported(s, masked) &&
           (long long)s.B * s.K <= kDirectMaxSegments && s.max_blocks_per_seq <= max_tiles;
}

gqa_status attention_plan(const gqa_shape& s, bool masked, AttnPlan* plan) {
    // masked: a tree mask will be passed (the general kernel variant)
    if (s.B < 0 || s.T < 1 || s.N < 1 || s.K < 1 || s.N % s.K != 0) return GQA_ERR_SHAPE;
    if (s.H != 64 && s.H != 128) return GQA_ERR_SHAPE;
    if (s.block_size != 16 || s.num_blocks < 1 || s.max_blocks_per_seq < 1) return GQA_ERR_SHAPE;
    if ((long long)s.num_blocks * 16 > (1ll << 31) - 1) return GQA_ERR_SHAPE;
    if ((long long)s.max_blocks_per_seq * 16 > (1ll << 30)) return GQA_ERR_SHAPE;
    if (s.dtype != GQA_F16 && s.dtype != GQA_BF16) return GQA_ERR_DTYPE;
    if (s.window < 0) return GQA_ERR_SHAPE;
    const int G = s.N / s.K;
    const long long R = (long long)s.T * G;
    if (R > kMaxRows) return GQA_ERR_SHAPE;
    // Row chunks of at most 48 rows, as even as multiples of 8 allow.
    const int chunks = (int)((R + 8 * kMaxRowWarps - 1) / (8 * kMaxRowWarps));
    const int rows_per_chunk = (int)(((R + chunks - 1) / chunks + 7) / 8 * 8);
    // One 8-row tile per warp.  (Two tiles per warp -- each K/V fragment read
    // from shared memory serving 16 rows -- measured slower on the 40-row verify
    // workload: fewer warps hide less latency.  The kernel keeps both forms.)
    const int nw = 1;
    const int nt = (rows_per_chunk + 8 * nw - 1) / (8 * nw);
    const int kvq = s.kv_dtype;
    const int groups = groups_for(nt, kvq);
    int stages = default_stages(s.H, kvq);
    size_t smem = smem_for(s.H, nt, nw, stages, kvq, groups);
    const bool general = masked || s.window > 0 || chunks > 1;
    // the one-byte caches have kernels for H = 128 only
    if (kvq != GQA_KV_SAME && s.H != 128) return GQA_ERR_SHAPE;
    const bool bf16 = s.dtype == GQA_BF16;
    int occ = resident_ctas(s.H, bf16, nt, nw, general, kvq, groups, smem);
    if (occ < 1) return GQA_ERR_CUDA;
    if (kvq != GQA_KV_SAME) {
        // the shallower ring where it fits more CTAs per SM (each CTA issues
        // its stages one at a time, so more CTAs keep more stages in flight)
        for (int st = stages - 1; st >= 2; --st) {
            const size_t sm = smem_for(s.H, nt, nw, st, kvq, groups);
            const int o = resident_ctas(s.H, bf16, nt, nw, general, kvq, groups, sm);
            if (o > occ) {
                occ = o;
                stages = st;
                smem = sm;
            }
        }
    }
    const int sms = device_sm_count();
    if (sms < 1) return GQA_ERR_CUDA;
    // As many CTAs as fit on the GPU, also for small problems: one CTA per SM
    // there (fewer split sequences, room for the next launch's CTAs under
    // programmatic dependent launch) measured slower -- 24 layers of 14 MB
    // 396 vs 371 us, the local/global layer mix 382 vs 317 us -- than
    // shorter per-CTA chains on more CTAs.
    long long blocks_max = s.max_blocks_per_seq;  // per sequence, window included
    if (s.window > 0)
        blocks_max = std::min<long long>(blocks_max, ((long long)s.window + s.T + 14) / 16 + 1);
    const long long tiles_max = (long long)s.B * s.K * chunks * (blocks_max + kSegUnits);
    const int threads = 32 * (groups * nt + 1);
    long long grid = (long long)sms * occ;
    grid = std::min<long long>(grid, std::max<long long>(1, (tiles_max + kQuotaMin - 1) / kQuotaMin));
    plan->grid = (int)grid;
    plan->consumer_warps = nt;
    plan->threads = threads;
    plan->smem = smem;
    plan->stages = stages;
    plan->groups = groups;
    plan->tiles_per_warp = nw;
    plan->general = general;
    plan->chunks = chunks;
    plan->rows_per_chunk = rows_per_chunk;
    // The tickets of split segments live in a fixed region at the start of
    // every workspace, whatever the shape, and partial results always start
    // after it: partial data of one call can then never sit where a later
    // call of another shape expects zeroed tickets.
    if (grid * nt > kMaxFlags) return GQA_ERR_SHAPE;
    plan->flags_bytes = (size_t)kMaxFlags * 4;
    plan->partial_floats_per_cta = 2 * section_floats(s.H) * nt * nw;  // two slots
    plan->workspace = plan->flags_bytes + (size_t)grid * plan->partial_floats_per_cta * 4;
    // The direct kernel, where it serves the call (the workspace stays sized
    // for the persistent kernel: one size for every kernel a shape may take).
    plan->direct = direct_attention_preferred(s, masked);
    if ((s.flags & GQA_FLAG_DIRECT) != 0 && !plan->direct) return GQA_ERR_SHAPE;
    if (plan->direct) {
        if (!direct_ready(s.H, bf16)) return GQA_ERR_CUDA;
        plan->grid = s.B * s.K;
        plan->threads = 32 * (s.H == 64 ? Direct<64>::kWarps : Direct<128>::kWarps);
        plan->smem = s.H == 64 ? direct_smem_of<64>() : direct_smem_of<128>();
    }
    return GQA_OK;
}

gqa_status launch_attention(const gqa_shape& s, const AttnPlan& plan, const void* q,
                            const void* k_new, const void* v_new, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables,
                            const int32_t* context_lens, const uint64_t* tree_mask,
                            const float* k_scale, const float* v_scale, void* out,
                            void* workspace, int32_t* dev_status, cudaStream_t stream) {
    if (s.B == 0) return GQA_OK;
    CUtensorMap tmk, tmv;  // (the direct kernel copies with cp.async: no tensor maps)
    if (!plan.direct &&
        (!encode_cache_map(&tmk, k_cache, s) || !encode_cache_map(&tmv, v_cache, s)))
        return GQA_ERR_CUDA;
    AttnParams p;
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.flags = static_cast<int32_t*>(workspace);
    p.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.flags_bytes);
    p.status = dev_status;
    p.B = s.B;
    p.T = s.T;
    p.N = s.N;
    p.K = s.K;
    p.G = s.N / s.K;
    p.R = s.T * p.G;
    p.C = plan.chunks;
    p.Rc = plan.rows_per_chunk;
    p.KC = s.K * plan.chunks;
    p.nt = plan.consumer_warps;
    p.stages = plan.stages;
    p.groups = plan.groups;
    p.max_blocks = s.max_blocks_per_seq;
    p.num_blocks = s.num_blocks;
    const double scale = s.scale > 0.f ? (double)s.scale : 1.0 / sqrt((double)s.H);
    p.scale_log2 = (float)(scale * 1.4426950408889634);  // log2(e)
    p.early_kv = (s.flags & GQA_FLAG_EARLY_KV) ? 1 : 0;
    p.window = s.window;
    p.tree_mask = tree_mask;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    if ((s.kv_dtype != GQA_KV_SAME) != (k_scale != nullptr)) return GQA_ERR_NULL;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache = const_cast<void*>(k_cache);
    p.v_cache = const_cast<void*>(v_cache);
    const bool pdl = (s.flags & (GQA_FLAG_PDL | GQA_FLAG_EARLY_KV)) != 0;
    const bool bf16 = s.dtype == GQA_BF16;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(plan.threads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (plan.direct) {
        if (tree_mask || s.window > 0 || s.kv_dtype != GQA_KV_SAME)
            return GQA_ERR_SHAPE;  // plan made for another call
        void* dargs[] = {&p};
        const cudaError_t e = cudaLaunchKernelExC(&cfg, direct_ptr(s.H, bf16), dargs);
        return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
    }
    const int nw = plan.tiles_per_warp;
    if ((tree_mask || s.window > 0 || plan.chunks > 1) && !plan.general)
        return GQA_ERR_SHAPE;  // plan made for another call
    const void* kern = pick_kernel(s.H, bf16, nw, plan.general, s.kv_dtype);
    void* args[] = {&tmk, &tmv, &p};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, kern, args);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
