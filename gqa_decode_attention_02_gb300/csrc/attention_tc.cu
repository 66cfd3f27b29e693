// attention_tc.cu -- decode / verify / tree-verify attention on the fifth-
// generation tensor cores: tcgen05.mma with its accumulators in tensor memory.
//
// Head size 64 or 128.  Same computation as attention.cu (CS336 lecture 10 §"Арифметическая
// интенсивность инференса": Y = softmax(Q K^T) V of the new tokens over the
// cached keys and values, GQA from §"Уменьшаем KV-кэш", paged reads from
// §"PagedAttention"; the tree mask of "Болжау арқылы Sonar модельдерін
// жылдамдату" §"EAGLE").  It serves the shapes where the contraction is dense:
// many query rows per KV head (long drafts, draft trees, MQA with many query
// heads), where the warp-level mma of attention.cu runs out of issue slots.
//
// Work order.  As in attention.cu: segments (sequence b, virtual head v) in
// b-major order, a virtual head being a KV head and a chunk of at most 128 of
// its T*G query rows; each segment is ceil(ctx_b / 16) tiles (cache blocks).
// CTA c takes units [c*quota, (c+1)*quota) of that order (one CTA per SM),
// a segment being its tiles plus a few units for its start-up, so every SM
// streams about the same bytes and pays about the same per-segment costs
// however ragged the batch.  A
// segment cut by range boundaries is split into pieces: every piece's softmax
// warps publish their partial result (O unnormalized, running max, sum) in the
// workspace and take a ticket (an acq_rel atomicAdd); the warp that draws the
// last ticket folds the pieces in piece order (the same arithmetic in
// whichever CTA it runs: a deterministic result) with log-sum-exp weights --
// the context split of FlashDecoding named in §"PagedAttention" -- and stores
// its rows.  No CTA waits for another.
//
// One CTA: warp 0 MMA issuer and tensor-memory owner, warps 1..2 producers
// (TMA), warps 3..10 softmax in two groups of four warps (one thread per query
// row each; tensor-memory lane = row).  Group g takes the stages st = g, g + 2,
// ... of every piece with its own S, P and O in tensor memory, so the two
// groups' online softmaxes run side by side and meet once per piece (a
// log-sum-exp merge of two partial results, like the context split).
// A stage is up to 64 tokens (four 16-token cache blocks of one piece):
//   S_g[128 x 64]   = Q[128 x 128] . K^T   8 MMAs, Q from tensor memory, K K-major
//   rows: mask (causal, tree, past the context) as one 64-bit word, running
//         max with a lazy rescale of O_g, P = exp2(S*scale - max) in q's dtype
//   O_g[128 x 128] += P_g[128 x 64] . V    4 MMAs, P from tensor memory, V MN-major
// Tensor memory (512 columns, lane = query row) holds O_0, O_1, S_0, S_1,
// P_0, P_1 and the piece's Q.  The MMA issuer starts PV(n) as soon as P(n) is
// written and QK^T(n + 2) right after it (S_g is free once P_g is written), so
// the tensor pipe and both groups stay busy.  Shared memory holds a ring of
// four stages (K and V, each two 64-dim halves of 64 token rows x 128 B,
// 128-byte swizzled: 128 KB), the piece's Q box (TMA, then copied into tensor
// memory) and the output staging box (TMA store).  V rows of a stage that hold no data
// (past the context, or unused tiles) are zeroed before the PV product: their
// probabilities are 0, but stale bytes could be NaN.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "launch.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace gqa {
namespace {

constexpr int kRowsTc = 128;                     // query rows per segment (MMA M)
constexpr int kStagesTc = 4;                     // (6 measured no faster: the pipeline, not memory, bounds it)
constexpr int kProducerWarps = 1;                // TMA issuer of the K / V stages
constexpr int kQWarp = 1 + kProducerWarps;       // TMA loads of Q (warp 0 issues the MMAs)
constexpr int kSoftmaxWarp0 = kQWarp + 1;
constexpr int kSoftmaxThreads = 256;             // eight softmax warps, two groups
constexpr int kGroupThreads = 128;               // one softmax group: a thread per row
constexpr int kThreadsTc = 32 * kSoftmaxWarp0 + kSoftmaxThreads;
constexpr int kHalfBytes = 64 * 128;             // 64 rows of one 64-dim half: 8 KB
constexpr int kStageBytesTc = 4 * kHalfBytes;    // K then V, two halves each: 32 KB
constexpr int kRowHalfBytes = kRowsTc * 128;     // 128 rows x 64 dims of Q or of the output: 16 KB
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns (32 bits each; lane = query row), per softmax group g:
// O_g fp32 [128], S_g fp32 [64], P_g two 16-bit values per column [32]; the
// piece's Q two 16-bit values per column [64]
constexpr uint32_t kColO = 0, kColS = 256, kColP = 384, kColQ = 448;
constexpr uint32_t kColOStep = 128, kColSStep = 64, kColPStep = 32;
constexpr float kGapTc = 8.0f;                   // log2-domain slack before rescaling O
constexpr int kQuotaMinTc = 16;                  // tiles per CTA at least: fewer split pieces
// Start-up cost of a segment in the partition, in tiles: every segment
// occupies its tiles plus kSegCost units at its start, so a CTA that starts
// many segments (each with its own epilogue, ~2 us) streams fewer tiles.
constexpr int kSegCost = 6;
constexpr int kPartFloats = 132 * kRowsTc;       // a partial: O^T [128][128], (max, sum) per half
constexpr int kTcMinRows = 32;                   // rows per KV head from which it is picked
                                                 // (measured faster than mma.sync from 32 rows;
                                                 // at H = 64 70.6 vs 82.1 us at 40 rows and
                                                 // 77.0 vs 141.3 at 64, a 16-sequence verify)
constexpr int kCtxCache = 128;                   // context lengths cached from the CTA's first sequence
constexpr unsigned FULLM = 0xffffffffu;

struct TcParams {
    const void* q;
    void* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const uint64_t* tree_mask;  // nullptr: causal chain among the new tokens
    int32_t* status;
    int32_t* flags;             // tickets: per (CTA holding a first piece, softmax warp)
    float* partials;            // [grid][2][kPartFloats]: per CTA, slot 0 its first
                                // segment (a later piece), slot 1 its last (a first piece)
    int B, T, N, K, G;
    // A row chunk (virtual head) is a box of tpc new tokens x hpc query heads of
    // one KV head, Rc = tpc * hpc <= 128 rows (row = token-in-box * hpc +
    // head-in-box); a KV head has C chunks: cpt per token block (G > 128)
    // times ceil(T / tpc) token blocks.
    int tpc, hpc, cpt, C, Rc, KC;
    int max_blocks, num_blocks;
    int early;                  // GQA_FLAG_EARLY_KV: plan and stream older positions before the wait
    int window;                 // local attention: each query sees its last `window` positions (0: all)
    float scale_log2;
};

struct TcSmem {
    uint64_t full[kStagesTc];   // stage data landed (TMA transaction bytes)
    uint64_t empty[kStagesTc];  // the PV product of the stage completed
    uint64_t q_full;            // the piece's Q box landed in shared memory (TMA bytes)
    uint64_t q_free;            // every QK^T of the previous piece completed
    uint64_t o_free;            // the softmax threads read O_0 / O_1 of the previous piece (256)
    uint64_t s_ready[2];        // QK^T of a stage of group g completed
    uint64_t p_ready[2];        // group g wrote P_g (and zeroed stale V rows)
    uint64_t o_ready[2];        // PV of a stage of group g completed
    uint64_t done;              // every MMA completed (before freeing tensor memory)
    uint64_t pair[4];           // the two threads of each row of a lane quarter (64)
    uint64_t all;               // every softmax thread (256)
    long long c0, c1, base;     // the CTA's tile range; first tile of segment (b0, 0)
    int b0, quota;
    uint32_t tmem_base;
    int bad[kStagesTc];         // the stage's blocks include an invalid id
    volatile int abort_flag;
    float xm[2][kRowsTc];       // per group: running max of each row at the piece's end
    float xl[2][kRowsTc];       // per group: sum of each row
    int xb[2][kRowsTc];         // per group: a stage held an invalid block id
    int ctxc[kCtxCache];        // context_lens[b0 + i]: no dependent global load at a piece change
};

// First logical block a segment reads: the one holding the earliest position
// any of its T new tokens sees (0 without a window).
__device__ __forceinline__ int tc_first(const TcParams& p, int ctx) {
    return p.window > 0 ? max(0, ctx - p.T - p.window + 1) >> 4 : 0;
}
// Tiles of a segment: logical blocks tc_first .. ceil(ctx / 16) - 1 (0 for an
// invalid length).
__device__ __forceinline__ int tc_nblk_of(const TcParams& p, int ctx) {
    return (ctx >= p.T && ctx >= 1 && ctx <= p.max_blocks * 16)
               ? ((ctx + 15) >> 4) - tc_first(p, ctx)
               : 0;
}
__device__ __forceinline__ int tc_nblk(const TcParams& p, int b) {
    return tc_nblk_of(p, __ldg(p.context_lens + b));
}
// context_lens[b] from the shared-memory copy where it holds b
__device__ __forceinline__ int tc_ctx(const TcSmem& sm, const TcParams& p, int b) {
    const int i = b - sm.b0;
    return (i >= 0 && i < kCtxCache) ? sm.ctxc[i] : __ldg(p.context_lens + b);
}

__device__ __forceinline__ void tc_abort(TcSmem& sm, const TcParams& p) {
    report(p.status, GQA_ERR_TIMEOUT);
    sm.abort_flag = 1;
}

// Ticket of a split segment (GPU scope): a warp stores its partial, then
// (after __syncwarp) lane 0 takes a ticket with an acq_rel atomic; the warp
// that draws the last ticket has acquired every earlier piece's stores.
__device__ __forceinline__ unsigned tc_ticket(int32_t* t) {
    unsigned v;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(v)
                 : "l"(t)
                 : "memory");
    return v;
}
// Tickets drawn so far (acquire: the pieces that drew them are visible).
__device__ __forceinline__ unsigned tc_ticket_seen(const int32_t* t) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(t) : "memory");
    return v;
}

// Waits until stage n has landed.
__device__ __forceinline__ bool stage_landed(TcSmem& sm, int n) {
    return mbar_wait(smem_addr(&sm.full[n % kStagesTc]), (n / kStagesTc) & 1);
}

// All softmax threads meet on an mbarrier (arrive, then a bounded wait for
// the phase): a thread that gave up on an earlier wait cannot leave the
// others waiting without limit, as a named barrier would.  `ph` counts this
// thread's uses.
__device__ __forceinline__ bool softmax_bar(TcSmem& sm, int& ph) {
    mbar_arrive(smem_addr(&sm.all));
    const bool ok = mbar_wait(smem_addr(&sm.all), ph & 1);
    ++ph;
    return ok;
}

// One piece: tiles [t0, t1) of segment (b, v), whose first tile is number
// `first` of the whole order and which has nb tiles.
struct TcPiece {
    int b, v, nb, t0, t1;
    int f0;  // logical block of the segment's tile 0 (the window's first block)
    long long first;
};

// Walks the pieces of the CTA's range in order (every role walks the same).
struct TcWalker {
    long long pos, c1, base;
    int b, v, nb;
    const TcSmem* sm;
    __device__ void init(const TcSmem& s, const TcParams& p) {
        sm = &s;
        pos = s.c0;
        c1 = s.c1;
        base = s.base;
        b = s.b0;
        v = 0;
        nb = (pos < c1) ? tc_nblk_of(p, tc_ctx(s, p, b)) : 0;
    }
    // segment (b, v) occupies units [first, first + nb + kSegCost); its tiles
    // are the units from first + kSegCost on
    __device__ bool next(const TcParams& p, TcPiece& pc) {
        while (pos < c1) {
            const long long units = nb > 0 ? nb + kSegCost : 0;
            const long long first = base + (long long)v * units;
            if (nb > 0 && pos < first + units) {
                const long long e = min(c1, first + units);
                const long long tile0 = first + kSegCost;
                const long long s0 = max(pos, tile0);
                pos = e;
                if (e <= s0) continue;  // only start-up units in this range (pos is c1 now)
                pc.b = b;
                pc.v = v;
                pc.nb = nb;
                pc.t0 = (int)(s0 - tile0);
                pc.t1 = (int)(e - tile0);
                pc.f0 = p.window > 0 ? tc_first(p, tc_ctx(*sm, p, b)) : 0;
                pc.first = tile0;
                return true;
            }
            if (nb > 0 && ++v < p.KC) continue;
            base += (long long)p.KC * units;
            v = 0;
            if (++b >= p.B) break;
            nb = tc_nblk_of(p, tc_ctx(*sm, p, b));
        }
        pos = c1;
        return false;
    }
};

// Warp 0, all lanes: tiles per sequence, their prefix sum, this CTA's range
// and the sequence it starts in.
__device__ void tc_plan(const TcParams& p, TcSmem& sm) {
    const int lane = threadIdx.x & 31;
    const int per = (p.B + 31) / 32;
    const int lo = min(p.B, lane * per), hi = min(p.B, lo + per);
    int local = 0;  // units of this lane's sequences (per virtual head)
    for (int b = lo; b < hi; ++b) {
        const int nb = tc_nblk(p, b);
        local += nb > 0 ? nb + kSegCost : 0;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(FULLM, incl, o);
        if (lane >= o) incl += x;
    }
    const int excl = incl - local;
    const long long total = (long long)p.KC * __shfl_sync(FULLM, incl, 31);
    const int quota = (int)max((total + gridDim.x - 1) / gridDim.x, (long long)kQuotaMinTc);
    const long long c0 = (long long)blockIdx.x * quota;
    const long long c1 = min(total, c0 + quota);
    const bool mine = c0 < c1 && (long long)p.KC * excl <= c0 && c0 < (long long)p.KC * incl;
    const unsigned owners = __ballot_sync(FULLM, mine);
    if (lane == 0) {
        sm.c0 = c0;
        sm.c1 = c0 < c1 ? c1 : c0;
        sm.quota = quota;
        sm.b0 = 0;
        sm.base = 0;
    }
    __syncwarp();
    if (owners != 0 && lane == __ffs(owners) - 1) {
        long long acc = (long long)p.KC * excl;
        for (int b = lo; b < hi; ++b) {
            const int nb = tc_nblk(p, b);
            const long long n = (long long)p.KC * (nb > 0 ? nb + kSegCost : 0);
            if (c0 < acc + n) {
                sm.b0 = b;
                sm.base = acc;
                break;
            }
            acc += n;
        }
    }
    __syncwarp();
    const int b0 = sm.b0;
    for (int i = lane; i < kCtxCache; i += 32)
        sm.ctxc[i] = (b0 + i < p.B) ? __ldg(p.context_lens + b0 + i) : 0;
}

// ---------------------------------------------------------------------------
// kProducerWarps warps (one) share each stage: warp pw loads the blocks j of
// the stage with j % kProducerWarps == pw (K and V, two 64-dim halves each,
// one box per lane) and arrives on the stage's barrier with its own byte count.
// Block ids are read 32 at a time (a window of eight stages, one id per lane),
// the next window while the current one is in use.
template <int H>
__device__ void tc_producer(const CUtensorMap* tmk, const CUtensorMap* tmv, const TcParams& p,
                            uint8_t* stages, TcSmem& sm, int pw) {
    const int lane = threadIdx.x & 31;
    if (lane == 0 && pw == 0) {
        tma_prefetch_desc(tmk);
        tma_prefetch_desc(tmv);
    }
    // row chunks read a block once per chunk: keep it in L2 for them
    const uint64_t pol = p.C > 1 ? policy_evict_normal() : policy_evict_first();
    // this lane's box: block bj of the stage, K (kvsel 0) or V, half bh
    constexpr int kBlocksPerWarp = 4 / kProducerWarps;
    const int bj = pw + kProducerWarps * (lane >> 2), kvsel = (lane >> 1) & 1, bh = lane & 1;
    // (H = 64: one 64-dim half per block, K and V)
    const bool boxer = lane < 4 * kBlocksPerWarp && (H == 128 || bh == 0);
    const CUtensorMap* tm = kvsel ? tmv : tmk;
    TcWalker wk;
    wk.init(sm, p);
    TcPiece pc;
    int it = 0;
    bool aborted = false;
    bool waited = !p.early;  // with early KV: only positions below ctx - T before the wait
    while (!aborted && wk.next(p, pc)) {
        const int kv = pc.v / p.C;
        const int32_t* table = p.block_tables + (size_t)pc.b * p.max_blocks + pc.f0;
        const int newpos = tc_ctx(sm, p, pc.b) - p.T;  // the first of the T newest positions
        int win = pc.t0;  // first tile of the current window
        int ids = (win + lane < pc.t1) ? __ldg(table + win + lane) : 0;
        int nxt = (win + 32 + lane < pc.t1) ? __ldg(table + win + 32 + lane) : 0;
        for (int blk0 = pc.t0; blk0 < pc.t1; blk0 += 4) {
            if (blk0 - win == 32) {  // next window; fetch the one after it
                win = blk0;
                ids = nxt;
                nxt = (win + 32 + lane < pc.t1) ? __ldg(table + win + 32 + lane) : 0;
            }
            const int tiles = min(4, pc.t1 - blk0);
            if (!waited && (pc.f0 + blk0 + tiles) * 16 > newpos) {  // the stage holds a new position
                griddep_wait();
                waited = true;
            }
            const int w0 = blk0 - win;
            const int id = __shfl_sync(FULLM, ids, (w0 + (lane & 3)) & 31);
            const bool bad =
                __any_sync(FULLM, lane < tiles && (id < 0 || id >= p.num_blocks));
            const int my_id = __shfl_sync(FULLM, ids, (w0 + (bj & 3)) & 31);
            const int s = it % kStagesTc;
            if (lane == 0) {
                bool ok = true;
                if (it >= kStagesTc)
                    ok = mbar_wait(smem_addr(&sm.empty[s]), ((it / kStagesTc) - 1) & 1);
                if (!ok) tc_abort(sm, p);
                aborted = !ok || sm.abort_flag;
                if (!aborted) {
                    if (pw == 0) sm.bad[s] = bad ? 1 : 0;
                    if (bad && pw == 0) report(p.status, GQA_ERR_BLOCK_ID);
                    // each producer warp arrives once, expecting its own boxes' bytes
                    const int mine =
                        tiles > pw ? (tiles - pw + kProducerWarps - 1) / kProducerWarps : 0;
                    if (bad || mine == 0)
                        mbar_arrive(smem_addr(&sm.full[s]));
                    else
                        mbar_arrive_expect_tx(smem_addr(&sm.full[s]),
                                              (uint32_t)(mine * 2 * (H / 64) * 2048));
                }
            }
            aborted = __shfl_sync(FULLM, aborted, 0);
            if (aborted) break;
            // the stage's barrier expects this warp's bytes before its boxes are issued
            if (!bad && boxer && bj < tiles) {
                const uint32_t dst = smem_addr(stages + (size_t)s * kStageBytesTc) +
                                     (2 * kvsel + bh) * kHalfBytes + bj * 2048;
                tma_load_3d(dst, tm, smem_addr(&sm.full[s]), bh * 64, kv, my_id * 16, pol);
            }
            ++it;
        }
    }
    if (lane == 0 && aborted) {  // let copies already issued land before the CTA exits
        for (int j = max(0, it - kStagesTc); j < it; ++j)
            stage_landed(sm, j);
    }
}

// ---------------------------------------------------------------------------
// Box of a row chunk in the 5-D view (dim, head in group, KV head, token,
// sequence) of q and out.
struct TcBox {
    int h0, t0;  // first query head (within the group) and first new token of the chunk
};
__device__ __forceinline__ TcBox tc_box(const TcParams& p, int chunk) {
    TcBox x;
    x.h0 = (chunk % p.cpt) * p.hpc;
    x.t0 = (chunk / p.cpt) * p.tpc;
    return x;
}

// Lane 0 of warp kQWarp: the Q box of every piece, two 64-dim halves by TMA
// into the shared Q buffer (128-byte swizzled, as an MMA operand; rows past
// the box keep stale bytes: their S, P and O rows are never read).  The box
// of piece k is loaded once the MMA issuer's copy of box k - 1 into tensor
// memory has completed.
template <int H>
__device__ void tc_qloader(const CUtensorMap* tmq, const TcParams& p, uint8_t* qbuf, TcSmem& sm) {
    if ((threadIdx.x & 31) != 0) return;
    tma_prefetch_desc(tmq);
    if (p.early) griddep_wait();  // q follows earlier kernels
    TcWalker wk;
    wk.init(sm, p);
    TcPiece pc;
    int k = 0;
    const uint32_t bytes = (uint32_t)(H / 64) * 128u * (uint32_t)p.Rc;
    bool aborted = false;
    while (!aborted && wk.next(p, pc)) {
        if (k >= 1 && !mbar_wait(smem_addr(&sm.q_free), (k - 1) & 1)) tc_abort(sm, p);
        aborted = sm.abort_flag != 0;
        if (aborted) break;
        const TcBox x = tc_box(p, pc.v % p.C);
        const int kv = pc.v / p.C;
        mbar_arrive_expect_tx(smem_addr(&sm.q_full), bytes);
        for (int h = 0; h < H / 64; ++h)
            tma_load_5d(smem_addr(qbuf) + h * kRowHalfBytes, tmq, smem_addr(&sm.q_full), 64 * h, x.h0,
                        kv, x.t0, pc.b);
        ++k;
    }
    if (aborted && k >= 1) mbar_wait(smem_addr(&sm.q_full), (k - 1) & 1);  // the last box landed
}

// ---------------------------------------------------------------------------
// One elected thread issues every MMA.  Stage st of a piece belongs to
// softmax group g = st % 2.  When the piece's Q box has landed -- typically
// long before, right after the previous piece's last PVs have been issued --
// the issuer copies it into tensor memory (tcgen05.cp, in issue order after
// the previous piece's QK^T products that read the old Q; a commit then frees
// the shared buffer for the next box) and issues QK^T of the first two
// stages, which run while the softmax threads finish the previous piece; then,
// per stage, PV(st) as soon as group g has written P_g(st), and right after
// it QK^T(st + 2) into S_g, which group g has finished reading (it wrote P_g
// from it) once stage st + 2 has landed.  PV(st) goes first because its
// completion frees the ring slot of stage st for the producer (waiting for
// stage st + 2 before it would make the ring two stages shallower).  The first
// PV of a piece overwrites O_g and so also waits until the softmax threads
// have read the previous piece's O.  (Q is read from
// tensor memory, not shared memory, which keeps the A operand off the shared
// memory port that the ring's TMA writes also use.)  Operand descriptors are
// built once and only constants are added per instruction: an MMA whose
// descriptors were rebuilt in the issuing loop measured 130-200 cycles of
// issue each, and the issuer's queue holds only a few MMAs (the 14-bit address
// field cannot carry: shared memory ends below 256 KB).
template <bool BF16, int H>
__device__ void tc_mma(const TcParams& p, uint8_t* stages, uint8_t* qbuf, TcSmem& sm,
                       uint32_t tmem) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        constexpr uint32_t id_s = umma_idesc_ct(BF16, kRowsTc, 64, false);  // S = Q . K^T
        constexpr uint32_t id_o = umma_idesc_ct(BF16, kRowsTc, H, true);  // O += P . V
        const uint32_t st0 = smem_addr(stages);
        const uint64_t dk0 = umma_desc_sw128(st0, 16, 1024);                        // K, K-major
        const uint64_t dv0 = umma_desc_sw128(st0 + 2 * kHalfBytes, kHalfBytes, 1024); // V, MN-major
        const uint64_t dq = umma_desc_sw128(smem_addr(qbuf), 16, 1024);             // Q, K-major
        const uint32_t tQ = tmem + kColQ;
        // S_g = Q . K(n)^T (stage n came by TMA; Q is in tensor memory)
        auto issue_qk = [&](int n, int g) {
            const uint32_t tS = tmem + kColS + g * kColSStep;
            const uint64_t dk = dk0 + (uint64_t)((n % kStagesTc) * (kStageBytesTc >> 4));
#pragma unroll
            for (int kk = 0; kk < H / 16; ++kk)  // 16 head dims per MMA, 32 B along the 128-B row
                umma_ts(tS, tQ + 8 * kk, dk + (uint64_t)(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4),
                        id_s, kk > 0);
            umma_commit(smem_addr(&sm.s_ready[g]));
        };
        TcWalker wk;
        wk.init(sm, p);
        TcPiece pc;
        int n = 0, k = 0;
        int kp0 = 0, kp1 = 0;  // P_0 / P_1 writes consumed so far (barrier phases)
        bool ok = true;
        while (ok && wk.next(p, pc)) {
            const int nst = (pc.t1 - pc.t0 + 3) / 4;
            ok = mbar_wait(smem_addr(&sm.q_full), k & 1) && !sm.abort_flag && stage_landed(sm, n);
            if (ok) {
#pragma unroll
                for (int kk = 0; kk < H / 16; ++kk)  // the Q box into tensor memory, 32 B of each row at a time
                    tmem_cp_128x256b(tQ + 8 * kk,
                                     dq + (uint64_t)(((kk >> 2) * kRowHalfBytes + (kk & 3) * 32) >> 4));
                umma_commit(smem_addr(&sm.q_free));
                issue_qk(n, 0);
            }
            if (ok && nst > 1) {
                ok = stage_landed(sm, n + 1);
                if (ok) issue_qk(n + 1, 1);
            }
            for (int st = 0; st < nst && ok; ++st, ++n) {
                const int g = st & 1;
                const bool more = st + 2 < nst;
                ok = mbar_wait(smem_addr(&sm.p_ready[g]), (g ? kp1 : kp0) & 1) &&
                     (st >= 2 || k == 0 || mbar_wait(smem_addr(&sm.o_free), (k - 1) & 1));
                if (g)
                    ++kp1;
                else
                    ++kp0;
                if (!ok || sm.abort_flag) break;
                tc_fence_after();  // P_g was written by the softmax threads
                const uint32_t tO = tmem + kColO + g * kColOStep, tP = tmem + kColP + g * kColPStep;
                const uint64_t dv = dv0 + (uint64_t)((n % kStagesTc) * (kStageBytesTc >> 4));
                umma_ts(tO, tP, dv, id_o, st >= 2);
#pragma unroll
                for (int ks = 1; ks < 4; ++ks)  // 16 tokens per MMA
                    umma_ts(tO, tP + ks * 8, dv + (uint64_t)((ks * 2048) >> 4), id_o, true);
                umma_commit(smem_addr(&sm.o_ready[g]));
                umma_commit(smem_addr(&sm.empty[n % kStagesTc]));
                if (more) {
                    ok = stage_landed(sm, n + 2);
                    if (ok) issue_qk(n + 2, g);
                }
            }
            ++k;
            if (!ok) tc_abort(sm, p);
            if (sm.abort_flag) ok = false;
        }
        // every MMA issued so far has completed before tensor memory is freed
        umma_commit(smem_addr(&sm.done));
        if (!mbar_wait(smem_addr(&sm.done), 0)) tc_abort(sm, p);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// Pairwise reductions: a dependency depth of log2(N) instead of N.
template <int N>
__device__ __forceinline__ float max_tree(const float (&v)[N]) {
    float a[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) a[i] = fmaxf(v[2 * i], v[2 * i + 1]);
    if constexpr (N / 2 == 1) {
        return a[0];
    } else {
        return max_tree<N / 2>(a);
    }
}
template <int N>
__device__ __forceinline__ float sum_tree(const float (&v)[N]) {
    float a[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) a[i] = v[2 * i] + v[2 * i + 1];
    if constexpr (N / 2 == 1) {
        return a[0];
    } else {
        return sum_tree<N / 2>(a);
    }
}

// 32 output elements of this thread's row: fp32 values times inv, rounded to
// q's dtype.
template <bool BF16>
__device__ __forceinline__ void store_row32(uint4* dst, const uint32_t (&o)[32], float inv) {
    using E = Elt<BF16>;
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
        w[k] = E::pack(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

// Softmax group g = (warp - kSoftmaxWarp0) / 4: its warps reach tensor-memory
// lane quarters 3, 0, 1, 2 (a warp reaches lanes 32 * (warp % 4) .. + 31),
// one thread per query row.  The group runs the online softmax of the stages
// st = g, g + 2, ... of each piece into its own O_g.  At the piece's end the
// two threads of a row (one per group) exchange running max, sum and
// invalid-block flag through shared memory, each reads both groups' O over
// its half of the head dimension (g = 0: dims 0..63, g = 1: 64..127), frees
// O for the next piece's PV products, and combines them with log-sum-exp
// weights into the row's output -- staged in shared memory and written by
// one TMA store per half -- or into a split-segment partial.
template <bool BF16, int H>
__device__ void tc_softmax(const CUtensorMap* tmo, const TcParams& p, uint8_t* stages,
                           uint8_t* obuf, TcSmem& sm, uint32_t tmem) {
    using E = Elt<BF16>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int quarter = warp & 3;
    const int g = (warp - kSoftmaxWarp0) >> 2;  // softmax group; also its half of the output dims
    const int row = 32 * quarter + lane;
    const int tsm = threadIdx.x - 32 * kSoftmaxWarp0;  // 0..255 among the softmax threads
    const int tg = tsm & (kGroupThreads - 1);         // 0..127 within the group
    const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);
    const uint32_t tS = trow + kColS + g * kColSStep, tP = trow + kColP + g * kColPStep;
    const uint32_t tOg = trow + kColO + g * kColOStep;  // this group's accumulator
    // this thread's 128 bytes of the staged output (row, half g; 128-byte swizzle)
    const uint32_t ostage = smem_addr(obuf) + g * kRowHalfBytes + (row >> 3) * 1024 + (row & 7) * 128;
    if (tsm == 0) tma_prefetch_desc(tmo);
    if (p.early) griddep_wait();  // out, the workspace and the tree mask follow earlier kernels
    // sequences with an invalid length: zero outputs (CTA 0), status
    if (blockIdx.x == 0) {
        for (int b = tsm; b < p.B; b += kSoftmaxThreads) {
            if (tc_nblk(p, b) != 0) continue;
            report(p.status, GQA_ERR_CONTEXT);
            uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                (size_t)b * p.T * p.N * H);
            for (int i = 0; i < p.T * p.N * (H / 8); ++i) o[i] = make_uint4(0, 0, 0, 0);
        }
    }
    TcWalker wk;
    wk.init(sm, p);
    TcPiece pc;
    int n0 = 0;  // stages of earlier pieces
    int kg = 0;  // stages of this group so far (barrier phases of s_ready[g], o_ready[g])
    int pp = 0, ap = 0;  // phases of this thread's pair barrier and of the softmax barrier
    bool ok = true;
    // The staged rows (64 values of this thread's half, fp32 bit patterns)
    // times inv, in q's dtype, into the staging buffer; then, once every
    // softmax thread has written (and the store before has finished reading
    // the buffer), one thread stores the box by TMA.
    auto stage_row = [&](const uint32_t (&o)[64], float inv) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t w0 = E::pack(__uint_as_float(o[8 * j]) * inv, __uint_as_float(o[8 * j + 1]) * inv);
            const uint32_t w1 = E::pack(__uint_as_float(o[8 * j + 2]) * inv, __uint_as_float(o[8 * j + 3]) * inv);
            const uint32_t w2 = E::pack(__uint_as_float(o[8 * j + 4]) * inv, __uint_as_float(o[8 * j + 5]) * inv);
            const uint32_t w3 = E::pack(__uint_as_float(o[8 * j + 6]) * inv, __uint_as_float(o[8 * j + 7]) * inv);
            st_shared_v4(ostage + ((j ^ (row & 7)) << 4), make_uint4(w0, w1, w2, w3));
        }
        fence_proxy_async_shared();
    };
    auto store_box = [&](int b, int kv, const TcBox& x) {
        if (tsm == 0) {
            for (int h = 0; h < H / 64; ++h)
                tma_store_5d(tmo, smem_addr(obuf) + h * kRowHalfBytes, 64 * h, x.h0, kv, x.t0, b);
            bulk_commit();
        }
    };
    while (ok && wk.next(p, pc)) {
        __syncwarp();
        const int b = pc.b, kv = pc.v / p.C;
        const TcBox box = tc_box(p, pc.v % p.C);
        const int t = box.t0 + row / p.hpc, gg = box.h0 + row % p.hpc;
        const bool active = row < p.Rc && t < p.T && gg < p.G;
        // a warp whose rows are all padding skips the softmax arithmetic: the
        // lanes of its rows in S, P and O are never read out
        const bool warp_active = __any_sync(FULLM, active);
        const int ctx = tc_ctx(sm, p, b);
        const int nst = (pc.t1 - pc.t0 + 3) / 4;
        const int fn = ctx - p.T;             // position of the first new token
        const int lim = fn + (active ? t : 0);  // last position this row sees
        // tree rows: the new positions this row sees (its ancestors and itself)
        const uint64_t tmk = (p.tree_mask && active)
                                 ? (__ldg(p.tree_mask + (size_t)b * p.T + t) | (1ull << t))
                                 : 0ull;
        float m = -INFINITY, l = 0.f;
        bool bad = false;
        int mine = 0;  // this group's stages in this piece
        for (int st = g; st < nst && ok; st += 2, ++kg, ++mine) {
            const int n = n0 + st, s = n % kStagesTc;
            // stage n has landed (its bad-block flag and V rows are read below)
            ok = stage_landed(sm, n) && mbar_wait(smem_addr(&sm.s_ready[g]), kg & 1);
            ok = __all_sync(FULLM, ok);  // warp-collective tensor-memory accesses follow
            if (!ok) break;
            const int blk0 = pc.t0 + 4 * st;
            const int tok0 = (pc.f0 + blk0) * 16;
            const int tiles = min(4, pc.t1 - blk0);
            bad |= sm.bad[s] != 0;
            if (warp_active) {
                tc_fence_after();
                uint32_t sa[32], sb[32];
                tmem_ld32(tS, sa);
                tmem_ld32(tS + 32, sb);
                tmem_wait_ld();
                // visible columns of the stage as one word: loaded and causal ...
                const int vis_end = min(tiles * 16, lim + 1 - tok0);
                uint64_t vm = vis_end >= 64 ? ~0ull : vis_end <= 0 ? 0ull : (1ull << vis_end) - 1;
                if (p.window > 0) {  // ... above the row's window: lim - window < position
                    const int vis_beg = lim - p.window + 1 - tok0;
                    if (vis_beg > 0) vm &= vis_beg >= 64 ? 0ull : ~((1ull << vis_beg) - 1);
                }
                if (p.tree_mask) {  // ... and, among the new positions, on the row's tree path
                    const int d = fn - tok0;  // stage column of the first new token
                    if (d < 64) {
                        const uint64_t nbits = d >= 0 ? tmk << d : (-d < 64 ? tmk >> -d : 0ull);
                        const uint64_t nmask = d >= 0 ? ~0ull << d : ~0ull;
                        vm &= ~nmask | nbits;
                    }
                }
                float sv[64];
                if (__all_sync(FULLM, vm == ~0ull)) {  // a stage inside every row's context
#pragma unroll
                    for (int j = 0; j < 64; ++j) sv[j] = __uint_as_float(j < 32 ? sa[j] : sb[j - 32]);
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        sv[j] = (vm >> j) & 1ull ? __uint_as_float(j < 32 ? sa[j] : sb[j - 32]) : -INFINITY;
                }
                const float x = max_tree(sv) * p.scale_log2;
                // running max; O_g is rescaled (lazily) in tensor memory, warp by warp
                const bool need = x > m + kGapTc;
                if (__any_sync(FULLM, need)) {
                    const float f = (need && m != -INFINITY) ? fast_exp2(m - x) : 1.f;
                    if (mine > 0) {  // PV of this group's previous stage has completed
                        ok = __all_sync(FULLM, mbar_wait(smem_addr(&sm.o_ready[g]), (kg - 1) & 1));
                        if (!ok) break;
                        tc_fence_after();
    #pragma unroll 1
                        for (int c = 0; c < H / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tOg + 32 * c, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
                            tmem_st32(tOg + 32 * c, o);
                        }
                        tmem_wait_st();
                    }
                    if (need) {
                        l *= f;
                        m = x;
                    }
                }
                const float nref = (m == -INFINITY) ? 0.f : -m;
                uint32_t pw[32];
                float ps[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    pw[k] = E::pack(fast_exp2(fmaf(sv[2 * k], p.scale_log2, nref)),
                                         fast_exp2(fmaf(sv[2 * k + 1], p.scale_log2, nref)));
                    ps[k] = E::lo(pw[k]) + E::hi(pw[k]);
                }
                l += sum_tree(ps);
                if (mine > 0) {  // the previous PV of this group has read P_g
                    ok = __all_sync(FULLM, mbar_wait(smem_addr(&sm.o_ready[g]), (kg - 1) & 1));
                    if (!ok) break;
                    tc_fence_after();
                }
                tmem_st32(tP, pw);
                tmem_wait_st();
            }  // warp_active
            // V rows without data in this stage -- past the context, or below
            // every new token's window (a block partly inside it may hold
            // anything there): zero them (NaN-safe products)
            const int valid_rows = max(0, min(tiles * 16, ctx - tok0));
            const int low_rows =
                p.window > 0 ? min(valid_rows, max(0, fn - p.window + 1 - tok0)) : 0;
            if (valid_rows < 64 || low_rows > 0) {
                const uint32_t vb = smem_addr(stages + (size_t)s * kStageBytesTc) + 2 * kHalfBytes;
                const int nz = 64 - valid_rows + low_rows;  // rows [0, low) and [valid, 64)
                constexpr int kChunks = H / 8;  // 16-byte chunks per row
                for (int i = tg; i < nz * kChunks; i += kGroupThreads) {
                    const int k = i / kChunks;
                    const int rr = k < low_rows ? k : valid_rows + (k - low_rows);
                    const int c = i % kChunks, h = c >> 3, cc = c & 7;
                    st_shared_v4(vb + h * kHalfBytes + (rr >> 3) * 1024 + (rr & 7) * 128 +
                                     ((cc ^ (rr & 7)) << 4),
                                 make_uint4(0, 0, 0, 0));
                }
                fence_proxy_async_shared();
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&sm.p_ready[g]));
        }
        n0 += nst;
        // ---- the piece's rows: the two groups' results meet ------------------------
        // The first piece of a split segment ends its CTA's range, so the
        // other pieces have usually drawn their tickets by now: read the
        // count (its latency overlaps the meeting below).
        const int first_cta = (int)(pc.first / sm.quota);
        const int last_cta = (int)((pc.first + pc.nb - 1) / sm.quota);
        const int wi = warp - kSoftmaxWarp0;  // this warp's ticket among the CTA's eight
        unsigned seen = 0u;
        if (lane == 0 && first_cta != last_cta && (int)blockIdx.x == first_cta)
            seen = tc_ticket_seen(p.flags + 8 * first_cta + wi);
        if (ok && mine > 0) {  // this group's last PV has completed
            ok = mbar_wait(smem_addr(&sm.o_ready[g]), (kg - 1) & 1);
            tc_fence_after();
        }
        ok = __all_sync(FULLM, ok);
        sm.xm[g][row] = m;
        sm.xl[g][row] = l;
        sm.xb[g][row] = bad ? 1 : 0;
        tc_fence_before();
        mbar_arrive(smem_addr(&sm.pair[quarter]));
        ok = __all_sync(FULLM, ok && mbar_wait(smem_addr(&sm.pair[quarter]), pp & 1));
        ++pp;
        if (!ok) {
            tc_abort(sm, p);
            break;
        }
        tc_fence_after();  // both groups' last PVs (and so every MMA of the piece) completed
        const float m0 = sm.xm[0][row], m1 = sm.xm[1][row];
        const float M = fmaxf(m0, m1);
        const float w0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M);
        const float w1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M);
        float lt = w0 * sm.xl[0][row] + w1 * sm.xl[1][row];
        bad = (sm.xb[0][row] | sm.xb[1][row]) != 0;
        // this thread's half of the dims: w0 O_0 + w1 O_1 (a group without
        // stages in this piece has weight 0 and is not read); then O is free
        uint32_t o[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t a0[32], a1[32];
            tmem_ld32(trow + kColO + 64 * g + 32 * c, a0);
            tmem_ld32(trow + kColO + kColOStep + 64 * g + 32 * c, a1);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k)
                o[32 * c + k] = __float_as_uint((w0 != 0.f ? w0 * __uint_as_float(a0[k]) : 0.f) +
                                                (w1 != 0.f ? w1 * __uint_as_float(a1[k]) : 0.f));
        }
        tc_fence_before();
        mbar_arrive(smem_addr(&sm.o_free));
        // this thread's rows and dims of the output (H = 64: group 0 holds all
        // the dims, group 1 none -- it still takes its part in the meetings and
        // tickets below)
        const bool mine_out = active && 64 * g < H;
        if (first_cta == last_cta) {  // the whole segment: O / l in q's dtype
            const bool zero = bad || !(lt > 0.f);  // an invalid block id: zeros
            if (zero) {
#pragma unroll
                for (int k = 0; k < 64; ++k) o[k] = 0u;
            }
            if (tsm == 0) bulk_wait_read();  // the previous box has left the staging buffer
            ok = softmax_bar(sm, ap);
            if (mine_out) stage_row(o, zero ? 0.f : 1.f / lt);
            ok = __all_sync(FULLM, ok && softmax_bar(sm, ap));
            if (!ok) {
                tc_abort(sm, p);
                break;
            }
            store_box(b, kv, box);
            continue;
        }
        // ---- a piece of a split segment -------------------------------------------
        // If this is the first piece and every other piece's warp has drawn
        // its ticket, fold them in now.  Otherwise each warp publishes its
        // rows of the piece (partial O over its 64 dims, max, sum; slot 1 for
        // the segment's first piece, which ends its CTA's range, slot 0 for
        // the others, which start theirs) and takes a ticket, and the warp
        // that draws the last one folds.  The fold runs over the pieces in CTA
        // order from the first piece's state; the merging warp stores its 32
        // rows x 64 dims with plain stores and resets the ticket for the next
        // call.  No warp waits for another CTA.
        const int me = blockIdx.x;
        const int npieces = last_cta - first_cta + 1;
        const bool early = me == first_cta && __shfl_sync(FULLM, seen, 0) == (unsigned)(npieces - 1);
        if (mine_out && !early) {
            float* part = p.partials + ((size_t)me * 2 + (me == first_cta ? 1 : 0)) * kPartFloats;
#pragma unroll
            for (int k = 0; k < 64; ++k)
                __stcg(part + (64 * g + k) * kRowsTc + row, __uint_as_float(o[k]));
            __stcg(part + (128 + 2 * g) * kRowsTc + row, M);
            __stcg(part + (129 + 2 * g) * kRowsTc + row, bad ? -1.f : lt);  // -1: a bad block
        }
        __syncwarp();  // the lanes' stores before lane 0's ticket
        if (!early) {
            unsigned drawn = 0;
            if (lane == 0) drawn = tc_ticket(p.flags + 8 * first_cta + wi);
            drawn = __shfl_sync(FULLM, drawn, 0);
            if (drawn != (unsigned)(npieces - 1)) continue;  // another piece's warp merges
        }
        __syncwarp();  // lane 0's acquire before every lane's reads of the partials
        if (mine_out) {
            // online fold over the pieces in CTA order: running max MM, sum L
            // (< 0 marks a piece with an invalid block), unnormalized values o
            float MM = M, L = bad ? -1.f : lt;
            if (me != first_cta) {  // start from the first piece's stored state
                const float* pf = p.partials + ((size_t)first_cta * 2 + 1) * kPartFloats;
                MM = __ldcg(pf + (128 + 2 * g) * kRowsTc + row);
                L = __ldcg(pf + (129 + 2 * g) * kRowsTc + row);
#pragma unroll
                for (int k = 0; k < 64; ++k)
                    o[k] = __float_as_uint(__ldcg(pf + (64 * g + k) * kRowsTc + row));
            }
            bool any_bad = L < 0.f;
            for (int c = first_cta + 1; c <= last_cta; ++c) {
                const float* pp_ = p.partials + (size_t)c * 2 * kPartFloats;  // slot 0
                const float mc = __ldcg(pp_ + (128 + 2 * g) * kRowsTc + row);
                const float lc = __ldcg(pp_ + (129 + 2 * g) * kRowsTc + row);
                float v[64];
#pragma unroll
                for (int k = 0; k < 64; ++k) v[k] = __ldcg(pp_ + (64 * g + k) * kRowsTc + row);
                any_bad |= lc < 0.f;
                const float mn = fmaxf(MM, mc);
                const float a = MM == -INFINITY ? 0.f : fast_exp2(MM - mn);
                const float bw = mc == -INFINITY ? 0.f : fast_exp2(mc - mn);
#pragma unroll
                for (int k = 0; k < 64; ++k)
                    o[k] = __float_as_uint((a != 0.f ? a * __uint_as_float(o[k]) : 0.f) +
                                           (bw != 0.f ? bw * v[k] : 0.f));
                L = (a != 0.f ? a * L : 0.f) + (bw != 0.f ? bw * lc : 0.f);
                MM = mn;
            }
            const bool zero = any_bad || !(L > 0.f);
            // this row's 64 dims of half g, in q's dtype
            uint4* dst = reinterpret_cast<uint4*>(
                static_cast<uint16_t*>(p.out) +
                (((size_t)b * p.T + t) * p.N + (size_t)kv * p.G + gg) * H + 64 * g);
            const float inv = zero ? 0.f : 1.f / L;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t w4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w4[e] = zero ? 0u
                                 : E::pack(__uint_as_float(o[8 * j + 2 * e]) * inv,
                                           __uint_as_float(o[8 * j + 2 * e + 1]) * inv);
                dst[j] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
        __syncwarp();
        if (lane == 0) p.flags[8 * first_cta + wi] = 0;  // ready for the next call
    }
    if (tsm == 0) bulk_wait_read();  // the staging buffer is read before the CTA leaves
}

template <bool BF16, int H>
__global__ void __launch_bounds__(kThreadsTc, 1)
    tc_attention_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv,
                        const __grid_constant__ CUtensorMap tmq,
                        const __grid_constant__ CUtensorMap tmo, const TcParams p) {
    // shared memory (1024-byte aligned): the K / V ring, the Q box (A operand
    // of QK^T), the output staging box, the barriers and scratch
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = base;
    uint8_t* qbuf = stages + (size_t)kStagesTc * kStageBytesTc;
    uint8_t* obuf = qbuf + 2 * kRowHalfBytes;
    TcSmem& sm = *reinterpret_cast<TcSmem*>(obuf + 2 * kRowHalfBytes);
    const int warp = threadIdx.x >> 5;
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesTc; ++s) {
            mbar_init(smem_addr(&sm.full[s]), kProducerWarps);
            mbar_init(smem_addr(&sm.empty[s]), 1);
            sm.bad[s] = 0;
        }
        mbar_init(smem_addr(&sm.q_full), 1);
        mbar_init(smem_addr(&sm.q_free), 1);
        mbar_init(smem_addr(&sm.o_free), kSoftmaxThreads);
        for (int g = 0; g < 2; ++g) {
            mbar_init(smem_addr(&sm.s_ready[g]), 1);
            mbar_init(smem_addr(&sm.p_ready[g]), kGroupThreads);
            mbar_init(smem_addr(&sm.o_ready[g]), 1);
        }
        for (int q = 0; q < 4; ++q) mbar_init(smem_addr(&sm.pair[q]), 2 * 32);
        mbar_init(smem_addr(&sm.all), kSoftmaxThreads);
        mbar_init(smem_addr(&sm.done), 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
    // q, the caches, the lengths, the workspace and out follow earlier kernels;
    // with early KV the lengths and tables may be read now and the roles wait
    // before their first access to anything else (the MMA issuer touches no
    // global memory)
    if (!p.early) griddep_wait();
    if (warp == 0) tc_plan(p, sm);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    if (warp == 0)
        tc_mma<BF16, H>(p, stages, qbuf, sm, tmem);
    else if (warp < kQWarp)
        tc_producer<H>(&tmk, &tmv, p, stages, sm, warp - 1);
    else if (warp == kQWarp)
        tc_qloader<H>(&tmq, p, qbuf, sm);
    else
        tc_softmax<BF16, H>(&tmo, p, stages, obuf, sm, tmem);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

constexpr size_t kSmemTc =
    1024 + (size_t)kStagesTc * kStageBytesTc + 4 * (size_t)kRowHalfBytes + sizeof(TcSmem);
static_assert(kSmemTc <= 227 * 1024, "shared memory per CTA");

}  // namespace

bool tc_attention_supported(const gqa_shape& s) {
    return (s.H == 64 || s.H == 128) && s.kv_dtype == GQA_KV_SAME && s.block_size == 16 &&
           (long long)s.T * (s.N / s.K) <= 8192;
}

bool tc_attention_preferred(const gqa_shape& s) {
    return tc_attention_supported(s) && (long long)s.T * (s.N / s.K) >= kTcMinRows;
}

size_t tc_workspace_bytes(const gqa_shape& s, size_t flags_bytes) {
    if (!tc_attention_supported(s)) return 0;
    const int sms = device_sm_count();
    if (sms < 1) return 0;
    return flags_bytes + (size_t)sms * 2 * kPartFloats * sizeof(float);  // two slots per CTA
}

gqa_status launch_tc_attention(const gqa_shape& s, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               const int32_t* context_lens, const uint64_t* tree_mask, void* out,
                               void* workspace, size_t flags_bytes, int32_t* dev_status,
                               cudaStream_t stream) {
    if (!tc_attention_supported(s)) return GQA_ERR_SHAPE;
    if (s.B == 0) return GQA_OK;
    // the shared-memory opt-in, once per device (no attribute calls later, so
    // that launches can be captured into CUDA graphs)
    {
        static std::mutex mu;
        static bool done[64] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GQA_ERR_CUDA;
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            const void* kerns[4] = {reinterpret_cast<const void*>(&tc_attention_kernel<true, 128>),
                                    reinterpret_cast<const void*>(&tc_attention_kernel<false, 128>),
                                    reinterpret_cast<const void*>(&tc_attention_kernel<true, 64>),
                                    reinterpret_cast<const void*>(&tc_attention_kernel<false, 64>)};
            for (const void* k : kerns)
                if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemTc) != cudaSuccess)
                    return GQA_ERR_CUDA;
            done[dev] = true;
        }
    }
    // row chunks: boxes of tpc new tokens x hpc query heads of one KV head
    const int G = s.N / s.K;
    int tpc, hpc, cpt;
    if (G <= kRowsTc) {
        hpc = G;
        cpt = 1;
        tpc = std::min(s.T, kRowsTc / G);
    } else {
        cpt = (G + kRowsTc - 1) / kRowsTc;
        hpc = (G + cpt - 1) / cpt;
        tpc = 1;
    }
    CUtensorMap tmk, tmv, tmq, tmo;
    if (!make_cache_map(&tmk, k_cache, s) || !make_cache_map(&tmv, v_cache, s) ||
        !make_rows_map(&tmq, q, s, hpc, tpc) || !make_rows_map(&tmo, out, s, hpc, tpc))
        return GQA_ERR_CUDA;
    TcParams p;
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.tree_mask = tree_mask;
    p.status = dev_status;
    p.flags = static_cast<int32_t*>(workspace);
    p.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + flags_bytes);
    p.B = s.B;
    p.T = s.T;
    p.N = s.N;
    p.K = s.K;
    p.G = G;
    p.tpc = tpc;
    p.hpc = hpc;
    p.cpt = cpt;
    p.C = cpt * ((s.T + tpc - 1) / tpc);
    p.Rc = tpc * hpc;
    p.KC = s.K * p.C;
    p.max_blocks = s.max_blocks_per_seq;
    p.num_blocks = s.num_blocks;
    p.early = (s.flags & GQA_FLAG_EARLY_KV) ? 1 : 0;
    p.window = s.window;
    const double scale = s.scale > 0.f ? (double)s.scale : 1.0 / sqrt((double)s.H);
    p.scale_log2 = (float)(scale * 1.4426950408889634);
    const int sms = device_sm_count();
    if (sms < 1) return GQA_ERR_CUDA;
    // at most one CTA per SM, and no more than the tiles allow at the minimum
    // quota (upper bound: every sequence at full capacity)
    const long long tiles_max = (long long)s.B * p.KC * (s.max_blocks_per_seq + kSegCost);
    const long long grid = std::min<long long>(
        sms, std::max<long long>(1, (tiles_max + kQuotaMinTc - 1) / kQuotaMinTc));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreadsTc);
    cfg.dynamicSmemBytes = kSmemTc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (s.flags & (GQA_FLAG_PDL | GQA_FLAG_EARLY_KV)) ? 1 : 0;
    const cudaError_t e =
        s.dtype == GQA_BF16
            ? (s.H == 64 ? cudaLaunchKernelEx(&cfg, tc_attention_kernel<true, 64>, tmk, tmv, tmq, tmo, p)
                         : cudaLaunchKernelEx(&cfg, tc_attention_kernel<true, 128>, tmk, tmv, tmq, tmo, p))
            : (s.H == 64 ? cudaLaunchKernelEx(&cfg, tc_attention_kernel<false, 64>, tmk, tmv, tmq, tmo, p)
                         : cudaLaunchKernelEx(&cfg, tc_attention_kernel<false, 128>, tmk, tmv, tmq, tmo, p));
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
