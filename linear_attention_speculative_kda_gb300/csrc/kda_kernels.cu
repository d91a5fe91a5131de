// KDA speculative verify / commit / flush kernels and the C ABI (sm_103a).
//
// The operations are those of the RecoverSSM pages:
//  - verify: recoverssm.py `_verify_kernel` (one checkpoint read per row and
//    head, per-token recurrence, bf16 outputs, raw records, no state store),
//    plus the deferred fold of the Kimi-K3 context page (the next verify
//    replays the pending accepted tokens in the same pass);
//  - commit: `_prepare_commit_plan_kernel` (commit length and validity) and
//    the replay of `Glm5NextRecoverSSMCommitContext.commit`, restricted to
//    the accepted tokens, with the deferred variant of
//    `KDADeferredCommitContext.commit` (pending / eager);
//  - flush: `KDADeferredCommitContext.flush`;
//  - with correction records (the Kimi-K3 context page's fp32 corrections),
//    the verify also records each token's delta, and the commit, the fold
//    and the flush apply the deltas without the prediction S k^.
// A verify item with 5 or more new tokens computes its outputs in the
// window form (kda_device.cuh); every stored state is computed token by
// token.  The public contract is in include/kda.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "kda_align.cuh"
#include "kda_async.cuh"
#include "kda_device.cuh"
#include "../../include/kda.h"

namespace kda {

static_assert(kRecStride == KDA_RECORD_STRIDE, "record layout mismatch");
static_assert(kCorrBytes == KDA_CORRECTION_RECORD_BYTES, "correction record layout mismatch");
static_assert(kD == KDA_HEAD_DIM, "head dim mismatch");
static_assert(kMaxQ == KDA_MAX_WINDOW, "window mismatch");
static_assert(kBadLength == KDA_ROW_BAD_LENGTH && kBadSlot == KDA_ROW_BAD_SLOT &&
                  kBadRecord == KDA_ROW_BAD_RECORD && kBadPending == KDA_ROW_BAD_PENDING &&
                  kErrWaitTimeout == KDA_ERR_WAIT_TIMEOUT && kBadBlock == KDA_ROW_BAD_BLOCK,
              "error-word bits mismatch");

// Row metadata shared by all kernels: token range, slot and record slot,
// with the device-side checks.  Returns the error bits (0: usable row).
struct Row {
    int bos, T, slot, r;
};

__device__ __forceinline__ int read_row(const Params &p, int b, bool need_len, Row &row) {
    int bad = 0;
    row.bos = 0;
    row.T = 0;
    if (need_len) {
        row.bos = p.cu_seqlens[b];
        row.T = p.cu_seqlens[b + 1] - row.bos;
        if (row.T < 0 || row.T > p.Q) bad |= kBadLength;
    }
    row.slot = p.state_indices[b];
    if (row.slot >= p.S) bad |= kBadSlot;
    row.r = p.record_rows != nullptr ? p.record_rows[b] : b;
    if (row.r < -1 || row.r >= p.R) bad |= kBadRecord;
    return bad;
}

__device__ __forceinline__ __nv_bfloat16 *record_base(const Params &p, int r, int head) {
    return p.records + ((size_t)(r + 1) * p.H + head) * (size_t)p.Q * kRecStride;
}

// Correction records: kCorrBytes per token, same (r + 1, head, token) order.
__device__ __forceinline__ unsigned char *corr_base(const Params &p, int r, int head) {
    return reinterpret_cast<unsigned char *>(p.records) +
           ((size_t)(r + 1) * p.H + head) * (size_t)p.Q * kCorrBytes;
}

// ------------------------------------------------------------- work items --
//
// A work item is one (row, head) tile with something to do.  Mode decides
// what: the verify runs `p` folded (pending) record tokens then `T` new
// tokens; the commit and the flush replay `p` record tokens.  Every mode
// stores the state after the p-th token, to slot `dst` (the row's own slot,
// or the final block of an align-mode commit); an align-mode commit also
// stores the state after `mid_len` tokens to block `mid` (0: none).

enum class Mode { kVerify, kCommit, kFlush };

struct Work {
    int tile;  // -1: none
    int head, slot, r, bos, T, p;
    int dst, mid, mid_len;
};

// Align-mode targets of a committing row of request `req` (the plan is in
// kda_align.cuh): the final block, and the boundary block when the boundary
// comes before the last token (a boundary at the last token is the final
// block itself).  Returns the error bits; w.dst = 0 when the row commits
// nothing.
__device__ __forceinline__ int align_targets(const Params &p, int req, int n, Work &w) {
    const kda_blocks::Blocks bl = kda_blocks::plan(p.block_table + (long long)req * p.bt_stride,
                                                 p.bt_width, p.block_size, p.num_computed[req], n);
    if (bl.bad) return kBadBlock;
    if (bl.final_block >= p.S || bl.boundary >= p.S) return kBadSlot;
    w.dst = bl.final_block > 0 ? bl.final_block : 0;
    w.mid = (bl.boundary > 0 && bl.boundary_len < n) ? bl.boundary : 0;
    w.mid_len = w.mid > 0 ? bl.boundary_len : 0;
    return 0;
}

// Plan row b for head `head`: row checks, the commit plan (n = clamp(accepted,
// 0, min(T, Q)), valid iff slot > 0, n > 0, r >= 0), the deferred commit's
// pending write.  Every head of a row has the same plan.  The row's side
// effects (error bits, pending writes) are made only when `side_effects` is
// set, by the one thread of the grid that plans the row for that purpose.
template <Mode kMode>
__device__ __forceinline__ bool plan_row(const Params &p, int b, int head, bool side_effects,
                                         Work &w) {
    Row row;
    const int bad = read_row(p, b, kMode != Mode::kFlush, row);
    if (bad) {
        if (side_effects) {
            flag_error(p.err, bad);
            // a deferred commit clears the pending count of a skipped row
            // whose record slot is usable: its records are this step's, so
            // the previous step's count no longer describes them
            if (kMode == Mode::kCommit && p.pending_out != nullptr && !(bad & kBadRecord) &&
                row.r >= 0)
                p.pending_out[row.r] = 0;
        }
        return false;
    }
    int fold = 0, T = 0;
    if constexpr (kMode == Mode::kVerify) {
        if (row.slot <= 0) return false;  // null block: padding row
        if (p.pending_in != nullptr && row.r >= 0) {
            fold = p.pending_in[row.r];
            if (fold < 0 || fold > p.Q) {
                if (side_effects) flag_error(p.err, kBadPending);
                return false;
            }
        }
        T = row.T;
        if (T == 0 && fold == 0) return false;
    } else if constexpr (kMode == Mode::kCommit) {
        // align mode reads the accepted count, num_computed and the block
        // table of the row's request
        int req = b;
        if (p.block_table != nullptr) {
            if (p.request_indices != nullptr) req = p.request_indices[b];
            if (req < 0 || req >= p.num_requests) {
                if (side_effects) {
                    flag_error(p.err, kBadBlock);
                    if (p.pending_out != nullptr && row.r >= 0) p.pending_out[row.r] = 0;
                }
                return false;
            }
        }
        const int n = min(max(p.num_accepted[req], 0), min(row.T, p.Q));
        bool valid = row.slot > 0 && n > 0 && row.r >= 0;
        w.dst = row.slot;
        w.mid = 0;
        w.mid_len = 0;
        if (p.block_table != nullptr && valid) {
            const int bad_align = align_targets(p, req, n, w);
            if (bad_align) {
                if (side_effects) {
                    flag_error(p.err, bad_align);
                    if (p.pending_out != nullptr && row.r >= 0) p.pending_out[row.r] = 0;
                }
                return false;
            }
            valid = w.dst > 0;
        }
        if (p.pending_out != nullptr) {
            // deferred: eager rows commit now; in align mode so does a row
            // whose final block is not its own slot or that owes a boundary
            // block (the later fold stores to the row's slot only)
            bool now = p.eager != nullptr && p.eager[b] != 0;
            if (p.block_table != nullptr && valid) now = now || w.dst != row.slot || w.mid > 0;
            if (side_effects && row.r >= 0) p.pending_out[row.r] = (valid && !now) ? n : 0;
            if (!now) return false;
        }
        if (!valid) return false;
        fold = n;
    } else {
        if (row.slot <= 0 || row.r < 0) return false;
        const int n = p.pending_in[row.r];
        if (n < 0 || n > p.Q) {
            if (side_effects) flag_error(p.err, kBadPending);
            return false;
        }
        if (n == 0) return false;
        fold = n;
    }
    w.tile = b * p.H + head;
    w.head = head;
    w.slot = row.slot;
    w.r = row.r;
    w.bos = row.bos;
    w.T = T;
    w.p = fold;
    if constexpr (kMode != Mode::kCommit) {
        w.dst = row.slot;
        w.mid = 0;
        w.mid_len = 0;
    }
    return true;
}

// ------------------------------------------------------------------ roles --
//
// One CTA per SM, 384 threads in three warpgroups:
//  - consumers 0 and 1 (128 threads each) each own one tile in registers at
//    a time and run its tokens;
//  - the producer (4 warps) plans the CTA's work, asks the TMA unit to stage
//    each item's checkpoint into its consumer's shared-memory buffer, brings
//    the raw inputs in with cp.async and prepares the per-token vectors
//    ahead of the consumers (double-buffered when shared memory allows).
// Items alternate between the two consumers.  Hand-offs use mbarriers; every
// wait is bounded and gives up (error bit KDA_ERR_WAIT_TIMEOUT, all roles
// leave) instead of hanging.

constexpr int kConsumerThreads = 128;
constexpr int kProducerWarps = 4;
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr int kBlockThreads = 2 * kConsumerThreads + kProducerThreads;
constexpr int kProducerBarrier = 1;  // named barrier of the producer warps
// A verify item with at least this many new tokens runs them in window form
// (kWindow kernels).  Measured on GB300: items of 8 tokens gain (dflash7's
// verify 115 -> 103 us), mixed lengths gain when only their longer items
// take it (mixed's verify 297 -> 288 us; all items: no gain), and windows of
// 4 tokens lose (deferred2's verify 245 -> 272 us).
constexpr int kWindowMinT = 5;
// The tensor window form (window items' row products on the tensor core) is
// a build option, off by default: measured on the window-8 workload
// (256 requests x 16 heads) its verify took 111 us against 88 us for the
// FMA window form.  Per item, each of its 32 tcgen05.mma of 128 x 32 x 8
// takes about 80 to 130 cycles to issue, the staging buffer stays held until
// the products finish, and the coefficients and the solve, unchanged,
// dominate the consumer's chain.
#ifdef KDA_TENSOR_WINDOW
constexpr bool kTensorWindow = true;
#else
constexpr bool kTensorWindow = false;
#endif
constexpr int kPlanSize = kProducerThreads;
#ifdef KDA_TEST_WAIT_BUDGET
// a test build: a short budget, so that a wait the test starves runs out fast
constexpr long long kWaitBudget = KDA_TEST_WAIT_BUDGET;
#else
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (about 2 s)
#endif
constexpr int kSmemBudget = 227 * 1024;
constexpr int kLaunchRegs = 168;     // 65536 / 384, rounded down to a multiple of 8
constexpr int kConsumerRegs = 208;
constexpr int kProducerRegs = 88;
static_assert(2 * kConsumerThreads * kConsumerRegs + kProducerThreads * kProducerRegs <=
                  kBlockThreads * kLaunchRegs,
              "register split exceeds the launch allocation");

template <int N>
__device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

struct ItemInfo {
    int tile, slot, head, bos, T, p, end;
    int dst, mid, mid_len, r, pad;
};

struct WorkList {
    int tile[kPlanSize];
    int slot[kPlanSize];
    int r[kPlanSize];
    int bos[kPlanSize];
    int tp[kPlanSize];   // T | p << 8 | head << 16
    int dst[kPlanSize];
    int mid[kPlanSize];  // boundary block, or 0
    int mid_len[kPlanSize];
    int warp_count[kProducerWarps];
    int count;
    int rows_per_thread;  // balanced plan: rows each producer thread scans (0: strided plan)
    // balanced plan (when shared memory has room for it): mask[t] bit i
    // marks row t * rows_per_thread + i as having work; prefix[t] counts the
    // work rows of the threads before t
    unsigned *mask;
    int *prefix;
};

struct Balance {
    unsigned mask[kPlanSize];
    int prefix[kPlanSize + 1];
    int pad[3];
};

// Hand-off barriers and the abort flag.
struct Sync {
    uint64_t full_state[2];    // TMA of a consumer's checkpoint landed
    uint64_t empty_state[2];   // the consumer has copied it into registers
    uint64_t full_tok[2][2];   // token vectors of an item are ready
    uint64_t empty_tok[2][2];  // the consumer is done with them
    uint64_t group[2];         // a consumer's own barrier (window form)
    uint64_t mma_hi[2];        // a consumer's products from the staging buffer are complete
    uint64_t mma_done[2];      // all of a consumer's tensor-core products are complete
    ItemInfo info[2][2];
    uint32_t tmem_base;        // tensor memory of the CTA (tensor window form)
    int abort;
    int leave[2];   // per item parity: the producer threads leave (abort seen)
    int pad;
};

// Raw bf16 inputs and gate parameters of one item, in channel pairs.  With
// correction records a token's v slot is twice as wide (kD words): a recorded
// token's fp32 delta, or a new token's bf16 v in its first half.
template <bool kCorr>
struct RawView {
    static constexpr int kVWords = kCorr ? kD : kD / 2;  // 32-bit words per v slot
    uint32_t *k, *v, *g, *q;
    uint2 *tail;                // record tails: beta_raw bits in the low half
    float *bias;                // g_bias of the item's head (128)
    float *a_log;
    uint32_t *beta_new;         // beta_raw bits of the new tokens
    __device__ __forceinline__ RawView(unsigned char *base, int slots, int Q) {
        k = reinterpret_cast<uint32_t *>(base);
        v = k + slots * (kD / 2);
        g = v + slots * kVWords;
        q = g + slots * (kD / 2);
        tail = reinterpret_cast<uint2 *>(q + Q * (kD / 2));
        bias = reinterpret_cast<float *>(tail + ((Q + 1) / 2) * 2);
        a_log = bias + kD;
        beta_new = reinterpret_cast<uint32_t *>(a_log + 4);
    }
};

__host__ __device__ inline int raw_buffer_bytes(int slots, int Q, bool corr) {
    return slots * (corr ? 4 : 3) * (kD * 2) + Q * (kD * 2) + ((Q + 1) / 2) * 16 + kD * 4 + 16 +
           ((Q * 4 + 15) / 16) * 16;
}

// Shared-memory layout of a launch (window Q, whether the verify folds, the
// record format, whether it is a window kernel).  A window kernel of the
// tensor window form uses the head token layout: every token buffer and
// staging buffer sits on a 1024-byte boundary of the (1024-byte aligned)
// dynamic shared memory.
struct Layout {
    int slots, nbuf, tok_bytes, raw_bytes;
    int off_state, off_tok, off_raw, off_list, off_sync, off_bal, total;
    bool head;
};

__host__ __device__ inline Layout make_layout(int Q, bool fold, bool corr, bool window) {
    Layout l;
    l.slots = fold ? 2 * Q : Q;
    l.head = window && kTensorWindow;
    l.tok_bytes = tok_buffer_bytes(l.slots, Q, l.head);
    l.raw_bytes = raw_buffer_bytes(l.slots, Q, corr);
    l.off_state = 0;                                // 2 x 64 KiB staging
    l.off_tok = 2 * kD * kD * 4;
    const int fixed = l.off_tok + 2 * l.raw_bytes + (int)sizeof(WorkList) + (int)sizeof(Sync);
    l.nbuf = fixed + 4 * l.tok_bytes <= kSmemBudget ? 2 : 1;
    l.off_raw = l.off_tok + 2 * l.nbuf * l.tok_bytes;
    l.off_list = l.off_raw + 2 * l.raw_bytes;
    l.off_sync = l.off_list + (int)sizeof(WorkList);
    l.total = l.off_sync + (int)sizeof(Sync);
    // the balanced plan's arrays, where they fit (else the strided plan)
    l.off_bal = l.total + (int)sizeof(Balance) <= kSmemBudget ? l.total : -1;
    if (l.off_bal >= 0) l.total += (int)sizeof(Balance);
    return l;
}

// Bounded wait shared by all roles: gives up on timeout or when another
// role has given up.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, Sync &sy,
                                           const Params &p) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int *>(&sy.abort)) return false;
        if (clock64() - t0 > kWaitBudget) {
            *reinterpret_cast<volatile int *>(&sy.abort) = 1;
            flag_error(p.err, kErrWaitTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ void producer_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(kProducerBarrier), "n"(kProducerThreads) : "memory");
}

// Candidate tiles of this CTA: of the balanced plan's work tiles, or of all
// tiles (the strided plan), every gridDim.x-th from blockIdx.x.
__device__ __forceinline__ int num_candidates(const WorkList &list, int num_tiles, int H) {
    const int total = list.rows_per_thread > 0 ? list.prefix[kPlanSize] * H : num_tiles;
    const int first = (int)blockIdx.x;
    return first < total ? (total - first + (int)gridDim.x - 1) / (int)gridDim.x : 0;
}

// Balanced plan, for batches of at most kBalanceRows rows.  With the
// strided plan every CTA takes every gridDim.x-th tile, and rows without
// work (null rows, nothing accepted, deferred rows) leave some CTAs with
// far more work than others.  Here every CTA first scans all rows: producer
// thread t checks rows t R .. t R + R - 1 (R = ceil(B / kPlanSize)) and marks
// those with work; the work rows, in row order, times the heads are the work
// tiles, and every CTA takes every gridDim.x-th of them.  A row's side
// effects (error bits, pending writes) are made by one CTA, row b's by CTA
// b mod gridDim.x, during this scan.
constexpr int kBalanceRowsPerThread = 32;
constexpr int kBalanceRows = kPlanSize * kBalanceRowsPerThread;

template <Mode kMode>
__device__ void balance_scan(const Params &p, WorkList &list, Balance *bal, int pt) {
    // Commits and flushes only: their rows without work (nothing accepted,
    // deferred, no pending replay) are what unbalances the strided plan.  A
    // verify has work in almost every row, and there the scan measured
    // slower than the strided plan (mixed verify 266 -> 273 us, deferred2
    // fused verify 344 -> 349 us; commits 1 to 8 us faster).
    const int R = (kMode != Mode::kVerify && bal != nullptr && p.B <= kBalanceRows)
                      ? (p.B + kPlanSize - 1) / kPlanSize
                      : 0;
    if (pt == 0) {
        list.rows_per_thread = R;
        list.mask = bal != nullptr ? bal->mask : nullptr;
        list.prefix = bal != nullptr ? bal->prefix : nullptr;
    }
    if (R == 0) {
        producer_sync();
        return;
    }
    unsigned m = 0u;
#pragma unroll 4
    for (int i = 0; i < kBalanceRowsPerThread; ++i) {
        const int b = pt * R + i;
        if (i < R && b < p.B) {
            Work w;
            if (plan_row<kMode>(p, b, 0, b % (int)gridDim.x == (int)blockIdx.x, w)) m |= 1u << i;
        }
    }
    // exclusive prefix of the per-thread counts: a warp scan, then the warps'
    // totals
    const int lane = pt & 31, warp = pt >> 5;
    const int cnt = __popc(m);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) list.warp_count[warp] = incl;
    bal->mask[pt] = m;
    producer_sync();
    int before = 0;
#pragma unroll
    for (int i = 0; i < kProducerWarps; ++i)
        if (i < warp) before += list.warp_count[i];
    bal->prefix[pt] = before + incl - cnt;
    if (pt == kPlanSize - 1) bal->prefix[kPlanSize] = before + incl;
    producer_sync();
}

// Row of the rank-th work row of the balanced plan.
__device__ __forceinline__ int balanced_row(const WorkList &list, int rank) {
    int lo = 0, hi = kPlanSize;  // prefix[lo] <= rank < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (list.prefix[mid] <= rank)
            lo = mid;
        else
            hi = mid;
    }
    unsigned m = list.mask[lo];
    for (int j = rank - list.prefix[lo]; j > 0; --j) m &= m - 1u;  // drop the lowest j bits
    return lo * list.rows_per_thread + (__ffs(m) - 1);
}

// One planning round over candidates [k0, k0 + kPlanSize) by the producer
// threads; compacts the tiles with work, in order, into the list.
template <Mode kMode>
__device__ int plan_round(const Params &p, WorkList &list, int k0, int num_tiles, int pt) {
    const int K = num_candidates(list, num_tiles, p.H);
    Work w;
    bool has = false;
    const int k = k0 + pt;
    if (k < K) {
        const int c = (int)blockIdx.x + k * (int)gridDim.x;
        if (list.rows_per_thread > 0) {
            const int rank = c / p.H;
            const int head = c - rank * p.H;
            has = plan_row<kMode>(p, balanced_row(list, rank), head, false, w);
        } else {
            const int b = c / p.H;
            const int head = c - b * p.H;
            has = plan_row<kMode>(p, b, head, head == 0, w);
        }
    }
    const unsigned ballot = __ballot_sync(kFull, has);
    const int lane = pt & 31, warp = pt >> 5;
    if (lane == 0) list.warp_count[warp] = __popc(ballot);
    producer_sync();
    int before = 0, total = 0;
#pragma unroll
    for (int i = 0; i < kProducerWarps; ++i) {
        const int c = list.warp_count[i];
        if (i < warp) before += c;
        total += c;
    }
    if (has) {
        const int pos = before + __popc(ballot & ((1u << lane) - 1u));
        list.tile[pos] = w.tile;
        list.slot[pos] = w.slot;
        list.r[pos] = w.r;
        list.bos[pos] = w.bos;
        list.tp[pos] = w.T | (w.p << 8) | (w.head << 16);
        if constexpr (kMode == Mode::kCommit) {
            list.dst[pos] = w.dst;
            list.mid[pos] = w.mid;
            list.mid_len[pos] = w.mid_len;
        }
    }
    producer_sync();
    return total;
}

struct Cursor {
    int idx, count, next_k;
};

// The producer's next work item (planning a new round when needed), or a
// Work with tile -1 when the CTA has no more.
template <Mode kMode>
__device__ __forceinline__ Work next_work(const Params &p, WorkList &list, Cursor &c,
                                          int num_tiles, int pt) {
    Work w;
    w.tile = -1;
    while (c.idx >= c.count) {
        if (c.next_k >= num_candidates(list, num_tiles, p.H)) return w;
        c.count = plan_round<kMode>(p, list, c.next_k, num_tiles, pt);
        c.next_k += kPlanSize;
        c.idx = 0;
    }
    const int i = c.idx++;
    w.tile = list.tile[i];
    w.slot = list.slot[i];
    w.r = list.r[i];
    w.bos = list.bos[i];
    w.T = list.tp[i] & 0xff;
    w.p = (list.tp[i] >> 8) & 0xff;
    w.head = list.tp[i] >> 16;
    if constexpr (kMode == Mode::kCommit) {
        w.dst = list.dst[i];
        w.mid = list.mid[i];
        w.mid_len = list.mid_len[i];
    } else {  // the other modes store to the row's own slot
        w.dst = w.slot;
        w.mid = 0;
        w.mid_len = 0;
    }
    return w;
}

// Raw inputs and gate parameters of an item into a raw buffer (cp.async by
// the producer threads).
template <Mode kMode, bool kCorr>
__device__ __forceinline__ void fetch_raw(const Params &p, const Work &w, RawView<kCorr> rv,
                                          int pt) {
    const int lane = pt & 31, warp = pt >> 5;
    if constexpr (kCorr) {
        // recorded tokens: bf16 k and g_raw, fp32 delta (16 bytes per lane)
        const unsigned char *rec = corr_base(p, w.r, w.head);
        for (int c = warp; c < 3 * w.p; c += kProducerWarps) {
            const int u = c / 3;
            const int part = c - 3 * u;
            const unsigned char *tok = rec + (size_t)u * kCorrBytes;
            if (part == 1)
                cp_async16(rv.v + u * RawView<kCorr>::kVWords + 4 * lane,
                           reinterpret_cast<const uint4 *>(tok) + lane);
            else
                cp_async8((part == 0 ? rv.k : rv.g) + u * (kD / 2) + 2 * lane,
                          reinterpret_cast<const uint2 *>(tok + (part == 0 ? kCorrK : kCorrG)) +
                              lane);
        }
    } else {
        const __nv_bfloat16 *rec = record_base(p, w.r, w.head);
        for (int c = warp; c < 3 * w.p; c += kProducerWarps) {
            const int u = c / 3;
            const int part = c - 3 * u;
            const uint2 *src =
                reinterpret_cast<const uint2 *>(rec + (size_t)u * kRecStride + part * kD);
            uint32_t *dst = (part == 0 ? rv.k : (part == 1 ? rv.v : rv.g)) + u * (kD / 2);
            cp_async8(dst + 2 * lane, src + lane);
        }
        if (warp == 0 && lane < w.p)
            cp_async8(&rv.tail[lane], rec + (size_t)lane * kRecStride + kRecBeta);
    }
    if (warp == kProducerWarps - 2) {
        cp_async16(rv.bias + 4 * lane, p.g_bias + w.head * kD + 4 * lane);
        if (lane == 0) cp_async4(rv.a_log, p.A_log + w.head);
    }
    if constexpr (kMode == Mode::kVerify) {
        // producer warp w copies part w (k, v, g_raw, q) of every new token:
        // one source row and one destination slot per token
        static_assert(kProducerWarps == 4, "one activation part per producer warp");
        const __nv_bfloat16 *src;
        long long stride;
        uint32_t *dst;
        int dstep;
        if (warp == 0) {
            src = p.k, stride = p.stride_k, dst = rv.k + w.p * (kD / 2), dstep = kD / 2;
        } else if (warp == 1) {
            src = p.v, stride = p.stride_v, dst = rv.v + w.p * RawView<kCorr>::kVWords,
            dstep = RawView<kCorr>::kVWords;
        } else if (warp == 2) {
            src = p.g, stride = p.stride_g, dst = rv.g + w.p * (kD / 2), dstep = kD / 2;
        } else {
            src = p.q, stride = p.stride_q, dst = rv.q, dstep = kD / 2;
        }
        const uint2 *row = reinterpret_cast<const uint2 *>(src + (size_t)w.bos * stride +
                                                           w.head * kD) + lane;
        const long long rstep = stride / 4;  // uint2 per token (the stride is a multiple of 4)
        for (int t = 0; t < w.T; ++t) cp_async8(dst + t * dstep + 2 * lane, row + t * rstep);
    }
    cp_async_commit();
}

// Per-token vectors of an item: token u is prepared by producer warp
// (u mod 4), four channels per lane, the norms summed across the warp; every
// token is computed the same way however many tokens the item has.  The
// verify also writes the new tokens' records (raw: k, v, g_raw, beta_raw;
// correction: k and g_raw, the consumer adds the delta).  An item in window
// form (window_item) needs no k^ . q^.
template <Mode kMode, bool kBounded, bool kCorr>
__device__ __forceinline__ void prep_item(const Params &p, const Work &w, RawView<kCorr> rv,
                                          const TokView &tv, int pt, bool window_item) {
    const int lane = pt & 31, warp = pt >> 5;
    const float a = expf(*rv.a_log);
    const float4 bias = *reinterpret_cast<const float4 *>(rv.bias + 4 * lane);
    for (int u = warp; u < w.p + w.T; u += kProducerWarps) {
        const bool is_new = kMode == Mode::kVerify && u >= w.p;
        const int t = u - w.p;
        const uint32_t *vslot = rv.v + u * RawView<kCorr>::kVWords;
        const uint2 kb = reinterpret_cast<const uint2 *>(rv.k + u * (kD / 2))[lane];
        const uint2 gb = reinterpret_cast<const uint2 *>(rv.g + u * (kD / 2))[lane];
        const float4 k = bf16x4_to_float4(kb);
        float s = __fmul_rn(k.x, k.x);
        s = __fmaf_rn(k.y, k.y, s);
        s = __fmaf_rn(k.z, k.z, s);
        s = __fmaf_rn(k.w, k.w, s);
        const float ik = inv_l2(warp_allsum(s));
        *reinterpret_cast<float4 *>(tv.kh + u * kD + 4 * lane) =
            make_float4(__fmul_rn(k.x, ik), __fmul_rn(k.y, ik), __fmul_rn(k.z, ik),
                        __fmul_rn(k.w, ik));
        const float4 g = bf16x4_to_float4(gb);
        float4 e;
        e.x = decay_factor(__fadd_rn(g.x, bias.x), a, kBounded, p.lower_bound);
        e.y = decay_factor(__fadd_rn(g.y, bias.y), a, kBounded, p.lower_bound);
        e.z = decay_factor(__fadd_rn(g.z, bias.z), a, kBounded, p.lower_bound);
        e.w = decay_factor(__fadd_rn(g.w, bias.w), a, kBounded, p.lower_bound);
        *reinterpret_cast<float4 *>(tv.e + u * kD + 4 * lane) = e;
        uint2 vb = make_uint2(0u, 0u);
        uint32_t bb = 0u;
        if (kCorr && !is_new) {
            // a recorded token's delta, as stored
            *reinterpret_cast<float4 *>(tv.v + u * kD + 4 * lane) =
                reinterpret_cast<const float4 *>(vslot)[lane];
        } else {
            vb = reinterpret_cast<const uint2 *>(vslot)[lane];
            bb = is_new ? rv.beta_new[t] : (rv.tail[u].x & 0xffffu);
            *reinterpret_cast<float4 *>(tv.v + u * kD + 4 * lane) = bf16x4_to_float4(vb);
            if (lane == 0) tv.beta[u] = sigmoidf_rn(bf16_bits_to_float(bb));
        }
        if (is_new) {
            const float4 q = bf16x4_to_float4(reinterpret_cast<const uint2 *>(rv.q + t * (kD / 2))[lane]);
            float sq = __fmul_rn(q.x, q.x);
            sq = __fmaf_rn(q.y, q.y, sq);
            sq = __fmaf_rn(q.z, q.z, sq);
            sq = __fmaf_rn(q.w, q.w, sq);
            const float iq = inv_l2(warp_allsum(sq));
            *reinterpret_cast<float4 *>(tv.qh + t * kD + 4 * lane) =
                make_float4(__fmul_rn(__fmul_rn(q.x, iq), p.scale),
                            __fmul_rn(__fmul_rn(q.y, iq), p.scale),
                            __fmul_rn(__fmul_rn(q.z, iq), p.scale),
                            __fmul_rn(__fmul_rn(q.w, iq), p.scale));
            if (!window_item) {
                // k^ . q^ from the raw dot product and the two norms
                float skq = __fmul_rn(k.x, q.x);
                skq = __fmaf_rn(k.y, q.y, skq);
                skq = __fmaf_rn(k.z, q.z, skq);
                skq = __fmaf_rn(k.w, q.w, skq);
                const float dkq = warp_allsum(skq);
                if (lane == 0) tv.kq[t] = __fmul_rn(__fmul_rn(__fmul_rn(dkq, ik), iq), p.scale);
            }
            if constexpr (kCorr) {
                unsigned char *tok = corr_base(p, w.r, w.head) + (size_t)t * kCorrBytes;
                reinterpret_cast<uint2 *>(tok + kCorrK)[lane] = kb;
                reinterpret_cast<uint2 *>(tok + kCorrG)[lane] = gb;
            } else {
                __nv_bfloat16 *rec = record_base(p, w.r, w.head);
                uint2 *dst = reinterpret_cast<uint2 *>(rec + (size_t)t * kRecStride);
                dst[lane] = kb;
                dst[kRecV / 4 + lane] = vb;
                dst[kRecG / 4 + lane] = gb;
                if (lane == 0)
                    reinterpret_cast<uint16_t *>(rec + (size_t)t * kRecStride)[kRecBeta] =
                        (uint16_t)bb;
            }
        }
    }
}

__device__ __forceinline__ void issue_state(const Params &p, const Work &w, float *dst,
                                            uint64_t *bar) {
    const float *src = p.pool + ((size_t)w.slot * p.H + w.head) * (size_t)(kD * kD);
    mbar_arrive_expect_tx(bar, kD * kD * 4);
    bulk_load(dst, src, kD * kD * 4, bar);
}

// The checkpoint of a tensor-window item, swizzled for the tensor core: four
// boxes of 32 columns x 128 rows through the pool's tensor map (rows of the
// pool viewed as (slot * H + head) * 128 + v).
__device__ __forceinline__ void issue_state_tc(const Params &p, const Work &w, float *dst,
                                               uint64_t *bar, const CUtensorMap *tmap) {
    const int row0 = (w.slot * p.H + w.head) * kD;
    mbar_arrive_expect_tx(bar, kD * kD * 4);
#pragma unroll
    for (int blk = 0; blk < 4; ++blk)
        tma_load_2d(dst + blk * (kD * 32), tmap, 32 * blk, row0, bar);
}

// A verify item in tensor window form: raw records, window kernel, the
// launch's tensor map valid and at least kWindowMinT new tokens.  Its
// checkpoint is staged swizzled.
template <bool kWindow>
__device__ __forceinline__ bool tensor_item(const Params &p, const unsigned char *smem, int T) {
    return kWindow && kTensorWindow && p.tc_window != 0 && T >= kWindowMinT &&
           (smem_u32(smem) & 1023u) == 0;
}

// Per-item duties of the producer warps, spread so that none carries two:
// warp 3 (the fewest tokens to prepare, token u going to warp u mod 4)
// stages the checkpoint, warp 2 copies g_bias and A_log, warp 1 waits for
// the token buffer, writes the item info and hands the item over, and warp 0
// copies the record tails.
constexpr int kStageThread = kProducerThreads - 32;
constexpr int kHandoffThread = 32;

template <Mode kMode, bool kBounded, bool kCorr, bool kWindow>
__device__ void run_producer(const Params &p, unsigned char *smem, const Layout &lay,
                             int num_tiles, int pt, const CUtensorMap *tmap) {
    using Raw = RawView<kCorr>;
    Sync &sy = *reinterpret_cast<Sync *>(smem + lay.off_sync);
    WorkList &list = *reinterpret_cast<WorkList *>(smem + lay.off_list);
    Cursor cursor{0, 0, 0};
    balance_scan<kMode>(p, list,
                        lay.off_bal >= 0 ? reinterpret_cast<Balance *>(smem + lay.off_bal) : nullptr,
                        pt);
    Work cur = next_work<kMode>(p, list, cursor, num_tiles, pt);
    int rb = 0;
    uint32_t beta_next = 0;
    if (cur.tile >= 0) {
        fetch_raw<kMode, kCorr>(p, cur, Raw(smem + lay.off_raw, lay.slots, p.Q), pt);
        if (kMode == Mode::kVerify && pt < cur.T)
            beta_next = reinterpret_cast<const uint16_t *>(
                p.beta)[(size_t)(cur.bos + pt) * p.stride_beta + cur.head];
    }
    int n = 0;
    bool ok = true;
    while (cur.tile >= 0) {
        const int c = n & 1;
        const int use_c = n >> 1;
        // checkpoint of `cur` into consumer c's staging buffer
        if (pt == kStageThread) {
            if (use_c > 0) ok = wait_phase(&sy.empty_state[c], (use_c - 1) & 1, sy, p);
            if (ok) {
                float *dst = reinterpret_cast<float *>(smem + lay.off_state) + c * kD * kD;
                if (tensor_item<kWindow>(p, smem, cur.T))
                    issue_state_tc(p, cur, dst, &sy.full_state[c], tmap);
                else
                    issue_state(p, cur, dst, &sy.full_state[c]);
            }
        }
        // raw inputs of `cur` have landed; start those of the next item
        Raw rv(smem + lay.off_raw + rb * lay.raw_bytes, lay.slots, p.Q);
        cp_async_wait_all();
        if (kMode == Mode::kVerify && pt < cur.T) rv.beta_new[pt] = beta_next;
        const Work nxt = next_work<kMode>(p, list, cursor, num_tiles, pt);  // has barriers
        if (nxt.tile >= 0) {
            fetch_raw<kMode, kCorr>(
                p, nxt, Raw(smem + lay.off_raw + (rb ^ 1) * lay.raw_bytes, lay.slots, p.Q), pt);
            if (kMode == Mode::kVerify && pt < nxt.T)
                beta_next = reinterpret_cast<const uint16_t *>(
                    p.beta)[(size_t)(nxt.bos + pt) * p.stride_beta + nxt.head];
        }
        // token vectors of `cur` into consumer c's buffer b, once it is free
        const int b = use_c % lay.nbuf;
        const int use_b = use_c / lay.nbuf;
        if (pt == kHandoffThread) {
            if (use_b > 0 && ok) ok = wait_phase(&sy.empty_tok[c][b], (use_b - 1) & 1, sy, p);
            // one thread decides for all whether to leave, so that they all do
            sy.leave[n & 1] = *reinterpret_cast<volatile int *>(&sy.abort);
        }
        producer_sync();
        if (sy.leave[n & 1]) {
            cp_async_wait_all();  // no copy into shared memory outlives the thread
            return;
        }
        TokView tv(smem + lay.off_tok + (c * lay.nbuf + b) * lay.tok_bytes, lay.slots, p.Q,
                   lay.head);
        // an item in either window form needs no k^ . q^ (the tensor build's
        // window items that cannot take the tensor form run token by token)
        const bool window_item = tensor_item<kWindow>(p, smem, cur.T) ||
                                 (kWindow && !kTensorWindow && cur.T >= kWindowMinT);
        prep_item<kMode, kBounded, kCorr>(p, cur, rv, tv, pt, window_item);
        if (pt == kHandoffThread) {
            ItemInfo &it = sy.info[c][b];
            it.head = cur.head;
            it.bos = cur.bos;
            it.T = cur.T;
            it.p = cur.p;
            it.end = 0;
            it.dst = cur.dst;
            it.mid = cur.mid;
            it.mid_len = cur.mid_len;
            it.r = cur.r;
        }
        producer_sync();  // all token vectors and the item info written
        if (pt == kHandoffThread) mbar_arrive(&sy.full_tok[c][b]);
        ++n;
        rb ^= 1;
        cur = nxt;
    }
    // end markers: the next buffer of each consumer says "no more items"
    if (pt == kHandoffThread) {
        for (int c = 0; c < 2; ++c) {
            const int use_c = (n + 1 - c) >> 1;
            const int b = use_c % lay.nbuf;
            const int use_b = use_c / lay.nbuf;
            if (use_b > 0 && !wait_phase(&sy.empty_tok[c][b], (use_b - 1) & 1, sy, p)) return;
#ifdef KDA_TEST_WITHHOLD_END_MARKER
            // a test build of the timeout path: consumer 0 of CTA 0 is never
            // told that its work is done, so its wait for a next item runs
            // out.  Every copy into this CTA's shared memory has landed by
            // then: the consumer waited for each checkpoint it loaded, and
            // the producer for each item's raw inputs.
            if (c == 0 && blockIdx.x == 0) continue;
#endif
            sy.info[c][b].end = 1;
            mbar_arrive(&sy.full_tok[c][b]);
        }
    }
}

template <Mode kMode, bool kCorr, bool kWindow>
__device__ void run_consumer(const Params &p, unsigned char *smem, const Layout &lay, int c,
                             int ct) {
    Sync &sy = *reinterpret_cast<Sync *>(smem + lay.off_sync);
    Lane L;
    L.lane = ct & 31;
    L.w = ct >> 5;
    L.g = L.lane >> 3;
    L.j = L.lane & 7;
    const float *staging = reinterpret_cast<const float *>(smem + lay.off_state) + c * kD * kD;
    // the group's barrier: an mbarrier, so that its wait is bounded like the
    // others and every thread leaves on an abort
    uint32_t group_uses = 0;
    uint32_t mma_uses = 0;  // tensor window items done (parity of mma_hi and mma_done)
    auto group_sync = [&]() -> bool {
        mbar_arrive(&sy.group[c]);
        return wait_phase(&sy.group[c], group_uses++ & 1, sy, p);
    };
    for (int k = 0;; ++k) {
        const int b = k % lay.nbuf;
        const int use_b = k / lay.nbuf;
        if (!wait_phase(&sy.full_tok[c][b], use_b & 1, sy, p)) return;
        const ItemInfo it = sy.info[c][b];
        if (it.end) return;
        const TokView tv(smem + lay.off_tok + (c * lay.nbuf + b) * lay.tok_bytes, lay.slots, p.Q,
                         lay.head);
        // tensor window form (window kernels): the outputs' row products on
        // the tensor core, from the swizzled staging buffer
        const bool tensor = tensor_item<kWindow>(p, smem, it.T);
        // the FMA window form; the tensor build has none (its window items
        // that cannot take the tensor form run token by token)
        const bool window = kWindow && !kTensorWindow && it.T >= kWindowMinT;
        unsigned char *stage = smem + lay.off_state + c * (kD * kD * 4);
        // the FMA window form's coefficients, before the tile occupies registers
        if constexpr (kWindow)
            if (window && !tensor && !window_prep(tv, it.p, it.T, p.Q, ct, group_sync)) return;
        if (!tensor || it.p > 0) {
            if (!wait_phase(&sy.full_state[c], k & 1, sy, p)) return;
            Tile h;
            if (tensor)
                load_tile_sw(h, stage, L);
            else
                load_tile(h, staging, L);
            if (!tensor) mbar_arrive(&sy.empty_state[c]);
            for (int u = 0; u < it.p; ++u) {
                if constexpr (kCorr)
                    token_corr(h, tv, u, L);
                else
                    token_plain(h, tv, u, L);
                if constexpr (kMode == Mode::kCommit) {
                    if (u + 1 == it.mid_len)  // align mode: the state at the block boundary
                        store_tile(h, p.pool + ((size_t)it.mid * p.H + it.head) * (size_t)(kD * kD),
                                   L);
                }
            }
            if (it.p > 0)
                store_tile(h, p.pool + ((size_t)it.dst * p.H + it.head) * (size_t)(kD * kD), L);
            if (tensor) {
                // the folded state back to the staging buffer, for the tensor core
                store_tile_sw(h, stage, L);
            } else {
                if (kWindow && window) {
                    window_outputs(h, tv, it.p, it.T, p.Q, L,
                                   p.out + ((size_t)it.bos * p.H + it.head) * kD, (size_t)p.H * kD);
                } else if constexpr (kMode == Mode::kVerify) {
                    // the state after the last new token is stored only as a
                    // trajectory output: without one, that token's update is
                    // left out (its output does not depend on it).  Not in
                    // the window kernels, where the second copy of the token
                    // code spills registers.
                    const int updated = (kWindow || p.traj != nullptr) ? it.T : it.T - 1;
                    auto record_delta = [&](int t, float vp) {
                        if constexpr (kCorr)  // the token's delta into its correction record
                            reinterpret_cast<float *>(corr_base(p, it.r, it.head) +
                                                      (size_t)t * kCorrBytes)[L.row(L.j)] = vp;
                    };
                    int t = 0;
                    for (; t < updated; ++t) {
                        const size_t tok = (size_t)(it.bos + t) * p.H + it.head;
                        record_delta(t, token_out<true>(h, tv, it.p + t, t, L, p.out + tok * kD));
                        if (p.traj != nullptr) store_tile(h, p.traj + tok * (size_t)(kD * kD), L);
                    }
                    if (t < it.T) {
                        const size_t tok = (size_t)(it.bos + t) * p.H + it.head;
                        record_delta(t, token_out<false>(h, tv, it.p + t, t, L, p.out + tok * kD));
                    }
                }
                mbar_arrive(&sy.empty_tok[c][b]);
                continue;
            }
        }
        if constexpr (kWindow && kTensorWindow) {
            // tensor window form, from here with no tile in registers
            float vrow[kMaxQ];
            if (!window_tc_prep(tv, it.p, it.T, p.Q, ct, vrow, group_sync)) return;
            if (it.p == 0 && !wait_phase(&sy.full_state[c], k & 1, sy, p)) return;
            const uint32_t tmem = sy.tmem_base + 256u * (uint32_t)c;  // this consumer's columns
            const uint32_t lanes = (uint32_t)(32 * (ct >> 5)) << 16;  // this warp's TMEM lanes
            const uint32_t a_cols = tmem + lanes + 128u;               // A: S, then S_lo
            const uint32_t mbar_parity = mma_uses & 1u;
            // the state's row into A (read by the tensor core as S_hi); the
            // staging buffer is free once every row is read
            s_row_to_tmem(stage, ct, a_cols);
            mbar_arrive(&sy.empty_state[c]);
            tmem_wait_st();
            tc_fence_before();
            if (!group_sync()) return;  // the operands X and A in place
            if (ct == 0) {
                tc_fence_after();
                window_tc_mma(tmem + 128u, smem_u32(tv.kh), tmem);  // D_hi
                umma_commit(&sy.mma_hi[c]);
            }
            // A takes S_lo once D_hi has read it.  The products finish in
            // microseconds whatever the other roles do, so a product in flight
            // is waited for before any thread leaves (TMEM must not be freed
            // under it).
            if (!mbar_wait_bounded(&sy.mma_hi[c], mbar_parity, kWaitBudget)) {
                *reinterpret_cast<volatile int *>(&sy.abort) = 1;
                flag_error(p.err, kErrWaitTimeout);
                return;
            }
            tc_fence_after();
            s_lo_in_tmem(a_cols);
            tmem_wait_st();
            tc_fence_before();
            if (!group_sync()) return;  // S_lo in place (no product in flight)
            if (ct == 0) {
                tc_fence_after();
                window_tc_mma(tmem + 128u, smem_u32(tv.kh), tmem + 32u);  // D_lo
                umma_commit(&sy.mma_done[c]);
            }
            if (!mbar_wait_bounded(&sy.mma_done[c], mbar_parity, kWaitBudget)) {
                *reinterpret_cast<volatile int *>(&sy.abort) = 1;
                flag_error(p.err, kErrWaitTimeout);
                return;
            }
            ++mma_uses;
            tc_fence_after();
            window_tc_solve(tv, it.p, it.T, p.Q, ct, vrow, tmem + lanes,
                            p.out + ((size_t)it.bos * p.H + it.head) * kD, (size_t)p.H * kD);
            tc_fence_before();  // this item's TMEM reads before the next item's writes
        }
        mbar_arrive(&sy.empty_tok[c][b]);
    }
}

// kWindow: items of the verify with at least kWindowMinT new tokens run them
// in window form (raw records, no trajectory output); the others, and every
// other kernel, token by token.
//
// With the tensor window form the window kernels allocate all 512 columns of
// tensor memory (256 per consumer: D_hi in columns 0..31, D_lo in 32..63,
// S_lo in 128..255); one CTA per SM, so the allocation never waits.
constexpr uint32_t kTmemCols = 512;

template <Mode kMode, bool kBounded, bool kCorr, bool kWindow>
__global__ void __launch_bounds__(kBlockThreads, 1)
    step_kernel(const Params p, int num_tiles, int fold, const __grid_constant__ CUtensorMap tmap) {
    static_assert(!kWindow || (kMode == Mode::kVerify && !kCorr), "window form: raw verify only");
    // the head layout's buffers (swizzled operands) need a 1024-byte aligned
    // base; tensor_item checks it
    extern __shared__ __align__(1024) unsigned char smem[];
    const Layout lay = make_layout(p.Q, fold != 0, kCorr, kWindow);
    Sync &sy = *reinterpret_cast<Sync *>(smem + lay.off_sync);
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int c = 0; c < 2; ++c) {
            mbar_init(&sy.full_state[c], 1);
            mbar_init(&sy.empty_state[c], kConsumerThreads);
            mbar_init(&sy.group[c], kConsumerThreads);
            mbar_init(&sy.mma_hi[c], 1);
            mbar_init(&sy.mma_done[c], 1);
            for (int b = 0; b < 2; ++b) {
                mbar_init(&sy.full_tok[c][b], 1);
                mbar_init(&sy.empty_tok[c][b], kConsumerThreads);
            }
        }
        sy.abort = 0;
        fence_mbar_init();
    }
    if constexpr (kWindow && kTensorWindow) {
        if (tid < 32) tmem_alloc(&sy.tmem_base, kTmemCols);
        tc_fence_before();
    }
    __syncthreads();
    if constexpr (kWindow && kTensorWindow) tc_fence_after();
    // let the next launch start its set-up, and wait for the previous one
    // before any global memory is touched
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Register split: the launch gives every thread kLaunchRegs; the producer
    // warpgroup hands registers back and the consumers take them, so that
    // 2 * 128 * kConsumerRegs + 128 * kProducerRegs == 384 * kLaunchRegs.
    if (tid < 2 * kConsumerThreads) {
        reg_alloc<kConsumerRegs>();
        run_consumer<kMode, kCorr, kWindow>(p, smem, lay, tid / kConsumerThreads,
                                            tid % kConsumerThreads);
    } else {
        reg_dealloc<kProducerRegs>();
        run_producer<kMode, kBounded, kCorr, kWindow>(p, smem, lay, num_tiles,
                                                      tid - 2 * kConsumerThreads, &tmap);
    }
    if constexpr (kWindow && kTensorWindow) {
        // every role has left (an abort included); the consumers waited for
        // their products, so the tensor memory is idle
        tc_fence_before();
        __syncthreads();
        if (tid < 32) {
            tc_fence_after();
            tmem_dealloc(sy.tmem_base, kTmemCols);
        }
    }
}

}  // namespace kda

// =================================================================== C ABI ==

namespace {

using kda::Params;

bool aligned(const void *ptr, uintptr_t bytes) {
    return (reinterpret_cast<uintptr_t>(ptr) & (bytes - 1)) == 0;
}

// Checks of the config common to all entry points.
kda_status check_config(const kda_config *cfg) {
    if (cfg == nullptr) return KDA_ERR_INVALID_ARG;
    if (cfg->num_heads < 1 || cfg->num_slots < 1 || cfg->record_slots < 0)
        return KDA_ERR_INVALID_ARG;
    if (cfg->window < 1) return KDA_ERR_INVALID_ARG;
    if (cfg->head_dim != KDA_HEAD_DIM || cfg->window > KDA_MAX_WINDOW) return KDA_ERR_UNSUPPORTED;
    if (cfg->num_heads > KDA_MAX_HEADS) return KDA_ERR_UNSUPPORTED;
    if (cfg->use_lower_bound != 0 && cfg->use_lower_bound != 1) return KDA_ERR_INVALID_ARG;
    if (cfg->use_lower_bound == 1 && !(cfg->lower_bound < 0.0f && isfinite(cfg->lower_bound)))
        return KDA_ERR_INVALID_ARG;
    if (!isfinite(cfg->scale)) return KDA_ERR_INVALID_ARG;
    if (cfg->record_format != KDA_RECORDS_RAW && cfg->record_format != KDA_RECORDS_CORRECTION)
        return KDA_ERR_INVALID_ARG;
    if (cfg->reserved != 0) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

Params base_params(const kda_config *cfg, int32_t B) {
    Params p{};
    p.H = cfg->num_heads;
    p.Q = cfg->window;
    p.S = cfg->num_slots;
    p.R = cfg->record_slots;
    p.B = B;
    p.bounded = cfg->use_lower_bound;
    p.lower_bound = cfg->lower_bound;
    p.scale = cfg->scale;
    p.stride_q = cfg->stride_q_t;
    p.stride_k = cfg->stride_k_t;
    p.stride_v = cfg->stride_v_t;
    p.stride_g = cfg->stride_g_t;
    p.stride_beta = cfg->stride_beta_t;
    return p;
}

kda_status check_common(const kda_config *cfg, const float *A_log, const float *g_bias,
                        const float *pool, const int32_t *state_indices, int32_t B,
                        const int32_t *record_rows, const void *records,
                        const int32_t *error_word) {
    if (!A_log || !g_bias || !pool || !state_indices || !records) return KDA_ERR_INVALID_ARG;
    if (!aligned(g_bias, 16) || !aligned(pool, 16) || !aligned(A_log, 4) ||
        !aligned(state_indices, 4) || !aligned(records, 16))
        return KDA_ERR_INVALID_ARG;
    // the kernels OR bits into the error word with a 32-bit atomic
    if (error_word != nullptr && !aligned(error_word, 4)) return KDA_ERR_INVALID_ARG;
    if (record_rows == nullptr && B > cfg->record_slots) return KDA_ERR_INVALID_ARG;
    if (record_rows != nullptr && !aligned(record_rows, 4)) return KDA_ERR_INVALID_ARG;
    if ((long long)B * cfg->num_heads > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

kda_status finish_launch() {
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

// The instantiation of a launch: gate, record format, and for a raw-record
// verify without a trajectory output whose window can hold kWindowMinT
// tokens, the kernel that runs such items in window form.
template <kda::Mode M>
void (*step_kernel_for(bool bounded, bool corr, bool traj, bool window))(const Params, int, int,
                                                                         const CUtensorMap) {
    using kda::step_kernel;
    if constexpr (M == kda::Mode::kVerify) {
        if (!corr && !traj && window)
            return bounded ? step_kernel<M, true, false, true> : step_kernel<M, false, false, true>;
    }
    if (corr) return bounded ? step_kernel<M, true, true, false> : step_kernel<M, false, true, false>;
    return bounded ? step_kernel<M, true, false, false> : step_kernel<M, false, false, false>;
}

#ifdef KDA_TENSOR_WINDOW
// The driver's tensor-map encoder, looked up once through the runtime (the
// library links no driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}
#endif

// Tensor map of the state pool for the tensor window form: the pool as a
// 2-D fp32 array of S * H * 128 rows of 128, read in boxes of 32 columns x
// 128 rows with the 128-byte swizzle.  False when it cannot be made (then
// the window items take the FMA form).
bool pool_tensor_map(const Params &p, CUtensorMap *map) {
#ifndef KDA_TENSOR_WINDOW
    (void)p, (void)map;
    return false;  // the tensor window form is a build option
#else
    const long long rows = (long long)p.S * p.H * kda::kD;
    if (rows >= 0x7fffffffLL) return false;  // row coordinates are 32-bit signed
    const EncodeTiledFn enc = encode_tiled();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kda::kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kda::kD * 4};
    const cuuint32_t box[2] = {32, (cuuint32_t)kda::kD};
    const cuuint32_t elem[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.pool, dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
#endif
}

// Launch the warp-specialized step kernel: one CTA per SM (or one per tile
// when there are fewer tiles), the shared-memory layout sized by the window.
template <kda::Mode M>
kda_status launch_step(const Params &p_in, const kda_config *cfg, bool fold, cudaStream_t stream) {
    Params p = p_in;
    const long long tiles = (long long)p.B * p.H;
    const int sms = sm_count();
    if (sms <= 0) return KDA_ERR_CUDA;
    const int grid = (int)(tiles < (long long)sms ? tiles : (long long)sms);
    const bool bounded = cfg->use_lower_bound != 0;
    const bool corr = cfg->record_format == KDA_RECORDS_CORRECTION;
    const bool window =
        M == kda::Mode::kVerify && !corr && p.traj == nullptr && p.Q >= kda::kWindowMinT;
    const kda::Layout lay = kda::make_layout(p.Q, fold, corr, window);
    void (*kern)(const Params, int, int, const CUtensorMap) =
        step_kernel_for<M>(bounded, corr, p.traj != nullptr, window);
    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    p.tc_window = window && pool_tensor_map(p, &map) ? 1 : 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return KDA_ERR_CUDA;
    // programmatic dependent launch: the next launch's CTAs may start their
    // set-up while this grid's last CTAs finish; they wait for it before
    // touching memory
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kda::kBlockThreads);
    lc.dynamicSmemBytes = lay.total;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (cudaLaunchKernelEx(&lc, kern, p, (int)tiles, fold ? 1 : 0, map) != cudaSuccess)
        return KDA_ERR_CUDA;
    return finish_launch();
}

// Host checks of an align description; fills the Params fields.
kda_status set_align(const kda_align *al, int window, Params &p) {
    if (al == nullptr || al->reserved != 0) return KDA_ERR_INVALID_ARG;
    if (!al->block_table || !al->num_computed) return KDA_ERR_INVALID_ARG;
    if (al->block_table_width < 1 || al->block_table_stride < al->block_table_width ||
        al->num_requests < 1 || al->block_size < window)
        return KDA_ERR_INVALID_ARG;
    if (!aligned(al->block_table, 4) || !aligned(al->num_computed, 4) ||
        (al->request_indices != nullptr && !aligned(al->request_indices, 4)))
        return KDA_ERR_INVALID_ARG;
    p.block_table = al->block_table;
    p.bt_stride = al->block_table_stride;
    p.bt_width = al->block_table_width;
    p.block_size = al->block_size;
    p.num_requests = al->num_requests;
    p.num_computed = al->num_computed;
    p.request_indices = al->request_indices;
    return KDA_OK;
}

}  // namespace

extern "C" {

size_t kda_records_bytes(int32_t num_heads, int32_t window, int32_t record_slots) {
    if (num_heads < 1 || window < 1 || window > KDA_MAX_WINDOW || record_slots < 0) return 0;
    return (size_t)(record_slots + 1) * (size_t)num_heads * (size_t)window *
           (size_t)KDA_RECORD_STRIDE * 2u;
}

size_t kda_correction_records_bytes(int32_t num_heads, int32_t window, int32_t record_slots) {
    if (num_heads < 1 || window < 1 || window > KDA_MAX_WINDOW || record_slots < 0) return 0;
    return (size_t)(record_slots + 1) * (size_t)num_heads * (size_t)window *
           (size_t)KDA_CORRECTION_RECORD_BYTES;
}

kda_status kda_verify(const kda_config *cfg, const void *q, const void *k, const void *v,
                      const void *g_raw, const void *beta_raw, const float *A_log,
                      const float *g_bias, float *state_pool, const int32_t *cu_seqlens,
                      const int32_t *state_indices, int32_t B, const int32_t *record_rows,
                      const int32_t *pending, void *records, void *out, float *trajectory_out,
                      int32_t *error_word, void *stream) {
    kda_status st = check_config(cfg);
    if (st != KDA_OK) return st;
    if (B < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;  // nothing to do; no pointer is inspected
    st = check_common(cfg, A_log, g_bias, state_pool, state_indices, B, record_rows, records,
                      error_word);
    if (st != KDA_OK) return st;
    if (!q || !k || !v || !g_raw || !beta_raw || !cu_seqlens || !out) return KDA_ERR_INVALID_ARG;
    if (!aligned(q, 8) || !aligned(k, 8) || !aligned(v, 8) || !aligned(g_raw, 8) ||
        !aligned(beta_raw, 2) || !aligned(out, 8) || !aligned(cu_seqlens, 4))
        return KDA_ERR_INVALID_ARG;
    if (trajectory_out != nullptr && !aligned(trajectory_out, 16)) return KDA_ERR_INVALID_ARG;
    if (pending != nullptr && !aligned(pending, 4)) return KDA_ERR_INVALID_ARG;
    const int64_t strides[4] = {cfg->stride_q_t, cfg->stride_k_t, cfg->stride_v_t, cfg->stride_g_t};
    for (int64_t s : strides)
        if (s < 1 || (s & 3) != 0) return KDA_ERR_INVALID_ARG;
    if (cfg->stride_beta_t < 1) return KDA_ERR_INVALID_ARG;

    Params p = base_params(cfg, B);
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.g = static_cast<const __nv_bfloat16 *>(g_raw);
    p.beta = static_cast<const __nv_bfloat16 *>(beta_raw);
    p.A_log = A_log;
    p.g_bias = g_bias;
    p.pool = state_pool;
    p.cu_seqlens = cu_seqlens;
    p.state_indices = state_indices;
    p.record_rows = record_rows;
    p.pending_in = pending;
    p.records = static_cast<__nv_bfloat16 *>(records);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.traj = trajectory_out;
    p.err = error_word;

    return launch_step<kda::Mode::kVerify>(p, cfg, pending != nullptr,
                                           static_cast<cudaStream_t>(stream));
}

kda_status kda_commit(const kda_config *cfg, const float *A_log, const float *g_bias,
                      float *state_pool, const int32_t *cu_seqlens, const int32_t *state_indices,
                      int32_t B, const int32_t *num_accepted, const int32_t *record_rows,
                      const void *records, int32_t *pending, const uint8_t *eager,
                      int32_t *error_word, void *stream) {
    kda_status st = check_config(cfg);
    if (st != KDA_OK) return st;
    if (B < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;  // nothing to do; no pointer is inspected
    st = check_common(cfg, A_log, g_bias, state_pool, state_indices, B, record_rows, records,
                      error_word);
    if (st != KDA_OK) return st;
    if (!cu_seqlens || !num_accepted) return KDA_ERR_INVALID_ARG;
    if (!aligned(cu_seqlens, 4) || !aligned(num_accepted, 4)) return KDA_ERR_INVALID_ARG;
    if (pending != nullptr && !aligned(pending, 4)) return KDA_ERR_INVALID_ARG;
    if (pending == nullptr && eager != nullptr) return KDA_ERR_INVALID_ARG;

    Params p = base_params(cfg, B);
    p.A_log = A_log;
    p.g_bias = g_bias;
    p.pool = state_pool;
    p.cu_seqlens = cu_seqlens;
    p.state_indices = state_indices;
    p.record_rows = record_rows;
    p.num_accepted = num_accepted;
    p.records = const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(records));
    p.pending_out = pending;
    p.eager = eager;
    p.err = error_word;

    return launch_step<kda::Mode::kCommit>(p, cfg, false, static_cast<cudaStream_t>(stream));
}

kda_status kda_commit_align(const kda_config *cfg, const float *A_log, const float *g_bias,
                            float *state_pool, const int32_t *cu_seqlens,
                            const int32_t *state_indices, int32_t B,
                            const int32_t *num_accepted, const int32_t *record_rows,
                            const void *records, const kda_align *align, int32_t *pending,
                            const uint8_t *eager, int32_t *error_word, void *stream) {
    kda_status st = check_config(cfg);
    if (st != KDA_OK) return st;
    if (B < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;  // nothing to do; no pointer is inspected
    st = check_common(cfg, A_log, g_bias, state_pool, state_indices, B, record_rows, records,
                      error_word);
    if (st != KDA_OK) return st;
    if (!cu_seqlens || !num_accepted) return KDA_ERR_INVALID_ARG;
    if (!aligned(cu_seqlens, 4) || !aligned(num_accepted, 4)) return KDA_ERR_INVALID_ARG;
    if (pending != nullptr && !aligned(pending, 4)) return KDA_ERR_INVALID_ARG;
    if (pending == nullptr && eager != nullptr) return KDA_ERR_INVALID_ARG;

    Params p = base_params(cfg, B);
    st = set_align(align, cfg->window, p);
    if (st != KDA_OK) return st;
    p.A_log = A_log;
    p.g_bias = g_bias;
    p.pool = state_pool;
    p.cu_seqlens = cu_seqlens;
    p.state_indices = state_indices;
    p.record_rows = record_rows;
    p.num_accepted = num_accepted;
    p.records = const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(records));
    p.pending_out = pending;
    p.eager = eager;
    p.err = error_word;

    return launch_step<kda::Mode::kCommit>(p, cfg, false, static_cast<cudaStream_t>(stream));
}

kda_status kda_flush(const kda_config *cfg, const float *A_log, const float *g_bias,
                     float *state_pool, const int32_t *state_indices, int32_t B,
                     const int32_t *record_rows, const void *records, const int32_t *pending,
                     int32_t *error_word, void *stream) {
    kda_status st = check_config(cfg);
    if (st != KDA_OK) return st;
    if (B < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;  // nothing to do; no pointer is inspected
    st = check_common(cfg, A_log, g_bias, state_pool, state_indices, B, record_rows, records,
                      error_word);
    if (st != KDA_OK) return st;
    if (!pending || !aligned(pending, 4)) return KDA_ERR_INVALID_ARG;

    Params p = base_params(cfg, B);
    p.A_log = A_log;
    p.g_bias = g_bias;
    p.pool = state_pool;
    p.state_indices = state_indices;
    p.record_rows = record_rows;
    p.records = const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(records));
    p.pending_in = pending;
    p.err = error_word;

    return launch_step<kda::Mode::kFlush>(p, cfg, false, static_cast<cudaStream_t>(stream));
}

const char *kda_status_string(kda_status status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    }
    return "KDA_ERR_UNKNOWN";
}

int32_t kda_abi_version(void) { return 4; }

}  // extern "C"
