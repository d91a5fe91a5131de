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
//  - flush: `KDADeferredCommitContext.flush`.
// The public contract is in include/kda.h.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kda_async.cuh"
#include "kda_device.cuh"
#include "../../include/kda.h"

namespace kda {

static_assert(kRecStride == KDA_RECORD_STRIDE, "record layout mismatch");
static_assert(kD == KDA_HEAD_DIM, "head dim mismatch");
static_assert(kMaxQ == KDA_MAX_WINDOW, "window mismatch");
static_assert(kBadLength == KDA_ROW_BAD_LENGTH && kBadSlot == KDA_ROW_BAD_SLOT &&
                  kBadRecord == KDA_ROW_BAD_RECORD && kBadPending == KDA_ROW_BAD_PENDING &&
                  kErrWaitTimeout == KDA_ERR_WAIT_TIMEOUT,
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

// ------------------------------------------------------------- work items --
//
// A work item is one (row, head) tile with something to do.  Mode decides
// what: the verify runs `p` folded (pending) record tokens then `T` new
// tokens; the commit and the flush replay `p` record tokens.  Every mode
// stores the state when p > 0.

enum class Mode { kVerify, kCommit, kFlush };

struct Work {
    int tile;  // -1: no more work for this CTA
    int head, slot, r, bos, T, p;
};

// Plan one tile: row checks, the commit plan (n = clamp(accepted, 0,
// min(T, Q)), valid iff slot > 0, n > 0, r >= 0), the deferred commit's
// pending write.  Side effects (error bits, pending writes) are made by the
// one thread that plans the tile.
template <Mode kMode>
__device__ __forceinline__ bool plan_tile(const Params &p, int tile, Work &w) {
    const int b = tile / p.H;
    const int head = tile - b * p.H;
    Row row;
    const int bad = read_row(p, b, kMode != Mode::kFlush, row);
    if (bad) {
        if (head == 0) flag_error(p.err, bad);
        return false;
    }
    int fold = 0, T = 0;
    if constexpr (kMode == Mode::kVerify) {
        if (row.slot <= 0) return false;  // null block: padding row
        if (p.pending_in != nullptr && row.r >= 0) {
            fold = p.pending_in[row.r];
            if (fold < 0 || fold > p.Q) {
                if (head == 0) flag_error(p.err, kBadPending);
                return false;
            }
        }
        T = row.T;
        if (T == 0 && fold == 0) return false;
    } else if constexpr (kMode == Mode::kCommit) {
        const int n = min(max(p.num_accepted[b], 0), min(row.T, p.Q));
        const bool valid = row.slot > 0 && n > 0 && row.r >= 0;
        if (p.pending_out != nullptr) {
            const bool now = p.eager != nullptr && p.eager[b] != 0;
            if (head == 0 && row.r >= 0) p.pending_out[row.r] = (valid && !now) ? n : 0;
            if (!now) return false;
        }
        if (!valid) return false;
        fold = n;
    } else {
        if (row.slot <= 0 || row.r < 0) return false;
        const int n = p.pending_in[row.r];
        if (n < 0 || n > p.Q) {
            if (head == 0) flag_error(p.err, kBadPending);
            return false;
        }
        if (n == 0) return false;
        fold = n;
    }
    w.tile = tile;
    w.head = head;
    w.slot = row.slot;
    w.r = row.r;
    w.bos = row.bos;
    w.T = T;
    w.p = fold;
    return true;
}

// ---------------------------------------------------------- shared memory --

constexpr int kPlanThreads = 128;   // candidates planned per round
constexpr int kListCap = kPlanThreads;

// The CTA's work list: candidate k of this CTA is tile blockIdx.x + k *
// gridDim.x.  A planning round plans kPlanThreads candidates at once, one per
// thread, and compacts the ones with work, in order, into the list.
struct WorkList {
    int tile[kListCap];
    int slot[kListCap];
    int r[kListCap];
    int bos[kListCap];
    int tp[kListCap];   // T | p << 8
    int warp_count[kPlanThreads / 32];
    int count;
};

// Raw bf16 inputs and gate parameters of one work item, brought in by
// cp.async: token slots [0, p) are the folded record tokens, [p, p + T) the
// new tokens.  Stored as channel pairs (one 32-bit word = 2 bf16).
struct RawSmem {
    uint32_t k[2 * kMaxQ][kD / 2];
    uint32_t v[2 * kMaxQ][kD / 2];
    uint32_t g[2 * kMaxQ][kD / 2];
    uint32_t q[kMaxQ][kD / 2];
    uint2 tail[kMaxQ];          // record tails: beta_raw bits in the low half
    float bias[kD];             // g_bias of the item's head
    float a_log;                // A_log of the item's head
    uint32_t beta_new[kMaxQ];   // beta_raw bits of the new tokens
};

struct __align__(16) StepSmem {
    float state[kD * kD];       // staging of the next item's checkpoint (TMA)
    TokenSmem tok;              // per-token vectors of the current item
    RawSmem raw;                // raw inputs of the current / next item
    float red_k[2 * kMaxQ][2];  // per-warp halves of |k|^2
    float red_q[kMaxQ][2];      // per-warp halves of |q|^2
    WorkList list;
    uint64_t bar;               // completion of the staging copy
    int ok;
};

constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (about 2 s)

__device__ __forceinline__ int num_candidates(int num_tiles) {
    const int first = (int)blockIdx.x;
    return first < num_tiles ? (num_tiles - first + (int)gridDim.x - 1) / (int)gridDim.x : 0;
}

// One planning round over candidates [k0, k0 + kPlanThreads); all threads
// take part (it contains barriers).  Returns the number of listed items.
template <Mode kMode>
__device__ int plan_round(const Params &p, StepSmem &sm, int k0, int num_tiles, int tid) {
    const int K = num_candidates(num_tiles);
    Work w;
    bool has = false;
    if (tid < kPlanThreads) {
        const int k = k0 + tid;
        if (k < K) has = plan_tile<kMode>(p, (int)blockIdx.x + k * (int)gridDim.x, w);
    }
    const unsigned ballot = __ballot_sync(kFull, has);
    const int lane = tid & 31, warp = tid >> 5;
    if (tid < kPlanThreads && lane == 0) sm.list.warp_count[warp] = __popc(ballot);
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int i = 0; i < kPlanThreads / 32; ++i) {
        const int c = sm.list.warp_count[i];
        if (i < warp) before += c;
        total += c;
    }
    if (has) {
        const int pos = before + __popc(ballot & ((1u << lane) - 1u));
        sm.list.tile[pos] = w.tile;
        sm.list.slot[pos] = w.slot;
        sm.list.r[pos] = w.r;
        sm.list.bos[pos] = w.bos;
        sm.list.tp[pos] = w.T | (w.p << 8);
    }
    __syncthreads();
    return total;
}

__device__ __forceinline__ Work list_item(const StepSmem &sm, int i, int H) {
    Work w;
    w.tile = sm.list.tile[i];
    w.head = w.tile % H;
    w.slot = sm.list.slot[i];
    w.r = sm.list.r[i];
    w.bos = sm.list.bos[i];
    const int tp = sm.list.tp[i];
    w.T = tp & 0xff;
    w.p = tp >> 8;
    return w;
}

// Cursor over the CTA's work: the list of the current round and where the
// next round starts.  Uniform across the CTA.
struct Cursor {
    int idx, count, next_k;
};

// Advance to the next listed item (planning a new round when the list is
// used up).  Returns its list index, or -1 when the CTA has no more work.
// The item stays readable in the list until the following call.
template <Mode kMode>
__device__ __forceinline__ int next_item(const Params &p, StepSmem &sm, Cursor &c, int num_tiles,
                                         int tid) {
    const int K = num_candidates(num_tiles);
    while (c.idx >= c.count) {
        if (c.next_k >= K) return -1;
        c.count = plan_round<kMode>(p, sm, c.next_k, num_tiles, tid);
        c.next_k += kPlanThreads;
        c.idx = 0;
    }
    return c.idx++;
}

__device__ __forceinline__ void issue_state(const Params &p, const Work &w, StepSmem &sm) {
    const float *src = p.pool + ((size_t)w.slot * p.H + w.head) * (size_t)(kD * kD);
    mbar_arrive_expect_tx(&sm.bar, kD * kD * 4);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        bulk_load(sm.state + c * (kD * kD / 4), src + c * (kD * kD / 4), kD * kD, &sm.bar);
}

// Raw inputs and gate parameters of an item into shared memory (cp.async).
template <Mode kMode>
__device__ __forceinline__ void fetch_raw(const Params &p, const Work &w, RawSmem &raw, int warp,
                                          int lane) {
    const __nv_bfloat16 *rec = record_base(p, w.r, w.head);
    for (int c = warp; c < 3 * w.p; c += kWarps) {
        const int u = c / 3;
        const int part = c - 3 * u;
        const uint2 *src = reinterpret_cast<const uint2 *>(rec + (size_t)u * kRecStride + part * kD);
        uint32_t *dst = part == 0 ? raw.k[u] : (part == 1 ? raw.v[u] : raw.g[u]);
        cp_async8(dst + 2 * lane, src + lane);
    }
    if (warp == kWarps - 1) {
        if (lane < w.p) cp_async8(&raw.tail[lane], rec + (size_t)lane * kRecStride + kRecBeta);
        if (lane == 31) cp_async4(&raw.a_log, p.A_log + w.head);
    }
    if (warp == kWarps - 2) cp_async16(&raw.bias[4 * lane], p.g_bias + w.head * kD + 4 * lane);
    if constexpr (kMode == Mode::kVerify) {
        for (int c = warp; c < 4 * w.T; c += kWarps) {
            const int t = c >> 2;
            const int part = c & 3;
            const size_t tok = (size_t)(w.bos + t);
            const __nv_bfloat16 *src;
            uint32_t *dst;
            if (part == 0) {
                src = p.k + tok * p.stride_k;
                dst = raw.k[w.p + t];
            } else if (part == 1) {
                src = p.v + tok * p.stride_v;
                dst = raw.v[w.p + t];
            } else if (part == 2) {
                src = p.g + tok * p.stride_g;
                dst = raw.g[w.p + t];
            } else {
                src = p.q + tok * p.stride_q;
                dst = raw.q[t];
            }
            cp_async8(dst + 2 * lane, reinterpret_cast<const uint2 *>(src + w.head * kD) + lane);
        }
    }
    cp_async_commit();
}

// Per-token vectors of an item, all 8 warps: token u is prepared by the 64
// threads of quarter (u & 3) in pass (u >> 2), two channels per thread, so
// every token is computed the same way however many tokens the item has.
// The verify also writes the new tokens' raw records.
template <Mode kMode, bool kBounded>
__device__ __forceinline__ void prep_item(StepSmem &sm, const Params &p, const Work &w, int tid) {
    const int quarter = tid >> 6;
    const int c2 = tid & 63;              // channels 2*c2, 2*c2 + 1
    const int half = c2 >> 5;             // which of the quarter's two warps
    const bool lead = (tid & 31) == 0;
    const int total = w.p + w.T;
    const int passes = (total + 3) >> 2;
    const float a = expf(sm.raw.a_log);
    const float2 bias = *reinterpret_cast<const float2 *>(&sm.raw.bias[2 * c2]);
    __nv_bfloat16 *rec = record_base(p, w.r, w.head);
    for (int pass = 0; pass < passes; ++pass) {
        const int u = 4 * pass + quarter;
        const bool active = u < total;
        const bool is_new = kMode == Mode::kVerify && u >= w.p;
        const int t = u - w.p;
        float2 k = make_float2(0.f, 0.f), q = make_float2(0.f, 0.f);
        if (active) {
            const uint32_t kb = sm.raw.k[u][c2], vb = sm.raw.v[u][c2], gb = sm.raw.g[u][c2];
            k = bf16x2_to_float2(kb);
            const float sk = warp_allsum(__fmaf_rn(k.y, k.y, __fmul_rn(k.x, k.x)));
            if (lead) sm.red_k[u][half] = sk;
            const float2 g = bf16x2_to_float2(gb);
            float2 e;
            e.x = decay_factor(__fadd_rn(g.x, bias.x), a, kBounded, p.lower_bound);
            e.y = decay_factor(__fadd_rn(g.y, bias.y), a, kBounded, p.lower_bound);
            *reinterpret_cast<float2 *>(&sm.tok.e[u][2 * c2]) = e;
            *reinterpret_cast<float2 *>(&sm.tok.v[u][2 * c2]) = bf16x2_to_float2(vb);
            const uint32_t bb = is_new ? sm.raw.beta_new[t] : (sm.raw.tail[u].x & 0xffffu);
            if (c2 == 0) sm.tok.beta[u] = sigmoidf_rn(bf16_bits_to_float(bb));
            if (is_new) {
                const uint32_t qb = sm.raw.q[t][c2];
                q = bf16x2_to_float2(qb);
                const float sq = warp_allsum(__fmaf_rn(q.y, q.y, __fmul_rn(q.x, q.x)));
                if (lead) sm.red_q[t][half] = sq;
                __nv_bfloat16 *dst = rec + (size_t)t * kRecStride;
                reinterpret_cast<uint32_t *>(dst)[c2] = kb;
                reinterpret_cast<uint32_t *>(dst + kRecV)[c2] = vb;
                reinterpret_cast<uint32_t *>(dst + kRecG)[c2] = gb;
                if (c2 == 0) reinterpret_cast<uint16_t *>(dst)[kRecBeta] = (uint16_t)bb;
            }
        }
        __syncthreads();  // both halves of the norms are in
        if (active) {
            const float ik = inv_l2(__fadd_rn(sm.red_k[u][0], sm.red_k[u][1]));
            *reinterpret_cast<float2 *>(&sm.tok.kh[u][2 * c2]) =
                make_float2(__fmul_rn(k.x, ik), __fmul_rn(k.y, ik));
            if (is_new) {
                const float iq = inv_l2(__fadd_rn(sm.red_q[t][0], sm.red_q[t][1]));
                *reinterpret_cast<float2 *>(&sm.tok.qh[t][2 * c2]) =
                    make_float2(__fmul_rn(__fmul_rn(q.x, iq), p.scale),
                                __fmul_rn(__fmul_rn(q.y, iq), p.scale));
            }
        }
    }
}

// ------------------------------------------------------------------ kernel --
//
// Persistent: gridDim.x CTAs (two per SM) walk the tiles b*H + head with a
// stride of gridDim.x, planned in rounds into a shared-memory work list.
// While a CTA computes one item from registers, the next item's checkpoint
// streams into shared memory through the TMA unit and its raw inputs and
// gate parameters through cp.async, so memory and arithmetic overlap.

template <Mode kMode, bool kBounded>
__global__ void __launch_bounds__(kThreads, 2) step_kernel(const Params p, int num_tiles) {
    extern __shared__ __align__(128) unsigned char smem_bytes[];
    StepSmem &sm = *reinterpret_cast<StepSmem *>(smem_bytes);
    const int tid = threadIdx.x;
    Lane L;
    L.lane = tid & 31;
    L.w = tid >> 5;
    L.g = L.lane >> 3;
    L.j = L.lane & 7;

    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    Cursor cursor{0, 0, 0};
    const int first = next_item<kMode>(p, sm, cursor, num_tiles, tid);
    if (first < 0) return;
    Work cur = list_item(sm, first, p.H);
    if (tid == 0) issue_state(p, cur, sm);
    fetch_raw<kMode>(p, cur, sm.raw, L.w, L.lane);
    uint32_t beta_next = 0;
    if (kMode == Mode::kVerify && tid < cur.T)
        beta_next = reinterpret_cast<const uint16_t *>(
            p.beta)[(size_t)(cur.bos + tid) * p.stride_beta + cur.head];
    uint32_t phase = 0;

    while (true) {
        // raw inputs of `cur` have landed (each thread waits for its own
        // copies; the barrier publishes them and frees the token vectors)
        cp_async_wait_all();
        if (kMode == Mode::kVerify && tid < cur.T) sm.raw.beta_new[tid] = beta_next;
        __syncthreads();

        prep_item<kMode, kBounded>(sm, p, cur, tid);

        // checkpoint of `cur`: staged by the TMA unit
        if (tid == 0) sm.ok = mbar_wait_bounded(&sm.bar, phase, kWaitBudget) ? 1 : 0;
        __syncthreads();  // also: token vectors ready, raw inputs consumed
        if (!sm.ok) {
            if (tid == 0) {
                flag_error(p.err, kErrWaitTimeout);
                mbar_wait_bounded(&sm.bar, phase, kWaitBudget);
            }
            return;
        }
        mbar_try_wait(&sm.bar, phase);  // completed phase: acquires the staged bytes
        phase ^= 1u;
        float4 h[4][4];
        load_tile(h, sm.state, L);
        __syncthreads();  // staging buffer free

        // start the next item's copies before computing this one
        const int nidx = next_item<kMode>(p, sm, cursor, num_tiles, tid);
        if (nidx >= 0) {
            const Work nxt = list_item(sm, nidx, p.H);
            if (tid == 0) issue_state(p, nxt, sm);
            fetch_raw<kMode>(p, nxt, sm.raw, L.w, L.lane);
            if (kMode == Mode::kVerify && tid < nxt.T)
                beta_next = reinterpret_cast<const uint16_t *>(
                    p.beta)[(size_t)(nxt.bos + tid) * p.stride_beta + nxt.head];
        }

        // replay the folded / accepted records, store the state once
        float *tile = p.pool + ((size_t)cur.slot * p.H + cur.head) * (size_t)(kD * kD);
        for (int u = 0; u < cur.p; ++u) token_step<false>(h, sm.tok, u, 0, L, nullptr);
        if (cur.p > 0) store_tile(h, tile, L);
        if constexpr (kMode == Mode::kVerify) {
            for (int t = 0; t < cur.T; ++t) {
                const size_t tok = (size_t)(cur.bos + t);
                token_step<true>(h, sm.tok, cur.p + t, t, L, p.out + (tok * p.H + cur.head) * kD);
                if (p.traj != nullptr)
                    store_tile(h, p.traj + (tok * p.H + cur.head) * (size_t)(kD * kD), L);
            }
        }
        if (nidx < 0) break;
        cur = list_item(sm, nidx, p.H);
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
    if (cfg->use_lower_bound != 0 && cfg->use_lower_bound != 1) return KDA_ERR_INVALID_ARG;
    if (cfg->use_lower_bound == 1 && !(cfg->lower_bound < 0.0f && isfinite(cfg->lower_bound)))
        return KDA_ERR_INVALID_ARG;
    if (!isfinite(cfg->scale)) return KDA_ERR_INVALID_ARG;
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
                        const int32_t *record_rows, const void *records) {
    if (!A_log || !g_bias || !pool || !state_indices || !records) return KDA_ERR_INVALID_ARG;
    if (!aligned(g_bias, 16) || !aligned(pool, 16) || !aligned(A_log, 4) ||
        !aligned(state_indices, 4) || !aligned(records, 16))
        return KDA_ERR_INVALID_ARG;
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

// Launch the persistent step kernel: two CTAs per SM (or one per tile when
// there are fewer tiles), each with the StepSmem layout in dynamic shared
// memory.
template <kda::Mode M>
kda_status launch_step(const Params &p, bool bounded, cudaStream_t stream) {
    const long long tiles = (long long)p.B * p.H;
    const int sms = sm_count();
    if (sms <= 0) return KDA_ERR_CUDA;
    const int grid = (int)(tiles < 2LL * sms ? tiles : 2LL * sms);
    const size_t smem = sizeof(kda::StepSmem);
    void (*kern)(const Params, int) =
        bounded ? kda::step_kernel<M, true> : kda::step_kernel<M, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return KDA_ERR_CUDA;
    kern<<<grid, kda::kThreads, smem, stream>>>(p, (int)tiles);
    return finish_launch();
}

}  // namespace

extern "C" {

size_t kda_records_bytes(int32_t num_heads, int32_t window, int32_t record_slots) {
    if (num_heads < 1 || window < 1 || window > KDA_MAX_WINDOW || record_slots < 0) return 0;
    return (size_t)(record_slots + 1) * (size_t)num_heads * (size_t)window *
           (size_t)KDA_RECORD_STRIDE * 2u;
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
    st = check_common(cfg, A_log, g_bias, state_pool, state_indices, B, record_rows, records);
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

    return launch_step<kda::Mode::kVerify>(p, cfg->use_lower_bound != 0,
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
    st = check_common(cfg, A_log, g_bias, state_pool, state_indices, B, record_rows, records);
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

    return launch_step<kda::Mode::kCommit>(p, cfg->use_lower_bound != 0,
                                           static_cast<cudaStream_t>(stream));
}

kda_status kda_flush(const kda_config *cfg, const float *A_log, const float *g_bias,
                     float *state_pool, const int32_t *state_indices, int32_t B,
                     const int32_t *record_rows, const void *records, const int32_t *pending,
                     int32_t *error_word, void *stream) {
    kda_status st = check_config(cfg);
    if (st != KDA_OK) return st;
    if (B < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;  // nothing to do; no pointer is inspected
    st = check_common(cfg, A_log, g_bias, state_pool, state_indices, B, record_rows, records);
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

    return launch_step<kda::Mode::kFlush>(p, cfg->use_lower_bound != 0,
                                          static_cast<cudaStream_t>(stream));
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

int32_t kda_abi_version(void) { return 1; }

}  // extern "C"
