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

#include "kda_device.cuh"
#include "../../include/kda.h"

namespace kda {

static_assert(kRecStride == KDA_RECORD_STRIDE, "record layout mismatch");
static_assert(kD == KDA_HEAD_DIM, "head dim mismatch");
static_assert(kMaxQ == KDA_MAX_WINDOW, "window mismatch");
static_assert(kBadLength == KDA_ROW_BAD_LENGTH && kBadSlot == KDA_ROW_BAD_SLOT &&
                  kBadRecord == KDA_ROW_BAD_RECORD && kBadPending == KDA_ROW_BAD_PENDING,
              "row-check bits mismatch");

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

// Prepare `count` recorded tokens into smem slots [0, count).
__device__ __forceinline__ void prep_records(TokenSmem &sm, const __nv_bfloat16 *rec, int count,
                                             const float4 bias, float a, bool bounded, float lb,
                                             int warp, int lane) {
    for (int t = warp; t < count; t += kWarps) {
        const RawToken raw = load_record(rec + (size_t)t * kRecStride, lane);
        prep_token(sm, t, raw, bias, a, bounded, lb, lane);
    }
}

// ------------------------------------------------------------------ verify --

template <bool kBounded>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const Params p) {
    __shared__ __align__(16) TokenSmem sm;
    const int b = blockIdx.x / p.H;
    const int head = blockIdx.x - b * p.H;
    const int tid = threadIdx.x;
    Lane L;
    L.lane = tid & 31;
    L.w = tid >> 5;
    L.g = L.lane >> 3;
    L.j = L.lane & 7;

    Row row;
    const int bad = read_row(p, b, true, row);
    if (bad) {
        if (head == 0 && tid == 0) flag_error(p.err, bad);
        return;
    }
    if (row.slot <= 0) return;  // null block: padding row
    int pend = 0;
    if (p.pending_in != nullptr && row.r >= 0) {
        pend = p.pending_in[row.r];
        if (pend < 0 || pend > p.Q) {
            if (head == 0 && tid == 0) flag_error(p.err, kBadPending);
            return;
        }
    }
    if (row.T == 0 && pend == 0) return;

    float *tile = p.pool + ((size_t)row.slot * p.H + head) * (size_t)(kD * kD);
    float4 h[4][4];
    load_tile(h, tile, L);  // in flight while the token vectors are prepared

    const float a = expf(p.A_log[head]);
    const float4 bias = *reinterpret_cast<const float4 *>(p.g_bias + head * kD + 4 * L.lane);
    __nv_bfloat16 *rec = record_base(p, row.r, head);

    if (pend > 0) {  // the recorded tokens must be read before they are overwritten
        prep_records(sm, rec, pend, bias, a, kBounded, p.lower_bound, L.w, L.lane);
        __syncthreads();
    }
    for (int t = L.w; t < row.T; t += kWarps) {
        const size_t tok = (size_t)(row.bos + t);
        RawToken raw;
        raw.k = *reinterpret_cast<const uint2 *>(p.k + tok * p.stride_k + head * kD + 4 * L.lane);
        raw.v = *reinterpret_cast<const uint2 *>(p.v + tok * p.stride_v + head * kD + 4 * L.lane);
        raw.g = *reinterpret_cast<const uint2 *>(p.g + tok * p.stride_g + head * kD + 4 * L.lane);
        raw.beta = L.lane == 0
                       ? (uint32_t) reinterpret_cast<const uint16_t *>(p.beta)[tok * p.stride_beta + head]
                       : 0u;
        const uint2 qraw =
            *reinterpret_cast<const uint2 *>(p.q + tok * p.stride_q + head * kD + 4 * L.lane);
        prep_token(sm, pend + t, raw, bias, a, kBounded, p.lower_bound, L.lane);
        prep_query(sm, t, qraw, p.scale, L.lane);
        store_record(rec + (size_t)t * kRecStride, raw, L.lane);
    }
    __syncthreads();

    // deferred fold: replay the pending records, store the folded checkpoint
    for (int t = 0; t < pend; ++t) token_step<false>(h, sm, t, 0, L, nullptr);
    if (pend > 0) store_tile(h, tile, L);

    for (int t = 0; t < row.T; ++t) {
        const size_t tok = (size_t)(row.bos + t);
        token_step<true>(h, sm, pend + t, t, L, p.out + (tok * p.H + head) * kD);
        if (p.traj != nullptr) store_tile(h, p.traj + (tok * p.H + head) * (size_t)(kD * kD), L);
    }
}

// --------------------------------------------------------- commit / flush --

enum class Replay { kCommit, kFlush };

template <bool kBounded, Replay kMode>
__global__ void __launch_bounds__(kThreads, 2) replay_kernel(const Params p) {
    __shared__ __align__(16) TokenSmem sm;
    const int b = blockIdx.x / p.H;
    const int head = blockIdx.x - b * p.H;
    const int tid = threadIdx.x;
    Lane L;
    L.lane = tid & 31;
    L.w = tid >> 5;
    L.g = L.lane >> 3;
    L.j = L.lane & 7;

    Row row;
    const int bad = read_row(p, b, kMode == Replay::kCommit, row);
    if (bad) {
        if (head == 0 && tid == 0) flag_error(p.err, bad);
        return;
    }
    int n;
    if constexpr (kMode == Replay::kCommit) {
        // commit plan: accepted count clamped to [0, T] and to the window
        n = min(max(p.num_accepted[b], 0), min(row.T, p.Q));
        const bool valid = row.slot > 0 && n > 0 && row.r >= 0;
        if (p.pending_out != nullptr) {
            const bool now = p.eager != nullptr && p.eager[b] != 0;
            if (head == 0 && tid == 0 && row.r >= 0) p.pending_out[row.r] = (valid && !now) ? n : 0;
            if (!now) return;
        }
        if (!valid) return;
    } else {
        if (row.slot <= 0 || row.r < 0) return;
        n = p.pending_in[row.r];
        if (n < 0 || n > p.Q) {
            if (head == 0 && tid == 0) flag_error(p.err, kBadPending);
            return;
        }
        if (n == 0) return;
    }

    float *tile = p.pool + ((size_t)row.slot * p.H + head) * (size_t)(kD * kD);
    float4 h[4][4];
    load_tile(h, tile, L);

    const float a = expf(p.A_log[head]);
    const float4 bias = *reinterpret_cast<const float4 *>(p.g_bias + head * kD + 4 * L.lane);
    prep_records(sm, record_base(p, row.r, head), n, bias, a, kBounded, p.lower_bound, L.w,
                 L.lane);
    __syncthreads();
    for (int t = 0; t < n; ++t) token_step<false>(h, sm, t, 0, L, nullptr);
    store_tile(h, tile, L);
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

    const dim3 grid((unsigned)(B * cfg->num_heads));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cfg->use_lower_bound)
        kda::verify_kernel<true><<<grid, kda::kThreads, 0, s>>>(p);
    else
        kda::verify_kernel<false><<<grid, kda::kThreads, 0, s>>>(p);
    return finish_launch();
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

    const dim3 grid((unsigned)(B * cfg->num_heads));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    using kda::Replay;
    if (cfg->use_lower_bound)
        kda::replay_kernel<true, Replay::kCommit><<<grid, kda::kThreads, 0, s>>>(p);
    else
        kda::replay_kernel<false, Replay::kCommit><<<grid, kda::kThreads, 0, s>>>(p);
    return finish_launch();
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

    const dim3 grid((unsigned)(B * cfg->num_heads));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    using kda::Replay;
    if (cfg->use_lower_bound)
        kda::replay_kernel<true, Replay::kFlush><<<grid, kda::kThreads, 0, s>>>(p);
    else
        kda::replay_kernel<false, Replay::kFlush><<<grid, kda::kThreads, 0, s>>>(p);
    return finish_launch();
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
