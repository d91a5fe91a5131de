// Device building blocks of the KDA verify / commit kernels (sm_103a).
//
// One CTA owns one (request row, head) state tile S (128 x 128 fp32, row v,
// column k) for the whole window, in registers.  256 threads = 8 warps; warp
// w owns rows 16w .. 16w+15.  Inside a warp, lane = 8*g + j: the thread owns
// the 4 rows 16w + 4g + i (i = 0..3) and, of each row, the 16 columns
// 32m + 4j + c (m = 0..3, c = 0..3), held as float4 h[i][m].  A row therefore
// lives in the 8 lanes that share g, and its dot products (S k^, S q^) are
// reduced across those 8 lanes with shuffles only: no shared memory and no
// block barrier inside the token loop.
//
// The per-token vectors that do not depend on the state (k^, q^, exp(g),
// beta, v) are computed once per CTA per token and kept in shared memory; the
// token loop reads them with conflict-free broadcast loads.
//
// Bit-exactness of commit against verify: the verify, the commit replay, the
// deferred fold and the flush all run `token_step` below with the same thread
// mapping, the same explicit round-to-nearest intrinsics (no contraction left
// to the compiler) and the same reduction tree, so the state after token n is
// the same bits whichever kernel computes it.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {

constexpr int kD = 128;             // head dim, K = V
constexpr int kThreads = 256;       // threads per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kMaxQ = 8;            // window limit
constexpr int kRecStride = 392;     // bf16 elements per token record
constexpr int kRecV = 128;          // offset of v inside a token record
constexpr int kRecG = 256;          // offset of g_raw
constexpr int kRecBeta = 384;       // offset of beta_raw
constexpr unsigned kFull = 0xffffffffu;

// Error-word bits (same values as the public header's macros).
constexpr int kBadLength = 1;
constexpr int kBadSlot = 2;
constexpr int kBadRecord = 4;
constexpr int kBadPending = 8;
constexpr int kErrWaitTimeout = 16;

// Everything a launch needs; passed by value as the kernel parameter.
struct Params {
    int H, Q, S, R, B;
    int bounded;
    float lower_bound;
    float scale;
    long long stride_q, stride_k, stride_v, stride_g, stride_beta;
    const __nv_bfloat16 *q, *k, *v, *g, *beta;
    const float *A_log, *g_bias;
    float *pool;
    const int *cu_seqlens, *state_indices, *record_rows;
    const int *pending_in;     // verify fold / flush
    int *pending_out;          // deferred commit
    const int *num_accepted;
    const uint8_t *eager;
    __nv_bfloat16 *records;
    __nv_bfloat16 *out;
    float *traj;
    int *err;
};

// Per-token vectors of one window, in shared memory.  Slots [0, p) hold the
// folded (recorded) tokens, [p, p + T) the new ones; q^ only for new tokens.
struct TokenSmem {
    float kh[2 * kMaxQ][kD];
    float e[2 * kMaxQ][kD];
    float v[2 * kMaxQ][kD];
    float qh[kMaxQ][kD];
    float beta[2 * kMaxQ];
};

// ---------------------------------------------------------------- helpers --

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// Butterfly sum over the 32 lanes: every lane ends with the same bits
// (IEEE addition is commutative, and each step pairs lanes symmetrically).
__device__ __forceinline__ float warp_allsum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(kFull, x, o));
    return x;
}

// 1 / sqrt(sum + 1e-6), correctly rounded sqrt and division.
__device__ __forceinline__ float inv_l2(float sum) {
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(sum, 1e-6f)));
}

// exp(g) for one channel, x = g_raw + g_bias, a = exp(A_log[h]).
// Bounded gate: g = lb * sigmoid(a x) = lb / (1 + exp(-a x)).
// Softplus gate: g = -a * softplus(x), softplus(x) = x for x > 20.
__device__ __forceinline__ float decay_factor(float x, float a, bool bounded, float lb) {
    float g;
    if (bounded) {
        g = __fdiv_rn(lb, __fadd_rn(1.0f, expf(-__fmul_rn(a, x))));
    } else {
        float sp = x > 20.0f ? x : log1pf(expf(x));
        g = -__fmul_rn(a, sp);
    }
    return expf(g);
}

__device__ __forceinline__ float sigmoidf_rn(float x) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-x)));
}

// ------------------------------------------------------------ state tile --

struct Lane {
    int w, g, j, lane;
    __device__ __forceinline__ int row(int i) const { return 16 * w + 4 * g + i; }
    __device__ __forceinline__ int col(int m) const { return 32 * m + 4 * j; }
};

__device__ __forceinline__ void load_tile(float4 (&h)[4][4], const float *tile, const Lane &L) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m)
            h[i][m] = *reinterpret_cast<const float4 *>(tile + L.row(i) * kD + L.col(m));
}

__device__ __forceinline__ void store_tile(const float4 (&h)[4][4], float *tile, const Lane &L) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m)
            *reinterpret_cast<float4 *>(tile + L.row(i) * kD + L.col(m)) = h[i][m];
}

// Packed pairs of fp32 operations (Blackwell's f32x2 forms): each lane does
// two independent round-to-nearest multiplies or fused multiply-adds per
// instruction, bit-identical to two scalar __fmul_rn / __fmaf_rn.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 unpack2(unsigned long long v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

__device__ __forceinline__ float2 mul2(float ax, float ay, float bx, float by) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack2(ax, ay)), "l"(pack2(bx, by)));
    return unpack2(d);
}

__device__ __forceinline__ float2 fma2(float ax, float ay, float bx, float by, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(pack2(ax, ay)), "l"(pack2(bx, by)), "l"(pack2(c.x, c.y)));
    return unpack2(d);
}

// Row dot products of the thread's 4 rows with a vector x (its 16 columns),
// in a fixed order: two interleaved partial sums per row (the even and the
// odd columns of each float4, one packed pair), then their sum.
__device__ __forceinline__ void row_partials(const float4 (&h)[4][4], const float4 (&x)[4],
                                             float (&part)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 a = mul2(h[i][0].x, h[i][0].y, x[0].x, x[0].y);
        a = fma2(h[i][0].z, h[i][0].w, x[0].z, x[0].w, a);
#pragma unroll
        for (int m = 1; m < 4; ++m) {
            a = fma2(h[i][m].x, h[i][m].y, x[m].x, x[m].y, a);
            a = fma2(h[i][m].z, h[i][m].w, x[m].z, x[m].w, a);
        }
        part[i] = __fadd_rn(a.x, a.y);
    }
}

// Sum the 4 row partials over the 8 lanes of the row group (lane bits 0..2)
// by a transpose-reduce: after it, lane j holds the full sum of row
// R(j) = 2*bit2(j) + bit1(j); lanes j and j^1 hold identical bits.
__device__ __forceinline__ float reduce_rows(const float (&part)[4], int j) {
    const bool hi = (j & 4) != 0;
    const float send0 = hi ? part[0] : part[2];
    const float send1 = hi ? part[1] : part[3];
    const float keep0 = hi ? part[2] : part[0];
    const float keep1 = hi ? part[3] : part[1];
    const float t0 = __fadd_rn(keep0, __shfl_xor_sync(kFull, send0, 4));
    const float t1 = __fadd_rn(keep1, __shfl_xor_sync(kFull, send1, 4));
    const bool mid = (j & 2) != 0;
    const float send = mid ? t0 : t1;
    const float keep = mid ? t1 : t0;
    const float u = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 2));
    return __fadd_rn(u, __shfl_xor_sync(kFull, u, 1));
}

__device__ __forceinline__ int reduced_row(int j) { return 2 * ((j >> 2) & 1) + ((j >> 1) & 1); }

// One token of the recurrence on the thread's part of the tile:
//   S <- S diag(e);  u = S k^;  v' = beta (v - u);  S <- S + v' k^T
// and, when kOut, o = S q^ written as bf16 to out_row (128 outputs).
template <bool kOut>
__device__ __forceinline__ void token_step(float4 (&h)[4][4], const TokenSmem &sm, int slot,
                                           int qslot, const Lane &L,
                                           __nv_bfloat16 *out_row) {
    float4 kk[4], ee[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        kk[m] = *reinterpret_cast<const float4 *>(&sm.kh[slot][L.col(m)]);
        ee[m] = *reinterpret_cast<const float4 *>(&sm.e[slot][L.col(m)]);
    }
    // decay along K
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float2 lo = mul2(h[i][m].x, h[i][m].y, ee[m].x, ee[m].y);
            const float2 hi = mul2(h[i][m].z, h[i][m].w, ee[m].z, ee[m].w);
            h[i][m] = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
    // u = S k^ for the 4 rows, reduced over the row group
    float part[4];
    row_partials(h, kk, part);
    const float u = reduce_rows(part, L.j);
    const int R = reduced_row(L.j);
    const float vr = sm.v[slot][L.row(R)];
    const float vp = __fmul_rn(sm.beta[slot], __fsub_rn(vr, u));
    // every lane of the group gets v' of its 4 rows (lanes 2i hold row i)
    const int base = L.lane & ~7;
    float vpi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) vpi[i] = __shfl_sync(kFull, vp, base + 2 * i);
    // rank-one update
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float2 lo =
                fma2(vpi[i], vpi[i], kk[m].x, kk[m].y, make_float2(h[i][m].x, h[i][m].y));
            const float2 hi =
                fma2(vpi[i], vpi[i], kk[m].z, kk[m].w, make_float2(h[i][m].z, h[i][m].w));
            h[i][m] = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
    if constexpr (kOut) {
        float4 qq[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
            qq[m] = *reinterpret_cast<const float4 *>(&sm.qh[qslot][L.col(m)]);
        float opart[4];
        row_partials(h, qq, opart);
        const float o = reduce_rows(opart, L.j);
        if ((L.j & 1) == 0) out_row[L.row(R)] = __float2bfloat16_rn(o);
    }
}

__device__ __forceinline__ void flag_error(int *err, int bits) {
    if (err != nullptr) atomicOr(err, bits);
}

}  // namespace kda
