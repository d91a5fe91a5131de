// Device building blocks of the KDA verify / commit kernels (sm_103a).
//
// A consumer group of 128 threads (4 warps) owns one (request row, head)
// state tile S (128 x 128 fp32, row v, column k) in registers for the whole
// window.  Warp w owns rows 32w .. 32w+31; inside a warp, lane = 8*g + j and
// the thread owns the 8 rows 32w + 8g + i (i = 0..7) and, of each row, the 16
// columns 32m + 4j + c (m = 0..3, c = 0..3), held as float4 h[i][m].  A row
// lives in the 8 lanes that share g, so its dot products (S k^, S q^) are
// reduced across those 8 lanes with shuffles only.
//
// The per-token vectors that do not depend on the state (k^, q^, exp(g),
// beta, v, or a recorded token's delta v') are prepared by producer warps
// into shared memory; the token loop reads them with conflict-free
// broadcast loads.
//
// Bit-exactness of commit against verify: the verify, the commit replay, the
// deferred fold and the flush all run the token pieces below with the same
// thread mapping, the same explicit round-to-nearest intrinsics (no
// contraction left to the compiler), the same reduction tree and the same
// token preparation, so the state after a token has the same bits whichever
// kernel computes it.  With correction records the replays skip the
// prediction and apply the v' the verify stored, through the same decay and
// rank-one pieces, so they reach the same bits too.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_tc.cuh"

namespace kda {

constexpr int kD = 128;             // head dim, K = V
constexpr int kMaxQ = 8;            // window limit
constexpr int kRecStride = 392;     // bf16 elements per token record
constexpr int kRecV = 128;          // offset of v inside a token record
constexpr int kRecG = 256;          // offset of g_raw
constexpr int kRecBeta = 384;       // offset of beta_raw
// Correction records (the fp32-correction form): per token 1024 bytes, the
// fp32 delta v' at byte 0, bf16 k at byte 512 and bf16 g_raw at byte 768.
constexpr int kCorrBytes = 1024;
constexpr int kCorrK = 512;
constexpr int kCorrG = 768;
constexpr unsigned kFull = 0xffffffffu;

// Error-word bits (same values as the public header's macros).
constexpr int kBadLength = 1;
constexpr int kBadSlot = 2;
constexpr int kBadRecord = 4;
constexpr int kBadPending = 8;
constexpr int kErrWaitTimeout = 16;
constexpr int kBadBlock = 32;

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
    // align-mode commit (block_table == nullptr: off)
    const int *block_table, *num_computed, *request_indices;
    long long bt_stride;
    int bt_width, block_size, num_requests;
    // verify window items with no folded token on the tensor core (the
    // launch's tensor map of the state pool is valid)
    int tc_window;
};

// ---------------------------------------------------------------- helpers --

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 u) {
    const float2 a = bf16x2_to_float2(u.x), b = bf16x2_to_float2(u.y);
    return make_float4(a.x, a.y, b.x, b.y);
}

// Butterfly sum over the 32 lanes: every lane ends with the same bits
// (IEEE addition is commutative, and each step pairs lanes symmetrically).
__device__ __forceinline__ float warp_allsum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(kFull, x, o));
    return x;
}

// 1 / sqrt(sum + 1e-6), with CUDA's rsqrtf (within 2 ulp).
__device__ __forceinline__ float inv_l2(float sum) {
    return rsqrtf(__fadd_rn(sum, 1e-6f));
}

// The gate's exponentials use CUDA's __expf intrinsic and its divisions the
// __fdividef intrinsic: their documented error bounds (2 + floor(|1.16 x|)
// ulp for __expf, 2 ulp for __fdividef in this range) cost the state a few
// ulp per token, far inside the state tolerance, and they take half the
// instructions of the accurate forms on the producer's path.  Verify and
// commit call the same functions, so their states stay bit-identical.
//
// softplus(x) = log(1 + e^x), taken as x itself for x > 20, evaluated as
// max(x, 0) + log1p(z) with z = e^{-|x|} in (0, 1] (an identity) and
// log1p(z) = z * P(z): P is a degree-9 least-squares fit of log1p(z) / z on
// [0, 1] (coefficients from softplus_poly.py), within 2 ulp of log1p in
// fp32.  A fixed chain of fused multiply-adds: no branch, no logarithm.
__device__ __forceinline__ float softplus(float x) {
    constexpr float c[10] = {0x1p+0f,        -0x1.ffffcp-2f,  0x1.554c9cp-2f, -0x1.ff11c2p-3f,
                             0x1.930202p-3f, -0x1.399642p-3f, 0x1.b2c2a2p-4f, -0x1.d3784ep-5f,
                             0x1.4628bp-6f,  -0x1.aad1eep-9f};
    const float z = __expf(-fabsf(x));
    float r = c[9];
#pragma unroll
    for (int i = 8; i >= 0; --i) r = __fmaf_rn(r, z, c[i]);
    const float l = __fmul_rn(z, r);
    const float sp = x > 0.0f ? __fadd_rn(x, l) : l;
    return x > 20.0f ? x : sp;
}

// exp(g) for one channel, x = g_raw + g_bias, a = exp(A_log[h]).
// Bounded gate: g = lb * sigmoid(a x) = lb / (1 + exp(-a x)).
// Softplus gate: g = -a * softplus(x).
__device__ __forceinline__ float decay_factor(float x, float a, bool bounded, float lb) {
    float g;
    if (bounded)
        g = __fdividef(lb, __fadd_rn(1.0f, __expf(-__fmul_rn(a, x))));
    else
        g = -__fmul_rn(a, softplus(x));
    return __expf(g);
}

__device__ __forceinline__ float sigmoidf_rn(float x) {
    return __fdividef(1.0f, __fadd_rn(1.0f, __expf(-x)));
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

__device__ __forceinline__ float4 ld4(const float *ptr) {
    return *reinterpret_cast<const float4 *>(ptr);
}

__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
    return make_float4(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y), __fmul_rn(a.z, b.z),
                       __fmul_rn(a.w, b.w));
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    float d = __fmul_rn(a.x, b.x);
    d = __fmaf_rn(a.y, b.y, d);
    d = __fmaf_rn(a.z, b.z, d);
    return __fmaf_rn(a.w, b.w, d);
}

// Sums 16 values over the 32 lanes of a warp: a reduce-scatter over lane bits
// 3..0 (each step keeps half of the values and adds the partner's other
// half), then one exchange across lane bit 4.  Lane l ends with the sum of
// value (l & 15) over all lanes, in a fixed order.
__device__ __forceinline__ float reduce16(const float (&x)[16], int lane) {
    float y8[8], y4[4], y2[2];
    const bool h8 = (lane & 8) != 0, h4 = (lane & 4) != 0, h2 = (lane & 2) != 0,
               h1 = (lane & 1) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        y8[i] = __fadd_rn(h8 ? x[i + 8] : x[i], __shfl_xor_sync(kFull, h8 ? x[i] : x[i + 8], 8));
#pragma unroll
    for (int i = 0; i < 4; ++i)
        y4[i] = __fadd_rn(h4 ? y8[i + 4] : y8[i],
                          __shfl_xor_sync(kFull, h4 ? y8[i] : y8[i + 4], 4));
#pragma unroll
    for (int i = 0; i < 2; ++i)
        y2[i] = __fadd_rn(h2 ? y4[i + 2] : y4[i],
                          __shfl_xor_sync(kFull, h2 ? y4[i] : y4[i + 2], 2));
    const float y1 = __fadd_rn(h1 ? y2[1] : y2[0], __shfl_xor_sync(kFull, h1 ? y2[0] : y2[1], 1));
    return __fadd_rn(y1, __shfl_xor_sync(kFull, y1, 16));
}

__device__ __forceinline__ void flag_error(int *err, int bits) {
    if (err != nullptr) atomicOr(err, bits);
}

// ------------------------------------------------------- token vectors --
//
// One buffer of per-token vectors (fp32): slots [0, p) are folded (recorded)
// tokens, [p, p + T) the new ones; q^ only for new tokens.  In the verify's
// window form (see window_outputs) a new token's kh and qh slots hold the
// decay-weighted G_t * k^_t and G_t * q^_t instead, and pa / pb the pair
// coefficients of the window (Q x Q each, row t, column s).
//
// Two layouts.  In the tail layout the vectors start at the buffer and the
// small arrays (beta, kq, pa, pb) follow them.  In the head layout (the
// window kernels of the tensor window form) the small arrays come first and
// the vectors start kTokHead bytes in, on a 1024-byte boundary, with at
// least kXBytes of them: a verify item in tensor window form
// (window_tc_prep) overwrites those bytes with its swizzled tensor-core
// operands.
constexpr int kTokHead = 1024;
constexpr int kXBytes = 2 * 16 * kD * 4;  // X_hi and X_lo: 16 vectors of 128 fp32 each
constexpr int kXBlock = 32 * 128;          // one 32-column block of the 32 operand rows

__host__ __device__ inline int tok_small_bytes(int slots, int Q) {
    return ((slots + 3) / 4) * 16 + ((Q + 3) / 4) * 16 + ((2 * Q * Q + 3) / 4) * 16;
}

struct TokView {
    float *kh, *e, *v, *qh, *beta, *kq, *pa, *pb;
    __device__ __forceinline__ TokView(unsigned char *base, int slots, int Q, bool head) {
        kh = reinterpret_cast<float *>(head ? base + kTokHead : base);
        e = kh + slots * kD;
        v = e + slots * kD;
        qh = v + slots * kD;
        beta = head ? reinterpret_cast<float *>(base) : qh + Q * kD;
        kq = beta + ((slots + 3) / 4) * 4;  // k^ . q^ of each new token
        pa = kq + ((Q + 3) / 4) * 4;
        pb = pa + Q * Q;
    }
};

__host__ __device__ inline int tok_buffer_bytes(int slots, int Q, bool head) {
    const int vec = (3 * slots + Q) * kD * 4;
    if (!head) return vec + tok_small_bytes(slots, Q);
    const int bytes = kTokHead + (vec > kXBytes ? vec : kXBytes);
    return (bytes + 1023) / 1024 * 1024;  // every buffer on a 1024-byte boundary
}

// ------------------------------------------------------------ state tile --

struct Lane {
    int w, g, j, lane;
    __device__ __forceinline__ int row(int i) const { return 32 * w + 8 * g + i; }
    __device__ __forceinline__ int col(int m) const { return 32 * m + 4 * j; }
};

using Tile = float4[8][4];

__device__ __forceinline__ void load_tile(Tile &h, const float *tile, const Lane &L) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m)
            h[i][m] = *reinterpret_cast<const float4 *>(tile + L.row(i) * kD + L.col(m));
}

__device__ __forceinline__ void store_tile(const Tile &h, float *tile, const Lane &L) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m)
            *reinterpret_cast<float4 *>(tile + L.row(i) * kD + L.col(m)) = h[i][m];
}

// The tile from / to a staging buffer in the tensor core's layout: four
// 32-column blocks of 128 rows, 128-byte swizzled (see kda_tc.cuh).
__device__ __forceinline__ void load_tile_sw(Tile &h, const unsigned char *staging, const Lane &L) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m)
            h[i][m] = *reinterpret_cast<const float4 *>(staging + m * 16384 +
                                                        sw128_offset(L.row(i), 4 * L.j));
}

__device__ __forceinline__ void store_tile_sw(const Tile &h, unsigned char *staging, const Lane &L) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m)
            *reinterpret_cast<float4 *>(staging + m * 16384 + sw128_offset(L.row(i), 4 * L.j)) =
                h[i][m];
}

__device__ __forceinline__ float4 ld_cols(const float *vec, const Lane &L, int m) {
    return *reinterpret_cast<const float4 *>(vec + L.col(m));
}

// Row dot products of the thread's 8 rows with a vector x (its 16 columns),
// in a fixed order: two interleaved partial sums per row (the even and the
// odd columns of each float4, one packed pair), then their sum.
__device__ __forceinline__ void row_partials(const Tile &h, const float *x, const Lane &L,
                                             float (&part)[8]) {
    float2 acc[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 xx = ld_cols(x, L, m);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (m == 0)
                acc[i] = mul2(h[i][0].x, h[i][0].y, xx.x, xx.y);
            else
                acc[i] = fma2(h[i][m].x, h[i][m].y, xx.x, xx.y, acc[i]);
            acc[i] = fma2(h[i][m].z, h[i][m].w, xx.z, xx.w, acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) part[i] = __fadd_rn(acc[i].x, acc[i].y);
}

// Row dot products with two vectors in one pass (each in the order of
// row_partials, so the first is bit-identical to row_partials(h, x)).
__device__ __forceinline__ void row_partials2(const Tile &h, const float *x, const float *y,
                                              const Lane &L, float (&px)[8], float (&py)[8]) {
    float2 ax[8], ay[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 xx = ld_cols(x, L, m);
        const float4 yy = ld_cols(y, L, m);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (m == 0) {
                ax[i] = mul2(h[i][0].x, h[i][0].y, xx.x, xx.y);
                ay[i] = mul2(h[i][0].x, h[i][0].y, yy.x, yy.y);
            } else {
                ax[i] = fma2(h[i][m].x, h[i][m].y, xx.x, xx.y, ax[i]);
                ay[i] = fma2(h[i][m].x, h[i][m].y, yy.x, yy.y, ay[i]);
            }
            ax[i] = fma2(h[i][m].z, h[i][m].w, xx.z, xx.w, ax[i]);
            ay[i] = fma2(h[i][m].z, h[i][m].w, yy.z, yy.w, ay[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        px[i] = __fadd_rn(ax[i].x, ax[i].y);
        py[i] = __fadd_rn(ay[i].x, ay[i].y);
    }
}

// Sum the 8 row partials over the 8 lanes of the row group (lane bits 0..2)
// by a transpose-reduce: after it, lane j holds the full sum of row j.
__device__ __forceinline__ float reduce_rows(const float (&part)[8], int j) {
    const bool hi = (j & 4) != 0;
    float t[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float send = hi ? part[q] : part[q + 4];
        const float keep = hi ? part[q + 4] : part[q];
        t[q] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 4));
    }
    const bool mid = (j & 2) != 0;
    float t2[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const float send = mid ? t[q] : t[q + 2];
        const float keep = mid ? t[q + 2] : t[q];
        t2[q] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 2));
    }
    const bool lo = (j & 1) != 0;
    const float send = lo ? t2[0] : t2[1];
    const float keep = lo ? t2[1] : t2[0];
    return __fadd_rn(keep, __shfl_xor_sync(kFull, send, 1));
}

// Pieces of one token of the recurrence on the thread's part of the tile:
//   S <- S diag(e);  u = S k^;  v' = beta (v - u);  S <- S + v' k^T;  o = S q^.

// Decay along K in place: S <- S diag(e).
__device__ __forceinline__ void decay(Tile &h, const float *e, const Lane &L) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 ee = ld_cols(e, L, m);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 lo = mul2(h[i][m].x, h[i][m].y, ee.x, ee.y);
            const float2 hi = mul2(h[i][m].z, h[i][m].w, ee.z, ee.w);
            h[i][m] = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
    }
}

// Rank-one update S <- S + v' k^T of the thread's 8 rows (vpi: their v').
__device__ __forceinline__ void rank_one(Tile &h, const float (&vpi)[8], const float *kh,
                                         const Lane &L) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 kk = ld_cols(kh, L, m);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 lo =
                fma2(vpi[i], vpi[i], kk.x, kk.y, make_float2(h[i][m].x, h[i][m].y));
            const float2 hi =
                fma2(vpi[i], vpi[i], kk.z, kk.w, make_float2(h[i][m].z, h[i][m].w));
            h[i][m] = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
    }
}

// Decay along K in place, then the partial sums of u = S k^ of the 8 rows.
__device__ __forceinline__ void decay_partials(Tile &h, const TokView &tv, int slot, const Lane &L,
                                               float (&part)[8]) {
    decay(h, tv.e + slot * kD, L);
    row_partials(h, tv.kh + slot * kD, L, part);
}

// v' = beta (v - u) for the lane's row, shared with the row group, then the
// rank-one update S <- S + v' k^T.  The lane's v' replaces its row's v in
// the token's v slot (no one reads that v again), and each thread reads its
// 8 rows' v' back as two float4: one store and two broadcast loads, where
// 8 shuffles measured 3 to 4% slower on the verify launches.
__device__ __forceinline__ void delta_update_vp(Tile &h, const TokView &tv, int slot, float vp,
                                                const Lane &L) {
    float *vs = tv.v + slot * kD;
    vs[L.row(L.j)] = vp;
    __syncwarp();
    const float4 d0 = *reinterpret_cast<const float4 *>(vs + L.row(0));
    const float4 d1 = *reinterpret_cast<const float4 *>(vs + L.row(0) + 4);
    const float vpi[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
    rank_one(h, vpi, tv.kh + slot * kD, L);
}

__device__ __forceinline__ void delta_update(Tile &h, const TokView &tv, int slot, float u,
                                             const Lane &L) {
    const float vr = tv.v[slot * kD + L.row(L.j)];
    delta_update_vp(h, tv, slot, __fmul_rn(tv.beta[slot], __fsub_rn(vr, u)), L);
}

// One token without output (commit replay, deferred fold, flush).
__device__ __forceinline__ void token_plain(Tile &h, const TokView &tv, int slot, const Lane &L) {
    float part[8];
    decay_partials(h, tv, slot, L, part);
    delta_update(h, tv, slot, reduce_rows(part, L.j), L);
}

// One token whose delta v' is known (a correction record, in the token
// vector's v slot): S <- S diag(e) + v' k^T with no prediction S k^.  These
// are the operations the verify made after it computed v', so the state has
// the bits of the verify's trajectory.  The thread reads its 8 rows' v'
// from shared memory (rows 32w + 8g .. +7, two aligned float4).
__device__ __forceinline__ void token_corr(Tile &h, const TokView &tv, int slot, const Lane &L) {
    decay(h, tv.e + slot * kD, L);
    const float4 *d = reinterpret_cast<const float4 *>(tv.v + slot * kD + L.row(0));
    const float4 d0 = d[0], d1 = d[1];
    const float vpi[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
    rank_one(h, vpi, tv.kh + slot * kD, L);
}

// One token with its output o = S' q^ (S' the state after the token) to
// out_row (bf16), from the decayed state D = S diag(e) in one pass:
// S' q^ = D q^ + v' (k^ . q^), so u = D k^ and D q^ share the pass and the
// reduction.  The state update is the one token_plain does (same bits);
// kUpdate false leaves it out (a verify's last new token, when no state
// after it is stored).  Returns the lane's v' (of row L.row(L.j)).
template <bool kUpdate>
__device__ __forceinline__ float token_out(Tile &h, const TokView &tv, int slot, int qslot,
                                           const Lane &L, __nv_bfloat16 *out_row) {
    decay(h, tv.e + slot * kD, L);
    float pu[8], po[8];
    row_partials2(h, tv.kh + slot * kD, tv.qh + qslot * kD, L, pu, po);
    const float u = reduce_rows(pu, L.j);
    const float dq = reduce_rows(po, L.j);
    const float vr = tv.v[slot * kD + L.row(L.j)];
    const float vp = __fmul_rn(tv.beta[slot], __fsub_rn(vr, u));
    out_row[L.row(L.j)] = __float2bfloat16_rn(__fmaf_rn(vp, tv.kq[qslot], dq));
    if constexpr (kUpdate) delta_update_vp(h, tv, slot, vp, L);
    return vp;
}

// ------------------------------------------------------------ window form --
//
// A verify never stores the state after its new tokens, so their outputs can
// be taken from the state S they start from (the checkpoint, or the state
// after the fold) without updating it.  With G_t = e_1 ... e_t and
// r_st = e_{s+1} ... e_t per channel (r_tt = 1), the recurrence unrolls to
//   S_t = S diag(G_t) + sum_{s<=t} v'_s (k^_s * r_st)^T,
// so token t's prediction is w_t + sum_{s<t} a_ts v'_s and its output
// o_t = y_t + sum_{s<=t} b_ts v'_s, where
//   w_t = S (G_t * k^_t),  y_t = S (G_t * q^_t),
//   a_ts = sum_c k^_s r_st k^_t,  b_ts = sum_c k^_s r_st q^_t.
// Each consumer prepares, for its own item and before its tile is loaded,
// G_t * k^_t and G_t * q^_t (into the kh and qh slots) and the pair
// coefficients (window_prep); it then takes the 2T row dot products with S,
// which do not depend on one another, and solves each row's deltas
// v'_t = beta_t (v_t - w_t - sum_{s<t} a_ts v'_s) in token order
// (window_outputs).  The outputs round differently from the token-by-token
// form; the states (the commit's, the fold's, the trajectory) are not
// computed this way.

// One row s of the pair coefficients, this lane's four channels: for
// t = s .. T-1, x = k^_s * r_st, b_ts = x . q^_t and (t > s) a_ts = x . k^_t,
// into val[] at slots 2d (b) and 2d - 1 (a) for d = t - s, or mirrored
// (15 - 2d and 16 - 2d) for a warp's second row.
template <bool kSecond>
__device__ __forceinline__ void pair_row(const TokView &tv, int p0, int T, int s, int lane,
                                         float (&val)[16]) {
    const float4 ks = ld4(tv.kh + (p0 + s) * kD + 4 * lane);
    float4 r = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
#pragma unroll
    for (int d = 0; d < kMaxQ; ++d) {
        if (s + d < T) {
            const int t = s + d;
            if (d > 0) r = mul4(r, ld4(tv.e + (p0 + t) * kD + 4 * lane));
            const float4 x = mul4(ks, r);
            val[kSecond ? 15 - 2 * d : 2 * d] = dot4(x, ld4(tv.qh + t * kD + 4 * lane));
            if (d > 0)
                val[kSecond ? 16 - 2 * d : 2 * d - 1] =
                    dot4(x, ld4(tv.kh + (p0 + t) * kD + 4 * lane));
        }
    }
}

// The window's coefficients of tokens p0 .. p0 + T - 1, by the 128 threads of
// a group (thread ct): warp wi the pair coefficients of rows s = wi and
// s = T - 1 - wi (2T values, so the warps are balanced), and each thread the
// decay-weighted G_t * k^_t and G_t * q^_t of channel ct, which replace k^_t
// and q^_t once every warp has read them.  group_sync() is the group's
// barrier; false means it gave up (the caller leaves), and so does this.
template <class GroupSync>
__device__ __forceinline__ bool window_prep(const TokView &tv, int p0, int T, int Q, int ct,
                                            GroupSync &&group_sync) {
    const int lane = ct & 31, warp = ct >> 5;
    if (warp < (T + 1) / 2) {
        float val[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) val[i] = 0.0f;
        const int s0 = warp, s1 = T - 1 - warp;
        pair_row<false>(tv, p0, T, s0, lane, val);
        if (s1 != s0) pair_row<true>(tv, p0, T, s1, lane, val);
        const float sum = reduce16(val, lane);
        if (lane < 16) {
            int s = -1, slot = lane;
            if (slot <= 2 * (T - 1 - s0)) {
                s = s0;
            } else if (s1 != s0 && slot >= 15 - 2 * (T - 1 - s1)) {
                s = s1;
                slot = 15 - slot;
            }
            if (s >= 0) {
                const int d = (slot + 1) >> 1;
                float *dst = (slot & 1) ? tv.pa : tv.pb;
                dst[(s + d) * Q + s] = sum;
            }
        }
    }
    float gk[kMaxQ], gq[kMaxQ];
    float G = 1.0f;
#pragma unroll
    for (int t = 0; t < kMaxQ; ++t) {
        if (t < T) {
            G = __fmul_rn(G, tv.e[(p0 + t) * kD + ct]);
            gk[t] = __fmul_rn(G, tv.kh[(p0 + t) * kD + ct]);
            gq[t] = __fmul_rn(G, tv.qh[t * kD + ct]);
        }
    }
    if (!group_sync()) return false;  // every read of k^ and q^ done
#pragma unroll
    for (int t = 0; t < kMaxQ; ++t) {
        if (t < T) {
            tv.kh[(p0 + t) * kD + ct] = gk[t];
            tv.qh[t * kD + ct] = gq[t];
        }
    }
    return group_sync();  // the coefficients and vectors are in place
}

// The T new tokens' outputs (row L.row(L.j) per thread) to
// out0 + t * out_stride.  The new tokens' e and v slots serve as per-row
// scratch (v - w and y): only this thread reads its row there.
__device__ __forceinline__ void window_outputs(const Tile &h, const TokView &tv, int p, int T,
                                               int Q, const Lane &L, __nv_bfloat16 *out0,
                                               size_t out_stride) {
    const int row = L.row(L.j);
    for (int t = 0; t < T; ++t) {
        float pw[8], py[8];
        row_partials2(h, tv.kh + (p + t) * kD, tv.qh + t * kD, L, pw, py);
        const float w = reduce_rows(pw, L.j);
        const float y = reduce_rows(py, L.j);
        const int ix = (p + t) * kD + row;
        tv.e[ix] = __fsub_rn(tv.v[ix], w);
        tv.v[ix] = y;
    }
    float vp[kMaxQ];
#pragma unroll
    for (int t = 0; t < kMaxQ; ++t) {
        if (t < T) {
            const int ix = (p + t) * kD + row;
            float acc = tv.e[ix];
#pragma unroll
            for (int s = 0; s < t; ++s) acc = __fmaf_rn(-tv.pa[t * Q + s], vp[s], acc);
            vp[t] = __fmul_rn(tv.beta[p + t], acc);
            float o = tv.v[ix];
#pragma unroll
            for (int s = 0; s <= t; ++s) o = __fmaf_rn(tv.pb[t * Q + s], vp[s], o);
            out0[(size_t)t * out_stride + row] = __float2bfloat16_rn(o);
        }
    }
}

// ----------------------------------------------------- tensor window form --
//
// The same window form with its 2T row dot products on the tensor core:
// D = S X^T, S the state the new tokens start from (128 x 128) and X
// the 16 operand vectors X_t = G_t * k^_t and X_{8+t} = G_t * q^_t (t < T;
// the rows of the other vectors are never read back), so that D[v][t] = w_t
// and D[v][8+t] = y_t of row v.  The products are tcgen05.mma of kind::tf32
// with fp32 accuracy: with S = S_hi + S_lo and X = X_hi + X_lo split at the
// TF32 precision the tensor core reads, the operand B holds X_hi in rows
// 0..15 and X_lo in rows 16..31 (N = 32), and
//   D_hi = S_hi [X_hi; X_lo]^T,   D_lo = S_lo [X_hi; X_lo]^T
// are accumulated apart (every product of the four parts, 16 K steps each)
// and added in fp32, the small terms first.  Operand A comes from TMEM: each
// thread copies its row of S there from the swizzled staging buffer (the
// staged checkpoint, or, after folded tokens, the folded state written back
// there), which frees the staging buffer at once; the tensor core reads the
// fp32 columns as TF32, that is S_hi.  Once D_hi is complete each thread
// replaces its row by S_lo in the same columns for D_lo.  X_hi and X_lo go
// to shared memory.  Thread ct of the consumer group owns channel ct of the
// vectors and row ct of S, D and the outputs.  New token t sits in slot
// p0 + t (p0 folded tokens first).

// Pair coefficients, then the operand vectors of the channel into shared
// memory (swizzled, K-major).  The thread keeps its row's v_t in vrow: the
// vectors' bytes are overwritten.  group_sync() as in window_prep.
template <class GroupSync>
__device__ __forceinline__ bool window_tc_prep(const TokView &tv, int p0, int T, int Q, int ct,
                                               float (&vrow)[kMaxQ], GroupSync &&group_sync) {
    const int lane = ct & 31, warp = ct >> 5;
    if (warp < (T + 1) / 2) {
        float val[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) val[i] = 0.0f;
        const int s0 = warp, s1 = T - 1 - warp;
        pair_row<false>(tv, p0, T, s0, lane, val);
        if (s1 != s0) pair_row<true>(tv, p0, T, s1, lane, val);
        const float sum = reduce16(val, lane);
        if (lane < 16) {
            int s = -1, slot = lane;
            if (slot <= 2 * (T - 1 - s0)) {
                s = s0;
            } else if (s1 != s0 && slot >= 15 - 2 * (T - 1 - s1)) {
                s = s1;
                slot = 15 - slot;
            }
            if (s >= 0) {
                const int d = (slot + 1) >> 1;
                float *dst = (slot & 1) ? tv.pa : tv.pb;
                dst[(s + d) * Q + s] = sum;
            }
        }
    }
    float gk[kMaxQ], gq[kMaxQ];
    float G = 1.0f;
#pragma unroll
    for (int t = 0; t < kMaxQ; ++t) {
        if (t < T) {
            G = __fmul_rn(G, tv.e[(p0 + t) * kD + ct]);
            gk[t] = __fmul_rn(G, tv.kh[(p0 + t) * kD + ct]);
            gq[t] = __fmul_rn(G, tv.qh[t * kD + ct]);
            vrow[t] = tv.v[(p0 + t) * kD + ct];
        }
    }
    if (!group_sync()) return false;  // every read of the vectors done
    // head layout: the operands take the vectors' bytes, from kh on; X_hi of
    // vector n in operand row n, X_lo in row 16 + n, the 32-column block of
    // channel ct
    unsigned char *xb = reinterpret_cast<unsigned char *>(tv.kh) + (ct >> 5) * kXBlock;
    const int col = ct & 31;
#pragma unroll
    for (int t = 0; t < kMaxQ; ++t) {
        if (t < T) {
            const float hk = tf32_hi(gk[t]), hq = tf32_hi(gq[t]);
            *reinterpret_cast<float *>(xb + sw128_offset(t, col)) = hk;
            *reinterpret_cast<float *>(xb + sw128_offset(16 + t, col)) = __fsub_rn(gk[t], hk);
            *reinterpret_cast<float *>(xb + sw128_offset(8 + t, col)) = hq;
            *reinterpret_cast<float *>(xb + sw128_offset(24 + t, col)) = __fsub_rn(gq[t], hq);
        }
    }
    fence_proxy_async_smem();  // the tensor core reads X through the async proxy
    return true;
}

// Row ct of S (the staging buffer, four swizzled 32-column blocks) into
// TMEM columns a .. a + 127 of the thread's lane, 16 at a time.  The tensor
// core reads these fp32 columns as TF32, that is S_hi.
__device__ __forceinline__ void s_row_to_tmem(const unsigned char *staging, int ct, uint32_t a) {
#pragma unroll
    for (int half = 0; half < 8; ++half) {
        uint32_t u[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float4 q = *reinterpret_cast<const float4 *>(
                staging + (half >> 1) * 16384 + sw128_offset(ct, 16 * (half & 1) + 4 * c));
            u[4 * c + 0] = __float_as_uint(q.x);
            u[4 * c + 1] = __float_as_uint(q.y);
            u[4 * c + 2] = __float_as_uint(q.z);
            u[4 * c + 3] = __float_as_uint(q.w);
        }
        tmem_st16(a + 16 * half, u);
    }
}

// S in TMEM columns a .. a + 127 of the thread's lane replaced by
// S_lo = S - tf32(S), in two halves of 64 columns (once the product that
// reads S from them has completed).
__device__ __forceinline__ void s_lo_in_tmem(uint32_t a) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t u[4][16];
#pragma unroll
        for (int i = 0; i < 4; ++i) tmem_ld16(a + 64u * h + 16u * i, u[i]);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float x = __uint_as_float(u[i][j]);
                u[i][j] = __float_as_uint(__fsub_rn(x, tf32_hi(x)));
            }
            tmem_st16(a + 64u * h + 16u * i, u[i]);
        }
    }
}

// D = A [X_hi; X_lo]^T over K = 128 (16 steps of 8), A from TMEM (one fp32
// per column: S, read as S_hi, or S_lo); by one thread.  A step's B
// descriptor is the first one plus its byte offset / 16 (the start address
// field does not overflow).
__device__ __forceinline__ void window_tc_mma(uint32_t a, uint32_t xbase, uint32_t d) {
    constexpr uint32_t idesc = tf32_idesc(128, 32);
    const uint64_t b0 = sw128_desc(xbase);
#pragma unroll
    for (int k = 0; k < 16; ++k)
        umma_tf32_ts(d, a + 8u * (uint32_t)k,
                     b0 + (((uint32_t)(k >> 2) * (uint32_t)kXBlock + (uint32_t)(k & 3) * 32u) >> 4),
                     idesc, k > 0);
}

// The solve of row ct from D_hi (32 columns at TMEM address d of the
// thread's lane) and D_lo (the 32 after them), as in window_outputs:
// v'_t = beta_t (v_t - w_t - sum_{s<t} a_ts v'_s), o_t = y_t + sum_{s<=t} b_ts v'_s.
__device__ __forceinline__ void window_tc_solve(const TokView &tv, int p0, int T, int Q, int ct,
                                                const float (&vrow)[kMaxQ], uint32_t d,
                                                __nv_bfloat16 *out0, size_t out_stride) {
    uint32_t h0[16], h1[16], l0[16], l1[16];  // D_hi: X_hi, X_lo columns; D_lo: the same
    tmem_ld16(d, h0);
    tmem_ld16(d + 16u, h1);
    tmem_ld16(d + 32u, l0);
    tmem_ld16(d + 48u, l1);
    tmem_wait_ld();
    auto dot = [&](int n) {  // the small terms first
        const float lo = __fadd_rn(__uint_as_float(l0[n]), __uint_as_float(l1[n]));
        return __fadd_rn(__uint_as_float(h0[n]), __fadd_rn(__uint_as_float(h1[n]), lo));
    };
    float vp[kMaxQ];
#pragma unroll
    for (int t = 0; t < kMaxQ; ++t) {
        if (t < T) {
            const float w = dot(t);
            const float y = dot(8 + t);
            float acc = __fsub_rn(vrow[t], w);
#pragma unroll
            for (int s = 0; s < t; ++s) acc = __fmaf_rn(-tv.pa[t * Q + s], vp[s], acc);
            vp[t] = __fmul_rn(tv.beta[p0 + t], acc);
            float o = y;
#pragma unroll
            for (int s = 0; s <= t; ++s) o = __fmaf_rn(tv.pb[t * Q + s], vp[s], o);
            out0[(size_t)t * out_stride + ct] = __float2bfloat16_rn(o);
        }
    }
}

}  // namespace kda
