// Conv-state compaction of a commit, as a plain copy kernel (sm_103a).
//
// recoverssm.py, `_compact_conv_state_kernel` (non-align form): after n
// accepted tokens the window of each channel that starts at column n - 1
// moves to column 0.  Every element a thread writes it has read itself (or,
// in the staged form, the CTA has read it into shared memory) before any
// write, so a window that overlaps its destination is moved correctly.
// Three forms, chosen on the host from the strides:
//  - channel-major and dense (column stride 1, channel stride = width): a
//    CTA stages a 16-byte-aligned run of whole channels in shared memory with
//    16-byte loads, moves each channel's window there and writes the run back
//    with 16-byte stores (the bytes of a channel are not 16-byte aligned on
//    their own, e.g. 6 bf16 columns);
//  - column-major (channel stride 1) with 16-byte rows: a thread moves 16
//    bytes of channels through the window's columns;
//  - anything else: a thread moves one channel, element by element.
// Align mode (paged blocks) copies from the source slot into the final and
// boundary blocks with the element-wise form.
// The public contract is in include/kda.h (kda_conv_compact).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_align.cuh"

namespace kda_conv {

constexpr int kThreads = 256;
constexpr int kMaxRowsPerGrid = 65535;

struct Params {
    unsigned char *conv;
    long long stride_slot, stride_dim, stride_col;
    int S, C, Q, hist, B, elem_bytes;
    const int32_t *cu, *slots, *acc;
    int *err;
};

// Row checks shared by the three forms: the commit count n, or 0 to skip.
__device__ __forceinline__ int row_count(const Params &p, int b) {
    const int len = p.cu[b + 1] - p.cu[b];
    const int slot = p.slots[b];
    const bool first = blockIdx.x == 0 && threadIdx.x == 0;
    if (len < 0 || len > p.Q) {
        if (first && p.err != nullptr) atomicOr(p.err, KDA_ROW_BAD_LENGTH);
        return 0;
    }
    if (slot >= p.S) {
        if (first && p.err != nullptr) atomicOr(p.err, KDA_ROW_BAD_SLOT);
        return 0;
    }
    const int n = min(max(p.acc[b], 0), min(len, p.Q));
    return slot > 0 ? n : 0;
}

// Any strides: one thread per channel, element by element.
template <typename T>
__global__ void __launch_bounds__(kThreads) compact_kernel(const Params p) {
    for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
        const int n = row_count(p, b);
        if (n <= 0) continue;
        T *base = reinterpret_cast<T *>(p.conv) + (long long)p.slots[b] * p.stride_slot;
        for (int d = blockIdx.x * kThreads + threadIdx.x; d < p.C; d += gridDim.x * kThreads) {
            T *ch = base + (long long)d * p.stride_dim;
            T w[KDA_MAX_CONV_HISTORY];
#pragma unroll
            for (int h = 0; h < KDA_MAX_CONV_HISTORY; ++h)
                if (h < p.hist) w[h] = ch[(long long)(n - 1 + h) * p.stride_col];
#pragma unroll
            for (int h = 0; h < KDA_MAX_CONV_HISTORY; ++h)
                if (h < p.hist) ch[(long long)h * p.stride_col] = w[h];
        }
    }
}

constexpr int kStageBytes = 16384;                  // shared-memory run of the staged form
constexpr int kStageVecs = kStageBytes / 16 / kThreads;  // 16-byte loads per thread

// Channel-major, dense: run r of a slot covers channels [r*run, (r+1)*run),
// `run` a multiple of the channels whose bytes make 16-byte units.
template <typename T>
__global__ void __launch_bounds__(kThreads) staged_kernel(const Params p, int run) {
    __shared__ __align__(16) unsigned char stage[kStageBytes];
    const int W = (int)p.stride_dim;  // = width
    for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
        const int n = row_count(p, b);
        if (n <= 0) continue;  // uniform over the CTA
        unsigned char *slot_base =
            p.conv + (long long)p.slots[b] * p.stride_slot * (long long)sizeof(T);
        for (int c0 = blockIdx.x * run; c0 < p.C; c0 += gridDim.x * run) {
            const int chans = min(run, p.C - c0);
            const int vecs = chans * W * (int)sizeof(T) / 16;
            const uint4 *src = reinterpret_cast<const uint4 *>(
                slot_base + (long long)c0 * W * (long long)sizeof(T));
            uint4 *sv = reinterpret_cast<uint4 *>(stage);
            uint4 r[kStageVecs];  // all loads in flight before the first store
#pragma unroll
            for (int j = 0; j < kStageVecs; ++j) {
                const int i = threadIdx.x + j * kThreads;
                if (i < vecs) r[j] = src[i];
            }
#pragma unroll
            for (int j = 0; j < kStageVecs; ++j) {
                const int i = threadIdx.x + j * kThreads;
                if (i < vecs) sv[i] = r[j];
            }
            __syncthreads();
            T *se = reinterpret_cast<T *>(stage);
            for (int d = threadIdx.x; d < chans; d += kThreads) {
                T w[KDA_MAX_CONV_HISTORY];
#pragma unroll
                for (int h = 0; h < KDA_MAX_CONV_HISTORY; ++h)
                    if (h < p.hist) w[h] = se[d * W + n - 1 + h];
#pragma unroll
                for (int h = 0; h < KDA_MAX_CONV_HISTORY; ++h)
                    if (h < p.hist) se[d * W + h] = w[h];
            }
            __syncthreads();
            uint4 *dst = reinterpret_cast<uint4 *>(
                slot_base + (long long)c0 * W * (long long)sizeof(T));
#pragma unroll
            for (int j = 0; j < kStageVecs; ++j) {
                const int i = threadIdx.x + j * kThreads;
                if (i < vecs) r[j] = sv[i];
            }
#pragma unroll
            for (int j = 0; j < kStageVecs; ++j) {
                const int i = threadIdx.x + j * kThreads;
                if (i < vecs) dst[i] = r[j];
            }
            __syncthreads();  // the stage is reused by the next run
        }
    }
}

// Channel-major, dense, small units: a unit is the fewest whole channels
// whose bytes make 16-byte pieces (at most 4 channels, 64 bytes).  A thread
// loads kUnits units with 16-byte loads into its own slice of shared memory,
// moves each channel's window there, and stores the units back: no barrier,
// and every load is in flight before the first store.  Piece v of unit k of
// thread t sits at 16 * ((4k + v) * kThreads + t), so a warp's 16-byte
// accesses fall on distinct banks.
constexpr int kUnitMaxBytes = 64;

template <typename T, int kUnits>
__global__ void __launch_bounds__(kThreads) unit_kernel(const Params p, int unit_chans) {
    __shared__ __align__(16) unsigned char stage[kThreads * kUnits * kUnitMaxBytes];
    const int W = (int)p.stride_dim;  // = width
    const int unit_bytes = unit_chans * W * (int)sizeof(T);
    const int uv = unit_bytes / 16;    // 16-byte pieces per unit, <= 4
    const int units = p.C / unit_chans;
    constexpr int kPieces = kUnitMaxBytes / 16;
    for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
        const int n = row_count(p, b);
        if (n <= 0) continue;
        unsigned char *slot_base =
            p.conv + (long long)p.slots[b] * p.stride_slot * (long long)sizeof(T);
        for (int u0 = blockIdx.x * kThreads * kUnits + threadIdx.x; u0 < units;
             u0 += gridDim.x * kThreads * kUnits) {
            uint4 r[kUnits][kUnitMaxBytes / 16];
#pragma unroll
            for (int k = 0; k < kUnits; ++k) {
                const int u = u0 + k * kThreads;
                const uint4 *src = reinterpret_cast<const uint4 *>(slot_base + (long long)u * unit_bytes);
#pragma unroll
                for (int v = 0; v < kUnitMaxBytes / 16; ++v)
                    if (u < units && v < uv) r[k][v] = src[v];
            }
            constexpr int kPer = 16 / (int)sizeof(T);  // elements per piece
#pragma unroll
            for (int k = 0; k < kUnits; ++k) {
                uint4 *sv = reinterpret_cast<uint4 *>(stage) + (k * kPieces) * kThreads + threadIdx.x;
#pragma unroll
                for (int v = 0; v < kPieces; ++v)
                    if (v < uv) sv[v * kThreads] = r[k][v];
                // element e of the unit: piece e / kPer, slot e % kPer
                T *se = reinterpret_cast<T *>(sv);
                for (int c = 0; c < unit_chans; ++c) {
                    T w[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int e = c * W + n - 1 + h;
                        if (h < p.hist) w[h] = se[(e / kPer) * kThreads * kPer + e % kPer];
                    }
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int e = c * W + h;
                        if (h < p.hist) se[(e / kPer) * kThreads * kPer + e % kPer] = w[h];
                    }
                }
#pragma unroll
                for (int v = 0; v < kPieces; ++v)
                    if (v < uv) r[k][v] = sv[v * kThreads];
            }
#pragma unroll
            for (int k = 0; k < kUnits; ++k) {
                const int u = u0 + k * kThreads;
                uint4 *dst = reinterpret_cast<uint4 *>(slot_base + (long long)u * unit_bytes);
#pragma unroll
                for (int v = 0; v < kUnitMaxBytes / 16; ++v)
                    if (u < units && v < uv) dst[v] = r[k][v];
            }
        }
    }
}

// Column-major with 16-byte rows: a thread moves kVec 16-byte pieces of
// channels (kVec * kThreads apart) through the window's columns, all loads
// before any store; kHist bounds the history.
template <int kHist, int kVec>
__global__ void __launch_bounds__(kThreads) column_kernel(const Params p) {
    const long long col_bytes = p.stride_col * p.elem_bytes;
    const int vecs = p.C * p.elem_bytes / 16;
    for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
        const int n = row_count(p, b);
        if (n <= 0) continue;
        unsigned char *slot_base = p.conv + (long long)p.slots[b] * p.stride_slot * p.elem_bytes;
        const uint4 *src = reinterpret_cast<const uint4 *>(slot_base + (n - 1) * col_bytes);
        uint4 *dst = reinterpret_cast<uint4 *>(slot_base);
        const long long col_vecs = col_bytes / 16;
        for (int i0 = blockIdx.x * kThreads * kVec + threadIdx.x; i0 < vecs;
             i0 += gridDim.x * kThreads * kVec) {
            uint4 w[kVec][kHist];
#pragma unroll
            for (int v = 0; v < kVec; ++v)
#pragma unroll
                for (int h = 0; h < kHist; ++h)
                    if (h < p.hist && i0 + v * kThreads < vecs)
                        w[v][h] = src[h * col_vecs + i0 + v * kThreads];
#pragma unroll
            for (int v = 0; v < kVec; ++v)
#pragma unroll
                for (int h = 0; h < kHist; ++h)
                    if (h < p.hist && i0 + v * kThreads < vecs)
                        dst[h * col_vecs + i0 + v * kThreads] = w[v][h];
        }
    }
}

// Align mode: per row, the window at column n - 1 of the source slot goes to
// the final block and the window at column boundary_len - 1 to the boundary
// block (when the step reaches one), both read before either is written.
struct AlignArgs {
    const int32_t *block_table, *num_computed, *request_indices;
    long long bt_stride;
    int bt_width, block_size, num_requests;
};

__device__ __forceinline__ void flag(const Params &p, int bits) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.err != nullptr) atomicOr(p.err, bits);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) align_kernel(const Params p, const AlignArgs a) {
    for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
        const int len = p.cu[b + 1] - p.cu[b];
        const int slot = p.slots[b];
        if (len < 0 || len > p.Q) {
            flag(p, KDA_ROW_BAD_LENGTH);
            continue;
        }
        if (slot >= p.S) {
            flag(p, KDA_ROW_BAD_SLOT);
            continue;
        }
        const int req = a.request_indices != nullptr ? a.request_indices[b] : b;
        if (req < 0 || req >= a.num_requests) {
            flag(p, KDA_ROW_BAD_BLOCK);
            continue;
        }
        const int n = min(max(p.acc[req], 0), min(len, p.Q));
        if (slot <= 0 || n <= 0) continue;
        const kda_blocks::Blocks bl =
            kda_blocks::plan(a.block_table + (long long)req * a.bt_stride, a.bt_width,
                             a.block_size, a.num_computed[req], n);
        if (bl.bad) {
            flag(p, KDA_ROW_BAD_BLOCK);
            continue;
        }
        if (bl.final_block >= p.S || bl.boundary >= p.S) {
            flag(p, KDA_ROW_BAD_SLOT);
            continue;
        }
        if (bl.final_block <= 0) continue;
        T *base = reinterpret_cast<T *>(p.conv);
        const long long src = (long long)slot * p.stride_slot;
        const long long fin = (long long)bl.final_block * p.stride_slot;
        const long long bnd = (long long)bl.boundary * p.stride_slot;
        for (int d = blockIdx.x * kThreads + threadIdx.x; d < p.C; d += gridDim.x * kThreads) {
            const long long ch = (long long)d * p.stride_dim;
            T wf[KDA_MAX_CONV_HISTORY], wb[KDA_MAX_CONV_HISTORY];
#pragma unroll
            for (int h = 0; h < KDA_MAX_CONV_HISTORY; ++h) {
                if (h < p.hist) {
                    wf[h] = base[src + ch + (long long)(n - 1 + h) * p.stride_col];
                    if (bl.boundary > 0)
                        wb[h] = base[src + ch + (long long)(bl.boundary_len - 1 + h) * p.stride_col];
                }
            }
            if (bl.boundary > 0) {
#pragma unroll
                for (int h = 0; h < KDA_MAX_CONV_HISTORY; ++h)
                    if (h < p.hist) base[bnd + ch + (long long)h * p.stride_col] = wb[h];
            }
#pragma unroll
            for (int h = 0; h < KDA_MAX_CONV_HISTORY; ++h)
                if (h < p.hist) base[fin + ch + (long long)h * p.stride_col] = wf[h];
        }
    }
}

bool aligned(const void *ptr, uintptr_t bytes) {
    return (reinterpret_cast<uintptr_t>(ptr) & (bytes - 1)) == 0;
}

// Checks shared by both entry points; fills p.  KDA_OK with p.B == 0 means
// there is nothing to launch.
kda_status conv_params(const kda_conv_config *cc, void *conv_state, const int32_t *cu_seqlens,
                       const int32_t *state_indices, int32_t B, const int32_t *num_accepted,
                       int32_t *error_word, Params &p) {
    p.B = 0;
    if (cc == nullptr) return KDA_ERR_INVALID_ARG;
    if (cc->num_slots < 1 || cc->conv_dim < 1 || cc->window < 1 || cc->reserved != 0)
        return KDA_ERR_INVALID_ARG;
    if (cc->window > KDA_MAX_WINDOW) return KDA_ERR_UNSUPPORTED;
    if (cc->elem_bytes != 2 && cc->elem_bytes != 4) return KDA_ERR_INVALID_ARG;
    if (cc->width < cc->window) return KDA_ERR_INVALID_ARG;
    const int hist = cc->width - cc->window + 1;
    if (hist > KDA_MAX_CONV_HISTORY) return KDA_ERR_UNSUPPORTED;
    if (cc->stride_slot < 1 || cc->stride_dim < 1 || cc->stride_col < 1)
        return KDA_ERR_INVALID_ARG;
    if (B < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;  // nothing to do; no pointer is inspected
    if (!conv_state || !cu_seqlens || !state_indices || !num_accepted)
        return KDA_ERR_INVALID_ARG;
    if (!aligned(conv_state, (uintptr_t)cc->elem_bytes) || !aligned(cu_seqlens, 4) ||
        !aligned(state_indices, 4) || !aligned(num_accepted, 4) ||
        (error_word != nullptr && !aligned(error_word, 4)))
        return KDA_ERR_INVALID_ARG;

    p.conv = static_cast<unsigned char *>(conv_state);
    p.stride_slot = cc->stride_slot;
    p.stride_dim = cc->stride_dim;
    p.stride_col = cc->stride_col;
    p.S = cc->num_slots;
    p.C = cc->conv_dim;
    p.Q = cc->window;
    p.hist = hist;
    p.B = B;
    p.cu = cu_seqlens;
    p.slots = state_indices;
    p.acc = num_accepted;
    p.err = error_word;
    p.elem_bytes = cc->elem_bytes;
    return KDA_OK;
}

}  // namespace kda_conv

extern "C" {

kda_status kda_conv_compact(const kda_conv_config *cc, void *conv_state,
                            const int32_t *cu_seqlens, const int32_t *state_indices,
                            int32_t B, const int32_t *num_accepted,
                            int32_t *error_word, void *stream) {
    using namespace kda_conv;
    Params p;
    const kda_status status = conv_params(cc, conv_state, cu_seqlens, state_indices, B,
                                          num_accepted, error_word, p);
    if (status != KDA_OK || p.B == 0) return status;
    const int rows = B < kMaxRowsPerGrid ? B : kMaxRowsPerGrid;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long eb = cc->elem_bytes;
    const bool slots16 = aligned(conv_state, 16) && (cc->stride_slot * eb) % 16 == 0;
    // channels per 16-byte unit of a dense channel-major slot
    const long long chan_bytes = (long long)cc->width * eb;
    long long unit = 1;
    while ((unit * chan_bytes) % 16 != 0) ++unit;
    if (slots16 && cc->stride_col == 1 && cc->stride_dim == cc->width &&
        cc->conv_dim % unit == 0 && unit <= 4 && unit * chan_bytes <= kUnitMaxBytes &&
        p.hist <= 4) {
        constexpr int kUnits = 2;
        const int units = (int)(cc->conv_dim / unit);
        const dim3 grid((units + kThreads * kUnits - 1) / (kThreads * kUnits), rows);
        if (cc->elem_bytes == 2)
            unit_kernel<uint16_t, kUnits><<<grid, kThreads, 0, st>>>(p, (int)unit);
        else
            unit_kernel<uint32_t, kUnits><<<grid, kThreads, 0, st>>>(p, (int)unit);
    } else if (slots16 && cc->stride_col == 1 && cc->stride_dim == cc->width &&
               cc->conv_dim % unit == 0 && unit * chan_bytes <= kStageBytes) {
        const int run = (int)(unit * (kStageBytes / (unit * chan_bytes)));
        const dim3 grid((cc->conv_dim + run - 1) / run, rows);
        if (cc->elem_bytes == 2)
            staged_kernel<uint16_t><<<grid, kThreads, 0, st>>>(p, run);
        else
            staged_kernel<uint32_t><<<grid, kThreads, 0, st>>>(p, run);
    } else if (slots16 && cc->stride_dim == 1 && ((long long)cc->conv_dim * eb) % 16 == 0 &&
               (cc->stride_col * eb) % 16 == 0) {
        const int vecs = (int)((long long)cc->conv_dim * eb / 16);
        if (p.hist <= 4) {
            constexpr int kVec = 4;
            const dim3 grid((vecs + kThreads * kVec - 1) / (kThreads * kVec), rows);
            column_kernel<4, kVec><<<grid, kThreads, 0, st>>>(p);
        } else {
            const dim3 grid((vecs + kThreads - 1) / kThreads, rows);
            column_kernel<KDA_MAX_CONV_HISTORY, 1><<<grid, kThreads, 0, st>>>(p);
        }
    } else {
        const dim3 grid((cc->conv_dim + kThreads - 1) / kThreads, rows);
        if (cc->elem_bytes == 2)
            compact_kernel<uint16_t><<<grid, kThreads, 0, st>>>(p);
        else
            compact_kernel<uint32_t><<<grid, kThreads, 0, st>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_conv_compact_align(const kda_conv_config *cc, void *conv_state,
                                  const int32_t *cu_seqlens, const int32_t *state_indices,
                                  int32_t B, const int32_t *num_accepted, const kda_align *align,
                                  int32_t *error_word, void *stream) {
    using namespace kda_conv;
    Params p;
    const kda_status st = conv_params(cc, conv_state, cu_seqlens, state_indices, B,
                                      num_accepted, error_word, p);
    if (st != KDA_OK || p.B == 0) return st;
    if (align == nullptr || align->reserved != 0 || !align->block_table || !align->num_computed)
        return KDA_ERR_INVALID_ARG;
    if (align->block_table_width < 1 || align->block_table_stride < align->block_table_width ||
        align->num_requests < 1 || align->block_size < cc->window)
        return KDA_ERR_INVALID_ARG;
    if (!aligned(align->block_table, 4) || !aligned(align->num_computed, 4) ||
        (align->request_indices != nullptr && !aligned(align->request_indices, 4)))
        return KDA_ERR_INVALID_ARG;
    AlignArgs a;
    a.block_table = align->block_table;
    a.num_computed = align->num_computed;
    a.request_indices = align->request_indices;
    a.bt_stride = align->block_table_stride;
    a.bt_width = align->block_table_width;
    a.block_size = align->block_size;
    a.num_requests = align->num_requests;
    const int rows = B < kMaxRowsPerGrid ? B : kMaxRowsPerGrid;
    const dim3 grid((cc->conv_dim + kThreads - 1) / kThreads, rows);
    cudaStream_t stv = static_cast<cudaStream_t>(stream);
    if (cc->elem_bytes == 2)
        align_kernel<uint16_t><<<grid, kThreads, 0, stv>>>(p, a);
    else
        align_kernel<uint32_t><<<grid, kThreads, 0, stv>>>(p, a);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
