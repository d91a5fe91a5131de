// Conv-state compaction of a commit, as a plain copy kernel (sm_103a).
//
// recoverssm.py, `_compact_conv_state_kernel` (non-align form): after n
// accepted tokens the window of each channel that starts at column n - 1
// moves to column 0.  Every element a thread writes it has read itself (or,
// in the bulk form, the CTA has loaded it into shared memory) before any
// write, so a window that overlaps its destination is moved correctly.
// A row with n = 1 keeps every window where it is and is skipped.  Three
// forms, chosen on the host from the strides:
//  - channel-major and dense (column stride 1, channel stride = width): a
//    CTA loads a 16-byte-aligned run of whole channels (up to 24 KiB) into
//    shared memory with one TMA bulk copy, moves each channel's window there
//    and writes the run back with one bulk copy (the bytes of a channel are
//    not 16-byte aligned on their own, e.g. 6 bf16 columns);
//  - column-major (channel stride 1) with 16-byte rows: a thread moves 16
//    bytes of channels through the window's columns;
//  - anything else: a thread moves one channel, element by element.
// Align mode (paged blocks) copies from the source slot into the final and
// boundary blocks: for channel-major dense pools a thread moves 16-byte
// units of channels through shared memory, otherwise element by element.
// The public contract is in include/kda.h (kda_conv_compact).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_align.cuh"
#include "kda_async.cuh"

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

// Row checks shared by the three forms: the commit count n, or 0 to skip
// (n = 1 moves the window at column 0 onto itself).
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
    return slot > 0 && n > 1 ? n : 0;
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

// Channel-major, dense, in bulk: CTA (x, row) moves run x of the row's slot,
// `run` whole channels (a multiple of the channels whose bytes make 16-byte
// units, at most kBulkBytes), with one bulk copy each way: thread 0 loads
// the run into shared memory on an mbarrier, every thread moves its
// channels' windows there, and thread 0 stores the run back and waits until
// the store has read shared memory before the stage is reused.
constexpr int kBulkBytes = 24576;
constexpr long long kBulkWaitBudget = 4000000000LL;  // clock cycles (about 2 s)

// One bulk copy shared -> global (a multiple of 16 bytes, both addresses
// 16-byte aligned) in this thread's bulk group; bulk_commit closes the
// group and bulk_wait_read waits until every committed bulk store of the
// thread has finished reading shared memory.
__device__ __forceinline__ void bulk_store(void *dst_gmem, const void *src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
                 "r"(kda::smem_u32(src_smem)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

template <typename T>
__global__ void __launch_bounds__(kThreads) bulk_kernel(const Params p, int run) {
    __shared__ __align__(128) unsigned char stage[kBulkBytes];
    __shared__ __align__(8) uint64_t bar;
    const int W = (int)p.stride_dim;  // = width
    if (threadIdx.x == 0) {
        kda::mbar_init(&bar, 1);
        kda::fence_mbar_init();
    }
    __syncthreads();
    uint32_t phase = 0;
    for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
        const int n = row_count(p, b);
        if (n <= 0) continue;  // uniform over the CTA
        const int c0 = blockIdx.x * run;
        if (c0 >= p.C) continue;
        const int chans = min(run, p.C - c0);
        const uint32_t bytes = (uint32_t)(chans * W * (int)sizeof(T));
        unsigned char *src = p.conv + ((long long)p.slots[b] * p.stride_slot +
                                       (long long)c0 * W) * (long long)sizeof(T);
        if (threadIdx.x == 0) {
            kda::mbar_arrive_expect_tx(&bar, bytes);
            kda::bulk_load(stage, src, bytes, &bar);
        }
        const bool landed = kda::mbar_wait_bounded(&bar, phase, kBulkWaitBudget);
        if (__syncthreads_or(!landed)) {
            // the load did not land in time: report it, give it one more
            // bounded wait so that no copy into shared memory outlives the
            // CTA, and leave with nothing written
            if (threadIdx.x == 0) {
                if (p.err != nullptr) atomicOr(p.err, KDA_ERR_WAIT_TIMEOUT);
                kda::mbar_wait_bounded(&bar, phase, kBulkWaitBudget);
                bulk_wait_read();
            }
            return;
        }
        phase ^= 1u;
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
        kda::fence_proxy_async_smem();  // the bulk store reads through the async proxy
        __syncthreads();
        if (threadIdx.x == 0) {
            bulk_store(src, stage, bytes);
            bulk_commit();
            bulk_wait_read();
        }
        __syncthreads();  // the stage is free for the next row
    }
    if (threadIdx.x == 0) bulk_wait_read();
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

// Row b's align-mode plan: its checks (flagged), n, its source slot and its
// blocks.  False: the row writes nothing.
__device__ __forceinline__ bool align_row(const Params &p, const AlignArgs &a, int b, int &n,
                                          int &slot, kda_blocks::Blocks &bl) {
    const int len = p.cu[b + 1] - p.cu[b];
    slot = p.slots[b];
    if (len < 0 || len > p.Q) {
        flag(p, KDA_ROW_BAD_LENGTH);
        return false;
    }
    if (slot >= p.S) {
        flag(p, KDA_ROW_BAD_SLOT);
        return false;
    }
    const int req = a.request_indices != nullptr ? a.request_indices[b] : b;
    if (req < 0 || req >= a.num_requests) {
        flag(p, KDA_ROW_BAD_BLOCK);
        return false;
    }
    n = min(max(p.acc[req], 0), min(len, p.Q));
    if (slot <= 0 || n <= 0) return false;
    bl = kda_blocks::plan(a.block_table + (long long)req * a.bt_stride, a.bt_width, a.block_size,
                          a.num_computed[req], n);
    if (bl.bad) {
        flag(p, KDA_ROW_BAD_BLOCK);
        return false;
    }
    if (bl.final_block >= p.S || bl.boundary >= p.S) {
        flag(p, KDA_ROW_BAD_SLOT);
        return false;
    }
    return bl.final_block > 0;
}

// Any strides: one thread per channel, element by element.
template <typename T>
__global__ void __launch_bounds__(kThreads) align_kernel(const Params p, const AlignArgs a) {
    for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
        int n, slot;
        kda_blocks::Blocks bl;
        if (!align_row(p, a, b, n, slot, bl)) continue;
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

// Channel-major and dense, units of at most kUnitMaxBytes (the fewest whole
// channels whose bytes make 16-byte pieces): a thread loads its unit of the
// source slot with 16-byte loads into its own slice of shared memory, then,
// for the boundary block (when there is one) and the final block in turn,
// loads the block's unit into a second slice, copies each channel's window
// from the source's copy into columns [0, history) and stores the unit
// back.  Both windows come from the source as it was before the call, and
// a block that is the source itself, or a boundary block that is the final
// block, ends with what the element-wise form leaves.  Piece v of a slice
// sits at 16 * (v * kThreads + t), so a warp's 16-byte accesses fall on
// distinct banks.
constexpr int kUnitMaxBytes = 64;

template <typename T>
__global__ void __launch_bounds__(kThreads) align_unit_kernel(const Params p, const AlignArgs a,
                                                              int unit_chans) {
    constexpr int kPieces = kUnitMaxBytes / 16;
    constexpr int kPer = 16 / (int)sizeof(T);  // elements per piece
    __shared__ __align__(16) unsigned char stage[2 * kPieces * kThreads * 16];
    const int W = (int)p.stride_dim;  // = width
    const int unit_bytes = unit_chans * W * (int)sizeof(T);
    const int uv = unit_bytes / 16;
    const int units = p.C / unit_chans;
    uint4 *s0 = reinterpret_cast<uint4 *>(stage) + threadIdx.x;                     // source
    uint4 *s1 = reinterpret_cast<uint4 *>(stage) + kPieces * kThreads + threadIdx.x;  // block
    // element e of a slice: piece e / kPer, position e % kPer
    auto at = [&](uint4 *slice, int e) -> T & {
        return reinterpret_cast<T *>(slice + (e / kPer) * kThreads)[e % kPer];
    };
    for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
        int n, slot;
        kda_blocks::Blocks bl;
        if (!align_row(p, a, b, n, slot, bl)) continue;
        const long long slot_bytes = p.stride_slot * (long long)sizeof(T);
        for (int u = blockIdx.x * kThreads + threadIdx.x; u < units; u += gridDim.x * kThreads) {
            const long long off = (long long)u * unit_bytes;
            const uint4 *src = reinterpret_cast<const uint4 *>(p.conv + slot * slot_bytes + off);
#pragma unroll
            for (int v = 0; v < kPieces; ++v)
                if (v < uv) s0[v * kThreads] = src[v];
            // the window at column `col` of the source's copy into `block`
            auto merge_into = [&](long long block, int col) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.conv + block * slot_bytes + off);
#pragma unroll
                for (int v = 0; v < kPieces; ++v)
                    if (v < uv) s1[v * kThreads] = dst[v];
                for (int c = 0; c < unit_chans; ++c) {
#pragma unroll
                    for (int h = 0; h < KDA_MAX_CONV_HISTORY; ++h)
                        if (h < p.hist) at(s1, c * W + h) = at(s0, c * W + col + h);
                }
#pragma unroll
                for (int v = 0; v < kPieces; ++v)
                    if (v < uv) dst[v] = s1[v * kThreads];
            };
            if (bl.boundary > 0) merge_into(bl.boundary, bl.boundary_len - 1);
            merge_into(bl.final_block, n - 1);
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
        cc->conv_dim % unit == 0 && unit * chan_bytes <= kBulkBytes) {
        const int run = (int)(unit * (kBulkBytes / (unit * chan_bytes)));
        const dim3 grid((cc->conv_dim + run - 1) / run, rows);
        if (cc->elem_bytes == 2)
            bulk_kernel<uint16_t><<<grid, kThreads, 0, st>>>(p, run);
        else
            bulk_kernel<uint32_t><<<grid, kThreads, 0, st>>>(p, run);
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
    cudaStream_t stv = static_cast<cudaStream_t>(stream);
    const long long eb = cc->elem_bytes;
    const bool slots16 = aligned(conv_state, 16) && (cc->stride_slot * eb) % 16 == 0;
    const long long chan_bytes = (long long)cc->width * eb;
    long long unit = 1;
    while ((unit * chan_bytes) % 16 != 0) ++unit;
    if (slots16 && cc->stride_col == 1 && cc->stride_dim == cc->width &&
        cc->conv_dim % unit == 0 && unit * chan_bytes <= kUnitMaxBytes) {
        const int units = (int)(cc->conv_dim / unit);
        const dim3 grid((units + kThreads - 1) / kThreads, rows);
        if (cc->elem_bytes == 2)
            align_unit_kernel<uint16_t><<<grid, kThreads, 0, stv>>>(p, a, (int)unit);
        else
            align_unit_kernel<uint32_t><<<grid, kThreads, 0, stv>>>(p, a, (int)unit);
    } else {
        const dim3 grid((cc->conv_dim + kThreads - 1) / kThreads, rows);
        if (cc->elem_bytes == 2)
            align_kernel<uint16_t><<<grid, kThreads, 0, stv>>>(p, a);
        else
            align_kernel<uint32_t><<<grid, kThreads, 0, stv>>>(p, a);
    }
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
