// Align-mode bookkeeping after a commit, as a plain integer kernel (sm_103a).
//
// recoverssm.py, `_record_state_block_kernel` / `record_state_blocks`: the
// commit in align mode leaves a request's state in the block that holds its
// last committed token, so the request's running state column is pointed
// there (min((num_computed + num_sampled - 1) / block_size, width - 1), the
// position clamped at 0) and its accepted count is reset to 1.  One thread
// per spec row; a few bytes per row, so the launch is latency-bound.
// The public contract is in include/kda.h (kda_record_state_blocks).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda_blocks_record {

constexpr int kThreads = 256;

struct Args {
    const int32_t *idx_mapping, *num_sampled, *num_computed, *request_indices;
    int32_t *state_column, *num_accepted, *err;
    int B, num_requests, num_states, block_size, width;
};

__global__ void __launch_bounds__(kThreads) record_kernel(const Args a) {
    const int i = blockIdx.x * kThreads + threadIdx.x;
    if (i >= a.B) return;
    const int q = a.request_indices != nullptr ? a.request_indices[i] : i;
    if (q < 0 || q >= a.num_requests) {
        if (a.err != nullptr) atomicOr(a.err, KDA_ROW_BAD_BLOCK);
        return;
    }
    const int s = a.idx_mapping[q];
    if (s < 0) return;  // the request records nothing
    if (s >= a.num_states) {
        if (a.err != nullptr) atomicOr(a.err, KDA_ROW_BAD_SLOT);
        return;
    }
    long long last = (long long)a.num_computed[q] + (long long)a.num_sampled[q] - 1;
    if (last < 0) last = 0;
    const long long col = last / a.block_size;
    a.state_column[s] = (int32_t)(col < a.width - 1 ? col : a.width - 1);
    a.num_accepted[s] = 1;
}

bool aligned4(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }

}  // namespace kda_blocks_record

extern "C" {

kda_status kda_record_state_blocks(const kda_align *align, const int32_t *idx_mapping,
                                   const int32_t *num_sampled, int32_t B,
                                   int32_t *state_column, int32_t *num_accepted,
                                   int32_t num_states, int32_t *error_word, void *stream) {
    using namespace kda_blocks_record;
    if (B < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;  // nothing to do; no pointer is inspected
    if (align == nullptr || align->block_size < 1 || align->block_table_width < 1 ||
        align->num_requests < 1 || align->reserved != 0 || num_states < 1)
        return KDA_ERR_INVALID_ARG;
    if (!idx_mapping || !num_sampled || !align->num_computed || !state_column || !num_accepted)
        return KDA_ERR_INVALID_ARG;
    if (!aligned4(idx_mapping) || !aligned4(num_sampled) || !aligned4(align->num_computed) ||
        !aligned4(state_column) || !aligned4(num_accepted) ||
        (align->request_indices != nullptr && !aligned4(align->request_indices)) ||
        (error_word != nullptr && !aligned4(error_word)))
        return KDA_ERR_INVALID_ARG;
    Args a;
    a.idx_mapping = idx_mapping;
    a.num_sampled = num_sampled;
    a.num_computed = align->num_computed;
    a.request_indices = align->request_indices;
    a.state_column = state_column;
    a.num_accepted = num_accepted;
    a.err = error_word;
    a.B = B;
    a.num_requests = align->num_requests;
    a.num_states = num_states;
    a.block_size = align->block_size;
    a.width = align->block_table_width;
    const int grid = (B + kThreads - 1) / kThreads;
    record_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
