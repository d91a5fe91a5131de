// Align-mode block plan shared by the recurrent commit and the conv
// compaction (recoverssm.py, `_prepare_commit_plan_kernel` align branch).
#pragma once

namespace kda_blocks {

// Blocks a committing row writes.  Token t of the step sits at position
// c + t, c = num_computed of the row's request.  The state after the n-th
// accepted token belongs to the block holding position c + n - 1, column
// (c + n - 1) / block_size clamped to the table.  The first block boundary
// after c is (c / block_size + 1) * block_size; when the step reaches it
// (c + n >= boundary), the state after boundary_len = boundary - c tokens
// belongs to the block that ends there.
struct Blocks {
    int final_block;   // block_table entry, may be <= 0 (then nothing is written)
    int boundary;      // block_table entry of the reached boundary, or 0
    int boundary_len;  // tokens up to that boundary (0: none reached)
    bool bad;          // negative c, or the boundary block is past the table
};

__device__ __forceinline__ Blocks plan(const int *row, int width, int block_size, int c, int n) {
    Blocks b{0, 0, 0, false};
    if (c < 0) {
        b.bad = true;
        return b;
    }
    const int end = c + n;
    b.final_block = row[min(max(end - 1, 0) / block_size, width - 1)];
    const int boundary = (c / block_size + 1) * block_size;
    if (end >= boundary) {
        const int col = boundary / block_size - 1;
        if (col >= width) {
            b.bad = true;
            return b;
        }
        b.boundary = row[col];
        b.boundary_len = boundary - c;
    }
    return b;
}

}  // namespace kda_blocks
