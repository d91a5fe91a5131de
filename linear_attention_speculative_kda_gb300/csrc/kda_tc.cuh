// Tensor-core helpers (inline PTX, sm_100a family / sm_103a): tensor-map TMA
// loads with the 128-byte swizzle, tensor memory (TMEM) allocation, loads and
// stores, and tcgen05.mma of kind::tf32 with its commit to an mbarrier.
//
// Operand layout used throughout: K-major with the 128-byte swizzle.  A
// matrix of R rows x 32 fp32 (128 bytes per row) is stored as R/8 atoms of
// 8 rows x 128 bytes, atom after atom (1024 bytes apart); inside an atom,
// the 16-byte chunk c of row r sits at chunk position c ^ (r mod 8).  Each
// atom must start on a 1024-byte boundary.  A K extent of 128 fp32 is four
// such blocks of 32 columns, one after the other.
#pragma once

#include <stdint.h>

#include "kda_async.cuh"

namespace kda {

// Byte offset of element (row, col) (col < 32) inside one 32-column block.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col) {
    return (uint32_t)row * 128u + ((uint32_t)(((col >> 2) ^ (row & 7)) << 4)) +
           ((uint32_t)(col & 3) << 2);
}

// 2-D tensor-map load of one box into shared memory, completing on `bar`.
// x (the inner coordinate, in elements) times the element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void *dst_smem, const void *tmap, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand with the 128-byte
// swizzle starting at `addr` (shared-space byte address): leading byte
// offset unused (16), stride byte offset 1024 (one atom of 8 rows), the
// descriptor version of this architecture (bit 46) and the swizzle mode
// (2 = 128-byte) in bits 61..63.  Advancing K by 8 fp32 inside a 128-byte
// atom adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3fffu) | ((uint64_t)(16u >> 4) << 16) |
           ((uint64_t)(1024u >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::tf32 with fp32 accumulation, both operands
// K-major, shape M x N (bits: D format 4..5, A format 7..9, B format 10..12,
// N >> 3 in 17..22, M >> 4 in 24..28).
__host__ __device__ constexpr uint32_t tf32_idesc(uint32_t M, uint32_t N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// --- tensor memory: one warp allocates and frees the CTA's columns ---------

__device__ __forceinline__ void tmem_alloc(uint32_t *holder_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(holder_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// Ordering of tcgen05 operations around thread synchronisation.
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// A TMEM address is (lane << 16) | column; warp w of a CTA may access lanes
// 32 (w mod 4) .. 32 (w mod 4) + 31.  32x32b shapes: thread t of the warp
// accesses lane (taddr lane) + t, 16 consecutive columns here.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&u)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]),
        "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]),
        "r"(u[15])
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&u)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]),
          "=r"(u[14]), "=r"(u[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// D (TMEM) [+]= A B^T for one K step of 8: A from shared memory (descriptor)
// or from TMEM (lane = row, one fp32 per column), B from shared memory.
// Issued by one thread.
__device__ __forceinline__ void umma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The mbarrier gets one arrival once every tcgen05.mma this thread issued
// before has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// The TF32 part of an fp32 value as the tensor core reads it (the low 13
// mantissa bits dropped), so that x = tf32_hi(x) + (x - tf32_hi(x)) exactly.
__device__ __forceinline__ float tf32_hi(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

}  // namespace kda
