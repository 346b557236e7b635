// si_tc.cuh -- 5th-generation tensor core (tcgen05) building blocks for sm_103a:
// tensor-memory allocation, shared-memory matrix descriptors, the 16-bit
// (kind::f16: fp16 or bf16) MMA with fp32 accumulation in tensor memory, its
// completion signal, and the tensor-memory loads of the epilogue.  Inline PTX
// (no library).
//
// Operand layout used throughout: K-major, 128-byte swizzle.  A tile of R rows
// x 64 16-bit values (128 bytes per row) occupies R*128 bytes, 1024-byte aligned; row r
// sits at byte r*128 and its 16-byte chunk c is stored at chunk c ^ (r & 7).
// Eight rows form one 1024-byte swizzle atom; atoms follow each other along
// the row (M or N) dimension.
#pragma once
#include <cstdint>

namespace si {
namespace tc {

// ---------------------------------------------------------------- TMEM
// Allocate `ncols` (power of two >= 32) tensor-memory columns for this CTA;
// the base address is written to shared memory at `dst_smem`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// Whole warp; every allocation is released before the CTA exits.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes (st.shared, cp.async) become visible to
// the tensor core (async proxy) only after this fence.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor, K-major with 128-byte swizzle: start
// address >> 4 in bits 0-13, leading byte offset >> 4 in 16-29 (unused for a
// K extent within one swizzle row; 16 bytes), stride byte offset >> 4 in
// 32-45 (1024: one eight-row atom), descriptor version 1 in 46-47, layout
// type 2 (128-byte swizzle) in 61-63.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr) {
    return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)(16 >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (7-9 = 1, 10-12 = 1), both K-major (15, 16 = 0), N >> 3 in 17-22,
// M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with A and B fp16 (type fields 0).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- MMA
// D[tmem] (+)= A[smem] * B[smem]^T, M x N x 16 (16-bit operands of the type
// the instruction descriptor names), issued by one thread.
__device__ __forceinline__ void mma_f16kind(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}
// Arrive on an mbarrier once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

// ---------------------------------------------------------------- TMEM -> registers
// Warp w of a warpgroup reads lanes 32*(w%4) .. +31; thread t gets 32
// consecutive 32-bit columns of lane 32*(w%4)+t starting at column `col`.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- CTA pairs (cta_group::2)
// Two CTAs of a cluster (ranks 2p, 2p+1) act as one MMA unit: an M = 256
// MMA issued by the even CTA reads rows 0-127 of A from its own shared
// memory and rows 128-255 from its peer's (same offset), columns 0..N/2-1 of B
// from its own shared memory and N/2..N-1 from its peer's, and accumulates
// rows 0-127 of D in its own tensor memory and 128-255 in the peer's.
// Allocation and release are collective: one warp of each CTA of the pair.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_pair_f16kind(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}
// One 64-wide K step of pair MMAs: four K = 16 MMAs whose operand
// descriptors advance by 32 bytes (2 in the descriptor's address field) within
// the 128-byte swizzle row; the first accumulates into D only if `acc`.
__device__ __forceinline__ void mma_pair_k64(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %11, 0;\n\t"
        "setp.eq.u32 q, %10, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %5, %9, p;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %2, %6, %9, q;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %3, %7, %9, q;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %4, %8, %9, q;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(a_desc + 2), "l"(a_desc + 4), "l"(a_desc + 6), "l"(b_desc), "l"(b_desc + 2), "l"(b_desc + 4),
        "l"(b_desc + 6), "r"(idesc), "r"(0u), "r"(acc)
        : "memory");
}
// Once every pair MMA this thread issued so far has completed, arrive on the
// mbarrier at shared-memory offset `mbar` in each CTA of `cta_mask`.
__device__ __forceinline__ void mma_pair_commit_mc(uint32_t mbar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            mbar),
        "h"(cta_mask)
        : "memory");
}

// Byte offset of 16-bit element (row r, k) of a K-major 128-byte-swizzled tile
// of 64-wide rows (k < 64).
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t k) {
    return r * 128u + ((((k >> 3) ^ (r & 7u)) & 7u) << 4) + ((k & 7u) << 1);
}

}  // namespace tc
}  // namespace si
