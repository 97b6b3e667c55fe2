// Fifth-generation tensor-core building blocks for the block-scaled MXFP4
// path on sm_103a: tensor memory (TMEM) allocation, tcgen05 block-scaled
// MMA with E2M1 weights and E4M3 activations (kind::mxf8f6f4, one E8M0 scale
// per 32 values on each operand), scale copies into TMEM, accumulator loads,
// and the shared-memory / instruction descriptors they take.
//
// Operand layouts these helpers assume (all K-major, 128-byte swizzle):
//   - an "atom" is 128 K values. In shared memory a row of an atom is 128
//     bytes: E4M3 one byte per value; E2M1 as the TMA unpacking load
//     (16U4_ALIGN16B) leaves it, 8 bytes of 16 packed codes then 8 bytes of
//     gap per 16 values. Rows are 128 B apart, groups of 8 rows 1024 B apart,
//     16-byte chunks XOR-swizzled by (row % 8). One MMA consumes 32 K values
//     of an atom (32 bytes of each row), so the four MMAs of an atom start
//     32 bytes apart.
//   - block scales in TMEM: one 32-bit word per (row, atom) holds the 4
//     E8M0 scales of the atom's four 32-value blocks, first block in the
//     low byte. The scale address an MMA takes is a multiple of 4 columns;
//     the MMA reads row r's word at lane r, column (scale address + r/32),
//     and takes the byte of its K block within the atom (the scale "ID" of
//     the instruction descriptor). Words can be written by tcgen05.st (each
//     warp into its own 32-lane quarter) or copied from a 512-byte
//     shared-memory image of 32 lines x 16 bytes with a 32x128b.warpx4 copy,
//     which puts line m into lane m of every quarter, 4 columns.
//   - accumulator: row r of the 128-row tile in TMEM lane r, output column n
//     in TMEM column (base + n), fp32.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mxfp4 {
namespace tc {

// ------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor (sm_100 family format): start address,
// leading- and stride-dimension byte offsets (all >> 4), version 1 at bits
// 46-47, layout (swizzle) type at bits 61-63.
constexpr uint32_t kLayoutNone = 0;
constexpr uint32_t kLayoutSwizzle128 = 2;

__host__ __device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
           (static_cast<uint64_t>(layout & 7u) << 61);
}

// K-major, 128-byte swizzled operand tile starting at addr (1024-aligned
// atom base plus 32 bytes per MMA step): 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t operand_desc(uint32_t addr) { return smem_desc(addr, 16, 1024, kLayoutSwizzle128); }

// A 512-byte scale image: 32 contiguous 16-byte lines, no swizzle.
__device__ __forceinline__ uint64_t scale_image_desc(uint32_t addr) { return smem_desc(addr, 128, 128, kLayoutNone); }

constexpr uint32_t kFmtE4M3 = 0;
constexpr uint32_t kFmtE2M1 = 5;

// Instruction descriptor of a block-scaled MMA: B scale ID (bits 4-5), A
// and B formats (7-9, 10-12), N / 8 (17-22), E8M0 scales (bit 23), M / 16
// (24-28), A scale ID (29-30). Both operands K-major, no negation.
__host__ __device__ __forceinline__ uint32_t mma_idesc(uint32_t afmt, uint32_t bfmt, uint32_t m, uint32_t n,
                                                       uint32_t sf_id) {
    return (sf_id << 4) | (afmt << 7) | (bfmt << 10) | ((n >> 3) << 17) | (1u << 23) | ((m >> 4) << 24) |
           (sf_id << 29);
}

// ------------------------------------------------------------------ TMEM
// Warp-wide: allocate ncols columns (a power of two >= 32); the base address
// is written to the shared word at slot.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tcgen05 operations around thread synchronisation.
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ------------------------------------------------------------------- MMA
// D[128 x N] (+)= A[128 x 32] * B[N x 32]^T with per-32 block scales from
// TMEM; accumulate = false overwrites D.
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(static_cast<uint32_t>(accumulate))
        : "memory");
}

// Both operands packed E2M1 (two codes per byte, the even K index in the low
// nibble, as stored in HBM): D[128 x N] (+)= A[128 x 64] * B[N x 64]^T with
// one E8M0 scale per 32 values on each side (scale_vec::2X). The scale ID of
// the instruction descriptor picks bytes {0,1} (ID 0) or {2,3} (ID 2) of the
// 32-bit TMEM scale word, whose 4 bytes cover 128 consecutive K values.
constexpr uint32_t kFmtMxf4E2M1 = 1;

__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(static_cast<uint32_t>(accumulate))
        : "memory");
}

// Copy a 512-byte scale image from shared memory into 4 TMEM columns of all
// 128 lanes (each 32-lane quarter gets the same 32 lines).
__device__ __forceinline__ void copy_scales_to_tmem(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Arrive once on the mbarrier when every earlier tcgen05 operation of this
// thread has completed.
__device__ __forceinline__ void commit_to(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

// --------------------------------------------------------- TMEM -> regs
// Warp-wide: lane i of the warp's 32-lane quarter, N consecutive columns.
template <int N>
struct TmemLd;

template <>
struct TmemLd<16> {
    __device__ static void load(uint32_t taddr, uint32_t (&r)[16]) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr)
            : "memory");
    }
};

template <int N>
__device__ __forceinline__ void tmem_load(uint32_t taddr, uint32_t (&r)[N]) {
    static_assert(N % 16 == 0, "columns in multiples of 16");
#pragma unroll
    for (int c = 0; c < N / 16; ++c) TmemLd<16>::load(taddr + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&r[16 * c]));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Warp-wide: lane i of the warp's 32-lane quarter stores 16 consecutive
// columns starting at taddr (a multiple of 16 columns).
__device__ __forceinline__ void tmem_store16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ TMA
// 3D tiled tensor load (coordinates innermost first) completing on bar.
__device__ __forceinline__ void tma_load_3d_tc(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                               uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// Remote arrive (release, cluster scope) on an mbarrier of another CTA of
// the cluster (address from mapa).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

}  // namespace tc
}  // namespace mxfp4
