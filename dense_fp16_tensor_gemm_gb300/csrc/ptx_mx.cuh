// ptx_mx.cuh -- inline-PTX wrappers for block-scaled 8-bit MMA (kind::mxf8f6f4):
// plain bulk copies of scale-factor atoms, tcgen05.cp of an atom into Tensor
// Memory, and the block-scaled tcgen05.mma.  Written from the PTX ISA's
// descriptions of cp.async.bulk, tcgen05.cp and tcgen05.mma.
//
// Scale factors are E8M0 bytes, one per 32 consecutive K elements of a row.
// An "atom" is 512 bytes holding the scales of 128 rows for 4 consecutive
// 32-element K blocks (128 K elements, one stage of 8-bit data): byte
// 16*r + 4*q + s is the scale of row 32*q + r, K block s.  tcgen05.cp
// .32x128b.warpx4 copies the atom's 32 rows of 16 bytes into TMEM lanes r,
// 32+r, 64+r and 96+r, columns c..c+3 (column j holds bytes 4j..4j+3 of the
// row).  The block-scaled MMA reads the scale of row m of A from lane m,
// column (m / 32) of its A-scale address, and that of row n of B from lane
// n % 32, column (n / 32) of its B-scale address; the byte within the column
// is the scale-factor ID of the instruction descriptor (bits 29-30 for A, 4-5
// for B).  Both reads land on byte 4*(m/32) + s of atom row m % 32: the atom
// is the same for either operand.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace gnt {

// Contiguous global -> shared copy of `bytes` (a multiple of 16, both
// addresses 16-byte aligned), counted on `bar` like a tensor load.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// Shared-memory descriptor of one atom (32 rows of 16 bytes, no swizzle):
// 8-row core matrices of 128 contiguous bytes, 128 bytes apart.
__device__ __forceinline__ uint64_t atom_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128 >> 4) << 16;
    d |= static_cast<uint64_t>(128 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// Atom (shared) -> TMEM columns col..col+3 of all four lane quadrants.
__device__ __forceinline__ void tc_cp_atom(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Instruction descriptor for kind::mxf8f6f4 with E8M0 scales: bit 23 scale
// type (1 = UE8M0), 17-22 N >> 3, 24-28 M >> 4; the A/B formats (bits 7-9,
// 10-12) and majors (15, 16) are ORed in by the caller, the scale-factor IDs
// per instruction.  The accumulator is fp32.
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N)
{
    return (1u << 23) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= (A * scale_A) * (B * scale_B)^T over 32 elements of K.
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint32_t alo, uint32_t ahi, uint32_t blo, uint32_t bhi,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "setp.ne.b32 p, %8, 0;\n\t"
        "mov.b64 da, {%1, %2};\n\t"
        "mov.b64 db, {%3, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], da, db, %5, [%6], [%7], p;\n\t}" ::"r"(
            d_tmem),
        "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 4-D tiled load of scale atoms into this CTA's shared memory, completing on a
// barrier in either CTA of the pair (the pair kernel's stage barrier).
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int32_t c0,
                                                 int32_t c1, int32_t c2, int32_t c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// 5-D tiled load, completing on a barrier in either CTA of the pair: a scale
// map whose third dimension has stride 0 lands each atom several times over.
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int32_t c0,
                                                 int32_t c1, int32_t c2, int32_t c3, int32_t c4)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}

// Shared-memory descriptor of a 128-row x 32-byte source for tcgen05.cp
// .128x256b, no swizzle: row L's first 16 bytes at start + (L / 8) * 128 +
// (L % 8) * 16 (8-row core matrices of 128 contiguous bytes), its second 16
// bytes `lbo` bytes further on.
__device__ __forceinline__ uint64_t rows32_desc(uint32_t saddr, uint32_t lbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(lbo >> 4) << 16;
    d |= static_cast<uint64_t>(128 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// The pair forms (cta_group::2), issued by the leader CTA of a pair: the copy
// moves each CTA's atom at this shared offset into its own TMEM; each half of
// the MMA reads the scales of its 128 rows of A, and of all N rows of B, from
// its own CTA's TMEM.
__device__ __forceinline__ void tc_cp_atom_pair(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 128 rows of 32 bytes (shared) -> TMEM lane L, columns col..col+7, no
// replication: with the source holding two atoms four times over (copy q of
// atom h at h * lbo + 512 * q), every lane quadrant receives both atoms, as
// two .32x128b.warpx4 copies would give it, in one instruction.
__device__ __forceinline__ void tc_cp_rows32_pair(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tc_mma_pair_mx(uint32_t d_tmem, uint32_t alo, uint32_t ahi, uint32_t blo,
                                               uint32_t bhi, uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                               uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "setp.ne.b32 p, %8, 0;\n\t"
        "mov.b64 da, {%1, %2};\n\t"
        "mov.b64 db, {%3, %4};\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], da, db, %5, [%6], [%7], p;\n\t}" ::"r"(
            d_tmem),
        "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

}  // namespace gnt
