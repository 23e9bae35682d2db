// tc.cuh - hand-written PTX for the block-scaled 5th-generation tensor-core
// paths (tcgen05 kind::mxf4): shared-memory and instruction descriptors,
// the MMA, scale-factor copies into TMEM, TMA tile loads and TMEM loads.
#pragma once

#include "common.cuh"

namespace k3mx {
namespace {

// K-major operand in the 128-byte swizzle with a given stride between
// 8-row groups
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | (uint64_t)(16u >> 4) << 16 |
           (uint64_t)((sbo >> 4) & 0x3FFFu) << 32 | (uint64_t)1 << 46 | (uint64_t)2 << 61;
}
// K-major operand in the 64-byte swizzle: 8-row groups of 64-byte rows
// (512 bytes), 16-byte chunks XOR-permuted by (row / 2) % 4
__device__ __forceinline__ uint64_t desc_sw64(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | (uint64_t)(16u >> 4) << 16 |
           (uint64_t)((512u >> 4) & 0x3FFFu) << 32 | (uint64_t)1 << 46 | (uint64_t)4 << 61;
}
// tcgen05.cp source: 32 lines of 16 B in four 8-line groups `sbo` apart, no swizzle
__device__ __forceinline__ uint64_t desc_atom(uint32_t saddr, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | (uint64_t)((sbo >> 4) & 0x3FFFu) << 32 |
           (uint64_t)1 << 46;
}
// one scale-factor atom (32 lines x 16 B) into 4 TMEM columns of all 128
// lanes (each lane quarter gets the same copy); scale of row m, block kb of
// the atom: column m / 32, byte kb, line m % 32
__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
// 128 rows x 4 words into TMEM lanes 0..127, 4 columns (row r -> lane r);
// source: 128 rows of 16 B back to back (desc_atom with 8-row groups 128 B
// apart)
__device__ __forceinline__ void tmem_cp_rows16(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::1.128x128b [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
// tcgen05.cp.128x256b source: 128 rows of 32 B as [row / 8][16-byte half]
// [row % 8][16 B] (halves 128 B apart, 8-row groups 256 B apart), no swizzle
__device__ __forceinline__ uint64_t desc_rows32(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | (uint64_t)(128u >> 4) << 16 | (uint64_t)(256u >> 4) << 32 |
           (uint64_t)1 << 46;
}
// byte offset of 32-bit word j of row r in that source
__host__ __device__ constexpr uint32_t rows32_offset(int r, int j) {
    return (uint32_t)((r >> 3) * 256 + (j >> 2) * 128 + (r & 7) * 16 + (j & 3) * 4);
}
// 128 rows x 8 words into TMEM lanes 0..127, 8 columns (row r -> lane r).
// For an M = 128 block-scaled MMA the lanes of quarter q read their scale
// word at column (scale address + q), so word q of row r = 32 q + l feeds
// one matrix and word 4 + q another: two matrices' A scales in one copy.
__device__ __forceinline__ void tmem_cp_rows32(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
// instruction descriptor, kind::mxf4: e2m1 A and B, ue8m0 scales, K-major,
// M = 128, N = n; sf_id picks the byte pair of the scale columns
__device__ __forceinline__ uint32_t idesc_mxf4(int n, int sf_id) {
    return ((uint32_t)sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(128 >> 4) << 24) | ((uint32_t)sf_id << 29);
}
__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}
// instruction descriptor, kind::mxf8f6f4 with e2m1 A (each 16 packed codes
// spread over 16 bytes by the copy engine) and e4m3 B, ue8m0 scales, K-major, M = 128,
// N = n; sf_id picks the scale byte (the 32-column block of a K = 128 step)
__device__ __forceinline__ uint32_t idesc_e2m1_e4m3(int n, int sf_id) {
    return ((uint32_t)sf_id << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(128 >> 4) << 24) | ((uint32_t)sf_id << 29);
}
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa, uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}
// The same MMA, with three mbarrier phases polled (non-blocking) just ahead
// of it in the same instruction stream: the polls' shared-memory round trips
// overlap the MMA's issue.  True when all three phases had completed.
__device__ __forceinline__ bool mma_mxf8f6f4_poll3(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                   uint32_t sfa, uint32_t sfb, uint32_t acc, uint32_t bar0,
                                                   uint32_t par0, uint32_t bar1, uint32_t par1, uint32_t bar2,
                                                   uint32_t par2) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p, q0, q1, q2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q0, [%8], %9;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q1, [%10], %11;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q2, [%12], %13;\n\t"
        "setp.ne.b32 p, %7, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], %2, %3, %4, [%5], [%6], p;\n\t"
        "and.pred q0, q0, q1;\n\t"
        "and.pred q0, q0, q2;\n\t"
        "selp.u32 %0, 1, 0, q0;\n\t}"
        : "=r"(ok)
        : "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc), "r"(bar0), "r"(par0), "r"(bar1),
          "r"(par1), "r"(bar2), "r"(par2)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const void *map, int x, int y, uint32_t bar,
                                       uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}
// a box of a tensor map into L2 only (no shared memory, no barrier)
__device__ __forceinline__ void tma_prefetch_2d(const void *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_3d(uint32_t dst, const void *map, int x, int y, int z, uint32_t bar,
                                       uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&v)[N]);
template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr));
}
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
          "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
          "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
          "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// scale byte 255 (a group that contributes nothing) -> 0 (2^-127); the
// group's codes are zeroed in shared memory as well (zero_nan_groups_*), so
// the group adds exactly 0
__device__ __forceinline__ uint32_t drop_nan_scales(uint32_t w) { return w & ~__vcmpeq4(w, 0xFFFFFFFFu); }

// bytes 0xFF of a scale word (four groups) as 0xFF lanes, else 0
__device__ __forceinline__ uint32_t nan_scale_mask(uint32_t w) { return __vcmpeq4(w, 0xFFFFFFFFu); }

// Zero the 16 packed bytes (32 codes) of every group whose scale byte is 255,
// for row r of a weight tile of 128-byte rows in the 128-byte swizzle (a
// 256-column chunk: groups 0-3 from sc.x, 4-7 from sc.y).  Called after the
// tile's copy landed and before the tensor core reads it.
__device__ __forceinline__ void zero_nan_groups_sw128(uint32_t tile, int r, uint2 sc) {
    const uint32_t m[2] = {nan_scale_mask(sc.x), nan_scale_mask(sc.y)};
#pragma unroll
    for (int g = 0; g < 8; g++)
        if ((m[g >> 2] >> (8 * (g & 3))) & 1u)
            sts128(tile + (uint32_t)(r * 128) + (uint32_t)(((g ^ (r & 7)) & 7) << 4), 0u, 0u, 0u, 0u);
}

// The same for a tile of 64-byte rows in the 64-byte swizzle (a 128-column
// stage: groups 0-3 from the bytes of sc); chunk j of row r sits at
// j ^ ((r / 2) % 4)
__device__ __forceinline__ void zero_nan_groups_sw64(uint32_t tile, int r, uint32_t sc) {
    const uint32_t m = nan_scale_mask(sc);
#pragma unroll
    for (int g = 0; g < 4; g++)
        if ((m >> (8 * g)) & 1u)
            sts128(tile + (uint32_t)(r * 64) + (uint32_t)(((g ^ (r >> 1)) & 3) << 4), 0u, 0u, 0u, 0u);
}
// Tile of expanded e2m1 codes (rows of 128 codes in 128-byte rows, 128-byte
// swizzle; the copy engine puts each 16 packed codes into 8 bytes of a
// 16-byte chunk): the four 32-code groups of row r whose scale byte in `sc`
// is 255 get zero codes (both chunks of the group cleared).
__device__ __forceinline__ void zero_nan_groups_x128(uint32_t tile, int r, uint32_t sc) {
    const uint32_t row = tile + (uint32_t)r * 128;
#pragma unroll
    for (int g = 0; g < 4; g++)
        if (((sc >> (8 * g)) & 0xFFu) == 0xFFu) {
            sts128(row + (((uint32_t)(2 * g) ^ (uint32_t)r) & 7u) * 16, 0u, 0u, 0u, 0u);
            sts128(row + (((uint32_t)(2 * g + 1) ^ (uint32_t)r) & 7u) * 16, 0u, 0u, 0u, 0u);
        }
}


}  // namespace
}  // namespace k3mx
