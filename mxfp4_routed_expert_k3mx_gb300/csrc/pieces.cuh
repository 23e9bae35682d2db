// pieces.cuh - activation vectors as sums of MXFP4 pieces, written in the
// layout the block-scaled tensor-core MMA (tcgen05 kind::mxf4) reads.
//
// A vector v is split exactly into kPieces MXFP4 vectors plus a residual:
// piece i takes, per 32-column block, the ue8m0 scale 2^e that maps the
// block's largest residual |value| into (3, 6] and the nearest e2m1 value
// of every residual; the next residual is formed exactly in fp32.  Each
// piece cuts the block's largest residual at least fourfold.
//
// Piece image of a K-long vector (K a multiple of 256): B part
// [K/256][8 rows][128 B] (row p = piece p, 128-byte swizzle, 1024 B per
// 256 columns), then scale part [K/128][8 lines][16 B] (bytes 0-3 of line p:
// piece p's scales of the 4 blocks of that 128-column atom).
#pragma once

#include "common.cuh"

namespace k3mx {

constexpr int kPieces = 8;
constexpr int kPieceChunk = 256;
__host__ __device__ constexpr int img_b(int K) { return K / kPieceChunk * 1024; }
__host__ __device__ constexpr int img_s(int K) { return K / 128 * 128; }
__host__ __device__ constexpr int img_bytes(int K) { return img_b(K) + img_s(K); }


// 2^k for -126 <= k <= 127
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// index of the e2m1 magnitude nearest to a in [0, 6]: 0, .5, 1, 1.5, 2, 3, 4, 6
__device__ __forceinline__ int e2m1_index(float a) {
    return (a >= 0.25f) + (a >= 0.75f) + (a >= 1.25f) + (a >= 1.75f) + (a >= 2.5f) + (a >= 3.5f) +
           (a >= 5.0f);
}
__device__ __forceinline__ float e2m1_mag(int i) {
    return i < 2 ? 0.5f * (float)i : __uint_as_float((uint32_t)(126 + (i >> 1)) << 23 | (uint32_t)(i & 1) << 22);
}
// bits 0-7 of x to bits 0, 4, ..., 28
__device__ __forceinline__ uint32_t spread_nibbles(uint32_t x) {
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    x = (x | (x << 3)) & 0x11111111u;
    return x;
}

// The 32 values of a warp (lane = column of one 32-column block) split
// into NP MXFP4 pieces.  Lane p < NP receives piece p: its 16 packed bytes
// (`words`, the low nibble of byte i is lane 2i's code) and its ue8m0 scale
// byte.  Whole warp.  ROLLED keeps the loop body short (few instruction
// fetches where the body runs once per launch); otherwise it is unrolled.
template <int NP, bool ROLLED>
__device__ __forceinline__ void split_pieces(float r, uint4 &words, uint32_t &scale) {
    const int lane = threadIdx.x & 31;
    uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0, msb = 0;
#pragma unroll(ROLLED ? 1 : NP)
    for (int p = 0; p < NP; p++) {
        // the block's largest residual magnitude (non-negative floats order
        // as their bit patterns)
        const uint32_t mb = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(r)));
        const int E = (int)(mb >> 23) - 127;
        int code = 0;
        uint32_t sb = 0;
        if (E == 128) {
            sb = 255;                                   // Inf or NaN in the block: NaN scale
        } else if (E >= -124) {
            const int e = (mb & 0x7FFFFFu) <= 0x400000u ? E - 2 : E - 1;   // max / 2^e in (3, 6]
            const int i = e2m1_index(fabsf(r) * exp2i(-e));
            const float v = e2m1_mag(i) * exp2i(e);
            code = i | ((r < 0.f && i != 0) ? 8 : 0);
            r -= copysignf(v, r);                       // exact
            sb = (uint32_t)(e + 127);
        }
        const uint32_t b0 = __ballot_sync(0xffffffffu, code & 1), b1 = __ballot_sync(0xffffffffu, code & 2);
        const uint32_t b2 = __ballot_sync(0xffffffffu, code & 4), b3 = __ballot_sync(0xffffffffu, code & 8);
        if (lane == p) {
            m0 = b0;
            m1 = b1;
            m2 = b2;
            m3 = b3;
            msb = sb;
        }
    }
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; q++)
        w[q] = spread_nibbles((m0 >> (8 * q)) & 0xFFu) | spread_nibbles((m1 >> (8 * q)) & 0xFFu) << 1 |
               spread_nibbles((m2 >> (8 * q)) & 0xFFu) << 2 | spread_nibbles((m3 >> (8 * q)) & 0xFFu) << 3;
    words = make_uint4(w[0], w[1], w[2], w[3]);
    scale = msb;
}

// The 32 values of a warp (lane = column of one 32-column block `kb` of a
// vector) as kPieces MXFP4 pieces, stored into the vector's piece image
// (B part `ib`, scale part `is`).  Whole warp.
__device__ __forceinline__ void store_pieces(float r, uint8_t *ib, uint8_t *is, int kb) {
    const int lane = threadIdx.x & 31;
    uint4 w;
    uint32_t sb;
    // rolled: the body runs in epilogues while the weight stream keeps
    // memory busy, and a short body keeps its first instruction fetches few
    split_pieces<kPieces, true>(r, w, sb);
    if (lane < kPieces) {
        *reinterpret_cast<uint4 *>(ib + (kb >> 3) * 1024 + lane * 128 + (((kb & 7) ^ lane) << 4)) = w;
        is[(kb >> 2) * 128 + lane * 16 + (kb & 3)] = (uint8_t)sb;
    }
}

// Warp `w` of the x-image work (one 32-column block of one token): x
// (fp32 or bf16 bits) -> that block of the token's piece image.
__device__ __forceinline__ void ximg_block(const void *__restrict__ x, int bf16, int n_tokens,
                                           uint8_t *__restrict__ img, int w) {
    constexpr int NB = kD / 32;
    const int lane = threadIdx.x & 31;
    if (w >= n_tokens * NB) return;
    const int t = w / NB, kb = w % NB;
    const size_t i = (size_t)t * kD + (size_t)kb * 32 + lane;
    const float v = bf16 ? __uint_as_float((uint32_t)static_cast<const uint16_t *>(x)[i] << 16)
                         : static_cast<const float *>(x)[i];
    uint8_t *ib = img + (size_t)t * img_bytes(kD);
    store_pieces(v, ib, ib + img_b(kD), kb);
}

}  // namespace k3mx
