// prefill.cu - grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators) for many tokens with bf16 activations.
//
// Every unique expert of the batch is loaded once for all the tokens routed
// to it (Kimi K3 engine (c/kimi_k3.c), "Chunked prefill").  Per expert the
// problem is swapped so that weight rows are the MMA's M (128 per tile) and
// the expert's tokens are N (up to 128 per unit, padded to a multiple of 16):
//   gate/up: G = W1 X^T, U = W3 X^T over K = 3584, h = SiTU(G, U) -> H (f16)
//   down:    Y = W2 H^T over K = 3072, y[t] += w_tk * Y (fp32 atomics)
//
// MXFP4 -> f16 in shared memory.  tcgen05 kind::f16 takes A and B of one
// type; the weights are dequantised to f16 and the activations are f16 too
// (x is converted once: a bf16 value is exact in f16 from 2^-14 to 65504;
// larger ones overflow and smaller ones lose bits, so this path takes
// activations in that range, and h below 2^-14 loses bits the same way).
// An e2m1 code is exact in f16 (cvt.rn.f16x2.e2m1x2);
// its group scale 2^(s - 127) is split into a per-row reference 2^(sref-127),
// sref the row's largest scale, applied to the fp32 accumulator in the
// epilogue, and 2^(s - sref) <= 1 multiplied into the f16 value (exact while
// s - sref >= -24; smaller groups, 2^24 below the row's largest, round).  In
// a row whose scales span more than 24 binades, sref is the largest scale of
// a group with a nonzero code (a group of zero codes adds nothing whatever
// its scale, so it does not push the row's other groups out of range).
//
// Warp roles in a persistent CTA (one per SM):
//   warps 0-7   dequant: global packed bytes -> registers (4 chunks ahead)
//               -> f16 -> 128-byte-swizzled A tile in shared memory
//   warps 8-11  epilogue: tcgen05.ld of the accumulators (warp 8+q reads
//               TMEM lanes 32q..32q+31), SiTU or weighted accumulate
//   warps 12-13 B loader: cp.async of the tokens' f16 rows, swizzled
//   warp 14     TMEM owner; lane 0 issues the MMAs and commits
// A stage holds one 64-column K chunk of A (and W3 for gate/up) and of B;
// "full" counts the dequant and loader arrivals, "empty" is committed by the
// MMA thread.  Two accumulator buffers let the epilogue of one tile overlap
// the MMAs of the next.  Every wait is bounded.
#include "prefill.cuh"

namespace k3mx {
namespace {

enum : int { kPhaseGateUp = 0, kPhaseDown = 1 };

constexpr int kUnitTokens = 128;        // tokens per prefill work unit (MMA N <= 128)
constexpr int kBM = 128;                // weight rows per tile (MMA M)
constexpr int kBK = 64;                 // K per stage: 64 f16 = one 128-byte row
constexpr int kTileBytes = kBM * 128;   // 16 KB: one swizzled 128 x 64 f16 tile
constexpr int kThreads = 15 * 32;
constexpr int kDeqThreads = 256;
constexpr int kEpiWarp0 = 8;
constexpr int kLoadWarp0 = 12;
constexpr int kLoadThreads = 64;
constexpr int kMmaWarp = 14;
constexpr int kPF = 4;                  // K chunks of packed bytes in flight per dequant thread

template <int PH> struct PhaseCfg;
template <> struct PhaseCfg<kPhaseGateUp> {
    static constexpr int NMAT = 2, K = kD, M = kF, STAGES = 4, TMEM_COLS = 512;
};
template <> struct PhaseCfg<kPhaseDown> {
    static constexpr int NMAT = 1, K = kF, M = kD, STAGES = 6, TMEM_COLS = 256;
};

struct PArgs {
    const k3mx_expert *experts;
    const int32_t *units, *n_units, *perm;
    const float *w;            // routing weights by pair
    const __half *xh;          // [T][D] f16 activations
    __half *H;                 // [16T][F] f16 h rows in grouped order
    float *y;                  // [T][D]
    int *status;
};

__device__ __forceinline__ __half2 pow2_h2(int k) {
    // 2^k as f16 for -24 <= k <= 0 (subnormal below -14); 0 below -24
    uint32_t b;
    if (k < -24) b = 0;
    else if (k < -14) b = 1u << (k + 24);
    else b = (uint32_t)(k + 15) << 10;
    b |= b << 16;
    return *reinterpret_cast<__half2 *>(&b);
}

// spread of the f16 dequantisation below the row's reference scale
constexpr int kRefSpan = 24;

// a group of 16 packed bytes holds a nonzero code (codes 0 and 8 are +-0)
__device__ __forceinline__ bool group_nonzero(const uint8_t *g16) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(g16));
    return ((v.x | v.y | v.z | v.w) & 0x77777777u) != 0;
}

// The reference scale byte of a weight row (srow: its G scale bytes, prow:
// its packed bytes): the largest non-NaN scale, or, when the non-NaN scales
// span more than kRefSpan binades, the largest scale of a group with a
// nonzero code; 127 when no group qualifies.  One thread.
__device__ __forceinline__ int row_sref(const uint8_t *srow, const uint8_t *prow, int ngroups) {
    int mx = -1, mn = 256;
    for (int i = 0; i < ngroups; i += 16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(srow + i));
        const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; q++)
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int b = (ws[q] >> (8 * k)) & 0xFF;
                if (b != 255) {
                    mx = max(mx, b);
                    mn = min(mn, b);
                }
            }
    }
    if (mx - mn > kRefSpan) {
        mx = -1;
        for (int g = 0; g < ngroups; g++) {
            const int b = srow[g];
            if (b != 255 && b > mx && group_nonzero(prow + 16 * g)) mx = b;
        }
    }
    return mx < 0 ? 127 : mx;
}

struct SmemHeader {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t accf[2];
    uint64_t acce[2];
    uint64_t done;
    uint32_t tmem_base;
    int abort_flag;
};

template <int PH>
__global__ void __launch_bounds__(kThreads, 1) k_prefill(PArgs a) {
    using C = PhaseCfg<PH>;
    constexpr int NMAT = C::NMAT, K = C::K, M = C::M, S = C::STAGES;
    constexpr int KC = K / kBK;                     // K chunks per tile
    constexpr int MT = M / kBM;                     // row tiles per unit
    constexpr int G = K / 32;                       // scale groups per row
    constexpr uint32_t ROWB = K / 2;                // packed bytes per row
    constexpr uint32_t STAGE = (NMAT + 1) * kTileBytes;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SmemHeader *hd = reinterpret_cast<SmemHeader *>(smem);
    uint8_t *stage0 = smem + 1024;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const uint32_t full0 = smem_addr(hd->full), empty0 = smem_addr(hd->empty);
    const uint32_t accf0 = smem_addr(hd->accf), acce0 = smem_addr(hd->acce);

    if (tid == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(full0 + 8 * i, kDeqThreads + kLoadThreads);
            mbar_init(empty0 + 8 * i, 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(accf0 + 8 * i, 1);
            mbar_init(acce0 + 8 * i, 128);
        }
        mbar_init(smem_addr(&hd->done), 1);
        hd->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(smem_addr(&hd->tmem_base), C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = hd->tmem_base;
    volatile int *abort_flag = &hd->abort_flag;

    const int n_units = *a.n_units;
    const long long total = (long long)n_units * MT;
    const long long beg = total * blockIdx.x / gridDim.x;
    const long long end = total * (blockIdx.x + 1) / gridDim.x;

    if (warp < kEpiWarp0) {
        // ------------------------------------------------------ dequant --
        // Lanes 2i and 2i+1 take the two 16-byte halves (one 32-column
        // group each) of a row's 32 packed bytes per chunk, so a warp reads
        // 16 rows x 32 contiguous bytes.  Gate/up: threads 0-127 take W1 and
        // 128-255 W3, each thread two rows (r and r + 64); down: each thread
        // one row of W2.
        constexpr int RPT = NMAT;                      // rows per thread
        const int half = tid & 1;
        const int mat = NMAT == 2 ? (tid >> 7) : 0;
        const int rb = NMAT == 2 ? ((tid & 127) >> 1) : (tid >> 1);
        long long c = 0;                               // stage-use counter
        for (long long item = beg; item < end && !*abort_flag; item++) {
            const int unit = (int)(item / MT), mt = (int)(item % MT);
            const int e = a.units[3 * unit];
            const k3mx_expert ex = a.experts[e];
            const uint8_t *W = (PH == kPhaseGateUp) ? (mat ? ex.w3 : ex.w1) : ex.w2;
            const uint8_t *Sc = (PH == kPhaseGateUp) ? (mat ? ex.s3 : ex.s1) : ex.s2;
            if (((reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(Sc)) & 15u) != 0) {
                report_status(a.status, kStatusBadPointer, e);
                *abort_flag = 1;
                break;
            }
            const uint8_t *rowp[RPT];
            const uint8_t *srow[RPT];
            int sref[RPT];
#pragma unroll
            for (int i = 0; i < RPT; i++) {
                const int row = mt * kBM + rb + 64 * i;
                rowp[i] = W + (size_t)row * ROWB + 16 * half;
                srow[i] = Sc + (size_t)row * G;
                // the row's reference scale (row_sref): the lane pair scans
                // alternate 16-byte blocks of the row's G scale bytes
                int mx = -1, mn = 256;
                for (int blk = half; blk < G / 16; blk += 2) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(srow[i] + 16 * blk));
                    const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; q++)
#pragma unroll
                        for (int k = 0; k < 4; k++) {
                            const int bb = (ws[q] >> (8 * k)) & 0xFF;
                            if (bb != 255) {
                                mx = max(mx, bb);
                                mn = min(mn, bb);
                            }
                        }
                }
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
                if (mx - mn > kRefSpan) {
                    // a wide row (rare): the largest scale of a group with a
                    // nonzero code, the pair taking alternate groups
                    const unsigned pair = 3u << (lane & 30);
                    int m2 = -1;
                    const uint8_t *prow = W + (size_t)row * ROWB;
                    for (int gq = half; gq < G; gq += 2) {
                        const int b = srow[i][gq];
                        if (b != 255 && b > m2 && group_nonzero(prow + 16 * gq)) m2 = b;
                    }
                    mx = max(m2, __shfl_xor_sync(pair, m2, 1));
                }
                sref[i] = mx < 0 ? 127 : mx;
            }
            // packed bytes and the group's scale byte, kPF chunks ahead
            uint4 raw[kPF][RPT];
            uint32_t scb[kPF][RPT];
#pragma unroll
            for (int j = 0; j < kPF; j++)
#pragma unroll
                for (int i = 0; i < RPT; i++) {
                    raw[j][i] = ldg_stream(rowp[i] + (size_t)j * 32);
                    scb[j][i] = __ldg(srow[i] + 2 * j + half);
                }
            bool stop = false;
            for (int kc0 = 0; kc0 < KC && !stop; kc0 += kPF) {
#pragma unroll
                for (int j = 0; j < kPF; j++) {
                    const int kc = kc0 + j;
                    const int s = (int)(c % S);
                    const long long rnd = c / S;
                    if (*abort_flag) {
                        stop = true;
                        break;
                    }
                    if (rnd > 0 && !mbar_wait(empty0 + 8 * s, (uint32_t)((rnd - 1) & 1))) {
                        report_status(a.status, kStatusWaitTimeout, 200 + PH);
                        *abort_flag = 1;
                        stop = true;
                        break;
                    }
                    uint8_t *tile = stage0 + (size_t)s * STAGE + mat * kTileBytes;
#pragma unroll
                    for (int i = 0; i < RPT; i++) {
                        const int r = rb + 64 * i;
                        const int sb = (int)scb[j][i];
                        const __half2 m = sb == 255 ? pow2_h2(-100) : pow2_h2(sb - sref[i]);
                        const uint32_t words[4] = {raw[j][i].x, raw[j][i].y, raw[j][i].z, raw[j][i].w};
#pragma unroll
                        for (int wd = 0; wd < 4; wd++) {
                            uint32_t hv[4];
                            e2m1x8_to_h2x4(words[wd], hv);
                            uint32_t o[4];
#pragma unroll
                            for (int bq = 0; bq < 4; bq++) {
                                __half2 v = __hmul2(*reinterpret_cast<__half2 *>(&hv[bq]), m);
                                o[bq] = *reinterpret_cast<uint32_t *>(&v);
                            }
                            *reinterpret_cast<uint4 *>(tile + sw128_offset(r, 4 * half + wd)) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                        }
                        // refill this slot with the chunk kPF ahead
                        if (kc + kPF < KC) {
                            raw[j][i] = ldg_stream(rowp[i] + (size_t)(kc + kPF) * 32);
                            scb[j][i] = __ldg(srow[i] + 2 * (kc + kPF) + half);
                        }
                    }
                    fence_async_smem();
                    mbar_arrive(full0 + 8 * s);
                    c++;
                }
            }
        }
    } else if (warp < kLoadWarp0) {
        // ----------------------------------------------------- epilogue --
        const int q = warp - kEpiWarp0;                // TMEM lane quarter
        const int r = 32 * q + lane;                   // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        long long it = 0;
        for (long long item = beg; item < end; item++, it++) {
            const int unit = (int)(item / MT), mt = (int)(item % MT);
            const int e = a.units[3 * unit], off = a.units[3 * unit + 1], ntok = a.units[3 * unit + 2];
            const int npad = (ntok + 15) & ~15;
            const int ab = (int)(it & 1);
            if (*abort_flag) break;
            if (!mbar_wait(accf0 + 8 * ab, (uint32_t)((it >> 1) & 1))) {
                report_status(a.status, kStatusWaitTimeout, 210 + PH);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const k3mx_expert ex = a.experts[e];
            const int row = mt * kBM + r;
            if (PH == kPhaseGateUp) {
                const float f1 = ldexpf(1.f, row_sref(ex.s1 + (size_t)row * G, ex.w1 + (size_t)row * (K / 2), G) - 127);
                const float f3 = ldexpf(1.f, row_sref(ex.s3 + (size_t)row * G, ex.w3 + (size_t)row * (K / 2), G) - 127);
                const uint32_t tg = tmem + lane_base + (uint32_t)(ab * 256);
                for (int n0 = 0; n0 < npad; n0 += 16) {
                    uint32_t gv[16], uv[16];
                    tmem_ld16(tg + n0, gv);
                    tmem_ld16(tg + 128 + n0, uv);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const int n = n0 + j;
                        if (n < ntok) {
                            const float h = situ_glu(__uint_as_float(gv[j]) * f1, __uint_as_float(uv[j]) * f3);
                            a.H[(size_t)(off + n) * kF + row] = __float2half_rn(h);
                        }
                    }
                }
            } else {
                const float f2 = ldexpf(1.f, row_sref(ex.s2 + (size_t)row * G, ex.w2 + (size_t)row * (K / 2), G) - 127);
                const uint32_t td = tmem + lane_base + (uint32_t)(ab * 128);
                for (int n0 = 0; n0 < npad; n0 += 16) {
                    // the group's pairs and routing weights: lane j < 16
                    // loads token n0 + j's (one round trip for the group),
                    // shared by shuffles
                    int pj = 0;
                    float wj = 0.f;
                    if (lane < 16 && n0 + lane < ntok) {
                        pj = a.perm[off + n0 + lane];
                        wj = __ldg(a.w + pj);
                    }
                    uint32_t dv[16];
                    tmem_ld16(td + n0, dv);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const int p = __shfl_sync(0xffffffffu, pj, j);
                        const float wt = __shfl_sync(0xffffffffu, wj, j);
                        if (n0 + j < ntok) atomicAdd(a.y + (size_t)(p / kK) * kD + row, wt * __uint_as_float(dv[j]) * f2);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acce0 + 8 * ab);
        }
    } else if (warp < kMmaWarp) {
        // ---------------------------------------------------- B loader --
        const int lt = tid - 32 * kLoadWarp0;          // 0..63
        const int j = lt & 7;                          // 16-byte chunk of a 128-byte row
        const int nb = lt >> 3;                        // rows nb, nb + 8, ...
        long long c = 0;
        for (long long item = beg; item < end && !*abort_flag; item++) {
            const int unit = (int)(item / MT);
            const int off = a.units[3 * unit + 1], ntok = a.units[3 * unit + 2];
            const int npad = (ntok + 15) & ~15;
            const __half *src[kUnitTokens / 8];
#pragma unroll
            for (int k = 0; k < kUnitTokens / 8; k++) {
                const int n = nb + 8 * k;
                const int nn = n < ntok ? n : 0;
                if (PH == kPhaseGateUp) src[k] = a.xh + (size_t)(a.perm[off + nn] / kK) * kD;
                else src[k] = a.H + (size_t)(off + nn) * kF;
            }
            for (int kc = 0; kc < KC && !*abort_flag; kc++, c++) {
                const int s = (int)(c % S);
                const long long rnd = c / S;
                if (rnd > 0 && !mbar_wait(empty0 + 8 * s, (uint32_t)((rnd - 1) & 1))) {
                    report_status(a.status, kStatusWaitTimeout, 220 + PH);
                    *abort_flag = 1;
                    break;
                }
                const uint32_t btile = smem_addr(stage0 + (size_t)s * STAGE + NMAT * kTileBytes);
#pragma unroll
                for (int k = 0; k < kUnitTokens / 8; k++) {
                    const int n = nb + 8 * k;
                    if (n < npad)
                        cp_async16(btile + sw128_offset(n, j), src[k] + kc * kBK + 8 * j, n < ntok ? 16u : 0u);
                }
                cp_async_arrive(full0 + 8 * s);
            }
        }
        cp_async_wait_all();
    } else {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            long long c = 0, it = 0;
            for (long long item = beg; item < end && !*abort_flag; item++, it++) {
                const int unit = (int)(item / MT);
                const int ntok = a.units[3 * unit + 2];
                const int npad = (ntok + 15) & ~15;
                const uint32_t idesc = umma_idesc_f16(kBM, npad);
                const int ab = (int)(it & 1);
                if (it >= 2 && !mbar_wait(acce0 + 8 * ab, (uint32_t)(((it >> 1) - 1) & 1))) {
                    report_status(a.status, kStatusWaitTimeout, 230 + PH);
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem + (uint32_t)(ab * (PH == kPhaseGateUp ? 256 : 128));
                for (int kc = 0; kc < KC; kc++, c++) {
                    const int s = (int)(c % S);
                    if (*abort_flag) break;
                    if (!mbar_wait(full0 + 8 * s, (uint32_t)((c / S) & 1))) {
                        report_status(a.status, kStatusWaitTimeout, 240 + PH);
                        *abort_flag = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_addr(stage0 + (size_t)s * STAGE);
#pragma unroll
                    for (int k16 = 0; k16 < kBK / 16; k16++) {
                        const uint64_t bdesc = umma_desc_sw128(st + NMAT * kTileBytes + 32 * k16);
                        const uint32_t acc = (kc | k16) != 0;
                        umma_f16(d0, umma_desc_sw128(st + 32 * k16), bdesc, idesc, acc);
                        if (NMAT == 2)
                            umma_f16(d0 + 128, umma_desc_sw128(st + kTileBytes + 32 * k16), bdesc, idesc, acc);
                    }
                    umma_commit(empty0 + 8 * s);          // stage free once these MMAs finish
                }
                umma_commit(accf0 + 8 * ab);              // accumulators of this tile ready
            }
            // every MMA issued so far has completed before TMEM is released
            umma_commit(smem_addr(&hd->done));
            if (!mbar_wait_drain(smem_addr(&hd->done), 0)) report_status(a.status, kStatusWaitTimeout, 250 + PH);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// x (bf16 bits) -> f16 activations; y = 0
__global__ void k_prefill_prep(__half *xh, float *y, const uint16_t *x, size_t n) {
    const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i + 3 < n) {
        const uint2 v = *reinterpret_cast<const uint2 *>(x + i);
        const float f0 = __uint_as_float(v.x << 16), f1 = __uint_as_float(v.x & 0xFFFF0000u);
        const float f2 = __uint_as_float(v.y << 16), f3 = __uint_as_float(v.y & 0xFFFF0000u);
        __half2 h01 = __floats2half2_rn(f0, f1), h23 = __floats2half2_rn(f2, f3);
        *reinterpret_cast<uint2 *>(xh + i) =
            make_uint2(*reinterpret_cast<uint32_t *>(&h01), *reinterpret_cast<uint32_t *>(&h23));
        *reinterpret_cast<float4 *>(y + i) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Work units: every active expert's pair list cut into runs of at most 128
// pairs; one 1024-thread CTA, expert e handled by thread e.
__global__ void __launch_bounds__(1024) k_prefill_units(const int32_t *counts, const int32_t *offsets,
                                                        int32_t *units, int32_t *n_units) {
    __shared__ int tmp[33];
    const int e = threadIdx.x, lane = e % 32, wp = e / 32;
    const int cnt = e < kE ? counts[e] : 0;
    const int nu = (cnt + kUnitTokens - 1) / kUnitTokens;
    int incl = nu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) tmp[wp] = incl;
    __syncthreads();
    if (wp == 0) {
        const int ws = tmp[lane];
        int wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += v;
        }
        tmp[lane] = wi - ws;
        if (lane == 31) tmp[32] = wi;
    }
    __syncthreads();
    int pos = incl - nu + tmp[wp];
    if (e < kE) {
        const int o0 = offsets[e];
        for (int q = 0; q < cnt; q += kUnitTokens, pos++) {
            units[3 * pos + 0] = e;
            units[3 * pos + 1] = o0 + q;
            units[3 * pos + 2] = min(kUnitTokens, cnt - q);
        }
    }
    if (e == 0) *n_units = tmp[32];
}

template <int PH>
size_t prefill_smem() {
    return 1024 + 1024 + (size_t)PhaseCfg<PH>::STAGES * (PhaseCfg<PH>::NMAT + 1) * kTileBytes;
}

template <int PH>
cudaError_t launch_phase(const Ctx &c, const PArgs &a, long long max_items) {
    const size_t smem = prefill_smem<PH>();
    static std::atomic<uint64_t> configured{0};
    const cudaError_t e = ensure_smem((const void *)k_prefill<PH>, (int)smem, configured);
    if (e != cudaSuccess) return e;
    long long grid = c.num_sms;
    if (grid > max_items) grid = max_items;
    k_prefill<PH><<<(unsigned)grid, kThreads, smem, c.stream>>>(a);
    return cudaGetLastError();
}

inline size_t up256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace

cudaError_t set_wait_polls_prefill(uint32_t polls) { return set_wait_polls_here(polls); }

int prefill_max_units(int n_tokens) {
    const int pairs = n_tokens * kK;
    return pairs / kUnitTokens + (pairs < kE ? pairs : kE);
}

size_t prefill_scratch_bytes(int n_tokens) {
    const size_t T = n_tokens;
    return up256(T * kD * 2) + up256(T * kK * kF * 2) + up256((size_t)prefill_max_units(n_tokens) * 3 * 4) + 256;
}

cudaError_t launch_prefill(const Ctx &c, const PrefillArgs &p) {
    const size_t T = p.n_tokens;
    char *ws = static_cast<char *>(p.scratch);
    __half *xh = reinterpret_cast<__half *>(ws);
    __half *H = reinterpret_cast<__half *>(ws + up256(T * kD * 2));
    int32_t *units = reinterpret_cast<int32_t *>(ws + up256(T * kD * 2) + up256(T * kK * kF * 2));
    int32_t *n_units = units + up256((size_t)prefill_max_units(p.n_tokens) * 3 * 4) / 4;

    const size_t n = T * kD;
    cudaError_t err = traced("prefill_prep", c.stream, [&] {
        k_prefill_prep<<<(unsigned)((n / 4 + 255) / 256), 256, 0, c.stream>>>(xh, p.y, p.x, n);
        k_prefill_units<<<1, 1024, 0, c.stream>>>(p.counts, p.offsets, units, n_units);
        return cudaGetLastError();
    });
    if (err != cudaSuccess) return err;

    PArgs a{};
    a.experts = p.experts;
    a.units = units;
    a.n_units = n_units;
    a.perm = p.perm;
    a.w = p.w;
    a.xh = xh;
    a.H = H;
    a.y = p.y;
    a.status = c.status;
    const long long mu = prefill_max_units(p.n_tokens);
    err = traced("prefill_gate_up", c.stream, [&] { return launch_phase<kPhaseGateUp>(c, a, mu * (kF / kBM)); });
    if (err == cudaSuccess)
        err = traced("prefill_down", c.stream, [&] { return launch_phase<kPhaseDown>(c, a, mu * (kD / kBM)); });
    return err;
}

}  // namespace k3mx
