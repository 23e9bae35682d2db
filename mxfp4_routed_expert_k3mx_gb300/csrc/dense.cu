// dense.cu - the bf16 matrix products of the Stable LatentMoE block around
// the routed experts (Kimi K3 engine (c/kimi_k3.c), "Architecture notes":
// the sigmoid router [896, 7168] over the hidden state, the projections
// 7168 -> 3584 into the experts' latent and 3584 -> 7168 back, and the two
// fused full-width shared experts, inter 6144; the trunk is bf16):
//   y[t][col0 + r] = sum_c W[r][c] xin[t][c]  (+ add[t][col0 + r])
// with xin the input as given, SiTU-GLU of a (g | u) pair of rows, the
// RMSNorm of the input times its weight, or (the block's output product)
// both side by side against W_up's and W2s's rows side by side.  Every product of a bf16 weight
// and an fp32 value is exact in fp32; the sums are fp32.
//
// Few tokens, or fp32 inputs: k_gemv, persistent CTAs streaming their rows
// through a ring of bulk copies, one warp per row; HBM-bound on the weights.  Many bf16
// inputs: k_gemm on the tcgen05 tensor cores (kind::f16 with bf16 A and B,
// fp32 accumulators in TMEM); a CTA computes 128 weight rows x 256 tokens
// over the whole sum, its operands streamed by TMA (128-byte swizzle)
// through a 4-stage ring.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "dense.cuh"
#include "tmaps.cuh"

namespace k3mx {
namespace {

constexpr int kGemvTok = 3;                      // inputs per shared-memory chunk
constexpr int kGemvWarps = 8;                    // consumer warps, one weight row each at a time
constexpr int kGemvThreads = (kGemvWarps + 1) * 32;   // + the producer warp
constexpr int kGemvMaxSlots = 16;
constexpr float kRmsEps = 1e-5f;                 // K3Cfg rms_eps

template <int K>
struct GemvShape {
    static constexpr int VEC = K / 8;            // 16-byte vectors per row
    static constexpr int VPL = VEC / 32;         // per lane
    static constexpr int ROWB = K * 2;
    static constexpr int HDR = 2048;             // barriers and partial sums
    static constexpr int SMEM_MAX = 227 * 1024;
    // inputs per chunk (1..3) and row slots: the chunk takes what it needs,
    // the ring the rest (fewer inputs, more rows in flight)
    static constexpr int slots(int chunk) {
        const int fit = (SMEM_MAX - 1024 - HDR - chunk * K * 4) / ROWB;
        return fit > kGemvMaxSlots ? kGemvMaxSlots : fit;
    }
    static constexpr int smem(int chunk) { return 1024 + HDR + chunk * K * 4 + slots(chunk) * ROWB; }
    static_assert(VEC % 32 == 0 && slots(kGemvTok) >= 4, "row length");
    static_assert(smem(kGemvTok) <= SMEM_MAX && smem(1) <= SMEM_MAX, "shared memory budget");
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// four consecutive input values c4*4 .. c4*4+3 of token row `t`
template <int K, int XF>
__device__ __forceinline__ float4 input4(const GemvArgs &a, int t, int c4, float scale) {
    if (XF == kXfLatentOut && c4 >= kLatentOutK1 / 4) {
        constexpr int K2 = K - kLatentOutK1;
        const float *row = a.x2 + (size_t)t * a.ldx2;
        const float4 g = reinterpret_cast<const float4 *>(row)[c4 - kLatentOutK1 / 4];
        const float4 u = reinterpret_cast<const float4 *>(row + K2)[c4 - kLatentOutK1 / 4];
        return make_float4(situ_glu(g.x, u.x), situ_glu(g.y, u.y), situ_glu(g.z, u.z), situ_glu(g.w, u.w));
    }
    if (XF == kXfSitu) {
        const float *row = static_cast<const float *>(a.x) + (size_t)t * a.ldx;
        const float4 g = reinterpret_cast<const float4 *>(row)[c4];
        const float4 u = reinterpret_cast<const float4 *>(row + K)[c4];
        return make_float4(situ_glu(g.x, u.x), situ_glu(g.y, u.y), situ_glu(g.z, u.z), situ_glu(g.w, u.w));
    }
    float4 v;
    if (a.x_bf16) {
        const uint2 q = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.x) + (size_t)t * a.ldx)[c4];
        v = make_float4(bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y));
    } else {
        v = reinterpret_cast<const float4 *>(static_cast<const float *>(a.x) + (size_t)t * a.ldx)[c4];
    }
    if (XF == kXfRmsNorm || XF == kXfLatentOut) {
        const uint2 q = reinterpret_cast<const uint2 *>(a.g)[c4];
        v = make_float4(v.x * scale * bf16_lo(q.x), v.y * scale * bf16_hi(q.x), v.z * scale * bf16_lo(q.y),
                        v.w * scale * bf16_hi(q.y));
    }
    return v;
}

// The weight row of product row gr (the segments are in row order, the
// first at row 0)
template <int K>
__device__ __forceinline__ const uint16_t *row_weights(const GemvArgs &a, int gr) {
    const uint16_t *w = a.seg[0].W + (size_t)gr * K;
#pragma unroll
    for (int k = 1; k < kGemvMaxSeg; k++)
        if (k < a.n_seg && gr >= a.seg[k].r0) w = a.seg[k].W + (size_t)(gr - a.seg[k].r0) * K;
    return w;
}

// Where product row gr of input t goes, and its addend (or null)
__device__ __forceinline__ float *row_out(const GemvArgs &a, int gr, int t, const float *&add) {
    size_t o = (size_t)t * a.seg[0].ldy + gr;
    float *y = a.seg[0].y + o;
    add = a.seg[0].add != nullptr ? a.seg[0].add + o : nullptr;
#pragma unroll
    for (int k = 1; k < kGemvMaxSeg; k++)
        if (k < a.n_seg && gr >= a.seg[k].r0) {
            o = (size_t)t * a.seg[k].ldy + (gr - a.seg[k].r0);
            y = a.seg[k].y + o;
            add = a.seg[k].add != nullptr ? a.seg[k].add + o : nullptr;
        }
    return y;
}

// Persistent, one CTA per SM over a contiguous range of weight rows.  The
// inputs (3 at a time) are staged in shared memory first, laid out so that
// lanes read consecutive 16-byte words (columns 8v..8v+3 at slot v,
// 8v+4..8v+7 at slot K/8 + v, vector v = lane + 32 i); then a producer warp
// streams the range's rows by bulk copies through a ring of up to 16 row
// slots while 8 consumer warps take one row each at a time.  Per lane, a
// vector's 8 products are two 4-term sums added, the vectors go to four
// running sums added pairwise, and the warp adds its lanes (about 20 fp32
// roundings deep at K = 7168).  RMSNorm inputs first reduce each token's
// sum of squares over the CTA.
template <int K, int XF>
__global__ void __launch_bounds__(kGemvThreads, 1) k_gemv(const GemvArgs a) {
    using Sh = GemvShape<K>;
    constexpr int VEC = Sh::VEC, VPL = Sh::VPL;
    const int chunk = min(kGemvTok, a.n_tokens);  // inputs staged at a time
    const int SLOTS = Sh::slots(chunk);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t full0 = smem_addr(smem), empty0 = full0 + 8 * kGemvMaxSlots;
    float *red = reinterpret_cast<float *>(smem + 16 * kGemvMaxSlots);   // [kGemvTok][kGemvWarps + 1]
    // the row each ring slot holds, set by the producer before the row's
    // copies: a consumer waits for its row's number first, so that its
    // parity wait is never two phases ahead of the slot (the consumer
    // warps take rows round robin, and the ring may hold fewer slots than
    // there are consumers)
    volatile int *seq = reinterpret_cast<volatile int *>(smem + 512);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 640);   // a wait gave up
    float4 *hs = reinterpret_cast<float4 *>(smem + Sh::HDR);             // [chunk][2 VEC]
    const int stage_b = chunk * K * 4;
    const uint32_t ring = smem_addr(smem) + Sh::HDR + stage_b;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int NW = kGemvWarps + 1;
    const int G = gridDim.x, b = blockIdx.x;
    const int rb = (int)((long long)a.rows * b / G), nr = (int)((long long)a.rows * (b + 1) / G) - rb;
    const int prefilled = min(nr, SLOTS);         // rows whose copies go out before anything else
    // a row's copies into ring slot `dst`: one bulk copy, or the two parts
    // of an output-product row
    auto issue_row = [&](int i, uint32_t dst, uint32_t bar, uint64_t pol) {
        mbar_arrive_expect_tx(bar, Sh::ROWB);
        if (XF == kXfLatentOut) {
            constexpr int K2 = K - kLatentOutK1;
            const size_t gr = (size_t)(rb + i);
            bulk_g2s(dst, a.seg[0].W + gr * kLatentOutK1, kLatentOutK1 * 2, bar, pol);
            bulk_g2s(dst + kLatentOutK1 * 2, a.Wt + gr * K2, K2 * 2, bar, pol);
        } else {
            bulk_g2s(dst, row_weights<K>(a, rb + i), Sh::ROWB, bar, pol);
        }
    };
    if (threadIdx.x == 0) {
        for (int i = 0; i < SLOTS; i++) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        // the weights are the call's own: the ring fills while the kernel
        // before finishes and the inputs are staged
        const uint64_t pol = l2_evict_first_policy();
        for (int i = prefilled; i < kGemvMaxSlots; i++) seq[i] = -1;
        for (int i = 0; i < prefilled; i++) {
            seq[i] = i;
            issue_row(i, ring + i * Sh::ROWB, full0 + 8 * i, pol);
        }
    }
    // the kernel behind may start its prologue
    pdl_launch_dependents();
    pdl_wait();                                   // the inputs, if a kernel before writes them
    int gbase = 0;                                // rows this CTA streamed in earlier chunks
    int g_next = prefilled;                       // producer: rows whose copies went out
    for (int t0 = 0; t0 < a.n_tokens; t0 += chunk, gbase += nr) {
        const int nt = min(chunk, a.n_tokens - t0);
        __syncthreads();                          // barriers set up; the previous chunk is consumed
        float scale[kGemvTok] = {1.f, 1.f, 1.f};
        // the normalised part's length
        constexpr int KN = XF == kXfLatentOut ? kLatentOutK1 : K;
        if (XF == kXfRmsNorm || XF == kXfLatentOut) {
            for (int j = 0; j < nt; j++) {
                const float *row = static_cast<const float *>(a.x) + (size_t)(t0 + j) * a.ldx;
                float ss = 0.f;
                for (int c4 = threadIdx.x; c4 < KN / 4; c4 += blockDim.x) {
                    const float4 v = reinterpret_cast<const float4 *>(row)[c4];
                    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                if (lane == 0) red[j * NW + warp] = ss;
            }
            __syncthreads();
            for (int j = 0; j < nt; j++) {
                float ss = 0.f;
                for (int w = 0; w < NW; w++) ss += red[j * NW + w];
                scale[j] = 1.0f / sqrtf(ss / (float)KN + kRmsEps);
            }
        }
        // 8 loads in flight per thread before the stores
        const int n4 = nt * (K / 4);
        for (int i0 = threadIdx.x; i0 < n4; i0 += 8 * (int)blockDim.x) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int i = i0 + u * (int)blockDim.x;
                if (i < n4) {
                    const int t = i / (K / 4), c4 = i % (K / 4);
                    const float sc = t == 0 ? scale[0] : (t == 1 ? scale[1] : scale[2]);
                    v[u] = input4<K, XF>(a, t0 + t, c4, sc);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int i = i0 + u * (int)blockDim.x;
                if (i < n4) {
                    const int t = i / (K / 4), c4 = i % (K / 4);
                    hs[t * (2 * VEC) + (c4 & 1) * VEC + (c4 >> 1)] = v[u];
                }
            }
        }
        __syncthreads();
        if (warp == kGemvWarps) {
            // ---------------------------------------------------- producer --
            if (lane == 0) {
                const uint64_t pol = l2_evict_first_policy();
                for (int i = gbase == 0 ? prefilled : 0; i < nr && !*abort_flag; i++) {
                    const int g = gbase + i, s = g % SLOTS;
                    if (g >= SLOTS && !mbar_wait(empty0 + 8 * s, ((g / SLOTS) - 1) & 1)) {
                        report_status(a.status, kStatusWaitTimeout, 311);
                        *abort_flag = 1;
                        break;
                    }
                    seq[s] = g;
                    issue_row(i, ring + s * Sh::ROWB, full0 + 8 * s, pol);
                    g_next = g + 1;
                }
            }
            continue;
        }
        // ------------------------------------------------------ consumers --
        for (int i = warp; i < nr && !*abort_flag; i += kGemvWarps) {
            const int g = gbase + i, s = g % SLOTS;
            // the slot carries this row once the producer has claimed it for
            // the row (polls back off like an mbarrier wait's suspend)
            bool ok = true;
            const uint32_t lim = wait_polls();
            for (uint32_t n = 0; seq[s] != g; n++) {
                if (n >= lim) {
                    ok = false;
                    break;
                }
                __nanosleep(256);
            }
            ok = ok && mbar_wait(full0 + 8 * s, (g / SLOTS) & 1);
            if (!ok) {
                // give up on this row and the rest: reading the slot or
                // arriving on its barrier would advance a phase that belongs
                // to another row
                if (lane == 0) {
                    report_status(a.status, kStatusWaitTimeout, 310);
                    *abort_flag = 1;
                }
                break;
            }
            const uint4 *wr = reinterpret_cast<const uint4 *>(smem + Sh::HDR + stage_b + s * Sh::ROWB);
            // four independent running sums per input (vectors i mod 4),
            // each vector's 8 products as two 4-term chains
            float acc[kGemvTok][4];
#pragma unroll
            for (int j = 0; j < kGemvTok; j++)
#pragma unroll
                for (int r = 0; r < 4; r++) acc[j][r] = 0.f;
#pragma unroll 2
            for (int v0 = 0; v0 < VPL; v0 += 4)
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    const int vi = v0 + r;
                    if (vi >= VPL) break;
                    const int v = lane + 32 * vi;
                    const uint4 q = wr[v];
                    const float w0 = bf16_lo(q.x), w1 = bf16_hi(q.x), w2 = bf16_lo(q.y), w3 = bf16_hi(q.y);
                    const float w4 = bf16_lo(q.z), w5 = bf16_hi(q.z), w6 = bf16_lo(q.w), w7 = bf16_hi(q.w);
#pragma unroll
                    for (int j = 0; j < kGemvTok; j++) {
                        if (j < nt) {
                            const float4 x0 = hs[j * (2 * VEC) + v], x1 = hs[j * (2 * VEC) + VEC + v];
                            float s0 = w0 * x0.x, s1 = w4 * x1.x;
                            s0 = fmaf(w1, x0.y, s0);
                            s1 = fmaf(w5, x1.y, s1);
                            s0 = fmaf(w2, x0.z, s0);
                            s1 = fmaf(w6, x1.z, s1);
                            s0 = fmaf(w3, x0.w, s0);
                            s1 = fmaf(w7, x1.w, s1);
                            acc[j][r] += s0 + s1;
                        }
                    }
                }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);      // the slot's row is read
#pragma unroll
            for (int j = 0; j < kGemvTok; j++) {
                float sum = (acc[j][0] + acc[j][1]) + (acc[j][2] + acc[j][3]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                if (lane == 0 && j < nt) {
                    const float *ad;
                    float *o = row_out(a, rb + i, t0 + j, ad);
                    if (ad != nullptr) sum += *ad;
                    *o = sum;
                }
            }
        }
    }
    // after a wait gave up, the ring's copies still in flight land before
    // the CTA leaves (the last row issued into each slot)
    __syncthreads();
    if (warp == kGemvWarps && lane == 0 && *abort_flag)
        for (int sl = 0; sl < SLOTS && sl < g_next; sl++) {
            const int gl = sl + SLOTS * ((g_next - 1 - sl) / SLOTS);
            mbar_wait_drain(full0 + 8 * sl, (gl / SLOTS) & 1);
        }
}

// ----------------------------------------------------- tensor-core GEMM --

constexpr int kGM = 128, kGN = 256, kGK = 64;    // tile: weight rows x tokens x K per stage
constexpr int kGStages = 4;
constexpr int kGABytes = kGM * kGK * 2, kGBBytes = kGN * kGK * 2;
constexpr int kGStage = kGABytes + kGBBytes;
constexpr int kGThreads = 192;                   // warp 0 TMA, 1 MMA, 2-5 epilogue
constexpr int kGSmem = 1024 + 1024 + kGStages * kGStage;

struct GHdr {
    uint64_t full[kGStages], empty[kGStages], accf;
    uint32_t tmem;
};

struct GemmOut {
    float *y;
    uint16_t *y_bf16;
    int ldy, col0;
    const float *add;
    int n_tokens;
    int *status;
    // rows from m_split on come from the second weight map and go to
    // columns col1 + (row - m_split) (two matrices over one input in a
    // launch; m_split = all rows for one matrix)
    int m_split, col1;
};

// bf16 A and B, f32 accumulator, both K-major, M x N
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tma_2d_plain(uint32_t dst, const void *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    const uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40u);   // NaN stays NaN
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

template <int K, bool ADD>
__global__ void __launch_bounds__(kGThreads, 1)
    k_gemm(const GemmOut o, const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap wmap2,
           const __grid_constant__ CUtensorMap xmap) {
    constexpr int KSTEPS = K / kGK;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GHdr *hd = reinterpret_cast<GHdr *>(smem);
    const uint32_t st0 = smem_addr(smem) + 1024;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t full0 = smem_addr(hd->full), empty0 = smem_addr(hd->empty), accf = smem_addr(&hd->accf);
    // token tiles vary fastest: the CTAs that share a weight tile run
    // together, and the input (at most 58.7 MB at 4096 tokens) stays in L2
    const int m0 = blockIdx.y * kGM, n0 = blockIdx.x * kGN;
    const bool second = m0 >= o.m_split;          // a tile of the second matrix
    const int ma = second ? m0 - o.m_split : m0;  // its first row there
    if (tid == 0) {
        for (int i = 0; i < kGStages; i++) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        mbar_init(accf, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_addr(&hd->tmem), kGN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = hd->tmem;
    pdl_launch_dependents();
    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            const CUtensorMap *wm = second ? &wmap2 : &wmap;
            // the weights are the call's own: the first stages' weight
            // tiles go out before the wait for the inputs
            const int pre = KSTEPS < kGStages ? KSTEPS : kGStages;
            for (int k = 0; k < pre; k++) {
                mbar_arrive_expect_tx(full0 + 8 * k, kGStage);
                tma_2d_plain(st0 + k * kGStage, wm, k * kGK, ma, full0 + 8 * k);
            }
            pdl_wait();                               // the inputs, if a kernel before writes them
            for (int k = 0; k < KSTEPS; k++) {
                const int s = k % kGStages;
                if (k >= kGStages && !mbar_wait(empty0 + 8 * s, ((k / kGStages) - 1) & 1)) {
                    report_status(o.status, kStatusWaitTimeout, 300);
                    break;
                }
                const uint32_t dst = st0 + s * kGStage;
                if (k >= pre) {
                    mbar_arrive_expect_tx(full0 + 8 * s, kGStage);
                    tma_2d_plain(dst, wm, k * kGK, ma, full0 + 8 * s);
                }
                tma_2d_plain(dst + kGABytes, &xmap, k * kGK, n0, full0 + 8 * s);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------- MMA issuer --
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kGM, kGN);
            for (int k = 0; k < KSTEPS; k++) {
                const int s = k % kGStages;
                if (!mbar_wait(full0 + 8 * s, (k / kGStages) & 1)) {
                    report_status(o.status, kStatusWaitTimeout, 301);
                    break;
                }
                tc_fence_after();
                const uint32_t a = st0 + s * kGStage, b = a + kGABytes;
#pragma unroll
                for (int k16 = 0; k16 < kGK / 16; k16++)
                    umma_f16(tmem, umma_desc_sw128(a + 32 * k16), umma_desc_sw128(b + 32 * k16), idesc,
                             (k > 0 || k16 > 0) ? 1u : 0u);
                umma_commit(empty0 + 8 * s);          // the stage is free once these finish
            }
            umma_commit(accf);                        // every MMA issued so far has finished
        }
    } else {
        // --------------------------------------------------- epilogue --
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const int r = (second ? o.col1 : o.col0) + ma + 32 * q + lane;   // output column of this TMEM lane
        if (mbar_wait(accf, 0)) {
            tc_fence_after();
            const uint32_t base = tmem + ((uint32_t)(32 * q) << 16);
            for (int c0 = 0; c0 < kGN; c0 += 16) {
                if (n0 + c0 >= o.n_tokens) break;
                // the addends first, all 16 loads in flight (the output
                // stores cannot then hold them back)
                float ad[16];
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const int t = n0 + c0 + j;
                    ad[j] = ADD && t < o.n_tokens ? __ldg(o.add + (size_t)t * o.ldy + r) : 0.f;
                }
                uint32_t v[16];
                tmem_ld16(base + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const int t = n0 + c0 + j;
                    if (t < o.n_tokens) {
                        const size_t at = (size_t)t * o.ldy + r;
                        const float val = ADD ? __uint_as_float(v[j]) + ad[j] : __uint_as_float(v[j]);
                        if (o.y_bf16 != nullptr) o.y_bf16[at] = f32_to_bf16_rn(val);
                        else o.y[at] = val;
                    }
                }
            }
        } else if (lane == 0) {
            report_status(o.status, kStatusWaitTimeout, 302);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kGN);
    }
}

// ---------------------------------------------------------- elementwise --

// one thread per 4 outputs
__global__ void __launch_bounds__(256) k_situ_bf16(const float *__restrict__ gu, int F, int n_tokens,
                                                   uint16_t *__restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long n4 = (long long)n_tokens * F / 4;
    pdl_launch_dependents();
    pdl_wait();
    if (i >= n4) return;
    const int t = (int)(i / (F / 4)), c4 = (int)(i % (F / 4));
    const float *row = gu + (size_t)t * 2 * F;
    const float4 g = reinterpret_cast<const float4 *>(row)[c4];
    const float4 u = reinterpret_cast<const float4 *>(row + F)[c4];
    const uint32_t lo = f32_to_bf16_rn(situ_glu(g.x, u.x)) | (uint32_t)f32_to_bf16_rn(situ_glu(g.y, u.y)) << 16;
    const uint32_t hi = f32_to_bf16_rn(situ_glu(g.z, u.z)) | (uint32_t)f32_to_bf16_rn(situ_glu(g.w, u.w)) << 16;
    reinterpret_cast<uint2 *>(out + (size_t)t * F)[c4] = make_uint2(lo, hi);
}

// one CTA per token
__global__ void __launch_bounds__(256) k_rmsnorm_bf16(const float *__restrict__ x, const uint16_t *__restrict__ g,
                                                      int D, uint16_t *__restrict__ out) {
    __shared__ float red[8];
    const int t = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_launch_dependents();
    pdl_wait();
    const float4 *row = reinterpret_cast<const float4 *>(x + (size_t)t * D);
    float ss = 0.f;
    for (int c4 = threadIdx.x; c4 < D / 4; c4 += blockDim.x) {
        const float4 v = row[c4];
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; w++) tot += red[w];
    const float scale = 1.0f / sqrtf(tot / (float)D + kRmsEps);
    for (int c4 = threadIdx.x; c4 < D / 4; c4 += blockDim.x) {
        const float4 v = row[c4];
        const uint2 q = reinterpret_cast<const uint2 *>(g)[c4];
        const uint32_t lo = f32_to_bf16_rn(v.x * scale * bf16_lo(q.x)) |
                            (uint32_t)f32_to_bf16_rn(v.y * scale * bf16_hi(q.x)) << 16;
        const uint32_t hi = f32_to_bf16_rn(v.z * scale * bf16_lo(q.y)) |
                            (uint32_t)f32_to_bf16_rn(v.w * scale * bf16_hi(q.y)) << 16;
        reinterpret_cast<uint2 *>(out + (size_t)t * D)[c4] = make_uint2(lo, hi);
    }
}

// bf16 [rows][K] row-major, boxes of box_rows x 64 (128 bytes, 128-byte swizzle)
bool encode_bf16_rows(CUtensorMap &m, const void *base, int K, uint64_t rows, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, rows}, strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kGK, box_rows}, es[2] = {1, 1};
    return enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int K, int XF>
cudaError_t gemv_t(const Ctx &c, const GemvArgs &a) {
    static std::atomic<uint64_t> done{0};
    const cudaError_t e = ensure_smem((const void *)k_gemv<K, XF>, GemvShape<K>::SMEM_MAX, done);
    if (e != cudaSuccess) return e;
    const int chunk = a.n_tokens < kGemvTok ? a.n_tokens : kGemvTok;
    // one CTA per SM, at least 4 rows each
    int grid = c.num_sms;
    if (grid > (a.rows + 3) / 4) grid = (a.rows + 3) / 4;
    if (grid < 1) grid = 1;
    return launch_pdl(k_gemv<K, XF>, dim3(grid), dim3(kGemvThreads), (size_t)GemvShape<K>::smem(chunk), c.stream, a);
}

// rows of W, then (o.m_split < rows) rows - o.m_split rows of W2
template <int K, bool ADD>
cudaError_t gemm_t(const Ctx &c, const uint16_t *W, const uint16_t *W2, int rows, const uint16_t *x,
                   const GemmOut &o) {
    static std::atomic<uint64_t> done{0};
    const cudaError_t e = ensure_smem((const void *)k_gemm<K, ADD>, kGSmem, done);
    if (e != cudaSuccess) return e;
    CUtensorMap wm, wm2, xm;
    const int rows2 = rows - o.m_split;
    if (!encode_bf16_rows(wm, W, K, (uint64_t)o.m_split, kGM) ||
        !encode_bf16_rows(wm2, rows2 > 0 ? W2 : W, K, (uint64_t)(rows2 > 0 ? rows2 : o.m_split), kGM) ||
        !encode_bf16_rows(xm, x, K, (uint64_t)o.n_tokens, kGN))
        return cudaErrorInvalidValue;
    const dim3 grid((o.n_tokens + kGN - 1) / kGN, rows / kGM);
    return launch_pdl(k_gemm<K, ADD>, grid, dim3(kGThreads), (size_t)kGSmem, c.stream, o, wm, wm2, xm);
}

}  // namespace

cudaError_t launch_dense_gemv(const Ctx &c, int K, int xf, const GemvArgs &a) {
    if (K == 7168 && xf == kXfPlain) return gemv_t<7168, kXfPlain>(c, a);
    if (K == 6144 && xf == kXfSitu) return gemv_t<6144, kXfSitu>(c, a);
    if (K == 3584 && xf == kXfRmsNorm) return gemv_t<3584, kXfRmsNorm>(c, a);
    if (K == kLatentOutK && xf == kXfLatentOut) {
        if (a.n_seg != 1 || a.x_bf16 || a.Wt == nullptr || a.x2 == nullptr) return cudaErrorInvalidValue;
        return gemv_t<kLatentOutK, kXfLatentOut>(c, a);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_dense_gemm(const Ctx &c, int K, const uint16_t *W, int rows, const uint16_t *x, int n_tokens,
                              float *y, uint16_t *y_bf16, int ldy, int col0, const float *add) {
    if (rows % kGM != 0 || n_tokens < 1) return cudaErrorInvalidValue;
    const GemmOut o{y, y_bf16, ldy, col0, add, n_tokens, c.status, rows, 0};
    if (add != nullptr) {
        if (K == 3584) return gemm_t<3584, true>(c, W, W, rows, x, o);
        return cudaErrorInvalidValue;
    }
    if (K == 7168) return gemm_t<7168, false>(c, W, W, rows, x, o);
    if (K == 6144) return gemm_t<6144, false>(c, W, W, rows, x, o);
    if (K == 3584) return gemm_t<3584, false>(c, W, W, rows, x, o);
    return cudaErrorInvalidValue;
}

cudaError_t launch_dense_gemm2(const Ctx &c, int K, const uint16_t *W1, const uint16_t *W2, int rows, const uint16_t *x,
                               int n_tokens, float *y, int ldy, int col1, int col2) {
    if (rows % kGM != 0 || n_tokens < 1 || K != 7168) return cudaErrorInvalidValue;
    const GemmOut o{y, nullptr, ldy, col1, nullptr, n_tokens, c.status, rows, col2};
    return gemm_t<7168, false>(c, W1, W2, 2 * rows, x, o);
}

cudaError_t launch_situ_bf16(const Ctx &c, const float *gu, int F, int n_tokens, uint16_t *out) {
    const long long n4 = (long long)n_tokens * F / 4;
    return launch_pdl(k_situ_bf16, dim3((unsigned)((n4 + 255) / 256)), dim3(256), 0, c.stream, gu, F, n_tokens, out);
}

cudaError_t launch_rmsnorm_bf16(const Ctx &c, const float *x, const uint16_t *g, int D, int n_tokens,
                                uint16_t *out) {
    return launch_pdl(k_rmsnorm_bf16, dim3(n_tokens), dim3(256), 0, c.stream, x, g, D, out);
}

// the router's logits: fp32 states or up to 16 bf16 ones on CUDA cores,
// more bf16 states on the tensor cores
cudaError_t launch_router_logits(const Ctx &c, float *logits, const void *h, int h_bf16, const uint16_t *W,
                                 int n_tokens) {
    constexpr int kH = 7168;
    if (h_bf16 && n_tokens >= kDenseGemmMinTokens)
        return launch_dense_gemm(c, kH, W, kE, static_cast<const uint16_t *>(h), n_tokens, logits, nullptr, kE, 0,
                                 nullptr);
    GemvArgs a{};
    a.seg[0] = GemvSeg{W, logits, nullptr, kE, 0};
    a.n_seg = 1;
    a.rows = kE;
    a.x = h;
    a.x_bf16 = h_bf16;
    a.ldx = kH;
    a.n_tokens = n_tokens;
    a.status = c.status;
    return launch_dense_gemv(c, kH, kXfPlain, a);
}

cudaError_t set_wait_polls_dense(uint32_t polls) { return set_wait_polls_here(polls); }

}  // namespace k3mx
