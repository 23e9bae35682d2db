// router.cu - the router logits: the sigmoid router of the Stable LatentMoE
// (Kimi K3 engine (c/kimi_k3.c), "Architecture notes": a [896, 7168] matrix
// over the 7168-wide hidden state; the trunk, router included, is bf16)
//   logits[t][e] = sum_c W[e][c] h[t][c]
// W is bf16 [896][7168] row-major, h fp32 or bf16 [T][7168].  Every product
// of a bf16 weight and an fp32 (or bf16) state is exact in fp32; the sums
// are fp32.  The top-16 of the logits is the routing kernels' work
// (route_group.cu), launched right behind as programmatic dependents.
//
// Few tokens (decode), or fp32 states: k_router_gemv, one warp per router
// row, the rows brought in by bulk copies; HBM-bound on the 12.8 MB of
// weights.
// Many bf16 states (prefill): k_router_gemm, the tcgen05 tensor cores
// (kind::f16 with bf16 A and B, fp32 accumulators in TMEM); a CTA computes
// 128 router rows x 256 tokens over the whole 7168-deep sum, its operands
// streamed by TMA (128-byte swizzle) through a 4-stage ring.
#include <cudaTypedefs.h>

#include "common.cuh"

namespace k3mx {
namespace {

constexpr int kH = 7168;                         // hidden width
constexpr int kRowVec = kH / 8;                  // 16-byte vectors per router row
constexpr int kVecPerLane = kRowVec / 32;        // 28
constexpr int kGemvTok = 3;                      // hidden states per shared-memory chunk
constexpr int kGemvWarps = 7;                    // one router row per warp: 128 CTAs
constexpr int kRowBytes = kH * 2;                // 14336
constexpr int kGemvSmem = 1024 + kGemvWarps * kRowBytes + kGemvTok * kH * 4;
static_assert(kE % kGemvWarps == 0 && kRowVec % 32 == 0 && kRowBytes % 16 == 0, "router shape");

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// One warp per router row.  The CTA's 8 rows (112 KB, contiguous) come in
// by bulk copies, one per row, issued before anything else; the hidden
// states pass through shared memory in chunks of 3, laid out so that the
// lanes read consecutive 16-byte words (columns 8v..8v+3 at slot v,
// 8v+4..8v+7 at slot kRowVec + v, vector v = lane + 32 i).  Per lane, a
// vector's 8 products are two 4-term sums added, the vectors go to four
// running sums (7 each) added pairwise, and the warp adds its lanes: a
// logit is at most 4 + 1 + 7 + 2 + 5 = 19 fp32 roundings deep.
__global__ void __launch_bounds__(kGemvWarps * 32, 1)
    k_router_gemv(float *__restrict__ logits, const void *__restrict__ h, int h_bf16,
                  const uint16_t *__restrict__ W, int n_tokens, int *status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    const uint8_t *rows = smem + 1024;
    float4 *hs = reinterpret_cast<float4 *>(smem + 1024 + kGemvWarps * kRowBytes);   // [kGemvTok][2 * kRowVec]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kGemvWarps + warp;
    const uint32_t b = smem_addr(bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(b, kGemvWarps * kRowBytes);
        const uint8_t *src = reinterpret_cast<const uint8_t *>(W) + (size_t)blockIdx.x * kGemvWarps * kRowBytes;
        for (int r = 0; r < kGemvWarps; r++)
            bulk_g2s(smem_addr(rows) + r * kRowBytes, src + (size_t)r * kRowBytes, kRowBytes, b,
                     l2_evict_first_policy());
    }
    // the routing kernel behind may start its prologue
    pdl_launch_dependents();
    pdl_wait();                                   // the hidden states, if a kernel before writes them
    const uint4 *wr = reinterpret_cast<const uint4 *>(rows + warp * kRowBytes);
    bool have_rows = false;
    for (int t0 = 0; t0 < n_tokens; t0 += kGemvTok) {
        const int nt = min(kGemvTok, n_tokens - t0);
        __syncthreads();                          // the barrier is set up; the previous chunk is consumed
        // 8 loads in flight per thread before the stores
        const int n4 = nt * (kH / 4);
        for (int i0 = threadIdx.x; i0 < n4; i0 += 8 * (int)blockDim.x) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int i = i0 + u * (int)blockDim.x;
                if (i < n4) {
                    const int t = i / (kH / 4), c4 = i % (kH / 4);
                    if (h_bf16) {
                        const uint2 q = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(h) +
                                                                        (size_t)(t0 + t) * kH)[c4];
                        v[u] = make_float4(bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y));
                    } else {
                        v[u] = reinterpret_cast<const float4 *>(static_cast<const float *>(h) +
                                                                (size_t)(t0 + t) * kH)[c4];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int i = i0 + u * (int)blockDim.x;
                if (i < n4) {
                    const int t = i / (kH / 4), c4 = i % (kH / 4);
                    hs[t * (2 * kRowVec) + (c4 & 1) * kRowVec + (c4 >> 1)] = v[u];
                }
            }
        }
        __syncthreads();
        if (!have_rows) {
            if (!mbar_wait(b, 0)) {
                if (lane == 0) report_status(status, kStatusWaitTimeout, 310);
                return;                           // every warp leaves: no barrier follows
            }
            have_rows = true;
        }
        // four independent running sums per token (vectors i mod 4), each
        // vector's 8 products as two 4-term chains: the iterations overlap
        float acc[kGemvTok][4];
#pragma unroll
        for (int j = 0; j < kGemvTok; j++)
#pragma unroll
            for (int r = 0; r < 4; r++) acc[j][r] = 0.f;
        static_assert(kVecPerLane % 4 == 0, "vectors per lane");
#pragma unroll 4
        for (int i = 0; i < kVecPerLane; i++) {
            const int v = lane + 32 * i;
            const uint4 q = wr[v];
            const float w0 = bf16_lo(q.x), w1 = bf16_hi(q.x), w2 = bf16_lo(q.y), w3 = bf16_hi(q.y);
            const float w4 = bf16_lo(q.z), w5 = bf16_hi(q.z), w6 = bf16_lo(q.w), w7 = bf16_hi(q.w);
#pragma unroll
            for (int j = 0; j < kGemvTok; j++) {
                if (j < nt) {
                    const float4 a = hs[j * (2 * kRowVec) + v], c = hs[j * (2 * kRowVec) + kRowVec + v];
                    float s0 = w0 * a.x, s1 = w4 * c.x;
                    s0 = fmaf(w1, a.y, s0);
                    s1 = fmaf(w5, c.y, s1);
                    s0 = fmaf(w2, a.z, s0);
                    s1 = fmaf(w6, c.z, s1);
                    s0 = fmaf(w3, a.w, s0);
                    s1 = fmaf(w7, c.w, s1);
                    acc[j][i & 3] += s0 + s1;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kGemvTok; j++) {
            float a = (acc[j][0] + acc[j][1]) + (acc[j][2] + acc[j][3]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0 && j < nt) logits[(size_t)(t0 + j) * kE + e] = a;
        }
    }
}

// ----------------------------------------------------- tensor-core GEMM --

constexpr int kGM = 128, kGN = 256, kGK = 64;    // tile: router rows x tokens x K per stage
constexpr int kGStages = 4;
constexpr int kGABytes = kGM * kGK * 2, kGBBytes = kGN * kGK * 2;
constexpr int kGStage = kGABytes + kGBBytes;
constexpr int kGKSteps = kH / kGK;               // 112
constexpr int kGThreads = 192;                   // warp 0 TMA, 1 MMA, 2-5 epilogue
constexpr int kGSmem = 1024 + 1024 + kGStages * kGStage;
constexpr int kGemmMinTokens = 17;               // from here on the tensor cores
static_assert(kE % kGM == 0 && kH % kGK == 0, "router tiles");

struct GHdr {
    uint64_t full[kGStages], empty[kGStages], accf;
    uint32_t tmem;
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

__global__ void __launch_bounds__(kGThreads, 1)
    k_router_gemm(float *__restrict__ logits, int n_tokens, int *status, const __grid_constant__ CUtensorMap wmap,
                  const __grid_constant__ CUtensorMap hmap) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GHdr *hd = reinterpret_cast<GHdr *>(smem);
    const uint32_t st0 = smem_addr(smem) + 1024;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t full0 = smem_addr(hd->full), empty0 = smem_addr(hd->empty), accf = smem_addr(&hd->accf);
    const int m0 = blockIdx.x * kGM, n0 = blockIdx.y * kGN;
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
    bool ok = true;
    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            pdl_wait();                               // the hidden states, if a kernel before writes them
            for (int k = 0; k < kGKSteps; k++) {
                const int s = k % kGStages;
                if (k >= kGStages && !mbar_wait(empty0 + 8 * s, ((k / kGStages) - 1) & 1)) {
                    report_status(status, kStatusWaitTimeout, 300);
                    ok = false;
                    break;
                }
                const uint32_t dst = st0 + s * kGStage;
                mbar_arrive_expect_tx(full0 + 8 * s, kGStage);
                tma_2d_plain(dst, &wmap, k * kGK, m0, full0 + 8 * s);
                tma_2d_plain(dst + kGABytes, &hmap, k * kGK, n0, full0 + 8 * s);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------- MMA issuer --
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kGM, kGN);
            for (int k = 0; k < kGKSteps; k++) {
                const int s = k % kGStages;
                if (!mbar_wait(full0 + 8 * s, (k / kGStages) & 1)) {
                    report_status(status, kStatusWaitTimeout, 301);
                    ok = false;
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
        const int e = m0 + 32 * q + lane;
        if (mbar_wait(accf, 0)) {
            tc_fence_after();
            const uint32_t base = tmem + ((uint32_t)(32 * q) << 16);
            for (int c0 = 0; c0 < kGN; c0 += 16) {
                if (n0 + c0 >= n_tokens) break;
                uint32_t v[16];
                tmem_ld16(base + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const int t = n0 + c0 + j;
                    if (t < n_tokens) logits[(size_t)t * kE + e] = __uint_as_float(v[j]);
                }
            }
        } else if (lane == 0) {
            report_status(status, kStatusWaitTimeout, 302);
        }
    }
    (void)ok;
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kGN);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 router_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// bf16 [rows][kH] row-major, boxes of box_rows x 64 (128 bytes, 128-byte swizzle)
bool encode_bf16_rows(CUtensorMap &m, const void *base, uint64_t rows, uint32_t box_rows) {
    auto enc = router_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kH, rows}, strides[1] = {(cuuint64_t)kH * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kGK, box_rows}, es[2] = {1, 1};
    return enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_router_logits(const Ctx &c, float *logits, const void *h, int h_bf16, const uint16_t *W,
                                 int n_tokens) {
    if (h_bf16 && n_tokens >= kGemmMinTokens) {
        static bool gconf = false;
        if (!gconf) {
            const cudaError_t e = cudaFuncSetAttribute(k_router_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
            if (e != cudaSuccess) return e;
            gconf = true;
        }
        CUtensorMap wm, hm;
        if (!encode_bf16_rows(wm, W, kE, kGM) || !encode_bf16_rows(hm, h, (uint64_t)n_tokens, kGN))
            return cudaErrorInvalidValue;
        const dim3 grid(kE / kGM, (n_tokens + kGN - 1) / kGN);
        return launch_pdl(k_router_gemm, grid, dim3(kGThreads), (size_t)kGSmem, c.stream, logits, n_tokens,
                          c.status, wm, hm);
    }
    static bool configured = false;
    if (!configured) {
        const cudaError_t e =
            cudaFuncSetAttribute(k_router_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(k_router_gemv, dim3(kE / kGemvWarps), dim3(kGemvWarps * 32), (size_t)kGemvSmem, c.stream,
                      logits, h, h_bf16, W, n_tokens, c.status);
}

}  // namespace k3mx
