// router.cu - the router logits: the sigmoid router of the Stable LatentMoE
// (Kimi K3 engine (c/kimi_k3.c), "Architecture notes": a [896, 7168] matrix
// over the 7168-wide hidden state; the trunk, router included, is bf16)
//   logits[t][e] = sum_c W[e][c] h[t][c]
// W is bf16 [896][7168] row-major, h fp32 or bf16 [T][7168].  Every product
// of a bf16 weight and an fp32 (or bf16) state is exact in fp32; the sums
// are fp32.  The top-16 of the logits is the routing kernels' work
// (route_group.cu), launched right behind as programmatic dependents.
//
// Few tokens (decode): k_router_gemv, one warp per router row with the row
// held in registers, HBM-bound on the 12.8 MB of weights.
#include "common.cuh"

namespace k3mx {
namespace {

constexpr int kH = 7168;                         // hidden width
constexpr int kRowVec = kH / 8;                  // 16-byte vectors per router row
constexpr int kVecPerLane = kRowVec / 32;        // 28
constexpr int kGemvTok = 4;                      // hidden states per shared-memory chunk
constexpr int kGemvWarps = 8;
constexpr int kGemvSmem = kGemvTok * kH * 4;
static_assert(kE % kGemvWarps == 0 && kRowVec % 32 == 0, "router shape");

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// read once: no L1 allocation
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// One warp per router row: the row's 14 KB sit in registers (28 16-byte
// vectors per lane, vector v = lane + 32 i holds columns 8v..8v+7); the
// hidden states pass through shared memory in chunks of 4, laid out so that
// the lanes read consecutive 16-byte words (columns 8v..8v+3 at slot v,
// 8v+4..8v+7 at slot kRowVec + v).  Per lane, 8-term sums per vector are
// added over its 28 vectors; the warp adds its lanes: a logit is at most 41
// fp32 roundings deep.
__global__ void __launch_bounds__(kGemvWarps * 32, 1)
    k_router_gemv(float *__restrict__ logits, const void *__restrict__ h, int h_bf16,
                  const uint16_t *__restrict__ W, int n_tokens) {
    extern __shared__ float4 hs[];                // [kGemvTok][2 * kRowVec]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kGemvWarps + warp;
    // the routing kernel behind may start its prologue
    pdl_launch_dependents();
    const uint4 *wr = reinterpret_cast<const uint4 *>(W + (size_t)e * kH);
    uint4 wv[kVecPerLane];
#pragma unroll
    for (int i = 0; i < kVecPerLane; i++) wv[i] = ld_stream(wr + lane + 32 * i);
    pdl_wait();                                   // the hidden states, if a kernel before writes them
    for (int t0 = 0; t0 < n_tokens; t0 += kGemvTok) {
        const int nt = min(kGemvTok, n_tokens - t0);
        __syncthreads();                          // the previous chunk is consumed
        for (int i = threadIdx.x; i < nt * (kH / 4); i += blockDim.x) {
            const int t = i / (kH / 4), c4 = i % (kH / 4);
            float4 v;
            if (h_bf16) {
                const uint2 b = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(h) +
                                                                (size_t)(t0 + t) * kH)[c4];
                v = make_float4(bf16_lo(b.x), bf16_hi(b.x), bf16_lo(b.y), bf16_hi(b.y));
            } else {
                v = reinterpret_cast<const float4 *>(static_cast<const float *>(h) + (size_t)(t0 + t) * kH)[c4];
            }
            hs[t * (2 * kRowVec) + (c4 & 1) * kRowVec + (c4 >> 1)] = v;
        }
        __syncthreads();
        float acc[kGemvTok];
#pragma unroll
        for (int j = 0; j < kGemvTok; j++) acc[j] = 0.f;
#pragma unroll
        for (int i = 0; i < kVecPerLane; i++) {
            const int v = lane + 32 * i;
            const uint4 q = wv[i];
            const float w0 = bf16_lo(q.x), w1 = bf16_hi(q.x), w2 = bf16_lo(q.y), w3 = bf16_hi(q.y);
            const float w4 = bf16_lo(q.z), w5 = bf16_hi(q.z), w6 = bf16_lo(q.w), w7 = bf16_hi(q.w);
#pragma unroll
            for (int j = 0; j < kGemvTok; j++) {
                if (j < nt) {
                    const float4 a = hs[j * (2 * kRowVec) + v], b = hs[j * (2 * kRowVec) + kRowVec + v];
                    float s8 = w0 * a.x;
                    s8 = fmaf(w1, a.y, s8);
                    s8 = fmaf(w2, a.z, s8);
                    s8 = fmaf(w3, a.w, s8);
                    s8 = fmaf(w4, b.x, s8);
                    s8 = fmaf(w5, b.y, s8);
                    s8 = fmaf(w6, b.z, s8);
                    s8 = fmaf(w7, b.w, s8);
                    acc[j] += s8;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kGemvTok; j++) {
            float a = acc[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0 && j < nt) logits[(size_t)(t0 + j) * kE + e] = a;
        }
    }
}

}  // namespace

cudaError_t launch_router_logits(const Ctx &c, float *logits, const void *h, int h_bf16, const uint16_t *W,
                                 int n_tokens) {
    static bool configured = false;
    if (!configured) {
        const cudaError_t e =
            cudaFuncSetAttribute(k_router_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(k_router_gemv, dim3(kE / kGemvWarps), dim3(kGemvWarps * 32), (size_t)kGemvSmem, c.stream,
                      logits, h, h_bf16, W, n_tokens);
}

}  // namespace k3mx
