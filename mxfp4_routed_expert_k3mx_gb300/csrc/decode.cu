// decode.cu - the single MXFP4 GEMV y = W x with fp32 activations, and the
// slot-order combine of the batched decode pass (sm_103a).
//
// y = W x with W read straight out of packed MXFP4 and never written back
// as floats (kimi-k3-in-c: 2.78 trillion parameters, one CPU, 8 GB of RAM,
// "Reduction one: the experts already ship at half a byte"): per group of 32
// columns the codes times the activations are summed in fp32 and the sum is
// multiplied by the group's scale 2^(s - 127); a scale of 255 adds nothing.
//
// Layout of the work.  A CTA takes a tile of R rows; its warps split the K
// dimension: warp w owns gpw <= 32 consecutive groups and its lane l the
// group w * gpw + l, for every row of the tile.  The lane's 32 activations
// stay in registers; a row's group is one 16-byte load (a warp's loads of
// one row are contiguous), and the tile's R loads per lane are all issued
// before the first is used, so a tile costs one round trip to memory and a
// matrix of 3072 rows is one wave of CTAs.  Per row the lane forms its
// scaled group sum; the R row sums are reduced over the lanes by a
// reduce-scatter of shuffles (R shuffles in all, each lane ending with one
// row) and over the warps through shared memory, in a fixed order, so the
// result does not depend on timing.
//
// Back-to-back calls overlap: the kernel is launched as a programmatic
// dependent of the kernel before it.  Before waiting for that kernel it
// prefetches its tile into L2 (every write on the device lands in L2, so a
// prefetch cannot return stale data) and lets the next kernel launch; after
// the wait it reads x and the weights into registers and writes y.
#include "common.cuh"

namespace k3mx {
namespace {

// ------------------------------------------------------------------ GEMV --

constexpr int kGvMaxWarps = 16;       // in <= 16384: 512 groups, at most 32 per warp

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// R row sums per lane -> lane l holds the warp's sum of row l / (32 / R)
// (both lanes of a pair for R = 16); sums taken in a fixed order
template <int R>
__device__ __forceinline__ float reduce_scatter(float (&v)[R], int lane) {
#pragma unroll
    for (int n = R, o = 16; n > 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; i++) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    // the remaining lanes of a row group (32 / R of them) hold partial sums
    float r = v[0];
#pragma unroll
    for (int o = 16 / R; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

template <int R>
__global__ void __launch_bounds__(R == 16 ? 256 : 512)
k_gemv(float *__restrict__ y, const float *__restrict__ x, const uint8_t *__restrict__ packed,
       const uint8_t *__restrict__ scales, int in, int rows, int gpw) {
    __shared__ float red[kGvMaxWarps][R];
    const int G = in / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const long long r0 = (long long)blockIdx.x * R;
    const int nr = (int)min((long long)R, rows - r0);
    const size_t rowb = (size_t)in / 2;
    if (threadIdx.x == 0) {
        prefetch_l2(packed + r0 * rowb, (uint32_t)(nr * rowb));
        const uint8_t *sp = scales + r0 * G;
        if ((reinterpret_cast<uintptr_t>(sp) & 15u) == 0 && ((nr * G) & 15) == 0) prefetch_l2(sp, (uint32_t)(nr * G));
    }
    pdl_launch_dependents();
    pdl_wait();                                       // x and the weights may come from the kernel before
    const int g = warp * gpw + lane;
    const bool active = lane < gpw && g < G;
    float v[R];
    if (active) {
        float2 xv[16];
        load_x_group(x, g, xv);
        uint4 wv[R];
        uint32_t sv[R];
#pragma unroll
        for (int r = 0; r < R; r++) {
            if (r < nr) {
                wv[r] = ldg_stream(packed + (r0 + r) * rowb + 16 * g);
                sv[r] = ldg_u8(scales + (r0 + r) * G + g);
            } else {
                wv[r] = make_uint4(0u, 0u, 0u, 0u);
                sv[r] = 255u;
            }
        }
#pragma unroll
        for (int r = 0; r < R; r++) v[r] = group_term(wv[r], sv[r], xv);
    } else {
#pragma unroll
        for (int r = 0; r < R; r++) v[r] = 0.f;
    }
    const float sum = reduce_scatter<R>(v, lane);
    const int row = lane / (32 / R);
    if (lane % (32 / R) == 0) red[warp][row] = sum;
    __syncthreads();
    if ((int)threadIdx.x < nr) {
        float t = 0.f;
        for (int w = 0; w < nwarps; w++) t += red[w][threadIdx.x];
        y[r0 + threadIdx.x] = t;
    }
}

// y[t][i] = sum_k w[t][k] * out[t*16 + k][i], slot order, fp32
__global__ void k_combine(float *__restrict__ y, const float *__restrict__ out,
                          const float *__restrict__ w, int n_tokens) {
    const int per_tok = kD / 4;
    const long long i4 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    pdl_wait();                                          // the per-pair rows come from the down pass
    if (i4 >= (long long)n_tokens * per_tok) return;
    const int t = (int)(i4 / per_tok), c = (int)(i4 % per_tok);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kK; k++) {
        const float wk = __ldg(w + (size_t)t * kK + k);
        if (wk == 0.f) continue;                         // a slot dropped by top-p has no row
        const float4 v = __ldg(reinterpret_cast<const float4 *>(out + ((size_t)t * kK + k) * kD) + c);
        acc.x = fmaf(wk, v.x, acc.x);
        acc.y = fmaf(wk, v.y, acc.y);
        acc.z = fmaf(wk, v.z, acc.z);
        acc.w = fmaf(wk, v.w, acc.w);
    }
    reinterpret_cast<float4 *>(y + (size_t)t * kD)[c] = acc;
}


}  // namespace

cudaError_t set_wait_polls_decode(uint32_t polls) { return set_wait_polls_here(polls); }

cudaError_t launch_gemv(const Ctx &c, float *y, const float *x, const uint8_t *packed,
                        const uint8_t *scales, int in, int rows) {
    const int G = in / 32;
    const int nwarps = (G + 31) / 32;                 // 1..16
    const int gpw = (G + nwarps - 1) / nwarps;        // groups per warp, <= 32
    // 16 rows per tile up to 8 warps (255 registers a thread), else 8
    if (nwarps <= 8) {
        const unsigned grid = (unsigned)((rows + 15) / 16);
        return launch_pdl(k_gemv<16>, dim3(grid), dim3(32 * nwarps), 0, c.stream, y, x, packed, scales, in, rows, gpw);
    }
    const unsigned grid = (unsigned)((rows + 7) / 8);
    return launch_pdl(k_gemv<8>, dim3(grid), dim3(32 * nwarps), 0, c.stream, y, x, packed, scales, in, rows, gpw);
}

cudaError_t launch_combine(const Ctx &c, float *y, const float *stage, const float *w,
                           int n_tokens) {
    const long long n4 = (long long)n_tokens * (kD / 4);
    const int threads = 256;
    return launch_pdl(k_combine, dim3((unsigned)((n4 + threads - 1) / threads)), dim3(threads), 0, c.stream, y,
                      stage, w, n_tokens);
}

}  // namespace k3mx
