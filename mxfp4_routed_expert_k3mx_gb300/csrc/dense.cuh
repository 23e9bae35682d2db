// dense.cuh - the bf16 matrix products of the LatentMoE block (dense.cu).
#pragma once
#include "common.cuh"

namespace k3mx {

constexpr int kXfPlain = 0;      // the input as given (fp32 or bf16)
constexpr int kXfSitu = 1;       // SiTU-GLU(g, u) of an fp32 [g | u] row pair (u at +K)
constexpr int kXfRmsNorm = 2;    // RMSNorm (eps 1e-5) of an fp32 row times a bf16 weight
// [RMSNorm(x) * g | SiTU-GLU(x2)]: the block's output product, W_up's
// 3584 columns and W2s's 6144 side by side (K = 9728), each row's two
// parts copied from the two matrices
constexpr int kXfLatentOut = 3;
constexpr int kLatentOutK1 = 3584, kLatentOutK = 3584 + 6144;
constexpr int kDenseGemmMinTokens = 17;   // bf16 inputs from here on: the tensor cores

// One weight matrix of a CUDA-core product: rows [r0, next segment's r0)
// of the product are the rows of W, written y[t * ldy + (r - r0)] (+ add at
// the same place).  Several matrices over the same input run in one launch.
constexpr int kGemvMaxSeg = 4;
struct GemvSeg {
    const uint16_t *W;           // weight rows [rows][K]
    float *y;
    const float *add;            // or null
    int ldy, r0;
};

struct GemvArgs {
    GemvSeg seg[kGemvMaxSeg];
    int n_seg, rows;             // segments in row order, their rows in all
    const void *x;               // input rows [T][ldx]
    int x_bf16, ldx;
    const uint16_t *g;           // RMSNorm weight (kXfRmsNorm, kXfLatentOut)
    const float *x2;             // kXfLatentOut: the g | u rows [T][ldx2] of the SiTU-GLU part
    int ldx2;
    const uint16_t *Wt;          // kXfLatentOut: the rows' second parts [rows][K - kLatentOutK1]
    int n_tokens;
    int *status;
};

// CUDA cores, any token count; K in {7168, 6144, 3584, 9728 (kXfLatentOut)}
cudaError_t launch_dense_gemv(const Ctx &c, int K, int xf, const GemvArgs &a);

// tcgen05 tensor cores: x bf16 [T][K] (row stride K), W bf16 [rows][K],
// rows a multiple of 128, K in {7168, 6144, 3584}; the output fp32 (y) or
// bf16 (y_bf16), y[t * ldy + col0 + r] (+ add, fp32 output only)
cudaError_t launch_dense_gemm(const Ctx &c, int K, const uint16_t *W, int rows, const uint16_t *x, int n_tokens,
                              float *y, uint16_t *y_bf16, int ldy, int col0, const float *add);

// two matrices W1, W2 [rows][K] (K = 7168, rows a multiple of 128) over one
// bf16 input in one launch: y[t * ldy + col1 + r] = W1 x, y[t * ldy + col2 +
// r] = W2 x (fp32)
cudaError_t launch_dense_gemm2(const Ctx &c, int K, const uint16_t *W1, const uint16_t *W2, int rows, const uint16_t *x,
                               int n_tokens, float *y, int ldy, int col1, int col2);
// SiTU-GLU of fp32 [T][2F] (g | u) rows into bf16 [T][F]
cudaError_t launch_situ_bf16(const Ctx &c, const float *gu, int F, int n_tokens, uint16_t *out);
// RMSNorm (eps 1e-5) of fp32 [T][D] rows times a bf16 weight, into bf16
cudaError_t launch_rmsnorm_bf16(const Ctx &c, const float *x, const uint16_t *g, int D, int n_tokens,
                                uint16_t *out);

}  // namespace k3mx
