// prefill.cuh - grouped tcgen05 GEMM path for bf16 activations (many tokens).
#pragma once
#include "common.cuh"

namespace k3mx {

struct PrefillArgs {
    float *y;                      // [T][D] fp32, written
    const uint16_t *x;             // [T][D] bf16 bits
    int n_tokens;
    const k3mx_expert *experts;    // device [896]
    const float *w;                // [T][16] routing weights (by pair id t*16 + k)
    const int32_t *counts, *offsets, *perm, *act, *n_active;
    int max_active;
    void *scratch;                 // prefill_scratch_bytes(n_tokens), 256-byte aligned:
                                   // f16 x, f16 h rows in grouped order, work units
};

// upper bound of the number of prefill work units (<= 128 pairs of one expert)
int prefill_max_units(int n_tokens);
size_t prefill_scratch_bytes(int n_tokens);
cudaError_t launch_prefill(const Ctx &c, const PrefillArgs &a);

// Block-scaled variant (px.cu): x and h as four MXFP4 pieces, the weights
// fed to kind::mxf4 MMAs as stored.  `scratch` holds
// prefill_mx_scratch_bytes(n_tokens) bytes, 256-byte aligned.
int prefill_mx_max_units(int n_tokens);
size_t prefill_mx_scratch_bytes(int n_tokens);
cudaError_t launch_prefill_mx(const Ctx &c, const PrefillArgs &a);

}  // namespace k3mx
