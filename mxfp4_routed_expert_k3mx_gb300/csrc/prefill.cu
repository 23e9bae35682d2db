// prefill.cu - placeholder until the tcgen05 grouped GEMM lands.
#include "prefill.cuh"

namespace k3mx {

size_t prefill_scratch_bytes(int n_tokens) { return (size_t)n_tokens * kK * kF * 2; }

cudaError_t launch_prefill(const Ctx &, const PrefillArgs &) { return cudaErrorNotSupported; }

}  // namespace k3mx
