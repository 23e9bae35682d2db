// tmaps.cuh - TMA tensor maps of the expert weight matrices.
//
// Every expert matrix (w1, w3: 3072 x 1792 packed bytes; w2: 3584 x 1536)
// is read through a 2-D tensor map over its packed bytes (uint8 elements,
// 128 x 128-byte boxes, 128-byte swizzle).  The host encodes one template
// per shape; the step's first kernel builds the per-expert maps on the
// device from the expert table (tensormap.replace of the global address,
// published to global memory for the tensor-map proxy), so the expert
// passes only acquire a ready map before their first weight copy.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace k3mx {

constexpr int kMapBytes = 128;
constexpr int kMapsPerExpert = 3;        // w1, w3, w2

// the driver's cuTensorMapEncodeTiled, looked up once per process
// (nullptr when unavailable)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// templates for the current device (encoded once per device); false when
// the driver entry point or the encoding is unavailable
bool weight_map_templates(CUtensorMap &w13, CUtensorMap &w2);

// bytes of the per-expert map table of n experts
inline size_t expert_maps_bytes(int n_experts) { return (size_t)n_experts * kMapsPerExpert * kMapBytes; }

// Map `i` of the table (expert i / 3, matrix i % 3) built by one warp with
// a 128-byte shared staging slot `smap`.  A weight pointer not aligned to
// `align` bytes (16, or 32 for maps that expand e2m1 codes) keeps the
// template's address (the passes skip that expert).
__device__ __forceinline__ void build_expert_map(uint8_t *table, int i, uint32_t smap, const k3mx_expert &ex,
                                                 const CUtensorMap &w13, const CUtensorMap &w2, uint32_t align) {
    const int lane = threadIdx.x & 31, mat = i % kMapsPerExpert;
    const CUtensorMap &tmpl = mat < 2 ? w13 : w2;
    const uint8_t *addr = mat == 0 ? ex.w1 : mat == 1 ? ex.w3 : ex.w2;
    if (lane < 8) {
        const uint4 v = reinterpret_cast<const uint4 *>(&tmpl)[lane];
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smap + 16 * lane), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
    }
    __syncwarp();
    if (lane == 0 && (reinterpret_cast<uintptr_t>(addr) & (uintptr_t)(align - 1)) == 0)
        asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;" ::"r"(smap),
                     "l"(reinterpret_cast<uint64_t>(addr))
                     : "memory");
    __syncwarp();
    asm volatile(
        "tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu.sync.aligned "
        "[%0], [%1], 128;" ::"l"(table + (size_t)i * kMapBytes),
        "r"(smap)
        : "memory");
}

// the consumer side: a map built by an earlier kernel, before its first use
__device__ __forceinline__ void acquire_map(const void *map) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
    // (no prefetch.tensormap: measured, a prefetch ahead of the first copy
    // delayed the next acquire and that copy by about 0.7 us each)
}

// Map-building CTAs: 8 warps (1 KB of static shared memory), each warp
// building kMapsPerWarp maps one after another, so few CTAs (and SMs) are
// taken: warp w of CTA b builds maps (8 b + w) * kMapsPerWarp + j of
// n_experts * 3.  `table` is the device expert table, or nullptr with `one`
// as expert 0.
constexpr int kMapsPerWarp = 8;
constexpr int kMapsPerCta = 8 * kMapsPerWarp;
__device__ __forceinline__ void build_maps_cta(uint8_t *maps, int n_experts, const k3mx_expert *table,
                                               const k3mx_expert &one, const CUtensorMap &w13,
                                               const CUtensorMap &w2, int cta, uint32_t align = 16) {
    __shared__ __align__(128) uint8_t stage[8][kMapBytes];
    const int warp = threadIdx.x >> 5;
    if (warp >= 8) return;
    for (int j = 0; j < kMapsPerWarp; j++) {
        const int i = (cta * 8 + warp) * kMapsPerWarp + j;
        if (i >= n_experts * kMapsPerExpert) return;
        const k3mx_expert ex = table != nullptr ? table[i / kMapsPerExpert] : one;
        build_expert_map(maps, i, (uint32_t)__cvta_generic_to_shared(stage[warp]), ex, w13, w2, align);
        __syncwarp();                     // the staging slot is reused
    }
}

}  // namespace k3mx
