// common.cuh - shapes, MXFP4 decoding helpers and launch plumbing shared by
// the sm_103a kernels of the MXFP4 routed-expert layer.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "k3mx.h"

namespace k3mx {

// Kimi-K3 routed-expert shapes (kimi-k3-in-c README, K3Cfg).
constexpr int kD = K3MX_LATENT;      // 3584
constexpr int kF = K3MX_INTER;       // 3072
constexpr int kE = K3MX_N_EXPERTS;   // 896
constexpr int kK = K3MX_TOPK;        // 16
constexpr int kG = K3MX_GROUP;       // 32 columns per ue8m0 scale

// device status word codes (first failure wins)
enum : int {
    kStatusOk = 0,
    kStatusBadIndex = 1,       // an expert index outside 0..895 reached a kernel
    kStatusWaitTimeout = 2,    // a bounded mbarrier / flag wait gave up
    kStatusBadPointer = 3,     // a weight pointer from a device table is not 16-byte aligned
};

// Per-launch context shared by the launchers: stream, SM count, status word.
struct Ctx {
    cudaStream_t stream;
    int num_sms;
    int *status;               // device int[4]: [0] first code, [1] detail
};

// ---------------------------------------------------------------- decoding --
//
// MXFP4 (Kimi K3 engine (c/kimi_k3.c), "Weights"): e2m1 codes two per byte,
// the low nibble is the even column, bit 3 is the sign; one ue8m0 byte per
// 32 columns, weight = value * 2^(s - 127), s = 255 contributes nothing.
//
// The decode uses the sm_100-family conversion cvt.rn.f16x2.e2m1x2, which
// turns one byte (two codes) into two exact halves: the low nibble lands in
// the low half.  Every e2m1 value is exact in f16 and in fp32.

__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t q, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(q));
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t h) {
    __half2 v = *reinterpret_cast<__half2 *>(&h);
    return __half22float2(v);
}

// 2^(s - 127) for a ue8m0 byte s in 0..254 (s = 0 is the fp32 subnormal 2^-127)
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
    return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}

// One 32-column group: sum_i v_i x_i in fp32.  `w` holds the group's 16
// packed bytes; `x` holds its 32 activations as 16 (even, odd) pairs.  Two
// packed-fp32 accumulators (bytes 0,2 and 1,3 of each word) keep the FMA
// chains short; they are added at the end in a fixed order.
__device__ __forceinline__ float group_dot(const uint4 &w, const float2 (&x)[16]) {
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
        uint32_t h[4];
        e2m1x8_to_h2x4(words[q], h);
        a0 = __ffma2_rn(h2_to_f2(h[0]), x[4 * q + 0], a0);
        a1 = __ffma2_rn(h2_to_f2(h[1]), x[4 * q + 1], a1);
        a0 = __ffma2_rn(h2_to_f2(h[2]), x[4 * q + 2], a0);
        a1 = __ffma2_rn(h2_to_f2(h[3]), x[4 * q + 3], a1);
    }
    return (a0.x + a1.x) + (a0.y + a1.y);
}

// the scaled contribution of one group; a NaN scale (255) contributes 0 even
// when the activations hold inf or NaN
__device__ __forceinline__ float group_term(const uint4 &w, uint32_t s, const float2 (&x)[16]) {
    const float d = group_dot(w, x);
    return s == 255u ? 0.f : d * e8m0_to_f32(s);
}

// 32 fp32 activations of group g from a row of fp32 values (read-only path)
__device__ __forceinline__ void load_x_group(const float *row, int g, float2 (&x)[16]) {
    const float4 *p = reinterpret_cast<const float4 *>(row + 32 * g);
#pragma unroll
    for (int j = 0; j < 8; j++) {
        float4 v = __ldg(p + j);
        x[2 * j] = make_float2(v.x, v.y);
        x[2 * j + 1] = make_float2(v.z, v.w);
    }
}

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    // weights are read once: do not keep them in L1
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_u8(const uint8_t *p) {
    return (uint32_t)__ldg(p);
}

// SiTU-GLU (Kimi K3 engine (c/kimi_k3.c), "Architecture notes"; betas 4.0 and
// 25.0 from K3Cfg): 4 tanh(g/4) sigma(g) * 25 tanh(u/25), in fp32.
__device__ __forceinline__ float situ_glu(float g, float u) {
    const float sig = 1.0f / (1.0f + expf(-g));
    return (4.0f * tanhf(g * 0.25f) * sig) * (25.0f * tanhf(u / 25.0f));
}

__device__ __forceinline__ void report_status(int *status, int code, int detail) {
    if (status != nullptr && atomicCAS(status, 0, code) == 0) status[1] = detail;
}

// --------------------------------------------- async copies and barriers --
//
// Hand-written PTX for the bulk-copy engine (cp.async.bulk) and mbarriers.
// Every wait is bounded: after a number of polls it gives up and the caller
// reports kStatusWaitTimeout instead of spinning forever.  Waits for work
// take g_wait_polls polls (kWaitLimit unless k3mx_set_wait_limit changed it
// on this device); the waits a CTA makes on its way out (its copies in
// flight, its last MMAs before TMEM is freed) always take kWaitLimit, so a
// short limit never frees TMEM under a running MMA or leaves a copy landing
// in a finished CTA's shared memory.

constexpr uint32_t kWaitLimit = 1u << 22;

// One copy per translation unit (device code is not linked across files);
// every copy is set by k3mx_set_wait_limit through set_wait_polls_here().
static __device__ uint32_t g_wait_polls = kWaitLimit;
__device__ __forceinline__ uint32_t wait_polls() { return __ldg(&g_wait_polls); }
static inline cudaError_t set_wait_polls_here(uint32_t polls) {
    return cudaMemcpyToSymbol(g_wait_polls, &polls, sizeof(polls));
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// one poll; the thread may sleep in hardware up to kWaitSuspendNs while the
// phase is incomplete, so waiting warps do not compete for issue slots
constexpr uint32_t kWaitSuspendNs = 2000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kWaitSuspendNs)
        : "memory");
    return ok != 0;
}

// true when the phase of parity `parity` completed, false after wait_polls()
// polls (the limit is read only when the first poll fails)
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint32_t lim = wait_polls();
    for (uint32_t i = 1; i < lim; i++)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// the same with kWaitLimit polls: for the waits on a CTA's way out
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; i++)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// On a CTA's way out: wait until the last copy issued into each of the `n`
// slots of a ring has landed.  Uses are counted from 0, use u goes to slot
// u % n and completes one phase of that slot's barrier.  False if a wait
// gave up.
__device__ __forceinline__ bool drain_ring(uint32_t bar0, uint32_t n, uint32_t issued) {
    bool ok = true;
    for (uint32_t s = 0; s < n && s < issued; s++) {
        const uint32_t last = s + n * ((issued - 1 - s) / n);
        ok = mbar_wait_drain(bar0 + 8 * s, (last / n) & 1) && ok;
    }
    return ok;
}

// L2 policy for data read exactly once (weights): evict first
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared; completion is counted on `bar` in bytes.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

// programmatic dependent launch: let the next kernel in the stream start its
// independent prologue; wait until the previous kernel's results are visible
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// launch `kernel` as a programmatic dependent of the previous kernel in the
// stream (it may start before that kernel ends and must call pdl_wait
// before reading its results)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------ tracing --
// Launch tracing (k3mx_trace_enable): an event pair on the launch stream
// around each traced launch.  Defined in abi.cu.
bool trace_begin(cudaStream_t s, int *slot);
void trace_end(cudaStream_t s, int slot, const char *name);

template <typename F>
cudaError_t traced(const char *name, cudaStream_t s, F launch) {
    int slot = 0;
    const bool on = trace_begin(s, &slot);
    const cudaError_t err = launch();
    if (on) trace_end(s, slot, name);
    return err;
}

// ------------------------------------------------------------ launchers --
// (defined in the .cu files; called by the C-ABI layer)

// Work units of the decode kernels: each active expert's pairs cut into
// runs of at most kUnitPairs, so one unit has one fixed token set.
constexpr int kUnitPairs = 4;
inline int max_units(int n_tokens) {
    const int pairs = n_tokens * kK;
    const int experts = pairs < kE ? pairs : kE;
    return pairs / kUnitPairs + experts;
}

struct GroupOut {
    int32_t *counts;     // [896]
    int32_t *offsets;    // [897]
    int32_t *perm;       // [16 T]
    int32_t *act;        // [896] active experts, increasing id
    int32_t *n_active;   // [1]
    int32_t *units;      // [max_units][3]: expert, first pair slot, end slot (or null)
    int32_t *n_units;    // [1] (or null)
};

// top_p > 0: the low-weight tail of each token's 16 experts is dropped
// (index -1, weight 0), the kept weights renormalised
cudaError_t launch_route(const Ctx &c, int32_t *idx, float *w, const float *logits,
                         const float *bias, int n_tokens, double top_p,
                         bool pdl = false);
// router logits [T][896] = W [896][7168] (bf16) times hidden [T][7168] (fp32
// or bf16), launched as a programmatic dependent
cudaError_t launch_router_logits(const Ctx &c, float *logits, const void *h, int h_bf16, const uint16_t *W,
                                 int n_tokens);
// routing with one CTA per token (n_tokens <= 64) plus, when x is given, the
// tokens' x piece images and the weight tensor maps of the expert table
// (mx path) in the same launch; a single token with `g_one` is also
// grouped there (else group with launch_group_small)
cudaError_t launch_route_prep(const Ctx &c, int32_t *idx, float *w, const float *logits,
                              const float *bias, int n_tokens, const void *x, int x_bf16,
                              uint8_t *ximg, const GroupOut *g_one, int *flags, int n_flags,
                              const k3mx_expert *experts, uint8_t *maps, double top_p,
                              bool pdl = false);
// grouping of n_tokens * 16 <= 1024 pairs, programmatic dependent of the routing
cudaError_t launch_group_small(const Ctx &c, const int32_t *idx, int n_tokens, const GroupOut &g);
size_t group_scratch_bytes(int n_tokens);
cudaError_t launch_group(const Ctx &c, const int32_t *idx, int n_tokens, const GroupOut &g,
                         void *scratch);

cudaError_t launch_gemv(const Ctx &c, float *y, const float *x, const uint8_t *packed,
                        const uint8_t *scales, int in, int rows);

// Decode path over the grouped pairs.  x: [T][D] fp32; gu: [16T][2][F] fp32
// (g = W1 x and u = W3 x per pair); stage: [16T][D] fp32 (W2 SiTU(g, u) per
// pair); y: [T][D] fp32.  When `single` is non-null the grouping arguments
// are ignored and the one expert runs for token 0.
struct DecodeExperts {
    const k3mx_expert *experts;   // device [896]
    const k3mx_expert *single;    // host struct, or nullptr
    const int32_t *units, *n_units, *perm;
    int max_units;                // upper bound of *n_units
};
cudaError_t launch_combine(const Ctx &c, float *y, const float *stage, const float *w,
                           int n_tokens);

// The poll limit of the bounded waits in each kernel file, on the current
// device (k3mx_set_wait_limit).
cudaError_t set_wait_polls_mx(uint32_t polls);
cudaError_t set_wait_polls_px(uint32_t polls);
cudaError_t set_wait_polls_prefill(uint32_t polls);
cudaError_t set_wait_polls_decode(uint32_t polls);
cudaError_t set_wait_polls_dense(uint32_t polls);

// Host side.  The library's lazily filled per-device state (device
// properties, CUDA function attributes, tensor-map templates, the fixed
// scratch array's address) is set up under one lock, with a flag read
// without the lock afterwards, so first calls from several host threads
// are safe.
std::mutex &setup_mutex();
// cudaFuncSetAttribute(max dynamic shared memory) once per kernel and
// device; `done` holds one bit per device
cudaError_t ensure_smem(const void *fn, int bytes, std::atomic<uint64_t> &done);
// the largest shared-memory carve-out for `fn`, once per device
cudaError_t ensure_max_carveout(const void *fn, std::atomic<uint64_t> &done);

// The library's fixed device scratch array (abi.cu): its address on the
// current device, looked up on first use, and its size.
void *library_scratch();
size_t library_scratch_bytes();

// Block-scaled tensor-core decode path (mx.cu).  Piece images: every token's
// x and every pair's h split exactly into MXFP4 pieces in the layout the
// MMA reads; tensor-map slots: per-CTA copies of the weight tensor maps.
size_t mx_ximg_bytes(int n_tokens);
size_t mx_himg_bytes(int n_pairs);
size_t mx_maps_bytes(int n_experts);
// stream-K hand-over region of single-token decode (flags + partials); the
// step's first kernel zeroes the mx_streamk_flag_count() flags at its start
size_t mx_streamk_bytes();
int mx_streamk_flag_count();
// x pieces of every token, the weight tensor maps of the expert table (or
// of the single expert `one`), and, with `sk`, the stream-K flags zeroed
cudaError_t launch_mx_ximg(const Ctx &c, const void *x, int x_bf16, int n_tokens, uint8_t *ximg, uint8_t *sk,
                           uint8_t *maps, const k3mx_expert *table, const k3mx_expert *one);
// gate/up: g, u -> gu [pair][2][F]; h = SiTU(g, u) -> piece images himg
cudaError_t launch_mx_gate_up(const Ctx &c, const DecodeExperts &d, const uint8_t *ximg, uint8_t *himg,
                              float *gu, uint8_t *maps);
// one token (a batch of one, or one expert with w = null): gate/up, down and
// the weighted sum in one persistent launch; y [D] written, per-pair rows
// in `stage` (with w), g and u in `gu`; a dependent of the step's first kernel
cudaError_t launch_mx_fused1(const Ctx &c, const DecodeExperts &d, const uint8_t *ximg, uint8_t *himg, float *gu,
                             float *stage, const float *w, float *y, const uint8_t *maps, uint8_t *sk);
// down: W2 h of every pair -> out [pair][D] (launched as a dependent of gate/up)
cudaError_t launch_mx_down(const Ctx &c, const DecodeExperts &d, const uint8_t *himg, float *out,
                           uint8_t *maps);

}  // namespace k3mx

namespace k3mx {

// ------------------------------------------------------- tcgen05 / TMEM --
//
// Hand-written PTX for the 5th-generation tensor cores (sm_100 family).

// shared-memory matrix descriptor, K-major operand in the 128-byte swizzled
// canonical layout: 8-row atoms of 128-byte rows (1024 bytes), 16-byte
// chunks XOR-permuted by row % 8; the stride between 8-row atoms is 1024.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)(16u >> 4) << 16;                   // leading byte offset (unused for SW128 K-major)
    d |= (uint64_t)(1024u >> 4) << 32;                 // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                            // descriptor version (sm_100)
    d |= (uint64_t)2 << 61;                            // layout: 128-byte swizzle
    return d;
}

// instruction descriptor, kind::f16: f16 A and B, f32 accumulator, both
// K-major, shape M x N
__device__ __forceinline__ uint32_t umma_idesc_f16(int m, int n) {
    return (1u << 4)                                   // D format f32
           | (0u << 7) | (0u << 10)                    // A, B format f16
           | ((uint32_t)(n >> 3) << 17)                // N / 8
           | ((uint32_t)(m >> 4) << 24);               // M / 16
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on `bar` once every tcgen05 operation issued so far by this thread completed
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// generic-proxy shared-memory writes become visible to the tensor core
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
        "[%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16-byte asynchronous copy global -> shared (bytes beyond src_bytes are zero)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
// arrive on `bar` once this thread's earlier cp.async copies landed
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// byte offset of 16-byte chunk j of row r inside a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128_offset(int r, int j) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

}  // namespace k3mx
