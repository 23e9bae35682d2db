// abi.cu - the extern "C" entry points of libk3mx.so: argument checks,
// workspace layout and kernel launches.  No entry point allocates device
// memory; scratch lives in the caller's workspace.
#include <initializer_list>
#include <cmath>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "dense.cuh"
#include "prefill.cuh"

namespace k3mx {
namespace {

__device__ int g_status[4];       // [0] first failure code, [1] detail

constexpr int kMaxDevices = 64;
struct DevInfo {
    std::atomic<bool> init;               // set last, after the fields below
    bool ok;
    int num_sms;
    int *status;
};
DevInfo g_dev[kMaxDevices];

// Per-device set-up on first use: capability check, SM count, and the device
// address of the status word.
k3mx_status device_ctx(cudaStream_t stream, Ctx &c) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return K3MX_ECUDA;
    DevInfo &di = g_dev[dev];
    if (!di.init.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(setup_mutex());
        if (!di.init.load(std::memory_order_relaxed)) {
            int major = 0, minor = 0, sms = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return K3MX_ECUDA;
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return K3MX_ECUDA;
            di.ok = (major == 10 && minor == 3);
            di.num_sms = sms;
            di.status = static_cast<int *>(p);
            di.init.store(true, std::memory_order_release);
        }
    }
    if (!di.ok) return K3MX_EDEVICE;
    c.stream = stream;
    c.num_sms = di.num_sms;
    c.status = di.status;
    return K3MX_OK;
}

// Scratch of k3mx_moe_decode_noalloc.  Callers that may not allocate
// device memory when they run the layer (a runtime that keeps the whole
// memory budget to itself and hands out no scratch, a loop that must not
// take the synchronisation an allocation can imply) use this fixed array
// instead of a workspace.  The decode path writes every scratch word
// before it reads it, so nothing here needs clearing between calls.
constexpr size_t kNoallocBytes = size_t(8) << 20;
__device__ __align__(256) unsigned char g_noalloc_ws[kNoallocBytes];
std::atomic<void *> g_noalloc_ptr[kMaxDevices];

}  // namespace

std::mutex &setup_mutex() {
    static std::mutex m;
    return m;
}

cudaError_t ensure_smem(const void *fn, int bytes, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const uint64_t bit = uint64_t(1) << dev;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    std::lock_guard<std::mutex> lock(setup_mutex());
    if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// A small kernel that precedes a large-shared-memory one (with programmatic
// dependent launch) asks for the largest shared-memory carve-out: an SM that
// runs it is then already configured for the next kernel's CTA, which can
// start there at once instead of waiting for the SM to drain.
cudaError_t ensure_max_carveout(const void *fn, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const uint64_t bit = uint64_t(1) << dev;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    std::lock_guard<std::mutex> lock(setup_mutex());
    if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Device address of the library's fixed scratch array on the current device
// (looked up once per device), or nullptr.
void *library_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void *p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(setup_mutex());
        p = g_noalloc_ptr[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess) return nullptr;
            g_noalloc_ptr[dev].store(p, std::memory_order_release);
        }
    }
    return p;
}
size_t library_scratch_bytes() { return kNoallocBytes; }

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline size_t up256(size_t n) { return (n + 255) & ~size_t(255); }

bool expert_ok(const k3mx_expert *e) {
    return e && e->w1 && e->s1 && e->w3 && e->s3 && e->w2 && e->s2 && aligned16(e->w1) &&
           aligned16(e->s1) && aligned16(e->w3) && aligned16(e->s3) && aligned16(e->w2) &&
           aligned16(e->s2);
}

// the last CUDA error a call of this thread reported as K3MX_ECUDA
thread_local cudaError_t g_last_cuda = cudaSuccess;

k3mx_status from_cuda(cudaError_t err) {
    if (err == cudaSuccess) return K3MX_OK;
    g_last_cuda = err;
    return K3MX_ECUDA;
}

// the device address of a page-locked host buffer mapped into the device's
// address space, or nullptr (pageable or unknown memory)
const void *mapped_host(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();                       // clear the sticky-free error state
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// ---------------------------------------------------------------- tracing --

constexpr int kTracePool = 8192;
struct TraceRec {
    const char *name;
    int slot;
};
bool g_trace_on = false;
cudaEvent_t g_ev[kTracePool][2];
int g_ev_made = 0;
TraceRec g_rec[kTracePool];
int g_nrec = 0;

}  // namespace

// The event pair of the next traced launch, or false when tracing is off or
// the pool is used up.
bool trace_begin(cudaStream_t s, int *slot) {
    if (!g_trace_on || g_nrec >= kTracePool) return false;
    const int k = g_nrec;
    if (k >= g_ev_made) {
        if (cudaEventCreate(&g_ev[k][0]) != cudaSuccess || cudaEventCreate(&g_ev[k][1]) != cudaSuccess)
            return false;
        g_ev_made = k + 1;
    }
    cudaEventRecord(g_ev[k][0], s);
    *slot = k;
    return true;
}

void trace_end(cudaStream_t s, int slot, const char *name) {
    cudaEventRecord(g_ev[slot][1], s);
    g_rec[g_nrec++] = TraceRec{name, slot};
}

namespace {

// ------------------------------------------------------- workspace layout --

struct MoeLayout {
    size_t idx, w, counts, offsets, act, n_active, units, n_units, perm, hist, ximg, himg, maps, sk, h,
        stage, total;
    // prefill-only regions
    size_t pre;
    // host-variant staging
    size_t x_in, logits_in, bias_in, y_out, total_host;
};

int resolve_path(int n_tokens, int x_dtype, int path) {
    if (path == K3MX_PATH_AUTO)
        return (x_dtype == K3MX_BF16 && n_tokens >= K3MX_PREFILL_MIN_TOKENS) ? K3MX_PATH_PREFILL_MX
                                                                             : K3MX_PATH_DECODE;
    return path;
}

MoeLayout moe_layout(int n_tokens, int x_dtype, int path) {
    MoeLayout L{};
    const size_t P = (size_t)n_tokens * kK;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += up256(bytes);
        return at;
    };
    L.idx = take(P * 4);
    L.w = take(P * 4);
    L.counts = take(kE * 4);
    L.offsets = take((kE + 1) * 4);
    L.act = take(kE * 4);
    L.n_active = take(4);
    L.units = take((size_t)max_units(n_tokens) * 3 * 4);
    L.n_units = take(4);
    L.perm = take(P * 4);
    L.hist = take(group_scratch_bytes(n_tokens));
    if (path == K3MX_PATH_DECODE) {
        L.ximg = take(mx_ximg_bytes(n_tokens));  // x of every token as MXFP4 pieces
        L.himg = take(mx_himg_bytes((int)P));    // h of every pair as MXFP4 pieces
        L.maps = take(mx_maps_bytes(kE));          // weight tensor maps of the expert table
        L.sk = n_tokens == 1 ? take(mx_streamk_bytes()) : 0;   // stream-K hand-over (one token)
        L.h = take(P * 2 * kF * 4);          // g and u per pair
        L.stage = take(P * kD * 4);
    } else if (path == K3MX_PATH_PREFILL_MX) {
        L.pre = take(prefill_mx_scratch_bytes(n_tokens));
    } else {
        L.pre = take(prefill_scratch_bytes(n_tokens));
    }
    L.total = o;
    L.x_in = take((size_t)n_tokens * kD * (x_dtype == K3MX_BF16 ? 2 : 4));
    L.logits_in = take((size_t)n_tokens * kE * 4);
    L.bias_in = take(kE * 4);
    L.y_out = take((size_t)n_tokens * kD * 4);
    L.total_host = o;
    return L;
}

template <typename T>
T *at(void *base, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(base) + off);
}

k3mx_status check_moe_args(const void *y, const void *x, int x_dtype, int n_tokens,
                           const k3mx_expert *experts, const float *logits, const float *bias,
                           int path) {
    if (!y || !x || !experts || !logits || !bias) return K3MX_EINVAL;
    if (x_dtype != K3MX_F32 && x_dtype != K3MX_BF16) return K3MX_EINVAL;
    if (path < K3MX_PATH_AUTO || path > K3MX_PATH_PREFILL_MX) return K3MX_EINVAL;
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return K3MX_ESHAPE;
    if (resolve_path(n_tokens, x_dtype, path) >= K3MX_PATH_PREFILL && x_dtype != K3MX_BF16)
        return K3MX_EINVAL;
    if (!aligned16(y) || !aligned16(x) || !aligned16(logits) || !aligned16(bias) ||
        !aligned16(experts))
        return K3MX_EALIGN;
    return K3MX_OK;
}

// The layer on device buffers; `ws` is already checked.
k3mx_status run_moe(const Ctx &c, float *y, const void *x, int x_dtype, int n_tokens,
                    const k3mx_expert *experts, const float *logits, const float *bias, int path,
                    int32_t *idx_out, float *w_out, void *ws, const MoeLayout &L, double top_p = 0.0) {
    int32_t *idx = idx_out ? idx_out : at<int32_t>(ws, L.idx);
    float *w = w_out ? w_out : at<float>(ws, L.w);
    GroupOut g{at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.perm),
               at<int32_t>(ws, L.act), at<int32_t>(ws, L.n_active), at<int32_t>(ws, L.units),
               at<int32_t>(ws, L.n_units)};
    cudaError_t err;
    const bool decode = path == K3MX_PATH_DECODE;
    uint8_t *ximg = decode ? at<uint8_t>(ws, L.ximg) : nullptr;
    uint8_t *sk = decode && n_tokens == 1 ? at<uint8_t>(ws, L.sk) : nullptr;
    const int x_bf16 = x_dtype == K3MX_BF16 ? 1 : 0;
    bool pieces_done = false;
    if (n_tokens * kK <= 1024) {
        // one CTA per token, the decode path's x pieces in the same launch;
        // grouping as a programmatic dependent.  Every block of the routing
        // kernel waits for the kernel before it first thing, so it too is
        // launched as a programmatic dependent (of whatever came before).
        const bool one = n_tokens == 1 && g.units != nullptr;
        err = traced("route", c.stream, [&] {
            return launch_route_prep(c, idx, w, logits, bias, n_tokens, decode ? x : nullptr, x_bf16, ximg,
                                     one ? &g : nullptr, reinterpret_cast<int *>(sk), mx_streamk_flag_count(),
                                     decode ? experts : nullptr, decode ? at<uint8_t>(ws, L.maps) : nullptr, top_p,
                                     true);
        });
        if (err == cudaSuccess && !one)
            err = traced("group_small", c.stream, [&] { return launch_group_small(c, idx, n_tokens, g); });
        pieces_done = decode;
    } else {
        err = traced("route", c.stream,
                     [&] { return launch_route(c, idx, w, logits, bias, n_tokens, top_p); });
        if (err == cudaSuccess)
            err = traced("group", c.stream,
                         [&] { return launch_group(c, idx, n_tokens, g, at<void>(ws, L.hist)); });
    }
    if (err != cudaSuccess) return from_cuda(err);
    const int max_active = n_tokens * kK < kE ? n_tokens * kK : kE;

    if (path == K3MX_PATH_PREFILL || path == K3MX_PATH_PREFILL_MX) {
        PrefillArgs a{};
        a.y = y;
        a.x = static_cast<const uint16_t *>(x);
        a.n_tokens = n_tokens;
        a.experts = experts;
        a.w = w;
        a.counts = g.counts;
        a.offsets = g.offsets;
        a.perm = g.perm;
        a.act = g.act;
        a.n_active = g.n_active;
        a.max_active = max_active;
        a.scratch = at<void>(ws, L.pre);
        // traced per kernel inside
        return from_cuda(path == K3MX_PATH_PREFILL_MX ? launch_prefill_mx(c, a) : launch_prefill(c, a));
    }

    DecodeExperts d{experts, nullptr, g.units, g.n_units, g.perm, max_units(n_tokens)};
    uint8_t *himg = at<uint8_t>(ws, L.himg), *maps = at<uint8_t>(ws, L.maps);
    float *gu = at<float>(ws, L.h);
    float *stage = at<float>(ws, L.stage);
    if (!pieces_done)
        err = traced("mx_pieces", c.stream,
                     [&] { return launch_mx_ximg(c, x, x_bf16, n_tokens, ximg, sk, maps, experts, nullptr); });
    if (err == cudaSuccess && n_tokens == 1) {
        // one token: gate/up, down and the weighted sum in one launch
        err = traced("decode_expert", c.stream,
                     [&] { return launch_mx_fused1(c, d, ximg, himg, gu, stage, w, y, maps, sk); });
        return from_cuda(err);
    }
    if (err == cudaSuccess)
        err = traced("decode_gate_up", c.stream,
                     [&] { return launch_mx_gate_up(c, d, ximg, himg, gu, maps); });
    if (err == cudaSuccess)
        err = traced("decode_down", c.stream,
                     [&] { return launch_mx_down(c, d, himg, stage, maps); });
    if (err == cudaSuccess)
        err = traced("combine", c.stream, [&] { return launch_combine(c, y, stage, w, n_tokens); });
    return from_cuda(err);
}

// ------------------------------------------------ the LatentMoE block --

constexpr int kHid = 7168, kFs = 6144;           // hidden width, fused shared experts' inter width
static_assert(kLatentOutK1 == kD && kLatentOutK == kD + kFs, "the output product's two parts");

struct LatentLayout {
    size_t logits, xlat, ylat, gu, ysh, act, z, moe, total;
    bool batched;
    int moe_path;
    MoeLayout moe_l;
};

LatentLayout latent_layout(int n_tokens, int h_dtype) {
    LatentLayout L{};
    const size_t T = (size_t)n_tokens;
    L.batched = h_dtype == K3MX_BF16 && n_tokens >= kDenseGemmMinTokens;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += up256(bytes);
        return o;
    };
    L.logits = take(T * kE * 4);
    L.xlat = take(T * kD * (L.batched ? 2 : 4));
    L.ylat = take(T * kD * 4);
    L.gu = take(T * 2 * kFs * 4);
    L.ysh = take(T * kHid * 4);
    L.act = L.batched ? take(T * kFs * 2) : 0;
    L.z = L.batched ? take(T * kD * 2) : 0;
    const int x_dtype = L.batched ? K3MX_BF16 : K3MX_F32;
    L.moe_path = resolve_path(n_tokens, x_dtype, K3MX_PATH_AUTO);
    L.moe_l = moe_layout(n_tokens, x_dtype, L.moe_path);
    L.moe = take(L.moe_l.total);
    L.total = off;
    return L;
}

}  // namespace
}  // namespace k3mx

using namespace k3mx;

extern "C" {

int k3mx_abi_version(void) { return (1 << 16) | 0; }

const char *k3mx_last_cuda_error(void) {
    return g_last_cuda == cudaSuccess ? "cudaSuccess" : cudaGetErrorName(g_last_cuda);
}

const char *k3mx_status_str(k3mx_status s) {
    switch (s) {
    case K3MX_OK: return "ok";
    case K3MX_EINVAL: return "invalid argument";
    case K3MX_EALIGN: return "pointer not aligned as required";
    case K3MX_ESHAPE: return "size out of range";
    case K3MX_EWORKSPACE: return "workspace missing or too small";
    case K3MX_ECUDA: return "CUDA error";
    case K3MX_ETIMEOUT: return "device wait timed out";
    case K3MX_EDEVICE: return "device is not sm_103";
    }
    return "unknown status";
}

k3mx_status k3mx_gemv(float *y, const float *x, const uint8_t *packed, const uint8_t *scales,
                      int in, int rows, k3mx_stream_t stream) {
    if (!y || !x || !packed || !scales) return K3MX_EINVAL;
    if (in < 32 || in > 16384 || in % 32 != 0 || rows < 1 || rows > (1 << 24)) return K3MX_ESHAPE;
    if (!aligned16(y) || !aligned16(x) || !aligned16(packed)) return K3MX_EALIGN;
    Ctx c;
    k3mx_status st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    return from_cuda(traced("gemv", c.stream,
                            [&] { return launch_gemv(c, y, x, packed, scales, in, rows); }));
}

// expert_ffn workspace: g and u [2][F] fp32, x and h piece images, tensor-map slots
size_t k3mx_expert_ffn_workspace_size(void) {
    return up256((size_t)2 * kF * sizeof(float)) + up256(mx_ximg_bytes(1)) + up256(mx_himg_bytes(1)) +
           up256(mx_maps_bytes(1)) + up256(mx_streamk_bytes());
}

k3mx_status k3mx_expert_ffn(float *y, const float *x, const k3mx_expert *expert, void *workspace,
                            size_t ws_bytes, k3mx_stream_t stream) {
    if (!y || !x || !expert) return K3MX_EINVAL;
    if (!expert_ok(expert))
        return expert->w1 && expert->s1 && expert->w3 && expert->s3 && expert->w2 && expert->s2
                   ? K3MX_EALIGN
                   : K3MX_EINVAL;
    if (!aligned16(y) || !aligned16(x)) return K3MX_EALIGN;
    if (!workspace || ws_bytes < k3mx_expert_ffn_workspace_size()) return K3MX_EWORKSPACE;
    if (!aligned256(workspace)) return K3MX_EALIGN;
    Ctx c;
    k3mx_status st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    DecodeExperts d{nullptr, expert, nullptr, nullptr, nullptr, 1};
    char *ws = static_cast<char *>(workspace);
    float *gu = reinterpret_cast<float *>(ws);
    uint8_t *ximg = reinterpret_cast<uint8_t *>(ws + up256((size_t)2 * kF * sizeof(float)));
    uint8_t *himg = ximg + up256(mx_ximg_bytes(1));
    uint8_t *maps = himg + up256(mx_himg_bytes(1));
    uint8_t *sk = maps + up256(mx_maps_bytes(1));
    cudaError_t err = traced("mx_pieces", c.stream,
                             [&] { return launch_mx_ximg(c, x, 0, 1, ximg, sk, maps, nullptr, expert); });
    if (err == cudaSuccess)
        err = traced("decode_expert", c.stream,
                     [&] { return launch_mx_fused1(c, d, ximg, himg, gu, nullptr, nullptr, y, maps, sk); });
    return from_cuda(err);
}

k3mx_status k3mx_route_topk(int32_t *idx, float *w, const float *logits, const float *bias,
                            int n_tokens, k3mx_stream_t stream) {
    if (!idx || !w || !logits || !bias) return K3MX_EINVAL;
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return K3MX_ESHAPE;
    if (!aligned16(idx) || !aligned16(w) || !aligned16(logits) || !aligned16(bias))
        return K3MX_EALIGN;
    Ctx c;
    k3mx_status st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    return from_cuda(traced("route", c.stream,
                            [&] { return launch_route(c, idx, w, logits, bias, n_tokens, 0.0); }));
}

k3mx_status k3mx_route_topp(int32_t *idx, float *w, const float *logits, const float *bias,
                            int n_tokens, float top_p, k3mx_stream_t stream) {
    if (!idx || !w || !logits || !bias) return K3MX_EINVAL;
    if (!(top_p == top_p) || top_p == INFINITY || top_p == -INFINITY) return K3MX_EINVAL;
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return K3MX_ESHAPE;
    if (!aligned16(idx) || !aligned16(w) || !aligned16(logits) || !aligned16(bias))
        return K3MX_EALIGN;
    Ctx c;
    k3mx_status st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    return from_cuda(traced("route", c.stream,
                            [&] { return launch_route(c, idx, w, logits, bias, n_tokens, (double)top_p); }));
}

k3mx_status k3mx_router(float *logits, int32_t *idx, float *w, const void *hidden, int h_dtype,
                        const uint16_t *router_w, const float *bias, int n_tokens, float top_p,
                        k3mx_stream_t stream) {
    if (!logits || !idx || !w || !hidden || !router_w || !bias) return K3MX_EINVAL;
    if (h_dtype != K3MX_F32 && h_dtype != K3MX_BF16) return K3MX_EINVAL;
    if (!(top_p == top_p) || top_p == INFINITY || top_p == -INFINITY) return K3MX_EINVAL;
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return K3MX_ESHAPE;
    if (!aligned16(logits) || !aligned16(idx) || !aligned16(w) || !aligned16(hidden) || !aligned16(router_w) ||
        !aligned16(bias))
        return K3MX_EALIGN;
    Ctx c;
    k3mx_status st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    cudaError_t err = traced("router", c.stream, [&] {
        return launch_router_logits(c, logits, hidden, h_dtype == K3MX_BF16 ? 1 : 0, router_w, n_tokens);
    });
    if (err != cudaSuccess) return from_cuda(err);
    // the top-16 as a programmatic dependent of the logits
    err = traced("route", c.stream, [&] {
        return n_tokens * kK <= 1024
                   ? launch_route_prep(c, idx, w, logits, bias, n_tokens, nullptr, 0, nullptr, nullptr, nullptr, 0,
                                       nullptr, nullptr, (double)top_p, true)
                   : launch_route(c, idx, w, logits, bias, n_tokens, (double)top_p, true);
    });
    return from_cuda(err);
}

size_t k3mx_latent_moe_workspace_size(int n_tokens, int h_dtype) {
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return 0;
    if (h_dtype != K3MX_F32 && h_dtype != K3MX_BF16) return 0;
    return latent_layout(n_tokens, h_dtype).total;
}

k3mx_status k3mx_latent_moe(float *y, const void *hidden, int h_dtype, int n_tokens, const k3mx_latent_block *blk,
                            const k3mx_expert *experts, float top_p, int32_t *idx_out, float *w_out,
                            void *workspace, size_t ws_bytes, k3mx_stream_t stream) {
    if (!y || !hidden || !blk || !experts) return K3MX_EINVAL;
    if (!blk->router_w || !blk->bias || !blk->w_dn || !blk->w_up || !blk->g_norm || !blk->w1s || !blk->w3s ||
        !blk->w2s)
        return K3MX_EINVAL;
    if (h_dtype != K3MX_F32 && h_dtype != K3MX_BF16) return K3MX_EINVAL;
    if (!(top_p == top_p) || top_p == INFINITY || top_p == -INFINITY) return K3MX_EINVAL;
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return K3MX_ESHAPE;
    if (!aligned16(y) || !aligned16(hidden) || !aligned16(experts) || !aligned16(blk->router_w) ||
        !aligned16(blk->bias) || !aligned16(blk->w_dn) || !aligned16(blk->w_up) || !aligned16(blk->g_norm) ||
        !aligned16(blk->w1s) || !aligned16(blk->w3s) || !aligned16(blk->w2s) ||
        (idx_out && !aligned16(idx_out)) || (w_out && !aligned16(w_out)))
        return K3MX_EALIGN;
    const LatentLayout L = latent_layout(n_tokens, h_dtype);
    if (!workspace || ws_bytes < L.total) return K3MX_EWORKSPACE;
    if (!aligned256(workspace)) return K3MX_EALIGN;
    Ctx c;
    k3mx_status st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    const int T = n_tokens;
    const int h_bf16 = h_dtype == K3MX_BF16 ? 1 : 0;
    float *logits = at<float>(workspace, L.logits), *ylat = at<float>(workspace, L.ylat);
    float *gu = at<float>(workspace, L.gu), *ysh = at<float>(workspace, L.ysh);
    void *xlat = at<void>(workspace, L.xlat);
    // a CUDA-core product over up to four weight matrices sharing one input
    auto gemv = [&](std::initializer_list<GemvSeg> segs, const void *x, int x_bf16, int ldx, int K, int xf,
                    const int *rows) {
        GemvArgs a{};
        int r = 0, k = 0;
        for (const GemvSeg &sg : segs) {
            a.seg[k] = sg;
            a.seg[k].r0 = r;
            r += rows[k++];
        }
        a.n_seg = k;
        a.rows = r;
        a.x = x;
        a.x_bf16 = x_bf16;
        a.ldx = ldx;
        a.g = blk->g_norm;
        a.n_tokens = T;
        a.status = c.status;
        return launch_dense_gemv(c, K, xf, a);
    };
    const uint16_t *hb = static_cast<const uint16_t *>(hidden);
    cudaError_t err = cudaSuccess;
    if (!L.batched) {
        // 1. every product over the hidden state in one launch: the router's
        // logits, the latent x = W_dn h (7168 -> 3584) and the fused shared
        // experts' g | u
        const int rows[4] = {kE, kD, kFs, kFs};
        err = traced("hidden_products", c.stream, [&] {
            return gemv({GemvSeg{blk->router_w, logits, nullptr, kE, 0},
                         GemvSeg{blk->w_dn, static_cast<float *>(xlat), nullptr, kD, 0},
                         GemvSeg{blk->w1s, gu, nullptr, 2 * kFs, 0}, GemvSeg{blk->w3s, gu + kFs, nullptr, 2 * kFs, 0}},
                        hidden, h_bf16, kHid, kHid, kXfPlain, rows);
        });
    } else {
        // 1. the router's logits, the latent x = W_dn h (7168 -> 3584) in bf16
        err = traced("router", c.stream,
                     [&] { return launch_router_logits(c, logits, hidden, h_bf16, blk->router_w, T); });
        if (err == cudaSuccess)
            err = traced("latent_down", c.stream, [&] {
                return launch_dense_gemm(c, kHid, blk->w_dn, kD, hb, T, nullptr, static_cast<uint16_t *>(xlat), kD,
                                         0, nullptr);
            });
    }
    if (err != cudaSuccess) return from_cuda(err);
    // 2. the routed experts on the latent: route, group, experts, weighted sum
    st = run_moe(c, ylat, xlat, L.batched ? K3MX_BF16 : K3MX_F32, T, experts, logits, blk->bias,
                 L.moe_path, idx_out, w_out, at<void>(workspace, L.moe), L.moe_l, (double)top_p);
    if (st != K3MX_OK) return st;
    // 3. the fused shared experts' g | u on the hidden state (tensor cores)
    if (L.batched)
        err = traced("shared_gate_up", c.stream, [&] {
            return launch_dense_gemm2(c, kHid, blk->w1s, blk->w3s, kFs, hb, T, gu, 2 * kFs, 0, kFs);
        });
    if (!L.batched) {
        // 4. y = W_up (RMSNorm(routed sum) * g_norm) + W2s SiTU-GLU(g, u) as
        // one product over the two inputs side by side (3584 -> 7168 and
        // the shared experts' 6144 -> 7168)
        if (err == cudaSuccess)
            err = traced("latent_out", c.stream, [&] {
                GemvArgs a{};
                a.seg[0] = GemvSeg{blk->w_up, y, nullptr, kHid, 0};
                a.n_seg = 1;
                a.rows = kHid;
                a.x = ylat;
                a.ldx = kD;
                a.g = blk->g_norm;
                a.x2 = gu;
                a.ldx2 = 2 * kFs;
                a.Wt = blk->w2s;
                a.n_tokens = T;
                a.status = c.status;
                return launch_dense_gemv(c, kLatentOutK, kXfLatentOut, a);
            });
        return from_cuda(err);
    }
    // 4. the shared experts' down projection of SiTU-GLU(g, u)
    if (err == cudaSuccess)
        err = traced("shared_down", c.stream, [&] {
            uint16_t *act = at<uint16_t>(workspace, L.act);
            cudaError_t e = launch_situ_bf16(c, gu, kFs, T, act);
            if (e == cudaSuccess) e = launch_dense_gemm(c, kFs, blk->w2s, kHid, act, T, ysh, nullptr, kHid, 0, nullptr);
            return e;
        });
    // 5. y = W_up RMSNorm(routed sum) + shared (3584 -> 7168)
    if (err == cudaSuccess)
        err = traced("latent_up", c.stream, [&] {
            uint16_t *z = at<uint16_t>(workspace, L.z);
            cudaError_t e = launch_rmsnorm_bf16(c, ylat, blk->g_norm, kD, T, z);
            if (e == cudaSuccess) e = launch_dense_gemm(c, kD, blk->w_up, kHid, z, T, y, nullptr, kHid, 0, ysh);
            return e;
        });
    return from_cuda(err);
}

size_t k3mx_group_workspace_size(int n_tokens) {
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return 0;
    return up256((kE + 1) * 4) + up256(kE * 4) + up256(group_scratch_bytes(n_tokens));
}

k3mx_status k3mx_group(int32_t *counts, int32_t *offsets, int32_t *perm, const int32_t *idx,
                       int n_tokens, void *workspace, size_t ws_bytes, k3mx_stream_t stream) {
    if (!counts || !offsets || !perm || !idx) return K3MX_EINVAL;
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return K3MX_ESHAPE;
    if (!aligned16(counts) || !aligned16(offsets) || !aligned16(perm) || !aligned16(idx))
        return K3MX_EALIGN;
    if (!workspace || ws_bytes < k3mx_group_workspace_size(n_tokens)) return K3MX_EWORKSPACE;
    if (!aligned16(workspace)) return K3MX_EALIGN;
    Ctx c;
    k3mx_status st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    // the active-expert list is a by-product of the scan: keep it in the workspace
    char *ws = static_cast<char *>(workspace);
    GroupOut g{counts, offsets, perm, reinterpret_cast<int32_t *>(ws + up256((kE + 1) * 4)),
               reinterpret_cast<int32_t *>(ws), nullptr, nullptr};
    return from_cuda(traced("group", c.stream, [&] {
        return launch_group(c, idx, n_tokens, g, ws + up256((kE + 1) * 4) + up256(kE * 4));
    }));
}

size_t k3mx_moe_workspace_size(int n_tokens, int x_dtype, int path) {
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return 0;
    if (x_dtype != K3MX_F32 && x_dtype != K3MX_BF16) return 0;
    return moe_layout(n_tokens, x_dtype, resolve_path(n_tokens, x_dtype, path)).total;
}

k3mx_status k3mx_moe_decode_noalloc(float *y, const void *x, int x_dtype, int n_tokens,
                                    const k3mx_expert *experts, const float *logits,
                                    const float *bias, int32_t *idx_out, float *w_out,
                                    k3mx_stream_t stream) {
    k3mx_status st =
        check_moe_args(y, x, x_dtype, n_tokens, experts, logits, bias, K3MX_PATH_DECODE);
    if (st != K3MX_OK) return st;
    if (n_tokens > K3MX_NOALLOC_MAX_TOKENS) return K3MX_ESHAPE;
    if ((idx_out && !aligned16(idx_out)) || (w_out && !aligned16(w_out))) return K3MX_EALIGN;
    const MoeLayout L = moe_layout(n_tokens, x_dtype, K3MX_PATH_DECODE);
    if (L.total > kNoallocBytes) return K3MX_EWORKSPACE;
    Ctx c;
    st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    void *scratch = library_scratch();
    if (!scratch) return K3MX_ECUDA;
    return run_moe(c, y, x, x_dtype, n_tokens, experts, logits, bias, K3MX_PATH_DECODE, idx_out,
                   w_out, scratch, L);
}

size_t k3mx_moe_host_workspace_size(int n_tokens, int x_dtype, int path) {
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return 0;
    if (x_dtype != K3MX_F32 && x_dtype != K3MX_BF16) return 0;
    return moe_layout(n_tokens, x_dtype, resolve_path(n_tokens, x_dtype, path)).total_host;
}

k3mx_status k3mx_moe_routed(float *y, const void *x, int x_dtype, int n_tokens,
                            const k3mx_expert *experts, const float *logits, const float *bias,
                            int path, int32_t *idx_out, float *w_out, void *workspace,
                            size_t ws_bytes, k3mx_stream_t stream) {
    k3mx_status st = check_moe_args(y, x, x_dtype, n_tokens, experts, logits, bias, path);
    if (st != K3MX_OK) return st;
    if ((idx_out && !aligned16(idx_out)) || (w_out && !aligned16(w_out))) return K3MX_EALIGN;
    path = resolve_path(n_tokens, x_dtype, path);
    const MoeLayout L = moe_layout(n_tokens, x_dtype, path);
    if (!workspace || ws_bytes < L.total) return K3MX_EWORKSPACE;
    if (!aligned256(workspace)) return K3MX_EALIGN;
    Ctx c;
    st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    return run_moe(c, y, x, x_dtype, n_tokens, experts, logits, bias, path, idx_out, w_out,
                   workspace, L);
}

k3mx_status k3mx_moe_routed_topp(float *y, const void *x, int x_dtype, int n_tokens,
                                 const k3mx_expert *experts, const float *logits, const float *bias,
                                 int path, float top_p, int32_t *idx_out, float *w_out, void *workspace,
                                 size_t ws_bytes, k3mx_stream_t stream) {
    if (!(top_p == top_p) || top_p == INFINITY || top_p == -INFINITY) return K3MX_EINVAL;
    k3mx_status st = check_moe_args(y, x, x_dtype, n_tokens, experts, logits, bias, path);
    if (st != K3MX_OK) return st;
    if ((idx_out && !aligned16(idx_out)) || (w_out && !aligned16(w_out))) return K3MX_EALIGN;
    path = resolve_path(n_tokens, x_dtype, path);
    const MoeLayout L = moe_layout(n_tokens, x_dtype, path);
    if (!workspace || ws_bytes < L.total) return K3MX_EWORKSPACE;
    if (!aligned256(workspace)) return K3MX_EALIGN;
    Ctx c;
    st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    return run_moe(c, y, x, x_dtype, n_tokens, experts, logits, bias, path, idx_out, w_out, workspace, L,
                   (double)top_p);
}

k3mx_status k3mx_moe_routed_host(float *y_host, const void *x_host, int x_dtype, int n_tokens,
                                 const k3mx_expert *experts, const float *logits_host,
                                 const float *bias_host, int path, void *workspace,
                                 size_t ws_bytes, k3mx_stream_t stream) {
    if (!y_host || !x_host || !logits_host || !bias_host || !experts) return K3MX_EINVAL;
    if (x_dtype != K3MX_F32 && x_dtype != K3MX_BF16) return K3MX_EINVAL;
    if (path < K3MX_PATH_AUTO || path > K3MX_PATH_PREFILL_MX) return K3MX_EINVAL;
    if (n_tokens < 1 || n_tokens > K3MX_MAX_TOKENS) return K3MX_ESHAPE;
    path = resolve_path(n_tokens, x_dtype, path);
    if (path >= K3MX_PATH_PREFILL && x_dtype != K3MX_BF16) return K3MX_EINVAL;
    if (!aligned16(experts)) return K3MX_EALIGN;
    const MoeLayout L = moe_layout(n_tokens, x_dtype, path);
    if (!workspace || ws_bytes < L.total_host) return K3MX_EWORKSPACE;
    if (!aligned256(workspace)) return K3MX_EALIGN;
    Ctx c;
    k3mx_status st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    // Page-locked host buffers mapped into the device's address space are
    // read and written in place by the decode kernels (over the CPU-GPU
    // link); other buffers, and the prefill paths (whose y is summed with
    // atomics), go through copies.
    if (path == K3MX_PATH_DECODE) {
        const void *xm = mapped_host(x_host), *lm = mapped_host(logits_host), *bm = mapped_host(bias_host);
        void *ym = const_cast<void *>(mapped_host(y_host));
        if (xm && lm && bm && ym && aligned16(xm) && aligned16(lm) && aligned16(bm) && aligned16(ym)) {
            st = run_moe(c, static_cast<float *>(ym), xm, x_dtype, n_tokens, experts, static_cast<const float *>(lm),
                         static_cast<const float *>(bm), path, nullptr, nullptr, workspace, L);
            if (st != K3MX_OK) return st;
            return cudaStreamSynchronize(c.stream) == cudaSuccess ? K3MX_OK : K3MX_ECUDA;
        }
    }
    const size_t xb = (size_t)n_tokens * kD * (x_dtype == K3MX_BF16 ? 2 : 4);
    void *x_dev = at<void>(workspace, L.x_in);
    float *logits_dev = at<float>(workspace, L.logits_in);
    float *bias_dev = at<float>(workspace, L.bias_in);
    float *y_dev = at<float>(workspace, L.y_out);
    cudaStream_t s = c.stream;
    if (cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(logits_dev, logits_host, (size_t)n_tokens * kE * 4, cudaMemcpyHostToDevice,
                        s) != cudaSuccess ||
        cudaMemcpyAsync(bias_dev, bias_host, kE * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return K3MX_ECUDA;
    st = run_moe(c, y_dev, x_dev, x_dtype, n_tokens, experts, logits_dev, bias_dev, path, nullptr,
                 nullptr, workspace, L);
    if (st != K3MX_OK) return st;
    if (cudaMemcpyAsync(y_host, y_dev, (size_t)n_tokens * kD * 4, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return K3MX_ECUDA;
    return K3MX_OK;
}

k3mx_status k3mx_trace_enable(int on) {
    g_trace_on = on != 0;
    return K3MX_OK;
}

int k3mx_trace_read(k3mx_trace_entry *out, int max_entries) {
    int n = 0;
    for (int i = 0; i < g_nrec; i++) {
        const TraceRec &r = g_rec[i];
        float ms = 0.f;
        if (cudaEventSynchronize(g_ev[r.slot][1]) != cudaSuccess ||
            cudaEventElapsedTime(&ms, g_ev[r.slot][0], g_ev[r.slot][1]) != cudaSuccess)
            continue;
        int j = 0;
        while (j < n && std::strncmp(out[j].name, r.name, sizeof(out[j].name)) != 0) j++;
        if (j == n) {
            if (n >= max_entries) continue;
            std::memset(&out[n], 0, sizeof(out[n]));
            std::strncpy(out[n].name, r.name, sizeof(out[n].name) - 1);
            n++;
        }
        out[j].launches++;
        out[j].total_ms += ms;
    }
    g_nrec = 0;
    return n;
}

k3mx_status k3mx_set_wait_limit(unsigned int polls) {
    Ctx c;
    k3mx_status st = device_ctx(nullptr, c);
    if (st != K3MX_OK) return st;
    const uint32_t p = polls == 0 ? kWaitLimit : (polls > kWaitLimit ? kWaitLimit : polls);
    for (cudaError_t (*set)(uint32_t) : {set_wait_polls_mx, set_wait_polls_px, set_wait_polls_prefill,
                                         set_wait_polls_decode, set_wait_polls_dense}) {
        const cudaError_t e = set(p);
        if (e != cudaSuccess) return from_cuda(e);
    }
    return K3MX_OK;
}

k3mx_status k3mx_device_status(k3mx_stream_t stream, int *detail) {
    Ctx c;
    k3mx_status st = device_ctx(reinterpret_cast<cudaStream_t>(stream), c);
    if (st != K3MX_OK) return st;
    if (cudaStreamSynchronize(c.stream) != cudaSuccess) return K3MX_ECUDA;
    int word[2] = {0, 0};
    if (cudaMemcpy(word, c.status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return K3MX_ECUDA;
    const int zero[2] = {0, 0};
    if (cudaMemcpy(c.status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return K3MX_ECUDA;
    if (detail) *detail = word[1];
    switch (word[0]) {
    case kStatusOk: return K3MX_OK;
    case kStatusBadIndex: return K3MX_EINVAL;
    case kStatusWaitTimeout: return K3MX_ETIMEOUT;
    case kStatusBadPointer: return K3MX_EALIGN;
    default: return K3MX_ECUDA;
    }
}

}  // extern "C"
