// decode.cu - CUDA-core MXFP4 GEMV kernels for fp32 activations (sm_103a).
//
// y = W x with W read straight out of packed MXFP4 and never written back
// as floats (kimi-k3-in-c: 2.78 trillion parameters, one CPU, 8 GB of RAM,
// "Reduction one: the experts already ship at half a byte").
//
// Layout of the work.  A weight row of `in` columns is in/32 groups of 16
// packed bytes plus one scale byte.  A CTA holds G x RS threads, G = in/32:
// thread (g, rs) owns group column g for the whole CTA, so its 32 activations
// of that group sit in registers and serve every row it touches, and a warp's
// 16-byte loads cover consecutive groups of one row (fully coalesced).  A
// tile is RS x U rows; each thread reads U rows of its group column, forms
// one scaled group sum per row, and the CTA adds the G group sums of a row
// in shared memory in a fixed order (deterministic).
//
// Expert kernels:
//   phase A: rows j of W1 and W3 together, h_j = SiTU(g_j, u_j), fp32 h
//   phase B: rows i of W2 times h, one fp32 output per (token, slot) pair
//   combine: y_t = sum_k w_tk * out_(t,k) in slot order
// Work items are (active expert, row tile), handed out in contiguous runs
// so a CTA mostly stays on one expert; all tokens routed to an expert reuse
// the weights it loaded (Kimi K3 engine (c/kimi_k3.c), "Chunked prefill").
#include "common.cuh"

namespace k3mx {
namespace {

// ------------------------------------------------------------- generic GEMV --

constexpr int kGemvU = 4;

__global__ void __launch_bounds__(512)
k_gemv(float *__restrict__ y, const float *__restrict__ x, const uint8_t *__restrict__ packed,
       const uint8_t *__restrict__ scales, int in, int rows, int rs_count) {
    extern __shared__ float red[];                    // [2][RT][G]
    const int G = in / 32;
    const int RT = rs_count * kGemvU;
    const int tid = threadIdx.x;
    const int g = tid % G, rs = tid / G;
    const bool worker = rs < rs_count;
    const int tiles = (rows + RT - 1) / RT;
    const int beg = (int)((long long)tiles * blockIdx.x / gridDim.x);
    const int end = (int)((long long)tiles * (blockIdx.x + 1) / gridDim.x);
    const size_t row_bytes = (size_t)in / 2;
    const int nwarps = blockDim.x / 32, warp = tid / 32, lane = tid % 32;

    float2 xv[16];
    if (worker) load_x_group(x, g, xv);

    int it = 0;
    for (int tile = beg; tile < end; tile++, it++) {
        float *rb = red + (size_t)(it & 1) * RT * G;
        if (worker) {
            uint4 wv[kGemvU];
            uint32_t sv[kGemvU];
#pragma unroll
            for (int u = 0; u < kGemvU; u++) {
                const int r = tile * RT + rs * kGemvU + u;
                if (r < rows) {
                    wv[u] = ldg_stream(packed + (size_t)r * row_bytes + 16 * g);
                    sv[u] = ldg_u8(scales + (size_t)r * G + g);
                } else {
                    wv[u] = make_uint4(0, 0, 0, 0);
                    sv[u] = 255u;
                }
            }
#pragma unroll
            for (int u = 0; u < kGemvU; u++)
                rb[(rs * kGemvU + u) * G + g] = group_term(wv[u], sv[u], xv);
        }
        __syncthreads();
        for (int row = warp; row < RT; row += nwarps) {
            float s = 0.f;
            for (int gg = lane; gg < G; gg += 32) s += rb[row * G + gg];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            const int r = tile * RT + row;
            if (lane == 0 && r < rows) y[r] = s;
        }
    }
}

// ------------------------------------------------------ streaming engine --
//
// One persistent CTA per SM.  A producer warp streams row tiles (packed bytes
// and scale bytes of RT consecutive rows, of one or two matrices) from HBM
// into a ring of shared-memory stages with 1-D bulk copies (cp.async.bulk),
// each stage guarded by a "full" mbarrier (bytes landed) and an "empty"
// mbarrier (consumers done).  Consumer thread (g, rs) owns group column g:
// it copies its U rows x 16 bytes out of the stage, releases the stage, and
// for every token routed to the tile's expert forms the scaled group sums
// against the token's 32 activations of that group, then the consumers add
// each row's G group sums in shared memory (fixed order) and write the
// epilogue.  Every wait is bounded; a wait that gives up sets the device
// status word and the CTA leaves after its copies in flight have landed.

enum : int { kModeGemv = 0, kModeGateUp = 1, kModeDown = 2 };

constexpr int kU = 4;                 // rows per consumer thread per tile
constexpr int kMaxStages = 8;
constexpr int kHeader = 256;          // mbarriers + abort flag

struct ExpertsDev {
    const k3mx_expert *experts;
    const int32_t *act, *n_active, *offsets, *perm;
    k3mx_expert one;
    int single;
};

struct StreamArgs {
    ExpertsDev d;                     // expert modes
    const uint8_t *packed, *scales;   // gemv mode
    int rows;                         // rows of each matrix
    int in;                           // columns of each matrix
    int rs;                           // row slices: RT = rs * kU rows per tile
    int stages;
    const float *xin;                 // gemv: x; gate/up: x [T][D]; down: h [16T][F]
    float *out;                       // gemv: y; gate/up: h [16T][F]; down: [16T][D]
    int *status;
};

__device__ __forceinline__ void item_expert(const ExpertsDev &d, int slot, k3mx_expert &ex,
                                            int &p0, int &p1) {
    if (d.single) {
        ex = d.one;
        p0 = 0;
        p1 = 1;
    } else {
        const int e = d.act[slot];
        ex = d.experts[e];
        p0 = d.offsets[e];
        p1 = d.offsets[e + 1];
    }
}

// largest block of each mode: consumers (G x rs rounded to warps) + producer warp
template <int MODE>
constexpr int max_threads() {
    return MODE == kModeGateUp ? 448 + 32 : (MODE == kModeDown ? 384 + 32 : 512 + 32);
}

template <int NMAT, int MODE>
__global__ void __launch_bounds__(max_threads<MODE>(), 1) k_stream(StreamArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int G = a.in / 32;
    const int RT = a.rs * kU;
    const int NC = ((G * a.rs + 31) / 32) * 32;       // consumer threads
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const uint32_t pk_bytes = (uint32_t)RT * (a.in / 2);
    const uint32_t sc_bytes = (uint32_t)RT * G;
    const uint32_t stage_bytes = NMAT * (pk_bytes + sc_bytes);
    const int S = a.stages;

    // header: full[8] and empty[8] mbarriers (128 B), the abort flag (at 128),
    // then the row-sum buffer and the stage ring
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 2 * kMaxStages * 8);
    float *red = reinterpret_cast<float *>(smem + kHeader);      // [2][NMAT][RT][G]
    const size_t red_bytes = ((size_t)2 * NMAT * RT * G * 4 + 127) & ~size_t(127);
    uint8_t *stage0 = smem + kHeader + red_bytes;
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kMaxStages);

    if (tid == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, NC / 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (MODE == kModeGateUp) pdl_launch_dependents();

    const int tpe = (a.rows + RT - 1) / RT;                      // tiles per matrix
    int n_units = 1;
    if (MODE != kModeGemv) n_units = a.d.single ? 1 : *a.d.n_active;
    const long long total = (long long)n_units * tpe;
    const long long beg = total * blockIdx.x / gridDim.x;
    const long long end = total * (blockIdx.x + 1) / gridDim.x;

    if (warp == NC / 32) {
        // ------------------------------------------------------- producer --
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            long long n_issued = 0;
            for (long long item = beg; item < end; item++, n_issued++) {
                const int s = (int)(n_issued % S);
                const long long round = n_issued / S;
                if (round > 0 && !mbar_wait(empty0 + 8 * s, (uint32_t)((round - 1) & 1))) {
                    report_status(a.status, kStatusWaitTimeout, 100 + MODE);
                    *abort_flag = 1;
                    break;
                }
                const int tile = (int)(item % tpe);
                const int r0 = tile * RT;
                const int nr = min(RT, a.rows - r0);
                const uint8_t *W[2], *Sc[2];
                if (MODE == kModeGemv) {
                    W[0] = a.packed;
                    Sc[0] = a.scales;
                } else {
                    k3mx_expert ex;
                    int p0, p1;
                    item_expert(a.d, (int)(item / tpe), ex, p0, p1);
                    if (MODE == kModeGateUp) {
                        W[0] = ex.w1; Sc[0] = ex.s1; W[1] = ex.w3; Sc[1] = ex.s3;
                    } else {
                        W[0] = ex.w2; Sc[0] = ex.s2;
                    }
                }
                bool aligned = true;
#pragma unroll
                for (int m = 0; m < NMAT; m++)
                    aligned &= ((reinterpret_cast<uintptr_t>(W[m]) | reinterpret_cast<uintptr_t>(Sc[m])) & 15u) == 0;
                if (!aligned) {
                    report_status(a.status, kStatusBadPointer, (int)(item / tpe));
                    *abort_flag = 1;
                    break;
                }
                const uint32_t st = smem_addr(stage0 + (size_t)s * stage_bytes);
                const uint32_t full = full0 + 8 * s;
                mbar_arrive_expect_tx(full, NMAT * (uint32_t)nr * (a.in / 2 + G));
#pragma unroll
                for (int m = 0; m < NMAT; m++) {
                    bulk_g2s(st + m * pk_bytes, W[m] + (size_t)r0 * (a.in / 2), nr * (a.in / 2), full, pol);
                    bulk_g2s(st + NMAT * pk_bytes + m * sc_bytes, Sc[m] + (size_t)r0 * G, nr * G, full, pol);
                }
            }
            // keep the CTA alive until every issued copy has landed
            for (long long k = (n_issued > S ? n_issued - S : 0); k < n_issued; k++) {
                if (!mbar_wait(full0 + 8 * (int)(k % S), (uint32_t)((k / S) & 1))) {
                    report_status(a.status, kStatusWaitTimeout, 110 + MODE);
                    break;
                }
            }
        }
        return;
    }

    // ----------------------------------------------------------- consumers --
    const bool worker = tid < G * a.rs;
    const int g = tid % G, rsi = tid / G;
    const int NCW = NC / 32;
    if (MODE == kModeDown) pdl_wait();                           // h comes from the gate/up pass
    int b = 0;
    long long n_done = 0;
    for (long long item = beg; item < end; item++, n_done++) {
        const int s = (int)(n_done % S);
        if (!mbar_wait(full0 + 8 * s, (uint32_t)((n_done / S) & 1))) {
            report_status(a.status, kStatusWaitTimeout, 120 + MODE);
            *abort_flag = 1;
        }
        const uint8_t *st = stage0 + (size_t)s * stage_bytes;
        const int tile = (int)(item % tpe);
        const int r0 = tile * RT;
        const int nr = min(RT, a.rows - r0);
        uint4 wv[NMAT][kU];
        uint32_t sv[NMAT][kU];
#pragma unroll
        for (int m = 0; m < NMAT; m++)
#pragma unroll
            for (int u = 0; u < kU; u++) {
                const int row = rsi * kU + u;
                if (worker && row < nr) {
                    wv[m][u] = lds128(st + m * pk_bytes + (size_t)row * (a.in / 2) + 16 * g);
                    sv[m][u] = st[NMAT * pk_bytes + m * sc_bytes + row * G + g];
                } else {
                    wv[m][u] = make_uint4(0, 0, 0, 0);
                    sv[m][u] = 255u;
                }
            }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);               // stage free for the producer

        int p0 = 0, p1 = 1;
        if (MODE != kModeGemv) {
            k3mx_expert ex;
            item_expert(a.d, (int)(item / tpe), ex, p0, p1);
        }
        for (int pi = p0; pi < p1; pi++) {
            int p = 0;
            if (MODE != kModeGemv && !a.d.single) p = a.d.perm[pi];
            const float *xrow = a.xin;
            if (MODE == kModeGateUp) xrow = a.xin + (size_t)(p / kK) * kD;
            if (MODE == kModeDown) xrow = a.xin + (size_t)p * kF;
            float *rb = red + (size_t)b * NMAT * RT * G;
            if (worker) {
                float2 xv[16];
                load_x_group(xrow, g, xv);
#pragma unroll
                for (int m = 0; m < NMAT; m++)
#pragma unroll
                    for (int u = 0; u < kU; u++)
                        rb[((size_t)m * RT + rsi * kU + u) * G + g] = group_term(wv[m][u], sv[m][u], xv);
            }
            named_sync(1, NC);
            if (*abort_flag) return;
            for (int row = warp; row < nr; row += NCW) {
                float acc[NMAT];
#pragma unroll
                for (int m = 0; m < NMAT; m++) {
                    float t = 0.f;
                    for (int gg = lane; gg < G; gg += 32) t += rb[((size_t)m * RT + row) * G + gg];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                    acc[m] = t;
                }
                if (lane == 0) {
                    if (MODE == kModeGemv) a.out[r0 + row] = acc[0];
                    if (MODE == kModeGateUp) a.out[(size_t)p * kF + r0 + row] = situ_glu(acc[0], acc[NMAT - 1]);
                    if (MODE == kModeDown) a.out[(size_t)p * kD + r0 + row] = acc[0];
                }
            }
            b ^= 1;
        }
    }
}

size_t stream_smem_bytes(int nmat, int in, int rs, int stages) {
    const size_t G = in / 32, RT = (size_t)rs * kU;
    const size_t red = (2 * nmat * RT * G * 4 + 127) & ~size_t(127);
    const size_t stage = nmat * RT * (in / 2 + G);
    return kHeader + red + stages * stage;
}

// y[t][i] = sum_k w[t][k] * out[t*16 + k][i], slot order, fp32
__global__ void k_combine(float *__restrict__ y, const float *__restrict__ out,
                          const float *__restrict__ w, int n_tokens) {
    const int per_tok = kD / 4;
    const long long i4 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i4 >= (long long)n_tokens * per_tok) return;
    const int t = (int)(i4 / per_tok), c = (int)(i4 % per_tok);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kK; k++) {
        const float wk = __ldg(w + (size_t)t * kK + k);
        const float4 v = __ldg(reinterpret_cast<const float4 *>(out + ((size_t)t * kK + k) * kD) + c);
        acc.x = fmaf(wk, v.x, acc.x);
        acc.y = fmaf(wk, v.y, acc.y);
        acc.z = fmaf(wk, v.z, acc.z);
        acc.w = fmaf(wk, v.w, acc.w);
    }
    reinterpret_cast<float4 *>(y + (size_t)t * kD)[c] = acc;
}

__global__ void k_bf16_to_f32(float *__restrict__ out, const uint16_t *__restrict__ in, size_t n) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = __uint_as_float((uint32_t)in[i] << 16);
}

int occupancy(const void *fn, int threads, size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 1)
        n = 1;
    return n;
}

ExpertsDev make_dev(const DecodeExperts &d) {
    ExpertsDev e{};
    e.experts = d.experts;
    e.act = d.act;
    e.n_active = d.n_active;
    e.offsets = d.offsets;
    e.perm = d.perm;
    if (d.single) {
        e.one = *d.single;
        e.single = 1;
    }
    return e;
}

constexpr size_t kSmemBudget = 220 * 1024;

template <int NMAT, int MODE>
cudaError_t launch_stream(const Ctx &c, StreamArgs a, long long max_items, bool pdl) {
    const int G = a.in / 32;
    const int threads = ((G * a.rs + 31) / 32) * 32 + 32;
    const size_t smem = stream_smem_bytes(NMAT, a.in, a.rs, a.stages);
    static size_t configured = 0;
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(k_stream<NMAT, MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    long long grid = c.num_sms;
    if (grid > max_items) grid = max_items;
    a.status = c.status;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_stream<NMAT, MODE>, a);
}

}  // namespace

cudaError_t launch_gemv(const Ctx &c, float *y, const float *x, const uint8_t *packed,
                        const uint8_t *scales, int in, int rows) {
    const int G = in / 32;
    // streaming path: group count a multiple of 16 (16-byte scale tiles) and
    // a 16-byte aligned scale array
    if (G % 16 == 0 && (reinterpret_cast<uintptr_t>(scales) & 15u) == 0) {
        StreamArgs a{};
        a.packed = packed;
        a.scales = scales;
        a.rows = rows;
        a.in = in;
        a.rs = G >= 512 ? 1 : (G >= 256 ? 2 : 4);
        const size_t stage = (size_t)a.rs * kU * (in / 2 + G);
        const size_t fixed = stream_smem_bytes(1, in, a.rs, 0);
        int st = (int)((kSmemBudget - fixed) / stage);
        a.stages = st > kMaxStages ? kMaxStages : st;
        a.xin = x;
        a.out = y;
        const long long tiles = (rows + a.rs * kU - 1) / (a.rs * kU);
        return launch_stream<1, kModeGemv>(c, a, tiles, false);
    }
    int rs = 256 / G;
    if (rs < 1) rs = 1;
    if (rs > 8) rs = 8;
    const int threads = ((G * rs + 31) / 32) * 32;
    const size_t smem = (size_t)2 * rs * kGemvU * G * sizeof(float);
    const int tiles = (rows + rs * kGemvU - 1) / (rs * kGemvU);
    static int occ_cache[1025] = {0};
    int occ = occ_cache[threads / 32];
    if (occ == 0) occ = occ_cache[threads / 32] = occupancy((const void *)k_gemv, threads, smem);
    int grid = c.num_sms * occ;
    if (grid > tiles) grid = tiles;
    k_gemv<<<grid, threads, smem, c.stream>>>(y, x, packed, scales, in, rows, rs);
    return cudaGetLastError();
}

cudaError_t launch_decode_phase_a(const Ctx &c, const DecodeExperts &d, const float *x, float *h) {
    StreamArgs a{};
    a.d = make_dev(d);
    a.rows = kF;
    a.in = kD;
    a.rs = 4;
    a.stages = 3;
    a.xin = x;
    a.out = h;
    const long long items = (long long)(d.single ? 1 : d.max_active) * (kF / (a.rs * kU));
    return launch_stream<2, kModeGateUp>(c, a, items, false);
}

cudaError_t launch_decode_phase_b(const Ctx &c, const DecodeExperts &d, const float *h,
                                  float *stage) {
    StreamArgs a{};
    a.d = make_dev(d);
    a.rows = kD;
    a.in = kF;
    a.rs = 4;
    a.stages = 6;
    a.xin = h;
    a.out = stage;
    const long long items = (long long)(d.single ? 1 : d.max_active) * (kD / (a.rs * kU));
    return launch_stream<1, kModeDown>(c, a, items, true);
}

cudaError_t launch_combine(const Ctx &c, float *y, const float *stage, const float *w,
                           int n_tokens) {
    const long long n4 = (long long)n_tokens * (kD / 4);
    const int threads = 256;
    k_combine<<<(int)((n4 + threads - 1) / threads), threads, 0, c.stream>>>(y, stage, w, n_tokens);
    return cudaGetLastError();
}

cudaError_t launch_bf16_to_f32(const Ctx &c, float *out, const uint16_t *in, size_t n) {
    const int threads = 256;
    k_bf16_to_f32<<<(unsigned)((n + threads - 1) / threads), threads, 0, c.stream>>>(out, in, n);
    return cudaGetLastError();
}

}  // namespace k3mx
