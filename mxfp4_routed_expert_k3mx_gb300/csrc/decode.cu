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
// The tensor-core GEMV (`k_mma`, GEMV mode) streams 16-row tiles through a
// bulk-copy ring and runs mma.sync against the activation split into two
// exact f16 pieces; `k_gemv` takes the shapes the streaming path does not.
// The `k_mma` template also holds expert modes (gate/up and down over
// grouped pairs); the layer runs its experts on the block-scaled kernels of
// mx.cu, so only the GEMV mode is instantiated.  `k_combine` forms
// y_t = sum_k w_tk * out_(t,k) in slot order for the batched decode passes.
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

// ------------------------------------------------- tensor-core streaming --
//
// One persistent CTA per SM: a producer warp streams row tiles (RT = 16 MT
// consecutive rows of one or two matrices, packed bytes and scale bytes) from
// HBM into a ring of shared-memory stages with 1-D bulk copies, each stage
// guarded by a "full" mbarrier (bytes landed) and an "empty" mbarrier
// (consumers done).  The NCW consumer warps split the K dimension: warp w owns
// gpw consecutive 32-column groups.  It copies its packed words and scale
// words out of the stage into registers, releases the stage, and multiplies
// on the tensor cores with mma.sync m16n8k16 (f16 x f16 -> f32):
//   A (16 rows x 16 columns) : e2m1 codes turned into f16 pairs, half of
//       them by cvt.rn.f16x2.e2m1x2 and half by integer bit moves (see
//       decode_word), so the conversion and integer pipes share the work;
//   B (16 columns x 8)       : the activations, each column one of two f16
//       pieces whose sum is the fp32 value (to 22 bits) divided by a power of
//       two (the vector's scale), two columns per token, four tokens per MMA.
// The k16 chunks of a group take its columns in a permuted order (thread c of
// a quad supplies columns 8c..8c+7, i.e. packed word c); the same order is
// used for A and B, and all 32 columns share one scale, so the sum is the
// group's sum.  Per group and row the fp32 MMA result is multiplied by
// 2^(s - 127) and accumulated (a NaN scale adds nothing).  At the end of a
// tile the warps' partial sums are added in shared memory in a fixed order.
// Every wait is bounded; a wait that gives up sets the device status word and
// the CTA leaves after its copies in flight have landed.

enum : int { kModeGemv = 0, kModeGateUp = 1, kModeDown = 2 };

constexpr int kMaxStages = 8;
constexpr int kHeader = 512;          // mbarriers (0..127), abort flag (128), per-warp maxima (256..511)
constexpr int kMaxConsumerWarps = 16;

struct ExpertsDev {
    const k3mx_expert *experts;
    const int32_t *units, *n_units, *perm;
    k3mx_expert one;
    int single;
};

struct MmaArgs {
    ExpertsDev d;                     // expert modes
    const uint8_t *packed, *scales;   // gemv mode
    int rows;                         // rows of each matrix
    int in;                           // columns of each matrix
    int ncw;                          // consumer warps
    int gpw;                          // groups per consumer warp (multiple of 4)
    int stages;
    const float *xin;                 // gemv: x; gate/up: x [T][D]; down: g,u [16T][2][F]
    float *out;                       // gemv: y; gate/up: g,u [16T][2][F]; down: [16T][D]
    int *status;
};

// the expert and pair-slot range [p0, p1) of work unit `unit`
__device__ __forceinline__ void unit_expert(const ExpertsDev &d, int unit, k3mx_expert &ex,
                                            int &p0, int &p1) {
    if (d.single) {
        ex = d.one;
        p0 = 0;
        p1 = 1;
    } else {
        const int *u = d.units + 3 * unit;
        ex = d.experts[u[0]];
        p0 = u[1];
        p1 = u[2];
    }
}

// The four A registers (two k16 chunks, rows gq or gq+8) of one packed word
// q = codes n0..n7 of columns 8c..8c+7.  Two registers come from the
// conversion pipe (bytes 0 and 2: codes n0,n1 and n4,n5, exact f16 values);
// two are assembled on the integer pipe from code pairs (n2,n6) and (n3,n7):
// magnitude bits to f16 bits 9..11, sign to bit 15, i.e. the f16 value
// v * 2^-14 (exponent field = e2m1 exponent, subnormal when it is 0).  The
// matching B entries carry the factor 2^14.  Register order per chunk:
//   chunk 0: a0 = (n0, n1), a2 = (n2, n6);  chunk 1: a0 = (n4, n5), a2 = (n3, n7).
__device__ __forceinline__ void decode_word(uint32_t q, uint32_t &c0a, uint32_t &c0b,
                                            uint32_t &c1a, uint32_t &c1b) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b2;\n\t}"
        : "=r"(c0a), "=r"(c1a)
        : "r"(q));
    c0b = ((q << 1) & 0x0E000E00u) | ((q << 4) & 0x80008000u);
    c1b = ((q >> 3) & 0x0E000E00u) | (q & 0x80008000u);
}

// position of column offset j (0..7 inside a thread's 8 columns) in the B
// piece row, and whether that column's A value carries the factor 2^-14
__device__ __forceinline__ int bpos(int j) { return j == 3 ? 6 : (j == 6 ? 3 : j); }
__device__ __forceinline__ bool alu_col(int j) { return j == 2 || j == 3 || j == 6 || j == 7; }

__device__ __forceinline__ uint32_t lds32(const uint8_t *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1, float c0, float c1,
                                        float c2, float c3) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2),
          "f"(c3));
}

// activation of pair `pair` at column `col`: gemv x; gate/up the token's x
// row; down h = SiTU(g, u) from the gate/up outputs [pair][2][F]
template <int MODE>
__device__ __forceinline__ float act_of(const MmaArgs &a, int pair, int col) {
    if (MODE == kModeGateUp) return __ldg(a.xin + (size_t)(pair / kK) * kD + col);
    if (MODE == kModeDown) {
        const float *gu = a.xin + (size_t)pair * 2 * kF;
        return situ_glu(__ldg(gu + col), __ldg(gu + kF + col));
    }
    return __ldg(a.xin + col);
}

template <int NMAT, int MT, int GPW, int NTOK, int MODE, int MAXT>
__global__ void __launch_bounds__(MAXT, 1) k_mma(MmaArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int G = a.in / 32;
    constexpr int RT = 16 * MT;
    const int NCW = a.ncw, NCT = 32 * NCW, S = a.stages;
    constexpr int gpw = GPW;
    // one bulk copy per tile: rows keep their global pitch in shared memory
    const uint32_t pitch = (uint32_t)(a.in / 2);
    const uint32_t pk_bytes = (uint32_t)RT * pitch;
    const uint32_t sc_bytes = (uint32_t)RT * G;
    const uint32_t stage_bytes = NMAT * (pk_bytes + sc_bytes);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);                  // full[8], empty[8]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 128);
    float *tmax = reinterpret_cast<float *>(smem + 256);                 // [16 warps][NTOK <= 4]
    float *red = reinterpret_cast<float *>(smem + kHeader);              // [2][NCW][NMAT][NTOK][RT]
    const size_t red_bytes = ((size_t)2 * NCW * NMAT * NTOK * RT * 4 + 127) & ~size_t(127);
    // activation pieces [NCW][NTOK][2][pp]: a piece row holds GPW*32 halves
    // plus 32 halves of padding (bank spread for the B-fragment loads)
    const int pp = gpw * 32 + 32;
    __half *pieces = reinterpret_cast<__half *>(smem + kHeader + red_bytes);
    const size_t pc_bytes = ((size_t)NCW * NTOK * 2 * pp * 2 + 127) & ~size_t(127);
    uint8_t *stage0 = smem + kHeader + red_bytes + pc_bytes;
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kMaxStages);

    if (tid == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, NCW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (MODE == kModeGateUp) pdl_launch_dependents();

    // work items: (expert slot, matrix, row tile); gate/up has W1 then W3
    constexpr int NM = MODE == kModeGateUp ? 2 : 1;
    const int tpm = (a.rows + RT - 1) / RT;                      // tiles per matrix
    const int tpe = NM * tpm;                                    // tiles per expert
    int n_units = 1;
    if (MODE != kModeGemv) n_units = a.d.single ? 1 : *a.d.n_units;
    const long long total = (long long)n_units * tpe;
    const long long beg = total * blockIdx.x / gridDim.x;
    const long long end = total * (blockIdx.x + 1) / gridDim.x;

    if (warp == NCW) {
        // ------------------------------------------------------- producer --
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            long long n_issued = 0;
            int cur_slot = -1;
            const uint8_t *Wm[2] = {a.packed, a.packed}, *Sm[2] = {a.scales, a.scales};
            for (long long item = beg; item < end; item++, n_issued++) {
                const int s = (int)(n_issued % S);
                const long long round = n_issued / S;
                const int slot = (int)(item / tpe);
                // resolve the expert's pointers once per expert (a dependent
                // chain of loads), before waiting for the free stage
                if (MODE != kModeGemv && slot != cur_slot) {
                    k3mx_expert ex;
                    int p0, p1;
                    unit_expert(a.d, slot, ex, p0, p1);
                    if (MODE == kModeGateUp) {
                        Wm[0] = ex.w1; Sm[0] = ex.s1; Wm[1] = ex.w3; Sm[1] = ex.s3;
                    } else {
                        Wm[0] = ex.w2; Sm[0] = ex.s2; Wm[1] = ex.w2; Sm[1] = ex.s2;
                    }
                    cur_slot = slot;
                }
                const int mat = (int)((item / tpm) % NM);
                const uint8_t *W[1] = {Wm[mat]}, *Sc[1] = {Sm[mat]};
                if (round > 0 && !mbar_wait(empty0 + 8 * s, (uint32_t)((round - 1) & 1))) {
                    report_status(a.status, kStatusWaitTimeout, 100 + MODE);
                    *abort_flag = 1;
                    break;
                }
                const int tile = (int)(item % tpm);
                const int r0 = tile * RT;
                const int nr = min(RT, a.rows - r0);
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
                    bulk_g2s(st + m * pk_bytes, W[m] + (size_t)r0 * pitch, nr * pitch, full, pol);
                    bulk_g2s(st + NMAT * pk_bytes + m * sc_bytes, Sc[m] + (size_t)r0 * G, nr * G, full, pol);
                }
            }
            for (long long k = (n_issued > S ? n_issued - S : 0); k < n_issued; k++) {
                if (!mbar_wait(full0 + 8 * (int)(k % S), (uint32_t)((k / S) & 1))) {
                    report_status(a.status, kStatusWaitTimeout, 110 + MODE);
                    break;
                }
            }
        }
        return;
    }
    if (warp > NCW) return;

    // ----------------------------------------------------------- consumers --
    const int gq = lane >> 2, c = lane & 3;                       // quad row, quad lane
    const int grp0 = warp * gpw;                                  // first group of this warp
    __half *mypc = pieces + (size_t)warp * NTOK * 2 * pp;
    if (MODE == kModeDown) pdl_wait();                           // h comes from the gate/up pass

    int cached_lo = -1, cached_hi = -1;
    int cur_slot = -1, p0 = 0, p1 = 1;                           // pair range of the current expert
    int pairs[NTOK];
#pragma unroll
    for (int j = 0; j < NTOK; j++) pairs[j] = 0;
    float tscale[NTOK];
#pragma unroll
    for (int j = 0; j < NTOK; j++) tscale[j] = 1.f;
    int par = 0;
    long long n_done = 0;
    for (long long item = beg; item < end; item++, n_done++) {
        const int s = (int)(n_done % S);
        if (!mbar_wait(full0 + 8 * s, (uint32_t)((n_done / S) & 1))) {
            report_status(a.status, kStatusWaitTimeout, 120 + MODE);
            *abort_flag = 1;
        }
        const uint8_t *st = stage0 + (size_t)s * stage_bytes;
        const int tile = (int)(item % tpm);
        const int mat = (int)((item / tpm) % NM);
        const int r0 = tile * RT;
        const int nr = min(RT, a.rows - r0);

        // this warp's packed words (rows gq and gq+8 of each m-tile) and the
        // group scales of those rows, decoded to fp32 (a NaN scale, 255,
        // becomes 0: with finite activations the group then adds exactly 0)
        uint32_t aw[NMAT][MT][2][GPW];
        uint32_t sw[NMAT][MT][2][GPW / 4];
        float sf[NMAT][MT][2][GPW];
#pragma unroll
        for (int m = 0; m < NMAT; m++)
#pragma unroll
            for (int mt = 0; mt < MT; mt++)
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int row = 16 * mt + gq + 8 * h;
                    const bool ok = row < nr;
                    const uint8_t *rp = st + m * pk_bytes + (size_t)row * pitch + 16 * grp0 + 4 * c;
                    const uint8_t *sp = st + NMAT * pk_bytes + m * sc_bytes + (size_t)row * G + grp0;
                    // Rows share bank alignment (the pitch is a multiple of
                    // 128 bytes), so at step i row gq reads group (i + gq) mod
                    // GPW: the warp's eight rows then touch eight different
                    // 16-byte bank groups.  A rotation by gq restores the
                    // group order.
                    uint32_t r[GPW];
#pragma unroll
                    for (int i = 0; i < GPW; i++)
                        r[i] = ok ? lds32(rp + 16 * ((i + gq) & (GPW - 1))) : 0u;
#pragma unroll
                    for (int bit = 1; bit < GPW; bit <<= 1) {
                        const bool rot = (gq & bit) != 0;
                        uint32_t t[GPW];
#pragma unroll
                        for (int i = 0; i < GPW; i++) t[i] = rot ? r[(i - bit) & (GPW - 1)] : r[i];
#pragma unroll
                        for (int i = 0; i < GPW; i++) r[i] = t[i];
                    }
#pragma unroll
                    for (int gi = 0; gi < GPW; gi++) aw[m][mt][h][gi] = r[gi];
#pragma unroll
                    for (int q = 0; q < GPW / 4; q++) sw[m][mt][h][q] = ok ? lds32(sp + 4 * q) : 0xFFFFFFFFu;
                }
        // scale bytes 1..254 decode with one shift; 0 (2^-127, subnormal) and
        // 255 (NaN: contributes 0) take the exact path when the warp sees any
        bool special = false;
#pragma unroll
        for (int m = 0; m < NMAT; m++)
#pragma unroll
            for (int mt = 0; mt < MT; mt++)
#pragma unroll
                for (int h = 0; h < 2; h++)
#pragma unroll
                    for (int q = 0; q < GPW / 4; q++) {
                        const uint32_t w = sw[m][mt][h][q];
                        const uint32_t zero = (w - 0x01010101u) & ~w & 0x80808080u;   // a 0x00 byte
                        const uint32_t nw = ~w;
                        const uint32_t ff = (nw - 0x01010101u) & ~nw & 0x80808080u;   // a 0xFF byte
                        special |= (zero | ff) != 0u;
                    }
        special = __any_sync(0xffffffffu, special);
#pragma unroll
        for (int m = 0; m < NMAT; m++)
#pragma unroll
            for (int mt = 0; mt < MT; mt++)
#pragma unroll
                for (int h = 0; h < 2; h++)
#pragma unroll
                    for (int q = 0; q < GPW / 4; q++)
#pragma unroll
                        for (int k = 0; k < 4; k++) {
                            const uint32_t sb = (sw[m][mt][h][q] >> (8 * k)) & 0xFFu;
                            float f = __uint_as_float(sb << 23);
                            if (special) f = sb == 255u ? 0.f : e8m0_to_f32(sb);
                            sf[m][mt][h][4 * q + k] = f;
                        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);               // stage free for the producer

        const int slot = (int)(item / tpe);
        if (MODE != kModeGemv && slot != cur_slot) {
            k3mx_expert ex;
            unit_expert(a.d, slot, ex, p0, p1);
            cur_slot = slot;
        }
        for (int pa = p0; pa < p1; pa += NTOK) {
            const int nt = min(NTOK, p1 - pa);

            // activation pieces of this pass's tokens (shared by the tiles
            // of one expert, rebuilt when the token set changes)
            if (pa != cached_lo || pa + nt != cached_hi) {
#pragma unroll
                for (int j = 0; j < NTOK; j++)
                    pairs[j] = (MODE == kModeGemv || a.d.single) ? 0 : a.d.perm[min(pa + j, p1 - 1)];
#pragma unroll
                for (int j = 0; j < NTOK; j++) {
                    float mx = 0.f;
                    if (j < nt)
                        for (int gi = 0; gi < gpw; gi++)
                            mx = fmaxf(mx, fabsf(act_of<MODE>(a, pairs[j], 32 * (grp0 + gi) + lane)));
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    if (lane == 0) tmax[warp * NTOK + j] = mx;
                }
                named_sync(1, NCT);
                // column of this lane inside its quad's 8 columns, and its
                // slot in the B piece row (see decode_word)
                const int jcol = lane & 7;
                const int slot = (lane & ~7) + bpos(jcol);
                const float colf = alu_col(jcol) ? 16384.f : 1.f;
#pragma unroll
                for (int j = 0; j < NTOK; j++) {
                    float mx = 0.f;
                    for (int w2 = 0; w2 < NCW; w2++) mx = fmaxf(mx, tmax[w2 * NTOK + j]);
                    int e = 0;
                    if (mx > 0.f && mx <= 3.0e38f) {
                        frexpf(mx, &e);
                        e = min(max(e, -100), 126);
                    }
                    tscale[j] = ldexpf(1.f, e);
                    const float inv = ldexpf(1.f, -e) * colf;
                    if (j < nt) {
                        for (int gi = 0; gi < gpw; gi++) {
                            const float u = act_of<MODE>(a, pairs[j], 32 * (grp0 + gi) + lane) * inv;
                            const __half h0 = __float2half_rn(u);
                            const __half h1 = __float2half_rn(u - __half2float(h0));
                            __half *dst = mypc + (size_t)j * 2 * pp + 32 * gi + slot;
                            dst[0] = h0;
                            dst[pp] = h1;
                        }
                    }
                }
                __syncwarp();
                cached_lo = pa;
                cached_hi = pa + nt;
            }

            // B column of this lane: token gq / 2, piece gq % 2
            const int btok = gq >> 1, bpiece = gq & 1;
            const bool bval = btok < nt;
            const __half *bsrc = mypc + ((size_t)btok * 2 + bpiece) * pp + 8 * c;

            float acc[NMAT][MT][4];
#pragma unroll
            for (int m = 0; m < NMAT; m++)
#pragma unroll
                for (int mt = 0; mt < MT; mt++)
#pragma unroll
                    for (int i = 0; i < 4; i++) acc[m][mt][i] = 0.f;

#pragma unroll
            for (int gi = 0; gi < GPW; gi++) {
                const uint4 bq = bval ? *reinterpret_cast<const uint4 *>(bsrc + 32 * gi)
                                      : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int m = 0; m < NMAT; m++)
#pragma unroll
                    for (int mt = 0; mt < MT; mt++) {
                        uint32_t r0a, r0b, r0c, r0d, r1a, r1b, r1c, r1d;
                        decode_word(aw[m][mt][0][gi], r0a, r0b, r0c, r0d);   // row gq
                        decode_word(aw[m][mt][1][gi], r1a, r1b, r1c, r1d);   // row gq + 8
                        float d[4];
                        mma_f16(d, r0a, r1a, r0b, r1b, bq.x, bq.y, 0.f, 0.f, 0.f, 0.f);
                        mma_f16(d, r0c, r1c, r0d, r1d, bq.z, bq.w, d[0], d[1], d[2], d[3]);
                        const float f0 = sf[m][mt][0][gi], f1 = sf[m][mt][1][gi];
                        acc[m][mt][0] = fmaf(d[0], f0, acc[m][mt][0]);
                        acc[m][mt][1] = fmaf(d[1], f0, acc[m][mt][1]);
                        acc[m][mt][2] = fmaf(d[2], f1, acc[m][mt][2]);
                        acc[m][mt][3] = fmaf(d[3], f1, acc[m][mt][3]);
                    }
            }

            // columns 2t and 2t+1 are the two pieces of token t = c: this
            // thread holds token c's partial sums of rows gq and gq+8
            float *rb = red + (size_t)par * NCW * NMAT * NTOK * RT;
            if (c < NTOK) {
#pragma unroll
                for (int m = 0; m < NMAT; m++)
#pragma unroll
                    for (int mt = 0; mt < MT; mt++) {
                        float *rw = rb + ((size_t)(warp * NMAT + m) * NTOK + c) * RT + 16 * mt + gq;
                        rw[0] = acc[m][mt][0] + acc[m][mt][1];
                        rw[8] = acc[m][mt][2] + acc[m][mt][3];
                    }
            }
            named_sync(1, NCT);
            if (*abort_flag) return;
            for (int o = lane * NCW + warp; o < nt * RT; o += NCT) {
                const int j = o / RT, row = o % RT;
                if (row < nr) {
                    float f[NMAT];
#pragma unroll
                    for (int m = 0; m < NMAT; m++) {
                        float t = 0.f;
                        for (int w2 = 0; w2 < NCW; w2++) t += rb[((w2 * NMAT + m) * NTOK + j) * RT + row];
                        f[m] = t * tscale[j];
                    }
                    if (MODE == kModeGemv) a.out[r0 + row] = f[0];
                    if (MODE == kModeGateUp) a.out[((size_t)pairs[j] * 2 + mat) * kF + r0 + row] = f[0];
                    if (MODE == kModeDown) a.out[(size_t)pairs[j] * kD + r0 + row] = f[0];
                }
            }
            par ^= 1;
        }
    }
}

size_t mma_smem_bytes(int nmat, int mt, int ntok, int in, int ncw, int gpw, int stages) {
    const size_t G = in / 32, RT = 16 * (size_t)mt;
    const size_t red = (2 * (size_t)ncw * nmat * ntok * RT * 4 + 127) & ~size_t(127);
    const size_t pc = ((size_t)ncw * ntok * 2 * (gpw * 32 + 32) * 2 + 127) & ~size_t(127);
    const size_t stage = nmat * RT * (in / 2 + G);
    return kHeader + red + pc + stages * stage;
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


int occupancy(const void *fn, int threads, size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 1)
        n = 1;
    return n;
}


constexpr size_t kSmemBudget = 224 * 1024;

template <int NMAT, int MT, int GPW, int NTOK, int MODE, int MAXT>
cudaError_t launch_mma(const Ctx &c, MmaArgs a, long long max_items, bool pdl) {
    if (32 * (a.ncw + 1) > MAXT || a.gpw != GPW) return cudaErrorInvalidValue;
    const size_t smem = mma_smem_bytes(NMAT, MT, NTOK, a.in, a.ncw, a.gpw, a.stages);
    static size_t configured = 0;
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(k_mma<NMAT, MT, GPW, NTOK, MODE, MAXT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    long long grid = c.num_sms;
    if (grid > max_items) grid = max_items;
    a.status = c.status;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)(32 * (a.ncw + 1)));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_mma<NMAT, MT, GPW, NTOK, MODE, MAXT>, a);
}

int stages_for(size_t fixed, size_t stage) {
    int st = (int)((kSmemBudget - fixed) / stage);
    return st > kMaxStages ? kMaxStages : st;
}

}  // namespace

cudaError_t launch_gemv(const Ctx &c, float *y, const float *x, const uint8_t *packed,
                        const uint8_t *scales, int in, int rows) {
    const int G = in / 32;
    // tensor-core streaming path: 16-byte scale tiles (G % 16 == 0), a
    // 16-byte aligned scale array, and K split over at most 16 warps with 4,
    // 8 or 16 groups each
    int gpw = 0;
    for (int q = 4; q <= 16; q *= 2)
        if (G % q == 0 && G / q <= kMaxConsumerWarps) {
            gpw = q;
            break;
        }
    if (gpw > 0 && G % 16 == 0 && (reinterpret_cast<uintptr_t>(scales) & 15u) == 0) {
        MmaArgs a{};
        a.packed = packed;
        a.scales = scales;
        a.rows = rows;
        a.in = in;
        a.gpw = gpw;
        a.ncw = G / gpw;
        const int ncw = a.ncw;
        const size_t stage = (size_t)16 * (in / 2 + G);
        a.stages = stages_for(mma_smem_bytes(1, 1, 1, in, ncw, a.gpw, 0), stage);
        a.xin = x;
        a.out = y;
        const long long tiles = (rows + 15) / 16;
        if (gpw == 4) return launch_mma<1, 1, 4, 1, kModeGemv, 17 * 32>(c, a, tiles, false);
        if (gpw == 8) return launch_mma<1, 1, 8, 1, kModeGemv, 17 * 32>(c, a, tiles, false);
        return launch_mma<1, 1, 16, 1, kModeGemv, 17 * 32>(c, a, tiles, false);
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

cudaError_t launch_combine(const Ctx &c, float *y, const float *stage, const float *w,
                           int n_tokens) {
    const long long n4 = (long long)n_tokens * (kD / 4);
    const int threads = 256;
    return launch_pdl(k_combine, dim3((unsigned)((n4 + threads - 1) / threads)), dim3(threads), 0, c.stream, y,
                      stage, w, n_tokens);
}

}  // namespace k3mx
