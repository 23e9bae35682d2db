// px.cu - prefill on block-scaled 5th-generation tensor-core MMAs
// (tcgen05 kind::mxf8f6f4): the grouped expert GEMMs of many tokens with the
// packed MXFP4 weights and their ue8m0 group scales fed to the tensor cores
// as stored (Kimi K3 engine (c/kimi_k3.c), "Weights"), with no per-weight
// work in registers: the copy engine spreads each 16 packed e2m1 codes of a
// weight tile over 16 bytes of shared memory (the operand layout this MMA
// kind reads for 4-bit types), the codes themselves untouched.
//
// Activations.  The MMA multiplies e2m1 weights by e4m3 activations, so
// every activation row (x of a token for gate/up, h of a pair for down) is
// split into two MXFP8 (e4m3) pieces per 32-column block: piece i takes the
// scale 2^e that maps the block's largest residual |value| into (224, 448]
// and the nearest e4m3 value of every residual / 2^e; the next residual is
// exact in fp32.  A piece keeps four significant bits of every value within
// 2^15 of the block's largest (e4m3's exponent range), so two pieces
// reproduce a bf16 x exactly in all but extreme blocks, and h (from an f16
// staging copy, 11 bits) to about 2^-9 of each value.  The two pieces of
// every pair of a work unit are one B operand side by side (N = 2 x the
// unit's box rows); the epilogue adds the two accumulator halves.
//
// Work.  A unit is one expert and at most kUT of its (token, slot) pairs,
// contiguous in the grouped order (Kimi K3 engine (c/kimi_k3.c), "Chunked
// prefill": each unique expert is loaded once for all its tokens).  Item =
// (unit, 128-row tile); a CTA per SM takes every grid-th item.  Per
// item K streams in 128-column stages:
//   warp 0      A producer: TMA of the weight tiles (128 rows x 128 codes:
//               64 B each in global memory, 128 B in shared memory, 128-byte
//               swizzle) through per-expert tensor maps into an A ring, the
//               tiles some stages ahead prefetched into L2
//   warp 1      scale loader: the tile's scale bytes (16 per row, four
//               stages ahead) from global into registers, then per stage the
//               scale source tcgen05.cp reads (one 128x256b source for both
//               gate/up matrices, one 128x128b source for down); a group of scale
//               255 gets scale 0 and its codes are zeroed once the tile has
//               landed, so it adds exactly 0
//   warp 2      TMEM owner; lane 0 copies the scales to TMEM and issues,
//               per stage, 4 K steps x NMAT MMAs (M = 128, N = 2 x the unit's
//               box rows, K = 32)
//   warp 3      B producer: one 3-D TMA per stage for both pieces of the
//               unit's rows (box of 8, 16, ..., 96 rows x 128 B) and the
//               stage's 1 KB block of B scales, copied four times (once per
//               TMEM lane quarter), into a B ring
//   warps 4-11  epilogue, two warps per TMEM lane quarter, each half the
//               unit's tokens: gate/up takes g and u into registers and
//               releases the accumulator, then h = SiTU(g, u) through the
//               item's shared h tile split into pieces (rows of the grouped
//               h planes + the unit's B scales for down); down y[t] +=
//               w_tk * Y (fp32 atomics)
// Down keeps two accumulator buffers, so the epilogue of one item overlaps
// the MMAs of the next; gate/up's two matrices leave TMEM room for one,
// released as soon as it is read.  Every wait is bounded; a timeout is
// reported on the device status word and every role leaves its loop.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "pieces.cuh"
#include "prefill.cuh"
#include "tc.cuh"
#include "tmaps.cuh"

namespace k3mx {
namespace {

constexpr int kPPx = 2;                 // e4m3 pieces of x (gate/up's B)
constexpr int kPPh = 2;                 // e4m3 pieces of h (down's B)
constexpr int kUT = 96;                 // pairs per unit (MMA N = 2 x rows <= 192)
constexpr int kKS = 128;                // K columns per stage
constexpr int kATile = 128 * 128;       // A tile in shared memory: 128 rows x 128 B (expanded codes)
constexpr int kATx = 128 * 64;          // the bytes one A tile copy moves (packed codes)
constexpr int kBPiece = kUT * 128;      // one piece of the unit's B: 96 rows x 128 B (e4m3)
constexpr int kBoxes = kUT / 8;
__host__ __device__ constexpr int b_rows(int i) { return 8 * (i + 1); }    // B box heights: 8, 16, ..., 96
// the B box of a unit of n pairs: the smallest height holding them
__host__ __device__ constexpr int b_sel(int n) { return n <= 8 ? 0 : (n + 7) / 8 - 1; }

// the B tensor maps of one pass, one per box height
struct PxBMaps {
    CUtensorMap m[kBoxes];
};
constexpr int kBScaleBlock = 1024;      // a stage's B scales for one lane quarter
constexpr int kPxThreads = 12 * 32;
constexpr int kAProd = 0, kSfW = 1, kMmaW = 2, kBProd = 3, kEpi0 = 4;
constexpr int kEpiThreads = 8 * 32;
constexpr int kPxSmemLimit = 227 * 1024;

template <int PH> struct PxCfg;
// PF: weight stages prefetched into L2 ahead of the copies into the A ring
// (the ring itself holds too few bytes in flight to cover HBM latency)
template <> struct PxCfg<0> {           // gate/up: g = W1 x, u = W3 x
    static constexpr int NMAT = 2, K = kD, M = kF, SA = 3, SB = 3, PP = kPPx, PF = 10;
};
template <> struct PxCfg<1> {           // down: Y = W2 h
    static constexpr int NMAT = 1, K = kF, M = kD, SA = 6, SB = 4, PP = kPPh, PF = 6;
};

template <int PH> struct PxShape {
    using C = PxCfg<PH>;
    static constexpr int NMAT = C::NMAT, K = C::K, M = C::M, SA = C::SA, SB = C::SB, PP = C::PP, PF = C::PF;
    static constexpr int KC = K / kKS, MT = M / 128, G = K / 32;
    // A stage: the tiles, then the scale source of one copy into TMEM:
    // gate/up 128 x 32 bytes for both matrices, down 128 x 16 bytes
    static constexpr int ASCALE = NMAT == 2 ? 128 * 32 : 128 * 16;
    static constexpr int ASTAGE = ((NMAT * kATile + ASCALE) + 1023) / 1024 * 1024;
    // B stage: both pieces' rows, then the stage's B scales as the 4 KB
    // source of one 128x256b copy into TMEM: a 1 KB block (kBScaleBlock)
    // four times, once per lane quarter (every quarter reads every column's
    // scale)
    static constexpr int BSTAGE = PP * kBPiece + 4 * kBScaleBlock;      // 28 KB
    // gate/up: the item's h tile, to turn (feature, token) into (token,
    // feature): per 32-feature block a plane of up to kUT tokens x 32 f16
    // (64 bytes a token), then the exponents [token][block]; a token's 32
    // values of a block are scaled by a power of two that puts their
    // largest magnitude in [2^14, 2^15), so h keeps 11 bits whatever its
    // size.  Planes lie 4 kUT + 1 16-byte units apart, so the eight lanes
    // of a 16-byte load phase (two tokens x four blocks) hit eight
    // different bank groups; a warp's f16 stores fill 64 contiguous bytes.
    static constexpr int HPLANE = (4 * kUT + 1) * 16;
    static constexpr int TRANS = PH == 0 ? 4 * HPLANE + kUT * 4 * 4 : 0;
    static constexpr int SMEM = 1024 + 1024 + SA * ASTAGE + SB * BSTAGE + TRANS;  // alignment slack, header
    // The two pieces side by side in one B operand (N = 2 x the box rows):
    // each accumulator holds a piece-0 and a piece-1 half that the epilogue
    // adds.  Gate/up's two matrices leave TMEM for one accumulator buffer:
    // its epilogue releases the buffer as soon as h is staged in shared
    // memory.
    static constexpr int NACC = 2 * kUT;                       // accumulator columns per matrix
    static constexpr int NBUF = PH == 0 ? 1 : 2;
    // TMEM: accumulators [NBUF][NMAT][NACC], A scales [SA][NMAT][4], B scales [SB][PP][4]
    static constexpr int ACC = NBUF * NMAT * NACC;
    static constexpr int SFA_COL = ACC;
    static constexpr int SFB_COL = SFA_COL + SA * NMAT * 4;
    static constexpr int TMEM_COLS = 512;
    static_assert(SFB_COL + SB * PP * 4 <= TMEM_COLS, "TMEM budget");
    static_assert(PP == 2, "the two pieces form one operand");
    static_assert(SMEM <= kPxSmemLimit, "shared memory budget");
    static_assert(K % (4 * kKS) == 0, "scale rows load in 16-byte groups of four stages");
    static_assert(ASTAGE % 1024 == 0 && BSTAGE % 1024 == 0, "stage alignment");
};

struct PxArgs {
    const int32_t *units;          // [unit][3]: expert, first slot, pairs
    const int32_t *n_units;
    const int32_t *perm;           // slot -> pair t * 16 + k
    const float *w;                // routing weights by pair
    const uint8_t *maps;           // per-expert weight tensor maps [expert][w1, w3, w2]
    const k3mx_expert *experts;    // device table [896]
    const uint8_t *b_atoms;        // B scales of the pass's input [unit][KC][1 KB] (atom_byte_pair)
    uint8_t *h_planes;             // gate/up: h pieces [kPPh][slots][F] (e4m3)
    uint8_t *h_atoms;              // gate/up: down's B scales [unit][F / 128][1 KB]
    size_t slots;                  // 16 T: rows of one piece plane
    float *y;                      // down: [T][D], accumulated
    int *status;
};

struct PxHdr {
    // afull: the A stage's scales (32 scale-loader lanes); atfull: its
    // weight tiles (the producer's expect_tx and the copies' bytes)
    // aempty[s] completes when the MMAs of the stage in slot s are done: the
    // A and B rings advance together (SA >= SB), so it frees B slots too
    uint64_t afull[16], atfull[16], aempty[16], bfull[8], accf[2], acce[2], done;
    // gate/up's h tile: written by all eight epilogue warps (hfull), read
    // by all eight (hfree); one arrival per warp
    uint64_t hfull, hfree;
    uint32_t tmem;
    int abort;
};

// SiTU-GLU for the prefill epilogue (Kimi K3 engine (c/kimi_k3.c),
// "Architecture notes": 4 tanh(g/4) sigma(g) 25 tanh(u/25)), sigma(g) =
// (1 + tanh(g/2)) / 2, for two tokens at once with the hardware tanh on
// f16 pairs (relative error about 2^-10; arguments below 2^-6 in magnitude
// give tanh(x) = x, within x^2 / 3, so small g and u keep their precision)
__device__ __forceinline__ int lane_id() { return (int)(threadIdx.x & 31); }
__device__ __forceinline__ uint4 shfl_u4(uint4 v, int from) {
    return make_uint4(__shfl_sync(0xffffffffu, v.x, from), __shfl_sync(0xffffffffu, v.y, from),
                      __shfl_sync(0xffffffffu, v.z, from), __shfl_sync(0xffffffffu, v.w, from));
}

__device__ __forceinline__ float2 tanh2_f16(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    uint32_t r;
    asm("tanh.approx.f16x2 %0, %1;" : "=r"(r) : "r"(*reinterpret_cast<const uint32_t *>(&h)));
    float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&r));
    if (fabsf(a) < 0.015625f) t.x = a;
    if (fabsf(b) < 0.015625f) t.y = b;
    return t;
}
__device__ __forceinline__ float2 situ_fast2(float g0, float u0, float g1, float u1) {
    const float2 t4 = tanh2_f16(0.25f * g0, 0.25f * g1), t2 = tanh2_f16(0.5f * g0, 0.5f * g1);
    const float2 tu = tanh2_f16(0.04f * u0, 0.04f * u1);
    return make_float2((4.0f * t4.x * (0.5f + 0.5f * t2.x)) * (25.0f * tu.x),
                       (4.0f * t4.y * (0.5f + 0.5f * t2.y)) * (25.0f * tu.y));
}

// The NP MXFP8 pieces of 32 values held by one lane (v, column order):
// piece p takes the scale 2^e that maps the largest remaining |v| into
// (224, 448] (2^-126 at least) and the nearest e4m3 value of every v / 2^e
// (hardware conversion, column j in byte j); v keeps the exact residual.
// bytes[p] are the piece's 32 bytes, scale[p] its ue8m0 byte (255 when the
// values hold Inf or NaN, with zero bytes; 0 when they are all zero).
template <int NP>
__device__ __forceinline__ void lane_pieces_e4m3(float (&v)[32], uint4 (&bytes)[NP][2], uint32_t (&scale)[NP]) {
#pragma unroll
    for (int p = 0; p < NP; p++) {
        // the largest |v| (non-negative floats order as their bit patterns;
        // Inf and NaN lie above every finite value)
        uint32_t mb = 0;
#pragma unroll
        for (int j = 0; j < 32; j++) mb = max(mb, __float_as_uint(fabsf(v[j])));
        const int E = (int)(mb >> 23) - 127;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        uint32_t sb = 0;
        if (E == 128) {
            sb = 255;
        } else if (mb != 0) {
            // 448 = 1.75 x 2^8: max / 2^e in (224, 448]
            const int e = max((mb & 0x7FFFFFu) <= 0x600000u ? E - 8 : E - 7, -126);
            const float down = exp2i(-e), up = exp2i(e);
#pragma unroll
            for (int j = 0; j < 16; j++) {
                uint32_t pair, h2;
                asm("{\n\t.reg .b16 t;\n\t"
                    "cvt.rn.satfinite.e4m3x2.f32 t, %2, %3;\n\t"
                    "cvt.u32.u16 %0, t;\n\t"
                    "cvt.rn.f16x2.e4m3x2 %1, t;\n\t}"
                    : "=r"(pair), "=r"(h2)
                    : "f"(v[2 * j + 1] * down), "f"(v[2 * j] * down));
                const float2 q = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
                v[2 * j] = fmaf(-q.x, up, v[2 * j]);             // exact
                v[2 * j + 1] = fmaf(-q.y, up, v[2 * j + 1]);
                w[j >> 1] |= (pair & 0xFFFFu) << (16 * (j & 1));
            }
            sb = (uint32_t)(e + 127);
        }
        bytes[p][0] = make_uint4(w[0], w[1], w[2], w[3]);
        bytes[p][1] = make_uint4(w[4], w[5], w[6], w[7]);
        scale[p] = sb;
    }
}

// byte of a pass's B scales: per (unit, stage c) one 1 KB block over the
// two pieces' combined rows r = p * rows + n (rows = the unit's box height),
// row r's scale bytes in word r / 32 of line r % 32 of a 128x256b copy
// source (rows32_offset), block kb4 of the stage the byte in the word
template <int PP>
__device__ __forceinline__ size_t atom_byte_pair(int unit, int kc_total, int c, int p, int n, int rows, int kb4) {
    static_assert(PP == 2, "two pieces");
    const int r = p * rows + n;
    return ((size_t)unit * kc_total + c) * kBScaleBlock + rows32_offset(r & 31, r >> 5) + kb4;
}

// an item's unit and whether its expert's pointers are usable (weights
// 32-byte aligned, as the expanding copies need, scales 16-byte aligned;
// the maps of another expert are never used)
// A work item as loaded: ntok < 0 marks a unit whose expert pointers are
// unusable (checked once by k_px_units).  Nothing here computes on the
// loaded values, so decoding the next item only issues its loads: a role
// does not wait for them until that item is its current one.
struct PxItem {
    int unit, mt, e, off, ntok;
    __device__ __forceinline__ bool ok() const { return ntok > 0; }
};
template <int MT>
__device__ __forceinline__ PxItem px_item(const PxArgs &a, long long item) {
    PxItem r;
    r.unit = (int)(item / MT);
    r.mt = (int)(item % MT);
    r.e = __ldg(a.units + 3 * r.unit);
    r.off = __ldg(a.units + 3 * r.unit + 1);
    r.ntok = __ldg(a.units + 3 * r.unit + 2);
    return r;
}
__device__ __forceinline__ const uint8_t *px_scales(const PxArgs &a, int e, int m, int ph) {
    // k3mx_expert fields in order: w1, s1, w3, s3, w2, s2
    const unsigned long long *q = reinterpret_cast<const unsigned long long *>(a.experts + e);
    return reinterpret_cast<const uint8_t *>(__ldg(q + (ph == 1 ? 5 : (m == 0 ? 1 : 3))));
}

__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <int PH>
__global__ void __launch_bounds__(kPxThreads, 1)
    k_px(const PxArgs a, const __grid_constant__ PxBMaps bmaps) {
    using Sh = PxShape<PH>;
    constexpr int NMAT = Sh::NMAT, KC = Sh::KC, MT = Sh::MT, G = Sh::G, SA = Sh::SA, SB = Sh::SB;
    static_assert(SA <= 16 && SB <= 8, "barrier slots");
    static_assert(SA >= SB, "a B slot is freed by the A ring's empty barrier");

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PxHdr *hd = reinterpret_cast<PxHdr *>(smem);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t ar0 = sbase + 1024;                      // A ring [SA][ASTAGE]
    const uint32_t br0 = ar0 + SA * Sh::ASTAGE;             // B ring [SB][BSTAGE]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t afull0 = smem_addr(hd->afull), aempty0 = smem_addr(hd->aempty);
    const uint32_t atfull0 = smem_addr(hd->atfull);
    const uint32_t bfull0 = smem_addr(hd->bfull);
    const uint32_t accf0 = smem_addr(hd->accf), acce0 = smem_addr(hd->acce);
    const uint32_t done = smem_addr(&hd->done);
    const uint32_t hfull = smem_addr(&hd->hfull), hfree = smem_addr(&hd->hfree);

    if (tid == 0) {
        for (int i = 0; i < SA; i++) {
            mbar_init(afull0 + 8 * i, 32);         // the scale loader's lanes
            mbar_init(atfull0 + 8 * i, 1);         // the producer's expect_tx
            mbar_init(aempty0 + 8 * i, 1);
        }
        for (int i = 0; i < SB; i++) {
            mbar_init(bfull0 + 8 * i, 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(accf0 + 8 * i, 1);
            mbar_init(acce0 + 8 * i, kEpiThreads);
        }
        mbar_init(done, 1);
        mbar_init(hfull, kEpiThreads / 32);
        mbar_init(hfree, kEpiThreads / 32);
        hd->abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaW) tmem_alloc(smem_addr(&hd->tmem), Sh::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = hd->tmem;
    volatile int *abort_flag = &hd->abort;
    // gate/up reads the prep kernels' results everywhere; down reads gate/up's
    // h only in the B producer (the weights and work units were ready before
    // gate/up started), so its weight stream starts as gate/up CTAs retire
    if (PH == 0) pdl_wait();
    pdl_launch_dependents();

    // Items are dealt round robin (item = CTA + k * grid): at any time the
    // CTAs work on a few consecutive units, so each unit's activation rows
    // come from HBM once and from L2 for its other row tiles.
    const long long items = (long long)__ldg(a.n_units) * MT;
    const long long i0 = blockIdx.x, istep = gridDim.x;
    auto fail = [&](int detail) {
        report_status(a.status, kStatusWaitTimeout, detail);
        *abort_flag = 1;
    };

    if (warp == kAProd) {
        // ------------------------------------------------- A producer --
        const uint64_t pol = l2_evict_first_policy();       // weights: read once
        uint32_t sa = 0;
        int cur_e = -1;
        const uint8_t *map0 = nullptr, *map1 = nullptr;
        // L2 prefetch cursor: Sh::PF stages ahead of the copies, over the
        // same sequence of (item, stage)
        long long pf_item = i0;
        int pf_c = 0, pf_e = -1;
        PxItem pit = pf_item < items ? px_item<MT>(a, pf_item) : PxItem{};
        auto prefetch_next = [&]() {
            while (pf_item < items && !pit.ok()) {
                pf_item += istep;
                pf_c = 0;
                if (pf_item < items) pit = px_item<MT>(a, pf_item);
            }
            if (pf_item >= items) return;
            if (lane == 0) {
                const uint8_t *em = a.maps + (size_t)pit.e * kMapsPerExpert * kMapBytes;
                const uint8_t *m0 = em + (PH == 0 ? 0 : 2) * kMapBytes, *m1 = em + kMapBytes;
                if (pit.e != pf_e) {
                    acquire_map(m0);
                    if (NMAT == 2) acquire_map(m1);
                }
                tma_prefetch_2d(m0, pf_c * kKS, pit.mt * 128);
                if (NMAT == 2) tma_prefetch_2d(m1, pf_c * kKS, pit.mt * 128);
            }
            pf_e = pit.e;
            if (++pf_c == KC) {
                pf_c = 0;
                pf_item += istep;
                if (pf_item < items) pit = px_item<MT>(a, pf_item);
            }
        };
        for (int k = 0; k < Sh::PF; k++) prefetch_next();
        PxItem nxt = i0 < items ? px_item<MT>(a, i0) : PxItem{};
        for (long long item = i0; item < items && !*abort_flag; item += istep) {
            const PxItem it = nxt;                 // decoded one item ahead (dependent loads)
            if (item + istep < items) nxt = px_item<MT>(a, item + istep);
            if (!it.ok()) {
                if (lane == 0 && it.mt == 0) report_status(a.status, kStatusBadPointer, it.e);
                continue;
            }
            if (it.e != cur_e) {
                const uint8_t *em = a.maps + (size_t)it.e * kMapsPerExpert * kMapBytes;
                map0 = em + (PH == 0 ? 0 : 2) * kMapBytes;
                map1 = em + 1 * kMapBytes;
                if (lane == 0) {
                    acquire_map(map0);
                    if (NMAT == 2) acquire_map(map1);
                }
                cur_e = it.e;
            }
            bool ok = true;
            for (int c = 0; c < KC; c++, sa++) {
                const int s = sa % SA;
                if (!mbar_wait(aempty0 + 8 * s, ((sa / SA) & 1) ^ 1)) {
                    if (lane == 0) fail(300 + PH);
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t dst = ar0 + s * Sh::ASTAGE;
                    mbar_arrive_expect_tx(atfull0 + 8 * s, NMAT * kATx);
                    tma_2d(dst, map0, c * kKS, it.mt * 128, atfull0 + 8 * s, pol);
                    if (NMAT == 2) tma_2d(dst + kATile, map1, c * kKS, it.mt * 128, atfull0 + 8 * s, pol);
                }
                prefetch_next();
                __syncwarp();
            }
            if (!ok) break;
        }
        // copies still in flight (after a wait gave up) land before the CTA leaves
        if (lane == 0 && !drain_ring(atfull0, SA, sa)) report_status(a.status, kStatusWaitTimeout, 370 + PH);
    } else if (warp == kSfW) {
        // ----------------------------------------------- scale loader --
        // Each weight row's scale bytes load 16 at a time (four stages) into
        // registers two groups ahead; per stage, lane l writes line l of
        // each matrix's atom: rows l, l + 32, l + 64, l + 96, four bytes each
        constexpr int NG = KC / 4;                            // 16-byte groups per row
        uint4 cur[NMAT][4], n1[NMAT][4], n2[NMAT][4];
        // the group sequence: (item, group) for every item of the range
        auto advance = [&](long long &item, int &g) -> bool {
            if (++g == NG) {
                g = 0;
                item += istep;
            }
            return item < items;
        };
        auto load_group = [&](long long item, int g, uint4 (&dst)[NMAT][4]) {
            const PxItem it = px_item<MT>(a, item);
            if (!it.ok()) return;
#pragma unroll
            for (int m = 0; m < NMAT; m++) {
                const uint8_t *base = px_scales(a, it.e, m, PH) + (size_t)(it.mt * 128 + lane) * G + 16 * g;
#pragma unroll
                for (int i = 0; i < 4; i++)
                    dst[m][i] = __ldg(reinterpret_cast<const uint4 *>(base + (size_t)32 * i * G));
            }
        };
        long long la_item = i0;
        int la_g = 0;
        bool have2 = la_item < items;
        if (have2) load_group(la_item, la_g, cur);
        have2 = have2 && advance(la_item, la_g);
        if (have2) load_group(la_item, la_g, n1);
        have2 = have2 && advance(la_item, la_g);
        if (have2) load_group(la_item, la_g, n2);
        uint32_t sa = 0;
        PxItem nxt = i0 < items ? px_item<MT>(a, i0) : PxItem{};
        for (long long item = i0; item < items && !*abort_flag; item += istep) {
            const PxItem it = nxt;                 // decoded one item ahead (dependent loads)
            if (item + istep < items) nxt = px_item<MT>(a, item + istep);
            bool ok = true;
            for (int g = 0; g < NG && ok; g++) {
                if (it.ok()) {
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const int s = (int)(sa % SA);
                        if (!mbar_wait(aempty0 + 8 * s, ((sa / SA) & 1) ^ 1)) {
                            if (lane == 0) fail(310 + PH);
                            ok = false;
                            break;
                        }
                        const uint32_t ast = ar0 + s * Sh::ASTAGE, at0 = ast + NMAT * kATile;
                        uint32_t wq[NMAT][4];
#pragma unroll
                        for (int m = 0; m < NMAT; m++)
#pragma unroll
                            for (int i = 0; i < 4; i++)
                                wq[m][i] = j == 0 ? cur[m][i].x : j == 1 ? cur[m][i].y : j == 2 ? cur[m][i].z : cur[m][i].w;
                        // groups with scale 255 contribute nothing: once the
                        // stage's weight tiles landed, their codes are zeroed
                        // (rare; most stages skip this)
                        uint32_t nan = 0;
#pragma unroll
                        for (int m = 0; m < NMAT; m++)
#pragma unroll
                            for (int i = 0; i < 4; i++) nan |= nan_scale_mask(wq[m][i]);
                        if (__any_sync(0xffffffffu, nan != 0)) {
                            if (!mbar_wait(atfull0 + 8 * s, (sa / SA) & 1)) {
                                if (lane == 0) fail(315 + PH);
                                ok = false;
                                break;
                            }
#pragma unroll
                            for (int m = 0; m < NMAT; m++)
#pragma unroll
                                for (int i = 0; i < 4; i++) zero_nan_groups_x128(ast + m * kATile, lane + 32 * i, wq[m][i]);
                        }
                        if (NMAT == 2) {
                            // row lane + 32 i: word i the gate's scales, word 4 + i the up's
#pragma unroll
                            for (int m = 0; m < NMAT; m++)
#pragma unroll
                                for (int i = 0; i < 4; i++)
                                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(at0 + rows32_offset(lane + 32 * i, 4 * m + i)),
                                                 "r"(drop_nan_scales(wq[m][i]))
                                                 : "memory");
                        } else {
                            // row lane + 32 i of a 128 x 16-byte source: word i its scales
#pragma unroll
                            for (int i = 0; i < 4; i++)
                                asm volatile("st.shared.u32 [%0], %1;" ::"r"(at0 + 16 * (lane + 32 * i) + 4 * i),
                                             "r"(drop_nan_scales(wq[0][i]))
                                             : "memory");
                        }
                        fence_async_smem();
                        mbar_arrive(afull0 + 8 * s);
                        sa++;
                    }
                }
                // rotate the register groups and load two ahead
#pragma unroll
                for (int m = 0; m < NMAT; m++)
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        cur[m][i] = n1[m][i];
                        n1[m][i] = n2[m][i];
                    }
                if (have2) {
                    have2 = advance(la_item, la_g);
                    if (have2) load_group(la_item, la_g, n2);
                }
            }
            if (!ok) break;
        }
    } else if (warp == kBProd) {
        // ------------------------------------------------- B producer --
        if (PH == 1) pdl_wait();                               // h of every pair is written
        const uint64_t pol = l2_evict_normal_policy();
        uint32_t sb = 0;
        PxItem nxt = i0 < items ? px_item<MT>(a, i0) : PxItem{};
        for (long long item = i0; item < items && !*abort_flag; item += istep) {
            const PxItem it = nxt;                 // decoded one item ahead (dependent loads)
            if (item + istep < items) nxt = px_item<MT>(a, item + istep);
            if (!it.ok()) continue;
            const int hsel = b_sel(it.ntok);
            const void *bm = &bmaps.m[hsel];
            const int rows = b_rows(hsel);
            bool ok = true;
            for (int c = 0; c < KC; c++, sb++) {
                const int s = sb % SB;
                // slot s last held stage sb - SB: its MMAs are done when
                // aempty of that stage's A slot completes phase (sb - SB) / SA
                // (that barrier cannot run a phase further ahead: it would
                // need stage sb - SB + SA >= sb, not yet filled here)
                if (sb >= (uint32_t)SB) {
                    const uint32_t j = sb - SB;
                    if (!mbar_wait(aempty0 + 8 * (j % SA), (j / SA) & 1)) {
                        if (lane == 0) fail(320 + PH);
                        ok = false;
                        break;
                    }
                }
                if (lane == 0) {
                    const uint32_t dst = br0 + s * Sh::BSTAGE;
                    const uint32_t bf = bfull0 + 8 * s;
                    mbar_arrive_expect_tx(bf, (uint32_t)(Sh::PP * rows * 128 + 4 * kBScaleBlock));
                    // pieces land `rows` rows apart: [piece][rows][128 B]
                    tma_3d(dst, bm, c * kKS, it.off, 0, bf, pol);
                    // the stage's scale block once per lane quarter
                    const uint8_t *sblk = a.b_atoms + ((size_t)it.unit * KC + c) * kBScaleBlock;
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        bulk_g2s(dst + Sh::PP * kBPiece + q * kBScaleBlock, sblk, kBScaleBlock, bf, pol);
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        if (lane == 0 && !drain_ring(bfull0, SB, sb)) report_status(a.status, kStatusWaitTimeout, 372 + PH);
    } else if (warp == kMmaW) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            uint32_t sa = 0, sb = 0, itn = 0;
            bool run = true;
            // the next stage's three barriers, polled while the last MMA of
            // a stage issues: when they had completed, that stage starts
            // without the waits' shared-memory round trips
            bool ready = false;
            PxItem nxt = i0 < items ? px_item<MT>(a, i0) : PxItem{};
            for (long long item = i0; item < items && run && !*abort_flag; item += istep) {
                const PxItem it = nxt;             // decoded one item ahead (dependent loads)
                if (item + istep < items) nxt = px_item<MT>(a, item + istep);
                if (!it.ok()) continue;
                // both pieces: N covers two box heights
                const int nmma = 2 * b_rows(b_sel(it.ntok));
                uint32_t idk[4];
#pragma unroll
                for (int ks = 0; ks < 4; ks++) idk[ks] = idesc_e2m1_e4m3(nmma, ks);
                const int b = itn % Sh::NBUF;
                if (!mbar_wait(acce0 + 8 * b, ((itn / Sh::NBUF) & 1) ^ 1)) {
                    fail(330 + PH);
                    break;
                }
                tc_fence_after();
                for (int c = 0; c < KC; c++, sa++, sb++) {
                    const int s_a = sa % SA, s_b = sb % SB;
                    if (!ready && (!mbar_wait(atfull0 + 8 * s_a, (sa / SA) & 1) ||
                                   !mbar_wait(afull0 + 8 * s_a, (sa / SA) & 1) ||
                                   !mbar_wait(bfull0 + 8 * s_b, (sb / SB) & 1))) {
                        fail(340 + PH);
                        run = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ast = ar0 + s_a * Sh::ASTAGE, bst = br0 + s_b * Sh::BSTAGE;
                    const uint32_t sfa = tmem + Sh::SFA_COL + s_a * NMAT * 4;
                    const uint32_t sfb = tmem + Sh::SFB_COL + s_b * Sh::PP * 4;
                    if (NMAT == 2)
                        tmem_cp_rows32(sfa, desc_rows32(ast + NMAT * kATile));
                    else
                        tmem_cp_rows16(sfa, desc_atom(ast + NMAT * kATile, 128));
                    // B scales: the 2 x rows combined rows of the operand, 8
                    // columns in one copy
                    tmem_cp_rows32(sfb, desc_rows32(bst + Sh::PP * kBPiece));
#pragma unroll
                    for (int m = 0; m < NMAT; m++)
#pragma unroll
                        for (int ks = 0; ks < 4; ks++) {
                            const uint32_t d = tmem + (b * NMAT + m) * Sh::NACC;
                            const uint64_t ad = umma_desc_sw128(ast + m * kATile + 32 * ks), bd = umma_desc_sw128(bst + 32 * ks);
                            const uint32_t acc = (c | ks) != 0 ? 1u : 0u;
                            if (m == NMAT - 1 && ks == 3) {
                                // the barriers of stage sa + 1 (of this item or the next)
                                const uint32_t na = (sa + 1) % SA, pa = ((sa + 1) / SA) & 1;
                                const uint32_t nb = (sb + 1) % SB, pb = ((sb + 1) / SB) & 1;
                                ready = mma_mxf8f6f4_poll3(d, ad, bd, idk[ks], sfa + m * 4, sfb, acc, atfull0 + 8 * na, pa,
                                                           afull0 + 8 * na, pa, bfull0 + 8 * nb, pb);
                            } else {
                                mma_mxf8f6f4(d, ad, bd, idk[ks], sfa + m * 4, sfb, acc);
                            }
                        }
                    umma_commit(aempty0 + 8 * s_a);
                }
                if (!run) break;
                umma_commit(accf0 + 8 * b);
                itn++;
            }
            umma_commit(done);
        }
        __syncwarp();
    } else {
        // --------------------------------------------------- epilogue --
        const int q4 = warp & 3, half = (warp - kEpi0) >> 2;
        (void)half;
        const int row_in_tile = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        uint32_t itn = 0, hit = 0;       // items done; gate/up items through the h tile
        PxItem nxt = i0 < items ? px_item<MT>(a, i0) : PxItem{};
        for (long long item = i0; item < items && !*abort_flag; item += istep) {
            const PxItem it = nxt;                 // decoded one item ahead (dependent loads)
            if (item + istep < items) nxt = px_item<MT>(a, item + istep);
            if (!it.ok()) continue;
            const int b = itn % Sh::NBUF;
            if (!mbar_wait(accf0 + 8 * b, (itn / Sh::NBUF) & 1)) {
                if (lane == 0) fail(350 + PH);
                break;
            }
            tc_fence_after();
            const int n0 = half * (kUT / 2), n1 = min(it.ntok, n0 + kUT / 2);
            const int row = it.mt * 128 + row_in_tile;
            if (PH == 0) {
                // Groups of 16 tokens, dealt alternately to the two warps of
                // a lane quarter (this warp: groups half, half + 2, half + 4).
                // First each group's g and u (piece-0 plus piece-1 columns)
                // into registers and the accumulator is released; then each
                // group's h, in f16 scaled per token and 32-feature block,
                // into the item's shared h tile; then the eight warps split
                // the tile by (token, 32-feature block) into the two pieces,
                // four neighbouring lanes storing a token's 128 bytes of a
                // piece row whole.
                const int hrows = b_rows(b_sel(it.ntok));         // the unit's B box height
                uint8_t *htile = smem + 1024 + SA * Sh::ASTAGE + SB * Sh::BSTAGE;
                int *hexp = reinterpret_cast<int *>(htile + 4 * Sh::HPLANE);
                const size_t plane = a.slots * kF;
                const int ng = (it.ntok + 15) >> 4;               // groups of the unit
                const int nslot = ng > half ? (ng - half + 1) >> 1 : 0;   // this warp's groups
                static_assert(kUT <= 6 * 16, "three groups of 16 tokens per epilogue warp");
                float gs[3][16], us[3][16];
#pragma unroll
                for (int i = 0; i < 3; i++) {
                    if (i < nslot) {
                        uint32_t p0[16], p1[16];
                        const uint32_t cg = tmem + lane_base + (uint32_t)(16 * (half + 2 * i)), cu = cg + Sh::NACC;
                        tmem_ld16(cg, p0);
                        tmem_ld16(cg + hrows, p1);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; j++) gs[i][j] = __uint_as_float(p0[j]) + __uint_as_float(p1[j]);
                        tmem_ld16(cu, p0);
                        tmem_ld16(cu + hrows, p1);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; j++) us[i][j] = __uint_as_float(p0[j]) + __uint_as_float(p1[j]);
                    }
                }
                tc_fence_before();
                mbar_arrive(acce0 + 8 * b);
                // the tile is free once every epilogue warp has read the
                // previous item's
                if (hit > 0 && !mbar_wait(hfree, (hit - 1) & 1)) {
                    if (lane == 0) fail(356);
                    break;
                }
#pragma unroll
                for (int i = 0; i < 3; i++) {
                    if (i < nslot) {
                        const int n0 = 16 * (half + 2 * i);           // the group's first token
                        float hv[16];
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            const float2 h2 = situ_fast2(gs[i][j], us[i][j], gs[i][j + 1], us[i][j + 1]);
                            hv[j] = h2.x;
                            hv[j + 1] = h2.y;
                        }
                        // each token's block of 32 features: its largest |h| sets the scale
                        uint32_t mb[16];
#pragma unroll
                        for (int j = 0; j < 16; j++) mb[j] = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv[j])));
#pragma unroll
                        for (int j = 0; j < 16; j++) {
                            const int E = (int)(mb[j] >> 23);
                            const int es = (E == 0 || E == 255) ? 0 : max(-100, min(100, E - 127 - 14));
                            *reinterpret_cast<__half *>(htile + q4 * Sh::HPLANE + (n0 + j) * 64 + 2 * lane) =
                                __float2half_rn(hv[j] * __int_as_float((127 - es) << 23));
                            if (lane == j) hexp[(n0 + j) * 4 + q4] = es;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(hfull);
                if (!mbar_wait(hfull, hit & 1)) {
                    if (lane == 0) fail(357);
                    break;
                }
                const int te = (warp - kEpi0) * 32 + lane;
                const int sub = lane & 3;                         // the lane's block within its token's four
#pragma unroll 1
                for (int k0 = 0; k0 < 4 * kUT; k0 += kEpiThreads) {
                    const int n = (k0 + te) >> 2;                 // token of the unit
                    const bool live = n < it.ntok;
                    float v[32];
                    if (live) {
                        const float up = __int_as_float((127 + hexp[n * 4 + sub]) << 23);
                        const uint8_t *src = htile + sub * Sh::HPLANE + n * 64;
#pragma unroll
                        for (int c = 0; c < 4; c++) {
                            const uint4 q = reinterpret_cast<const uint4 *>(src)[c];
                            const uint32_t ws[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                            for (int k = 0; k < 4; k++) {
                                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ws[k]));
                                v[8 * c + 2 * k] = f.x * up;
                                v[8 * c + 2 * k + 1] = f.y * up;
                            }
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; k++) v[k] = 0.f;
                    }
                    uint4 wds[kPPh][2];
                    uint32_t sc[kPPh];
                    lane_pieces_e4m3<kPPh>(v, wds, sc);
                    // the token's four lanes hold its 128 bytes of a piece row
                    // as 8 chunks of 16 (chunk c: half c % 2 of lane c / 2):
                    // the first store writes chunks 0-3, the second 4-7
                    const int g0 = lane & ~3;
                    uint8_t *dst = a.h_planes + ((size_t)it.off + n) * kF + (size_t)it.mt * 128 + 16 * sub;
#pragma unroll
                    for (int p = 0; p < kPPh; p++) {
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            const int from = g0 + 2 * h + (sub >> 1);
                            const uint4 lo = shfl_u4(wds[p][0], from), hi = shfl_u4(wds[p][1], from);
                            if (live) reinterpret_cast<uint4 *>(dst + p * plane + 64 * h)[0] = (sub & 1) ? hi : lo;
                        }
                        // the four blocks' scale bytes: one word of the stage's scale block
                        const uint32_t b1 = __shfl_down_sync(0xffffffffu, sc[p], 1), b2 = __shfl_down_sync(0xffffffffu, sc[p], 2);
                        const uint32_t b3 = __shfl_down_sync(0xffffffffu, sc[p], 3);
                        if (live && sub == 0)
                            *reinterpret_cast<uint32_t *>(a.h_atoms + atom_byte_pair<kPPh>(it.unit, kF / kKS, it.mt, p, n, hrows, 0)) =
                                (sc[p] & 0xFFu) | (b1 & 0xFFu) << 8 | (b2 & 0xFFu) << 16 | (b3 & 0xFFu) << 24;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(hfree);
                hit++;
            } else {
                // token n's sum: the even-piece column n plus the odd-piece
                // column rows + n
                const int rows = b_rows(b_sel(it.ntok));
                for (int nb = n0; nb < n1; nb += 16) {
                    // the group's pairs and routing weights: lane j < 16
                    // loads token nb + j's (one round trip for the group, not
                    // two dependent loads per token), shared by shuffles
                    const int nn = min(16, n1 - nb);
                    int pj = 0;
                    float wj = 0.f;
                    if (lane < nn) {
                        pj = __ldg(a.perm + it.off + nb + lane);
                        wj = __ldg(a.w + pj);
                    }
                    uint32_t dv[16], dw[16];
                    tmem_ld16(tmem + lane_base + (uint32_t)b * Sh::NACC + nb, dv);
                    tmem_ld16(tmem + lane_base + (uint32_t)b * Sh::NACC + rows + nb, dw);   // NMAT = 1
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const int pair = __shfl_sync(0xffffffffu, pj, j);
                        const float wt = __shfl_sync(0xffffffffu, wj, j);
                        if (j < nn) {
                            const float yv = __uint_as_float(dv[j]) + __uint_as_float(dw[j]);
                            atomicAdd(a.y + (size_t)(pair / kK) * kD + row, wt * yv);
                        }
                    }
                }
            }
            if (PH == 1) {
                tc_fence_before();
                mbar_arrive(acce0 + 8 * b);
            }
            itn++;
        }
    }

    __syncthreads();
    if (warp == kMmaW) {
        // no MMA may still be running when TMEM is released
        if (!mbar_wait_drain(done, 0) && lane == 0) report_status(a.status, kStatusWaitTimeout, 360 + PH);
        tc_fence_after();
        tmem_dealloc(tmem, Sh::TMEM_COLS);
    }
}

// ------------------------------------------------------------ preparation --

// Work units: every active expert's pairs cut into ceil(n / kUT) runs of
// nearly equal length (one 1024-thread CTA, expert e on thread e).
__global__ void __launch_bounds__(1024) k_px_units(const int32_t *counts, const int32_t *offsets,
                                                   int32_t *units, int32_t *n_units, int32_t *slot_of_pair,
                                                   int n_pairs, const k3mx_expert *experts) {
    __shared__ int tmp[33];
    const int e = threadIdx.x, lane = e & 31, wp = e >> 5;
    const int cnt = e < kE ? counts[e] : 0;
    const int nu = (cnt + kUT - 1) / kUT;
    int incl = nu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) tmp[wp] = incl;
    __syncthreads();
    if (wp == 0) {
        const int ws = tmp[lane];
        int wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += v;
        }
        tmp[lane] = wi - ws;
        if (lane == 31) tmp[32] = wi;
    }
    __syncthreads();
    const int pos = incl - nu + tmp[wp];
    // every pair's slot starts as "not grouped" (a slot dropped by top-p)
    for (int i = threadIdx.x; i < n_pairs; i += blockDim.x) slot_of_pair[i] = -1;
    if (e < kE && nu > 0) {
        const int o0 = offsets[e];
        // the expert's weights 32-byte and scales 16-byte aligned, else its
        // units carry minus their pair counts (reported, and skipped, by
        // the passes)
        const uint4 *q = reinterpret_cast<const uint4 *>(experts + e);
        const uint4 v0 = __ldg(q), v1 = __ldg(q + 1), v2 = __ldg(q + 2);
        const bool usable = ((v0.x | v1.x | v2.x) & 31u) == 0 && ((v0.z | v1.z | v2.z) & 15u) == 0;
        for (int k = 0; k < nu; k++) {
            const int lo = (int)((long long)cnt * k / nu), hi = (int)((long long)cnt * (k + 1) / nu);
            units[3 * (pos + k) + 0] = e;
            units[3 * (pos + k) + 1] = o0 + lo;
            units[3 * (pos + k) + 2] = usable ? hi - lo : lo - hi;       // 1 <= hi - lo <= kUT
        }
    }
    if (e == 0) *n_units = tmp[32];
}

// A pair's place in its unit, packed: unit u, row n < kUT, box height
// index b_sel(pairs of the unit) (u stays below 2^20 for any workspace that
// fits in memory)
__host__ __device__ constexpr int32_t pack_pair_un(int u, int n, int bsel) { return (u << 11) | (n << 4) | bsel; }
static_assert(kUT <= 128 && kBoxes <= 16, "pack_pair_un fields");

// CTAs below max_units: each pair of unit u gets its slot and its place in
// the unit; the CTAs after them build the weight tensor maps of the expert
// table.
__global__ void __launch_bounds__(256)
k_px_slots(const int32_t *units, const int32_t *n_units, const int32_t *perm, int32_t *pair_un,
           int32_t *slot_of_pair, int max_units, uint8_t *maps, const k3mx_expert *table,
           const __grid_constant__ CUtensorMap w13, const __grid_constant__ CUtensorMap w2) {
    if ((int)blockIdx.x < max_units) {
        const int u = blockIdx.x;
        if (u >= __ldg(n_units)) return;
        const int off = units[3 * u + 1], ntok = units[3 * u + 2];
        for (int n = threadIdx.x; n < ntok; n += blockDim.x) {
            const int slot = off + n, pair = perm[slot];
            pair_un[pair] = pack_pair_un(u, n, b_sel(ntok));
            slot_of_pair[pair] = slot;
        }
        return;
    }
    build_maps_cta(maps, kE, table, k3mx_expert{}, w13, w2, blockIdx.x - max_units, 32);
}


// One thread per (token, 32-column block): x (bf16) -> kPPx pieces, written
// to the token's 16 slots (rows of the piece planes and bytes of the units'
// B scale blocks); y of the token's block zeroed for the down pass's sums.
// A half-warp holds 16 blocks of one token (512 contiguous bytes of a piece
// row): per slot and piece the warp stores them in two fully used 512-byte
// runs, lane L writing 16 bytes of each.
__global__ void __launch_bounds__(256)
k_px_xprep(const uint16_t *__restrict__ x, int n_tokens, const int32_t *__restrict__ slot_of_pair,
           const int32_t *__restrict__ pair_un, uint8_t *__restrict__ planes, uint8_t *__restrict__ atoms,
           size_t slots, float *__restrict__ y) {
    constexpr int NB = kD / 32, KC = kD / kKS;
    static_assert(NB % 16 == 0, "a token's blocks fill whole half-warps");
    const long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    // every lane of the warp takes part in the shuffles below; lanes past the
    // last block (whole half-warps, as NB is a multiple of 16) only idle
    const bool active = w < (long long)n_tokens * NB;
    const int t = active ? (int)(w / NB) : 0, kb = active ? (int)(w % NB) : 0;
    const size_t i0 = (size_t)t * kD + (size_t)kb * 32;
    // the token's slots and places in units: independent loads, issued first
    int slot[kK], info[kK];
#pragma unroll
    for (int q = 0; q < kK / 4; q++) {
        const int4 s4 = active ? __ldg(reinterpret_cast<const int4 *>(slot_of_pair + (size_t)t * kK) + q)
                               : make_int4(-1, -1, -1, -1);
        const int4 u4 = active ? __ldg(reinterpret_cast<const int4 *>(pair_un + (size_t)t * kK) + q)
                               : make_int4(0, 0, 0, 0);
        slot[4 * q] = s4.x, slot[4 * q + 1] = s4.y, slot[4 * q + 2] = s4.z, slot[4 * q + 3] = s4.w;
        info[4 * q] = u4.x, info[4 * q + 1] = u4.y, info[4 * q + 2] = u4.z, info[4 * q + 3] = u4.w;
    }
    float v[32];
    const uint4 *src = reinterpret_cast<const uint4 *>(x + i0);
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const uint4 u = active ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            v[8 * q + 2 * k] = __uint_as_float(ws[k] << 16);
            v[8 * q + 2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
        }
    }
    if (active) {
        float4 *yz = reinterpret_cast<float4 *>(y + i0);
#pragma unroll
        for (int q = 0; q < 8; q++) yz[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint4 wds[kPPx][2];
    uint32_t sc[kPPx];
    lane_pieces_e4m3<kPPx>(v, wds, sc);
    // the four blocks of a 128-column stage are four consecutive lanes: their
    // scale bytes form one word of the stage's scale block, stored by the first
    uint32_t word[kPPx];
#pragma unroll
    for (int p = 0; p < kPPx; p++) {
        const uint32_t b1 = __shfl_down_sync(0xffffffffu, sc[p], 1), b2 = __shfl_down_sync(0xffffffffu, sc[p], 2);
        const uint32_t b3 = __shfl_down_sync(0xffffffffu, sc[p], 3);
        word[p] = (sc[p] & 0xFFu) | (b1 & 0xFFu) << 8 | (b2 & 0xFFu) << 16 | (b3 & 0xFFu) << 24;
    }
    // chunk L of half-warp h's 512 bytes (16 B): half L % 2 of lane 16 h + L / 2
    uint4 ch[kPPx][2];
#pragma unroll
    for (int p = 0; p < kPPx; p++)
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int from = 16 * h + (lane_id() >> 1);
            const uint4 lo = shfl_u4(wds[p][0], from), hi = shfl_u4(wds[p][1], from);
            ch[p][h] = (lane_id() & 1) ? hi : lo;
        }
    const int kb0 = __shfl_sync(0xffffffffu, kb, 0), kb1 = __shfl_sync(0xffffffffu, kb, 16);
    const bool first = active && (kb & 3) == 0;
#pragma unroll
    for (int k = 0; k < kK; k++) {
        // -1: a dropped pair (top-p) or a half-warp past the last token
        const int s0 = __shfl_sync(0xffffffffu, slot[k], 0), s1 = __shfl_sync(0xffffffffu, slot[k], 16);
#pragma unroll
        for (int p = 0; p < kPPx; p++) {
            uint8_t *plane = planes + (size_t)p * slots * kD + 16 * lane_id();
            if (s0 >= 0) *reinterpret_cast<uint4 *>(plane + (size_t)s0 * kD + (size_t)kb0 * 32) = ch[p][0];
            if (s1 >= 0) *reinterpret_cast<uint4 *>(plane + (size_t)s1 * kD + (size_t)kb1 * 32) = ch[p][1];
        }
        if (first && slot[k] >= 0) {
            const int u = info[k] >> 11, n = (info[k] >> 4) & 127, rows = b_rows(info[k] & 15);
#pragma unroll
            for (int p = 0; p < kPPx; p++)
                *reinterpret_cast<uint32_t *>(atoms + atom_byte_pair<kPPx>(u, KC, kb >> 2, p, n, rows, 0)) = word[p];
        }
    }
}

// ------------------------------------------------------------- launchers --

template <int PH>
cudaError_t launch_px_t(const Ctx &c, const PxArgs &a, const PxBMaps &bmaps, long long max_items) {
    using Sh = PxShape<PH>;
    static std::atomic<uint64_t> configured{0};
    const cudaError_t e = ensure_smem((const void *)k_px<PH>, Sh::SMEM, configured);
    if (e != cudaSuccess) return e;
    long long grid = c.num_sms;
    if (grid > max_items) grid = max_items;
    if (grid < 1) grid = 1;
    return launch_pdl(k_px<PH>, dim3((unsigned)grid), dim3(kPxThreads), (size_t)Sh::SMEM, c.stream, a, bmaps);
}

// 2-D map over a packed e2m1 matrix of `rows` rows of `cols` codes: boxes
// of 128 rows x 128 codes, each 16 packed codes (8 bytes) landing in a
// 16-byte chunk of shared memory (128-byte rows, 128-byte swizzle)
bool encode_e2m1_x128(CUtensorMap &m, const void *base, uint64_t cols, uint64_t rows) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows}, strides[1] = {cols / 2};
    const cuuint32_t box[2] = {128, 128}, es[2] = {1, 1};
    return enc(&m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// weight map templates of the prefill path, encoded once per device over
// the library's scratch array (any 32-byte aligned address works for a
// template; the device replaces it per expert)
bool px_weight_templates(CUtensorMap &w13, CUtensorMap &w2) {
    constexpr int kDevs = 64;
    static std::atomic<int> state[kDevs];  // 0 not tried, 1 ok, 2 failed
    static CUtensorMap t13[kDevs], t2[kDevs];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return false;
    if (state[dev].load(std::memory_order_acquire) == 0) {
        void *base = library_scratch();
        std::lock_guard<std::mutex> lock(setup_mutex());
        if (state[dev].load(std::memory_order_relaxed) == 0) {
            const bool ok = base != nullptr && library_scratch_bytes() >= (size_t)kD / 2 * kF &&
                            encode_e2m1_x128(t13[dev], base, kD, kF) && encode_e2m1_x128(t2[dev], base, kF, kD);
            state[dev].store(ok ? 1 : 2, std::memory_order_release);
        }
    }
    if (state[dev].load(std::memory_order_acquire) != 1) return false;
    w13 = t13[dev];
    w2 = t2[dev];
    return true;
}

// 3-D uint8 map over `planes` planes of `rows` rows of row_bytes: boxes of
// 128 bytes x box_rows rows x all planes, 128-byte swizzle
bool encode_planes(CUtensorMap &m, const void *base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows,
                   int planes) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {row_bytes, rows, (cuuint64_t)planes}, strides[2] = {row_bytes, row_bytes * rows};
    const cuuint32_t box[3] = {128, box_rows, (cuuint32_t)planes}, es[3] = {1, 1, 1};
    return enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t up256(size_t n) { return (n + 255) & ~size_t(255); }

struct PxLayout {
    size_t xplanes, hplanes, xatoms, hatoms, units, n_units, pair_un, slot_of_pair, maps, total;
};
PxLayout px_layout(int n_tokens) {
    PxLayout L{};
    const size_t S = (size_t)n_tokens * kK, U = (size_t)prefill_mx_max_units(n_tokens);
    size_t o = 0;
    auto take = [&](size_t b) {
        const size_t at = o;
        o += up256(b);
        return at;
    };
    L.xplanes = take(kPPx * S * kD);
    L.hplanes = take(kPPh * S * kF);
    L.xatoms = take(U * (kD / kKS) * kBScaleBlock);
    L.hatoms = take(U * (kF / kKS) * kBScaleBlock);
    L.units = take(U * 3 * 4);
    L.n_units = take(4);
    L.pair_un = take(S * 4);
    L.slot_of_pair = take(S * 4);
    L.maps = take(expert_maps_bytes(kE));
    L.total = o;
    return L;
}

}  // namespace

cudaError_t set_wait_polls_px(uint32_t polls) { return set_wait_polls_here(polls); }

int prefill_mx_max_units(int n_tokens) {
    const int pairs = n_tokens * kK;
    return pairs / kUT + (pairs < kE ? pairs : kE);
}

size_t prefill_mx_scratch_bytes(int n_tokens) { return px_layout(n_tokens).total; }

cudaError_t launch_prefill_mx(const Ctx &c, const PrefillArgs &p) {
    const PxLayout L = px_layout(p.n_tokens);
    char *ws = static_cast<char *>(p.scratch);
    auto at = [&](size_t off) { return ws + off; };
    const size_t S = (size_t)p.n_tokens * kK;
    const int U = prefill_mx_max_units(p.n_tokens);
    int32_t *units = reinterpret_cast<int32_t *>(at(L.units));
    int32_t *n_units = reinterpret_cast<int32_t *>(at(L.n_units));
    int32_t *pair_un = reinterpret_cast<int32_t *>(at(L.pair_un));
    int32_t *slot_of_pair = reinterpret_cast<int32_t *>(at(L.slot_of_pair));
    uint8_t *xplanes = reinterpret_cast<uint8_t *>(at(L.xplanes));
    uint8_t *hplanes = reinterpret_cast<uint8_t *>(at(L.hplanes));
    uint8_t *maps = reinterpret_cast<uint8_t *>(at(L.maps));

    CUtensorMap w13, w2;
    PxBMaps xmap, hmap;
    if (!px_weight_templates(w13, w2)) return cudaErrorNotSupported;
    for (int i = 0; i < kBoxes; i++)
        if (!encode_planes(xmap.m[i], xplanes, kD, S, b_rows(i), kPPx) ||
            !encode_planes(hmap.m[i], hplanes, kF, S, b_rows(i), kPPh))
            return cudaErrorNotSupported;

    cudaError_t err = traced("prefill_prep", c.stream, [&] {
        k_px_units<<<1, 1024, 0, c.stream>>>(p.counts, p.offsets, units, n_units, slot_of_pair, (int)S, p.experts);
        const int map_ctas = (kE * kMapsPerExpert + kMapsPerCta - 1) / kMapsPerCta;
        k_px_slots<<<(unsigned)(U + map_ctas), 256, 0, c.stream>>>(units, n_units, p.perm, pair_un, slot_of_pair, U,
                                                                     maps, p.experts, w13, w2);
        const long long threads = (long long)p.n_tokens * (kD / 32);
        k_px_xprep<<<(unsigned)((threads + 255) / 256), 256, 0, c.stream>>>(
            p.x, p.n_tokens, slot_of_pair, pair_un, xplanes, reinterpret_cast<uint8_t *>(at(L.xatoms)), S, p.y);
        return cudaGetLastError();
    });
    if (err != cudaSuccess) return err;

    PxArgs a{};
    a.units = units;
    a.n_units = n_units;
    a.perm = p.perm;
    a.w = p.w;
    a.maps = maps;
    a.experts = p.experts;
    a.h_planes = hplanes;
    a.h_atoms = reinterpret_cast<uint8_t *>(at(L.hatoms));
    a.slots = S;
    a.y = p.y;
    a.status = c.status;
    a.b_atoms = reinterpret_cast<const uint8_t *>(at(L.xatoms));
    err = traced("prefill_gate_up", c.stream, [&] { return launch_px_t<0>(c, a, xmap, (long long)U * (kF / 128)); });
    if (err != cudaSuccess) return err;
    a.b_atoms = reinterpret_cast<const uint8_t *>(at(L.hatoms));
    return traced("prefill_down", c.stream, [&] { return launch_px_t<1>(c, a, hmap, (long long)U * (kD / 128)); });
}

}  // namespace k3mx
