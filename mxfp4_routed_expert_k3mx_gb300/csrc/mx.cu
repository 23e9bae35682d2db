// mx.cu - the decode path of the routed-expert layer on block-scaled
// 5th-generation tensor-core MMAs (tcgen05 kind::mxf4): the packed MXFP4
// weights and their ue8m0 group scales reach the tensor cores exactly as
// they are stored (Kimi K3 engine (c/kimi_k3.c), "Weights"), with no
// per-weight work in registers.
//
// Activations.  kind::mxf4 multiplies e2m1 by e2m1, so the activation
// vector v (x for gate/up, h for down) is split exactly into kPieces MXFP4
// vectors, v = p_0 + ... + p_7 + r.  Piece i takes, per 32-column block,
// the ue8m0 scale 2^e that maps the block's largest residual |value| into
// (3, 6] and the nearest e2m1 value of every residual; the new residual is
// formed exactly in fp32.  Each piece cuts the block's largest residual by
// at least 4, so |r| <= 4^-8 of the block's largest |v|.  Every piece is one
// N column of the MMA, D[:, n] = W p_n, and the epilogue adds a token's
// eight columns in fp32.
//
// Work.  item = (unit, 128-row tile); a unit is one expert and at most four
// of its pairs (so one fixed token set).  A CTA per SM takes a contiguous
// range of items.  Per item the K dimension streams in 256-column chunks:
//   warp 0      TMA: each matrix's 128 x 128-byte tile (128-byte swizzle,
//               K-major) through the expert's tensor maps (built on the
//               device by the kernel before, one per matrix and expert);
//               bulk copies of the unit's piece images (B operand and its
//               scales) once per unit
//   warp 1      scale loader: the tile's 128 x 8 scale bytes per matrix into
//               the 32-row scale-factor atoms tcgen05.cp reads; a group of
//               scale 255 ("contributes nothing") gets scale 0 and, once the
//               tile has landed, its 32 codes are zeroed, so it adds exactly 0
//   warp 2      TMEM owner; lane 0 copies the scale atoms to TMEM and issues
//               four K=64 MMAs per matrix and chunk, M=128, N = 8 per token
//   warps 3-6   epilogue (TMEM lane quarter = warp % 4): adds the pieces;
//               gate/up writes g, u, h = SiTU(g, u) as piece images for the
//               down pass; down writes the per-pair rows of y
// Two accumulator buffers let the epilogue of one item overlap the MMAs of
// the next.  Every wait is bounded; a timeout is reported on the device
// status word and every role leaves its loop.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "pieces.cuh"
#include "tmaps.cuh"
#include "tc.cuh"

namespace k3mx {
namespace {

constexpr int kChunk = kPieceChunk;           // K columns per stage
constexpr int kTileBytes = 128 * 128;          // 128 rows x 128 packed bytes
constexpr int kAtomBytes = 512;                // scale-factor atom: 32 lines x 16 B
constexpr int kThreads = 7 * 32;
constexpr int kProdWarp = 0, kSfWarp = 1, kMmaWarp = 2;   // warps 3-6: epilogue
constexpr int kTmemCols = 512;
constexpr int kMaxGrid = 256;
constexpr int kSmemLimit = 227 * 1024;

template <int PH> struct MxCfg;
template <> struct MxCfg<0> { static constexpr int NMAT = 2, K = kD, M = kF; };   // gate/up
template <> struct MxCfg<1> { static constexpr int NMAT = 1, K = kF, M = kD; };   // down

template <int PH, int NTOK> struct MxShape {
    static constexpr int NMAT = MxCfg<PH>::NMAT, K = MxCfg<PH>::K, M = MxCfg<PH>::M;
    static constexpr int KC = K / kChunk, MT = M / 128, G = K / 32;
    static constexpr int NCOL = 8 * NTOK;                          // D columns per matrix
    static constexpr int STAGE = NMAT * (kTileBytes + 2 * kAtomBytes);
    static constexpr int TOKB = img_b(K), TOKS = img_s(K);
    static constexpr int SRAW = NMAT * 128 * G;                    // one tile's scale rows
    // one token: two scale-row buffers, so the next part's rows load during
    // the whole current part (a copy issued at the part boundary waits
    // behind the weight stream); several tokens: one (shared memory)
    static constexpr int SBUF = NTOK == 1 ? 2 : 1;
    // down with one token per unit: two piece-image buffers, so the next
    // pair's h images load while the current unit's MMAs run (gate/up keeps
    // the token's x images for every unit)
    static constexpr int BBUF = PH == 1 && NTOK == 1 ? 2 : 1;
    static constexpr int FIXED = 1024 + BBUF * NTOK * (TOKB + TOKS) + SBUF * SRAW;  // header, images, scales
    static constexpr int S_FIT = (kSmemLimit - 1024 - FIXED) / STAGE;
    static constexpr int S = S_FIT > 10 ? 10 : S_FIT;
    static constexpr int SMEM = 1024 + FIXED + S * STAGE;          // + 1024 alignment slack
    // TMEM columns: accumulators [2][NMAT][NCOL], A scales [S][NMAT][2 atoms][4],
    // B scales [K/128 atoms][4]
    static constexpr int SFA_COL = 2 * NMAT * NCOL;
    static constexpr int SFB_COL = SFA_COL + S * NMAT * 8;
    static_assert(S >= 3, "pipeline too shallow");
    static_assert(SFB_COL + (K / 128) * 4 <= kTmemCols, "TMEM budget");
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
};

struct MxArgs {
    const k3mx_expert *experts;     // device table [896], or nullptr: `one`, pair 0
    k3mx_expert one;
    const int32_t *units, *n_units, *perm;
    const uint8_t *img_in;          // gate/up: per-token x images; down: per-pair h images
    uint8_t *img_out;               // gate/up: per-pair h images
    float *gu;                      // gate/up: [pair][2][F]
    float *out;                     // down: [pair][D]
    const uint8_t *maps;            // per-expert weight tensor maps [expert][w1, w3, w2]
    float *partials;                // fused pass: stream-K hand-over sums [segment][grid][2][128], or null
    int *status;
    // fused single-token pass only
    const float *w;                 // routing weights [16] of the token (null: one expert, no sum)
    float *y;                       // [D]: the weighted sum (or the one expert's output)
    int *sync;                      // hand-over flags [segment][grid], h blocks done per pair [16],
                                    // y tiles done [28]; zeroed by the step's first kernel
};

struct Hdr {
    // full: the stage's scale atoms (32 scale-loader lanes); tfull: its weight
    // tiles (the producer's expect_tx and the copies' bytes)
    uint64_t full[10], tfull[10], empty[10], accf[2], acce[2], bfull[2], bempty[2], sfull[2], done;
    uint64_t table;                      // the single-token pass's staged expert table
    uint32_t tmem;
    int abort;
};

// x of every token -> its piece image; one warp per 32-column block
// x of every token -> its piece image (one warp per 32-column block); the
// CTAs after those build the weight tensor maps of the expert table (or of
// the single expert `one`); CTA 0 zeroes the stream-K flags
__global__ void __launch_bounds__(256) k_mx_ximg(const void *__restrict__ x, int bf16, int n_tokens,
                                                 uint8_t *__restrict__ img, int *flags, int n_flags,
                                                 int piece_ctas, uint8_t *maps, int n_map_experts,
                                                 const k3mx_expert *table, k3mx_expert one,
                                                 const __grid_constant__ CUtensorMap w13,
                                                 const __grid_constant__ CUtensorMap w2) {
    if (flags != nullptr && blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_flags; i += blockDim.x) flags[i] = 0;
    if ((int)blockIdx.x < piece_ctas)
        ximg_block(x, bf16, n_tokens, img, blockIdx.x * 8 + (threadIdx.x >> 5));
    else
        build_maps_cta(maps, n_map_experts, table, one, w13, w2, blockIdx.x - piece_ctas);
}

// ------------------------------------------------------------ work units --

struct Unit {
    int e, p0, p1;          // expert, pair slots [p0, p1) of perm
    k3mx_expert ex;
    bool ok;                // every pointer 16-byte aligned
};

__device__ __forceinline__ Unit unit_at(const MxArgs &a, int u) {
    Unit r;
    if (a.experts == nullptr) {
        r.e = 0;
        r.p0 = 0;
        r.p1 = 1;
        r.ex = a.one;
    } else {
        r.e = __ldg(a.units + 3 * u);
        r.p0 = __ldg(a.units + 3 * u + 1);
        r.p1 = __ldg(a.units + 3 * u + 2);
        const uint4 *q = reinterpret_cast<const uint4 *>(a.experts + r.e);
        const uint4 v0 = __ldg(q), v1 = __ldg(q + 1), v2 = __ldg(q + 2);
        r.ex.w1 = reinterpret_cast<const uint8_t *>((uint64_t)v0.y << 32 | v0.x);
        r.ex.s1 = reinterpret_cast<const uint8_t *>((uint64_t)v0.w << 32 | v0.z);
        r.ex.w3 = reinterpret_cast<const uint8_t *>((uint64_t)v1.y << 32 | v1.x);
        r.ex.s3 = reinterpret_cast<const uint8_t *>((uint64_t)v1.w << 32 | v1.z);
        r.ex.w2 = reinterpret_cast<const uint8_t *>((uint64_t)v2.y << 32 | v2.x);
        r.ex.s2 = reinterpret_cast<const uint8_t *>((uint64_t)v2.w << 32 | v2.z);
    }
    const uint64_t orp = reinterpret_cast<uint64_t>(r.ex.w1) | reinterpret_cast<uint64_t>(r.ex.s1) |
                         reinterpret_cast<uint64_t>(r.ex.w3) | reinterpret_cast<uint64_t>(r.ex.s3) |
                         reinterpret_cast<uint64_t>(r.ex.w2) | reinterpret_cast<uint64_t>(r.ex.s2);
    r.ok = (orp & 15u) == 0;
    return r;
}
__device__ __forceinline__ int pair_at(const MxArgs &a, int slot) {
    return a.experts == nullptr ? 0 : __ldg(a.perm + slot);
}

template <int PH, int NTOK>
__global__ void __launch_bounds__(kThreads, 1)
    k_mx(const MxArgs a) {
    using Sh = MxShape<PH, NTOK>;
    constexpr int NMAT = Sh::NMAT, KC = Sh::KC, MT = Sh::MT, G = Sh::G, S = Sh::S, NCOL = Sh::NCOL;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Hdr *hd = reinterpret_cast<Hdr *>(smem);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t st0 = sbase + 1024;                            // stages
    constexpr int BB = Sh::BBUF;
    const uint32_t bimg0 = st0 + S * Sh::STAGE;                   // unit's B images [BBUF][NTOK][TOKB]
    const uint32_t simg0 = bimg0 + BB * NTOK * Sh::TOKB;          // unit's scale images [BBUF][NTOK][TOKS]
    const uint32_t sraw0 = simg0 + BB * NTOK * Sh::TOKS;          // tile's scale rows [SBUF][NMAT][128][G]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t full0 = smem_addr(hd->full), empty0 = smem_addr(hd->empty);
    const uint32_t tfull0 = smem_addr(hd->tfull);
    const uint32_t accf0 = smem_addr(hd->accf), acce0 = smem_addr(hd->acce);
    const uint32_t bfull0 = smem_addr(hd->bfull), bempty0 = smem_addr(hd->bempty);
    const uint32_t sfull0 = smem_addr(hd->sfull);
    const uint32_t done = smem_addr(&hd->done);

    if (tid == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(full0 + 8 * i, 32);          // the scale loader's lanes
            mbar_init(tfull0 + 8 * i, 1);          // the producer's expect_tx
            mbar_init(empty0 + 8 * i, 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(accf0 + 8 * i, 1);
            mbar_init(acce0 + 8 * i, 128);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(bfull0 + 8 * i, 1);
            mbar_init(bempty0 + 8 * i, 1);
        }
        mbar_init(sfull0, 1);
        mbar_init(sfull0 + 8, 1);
        mbar_init(done, 1);
        hd->abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(smem_addr(&hd->tmem), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = hd->tmem;
    volatile int *abort_flag = &hd->abort;
    // Launched as a programmatic dependent: the prologue above overlapped
    // the previous kernel.  gate/up reads the work units, so it waits here;
    // down streams weights at once and waits (producer) only before the h
    // pieces.  Either lets the next kernel launch after this point.
    if (PH == 0) pdl_wait();
    pdl_launch_dependents();

    const int n_units = a.experts == nullptr ? 1 : __ldg(a.n_units);
    // This CTA's work is a contiguous range of whole items (item-major, KC
    // chunks per item).
    const long long items = (long long)n_units * MT;
    const long long q0 = items * blockIdx.x / gridDim.x * KC;
    const long long q1 = items * (blockIdx.x + 1) / gridDim.x * KC;
    auto fail = [&](int detail) {
        report_status(a.status, kStatusWaitTimeout, detail);
        *abort_flag = 1;
    };
    // the token set of a unit: the token (gate/up, one token per unit), else
    // the unit's slot range
    auto unit_key = [&](const Unit &u) -> long long {
        if (NTOK == 1 && PH == 0) return a.experts == nullptr ? 0 : __ldg(a.perm + u.p0) / kK;
        return (long long)u.p0 << 32 | (uint32_t)u.p1;
    };
    // parts: the chunks [lo, hi) of one item inside [q, q1); `next` skips
    // items of units with misaligned pointers (every role skips the same)
    struct Part {
        long long item;
        int lo, hi;
        Unit u;
    };
    auto next_part = [&](long long &q, Part &p) -> bool {
        while (q < q1) {
            p.item = q / KC;
            p.lo = (int)(q % KC);
            p.hi = (int)min((long long)KC, p.lo + (q1 - q));
            q += p.hi - p.lo;
            p.u = unit_at(a, (int)(p.item / MT));
            if (p.u.ok) return true;
            if (warp == kProdWarp && lane == 0 && p.lo == 0 && p.item % MT == 0)
                report_status(a.status, kStatusBadPointer, p.u.e);
        }
        return false;
    };

    if (warp == kProdWarp) {
        // ---------------------------------------------------- TMA producer --
        const uint64_t pol = l2_evict_first_policy();     // weights: read once
        const uint64_t pol_img = l2_evict_last_policy();   // piece images: read by every CTA
        int cur_e = -1;
        const uint8_t *map0 = nullptr, *map1 = nullptr;
        long long cur_key = -1, q = q0;
        uint32_t su = 0, bl = 0;
        bool waited = PH == 0;
        Part p;
        while (!*abort_flag && next_part(q, p)) {
            const Unit &u = p.u;
            const int mt = (int)(p.item % MT);
            if (u.e != cur_e) {
                const uint8_t *em = a.maps + (size_t)u.e * kMapsPerExpert * kMapBytes;
                map0 = em + (PH == 0 ? 0 : 2) * kMapBytes;
                map1 = em + 1 * kMapBytes;
                acquire_map(map0);
                if (NMAT == 2) acquire_map(map1);
                cur_e = u.e;
            }
            // the first weight tile goes out before the piece-image lookups
            auto issue_stage = [&](int c) -> bool {
                const int s = su % S;
                if (!mbar_wait(empty0 + 8 * s, ((su / S) & 1) ^ 1)) {
                    if (lane == 0) fail(2);
                    return false;
                }
                if (lane == 0) {
                    const uint32_t dst = st0 + s * Sh::STAGE;
                    mbar_arrive_expect_tx(tfull0 + 8 * s, NMAT * kTileBytes);
                    tma_2d(dst, map0, c * 128, mt * 128, tfull0 + 8 * s, pol);
                    if (NMAT == 2) tma_2d(dst + kTileBytes, map1, c * 128, mt * 128, tfull0 + 8 * s, pol);
                }
                __syncwarp();
                su++;
                return true;
            };
            if (!issue_stage(p.lo)) break;
            const long long key = unit_key(u);
            if (key != cur_key) {
                if (!waited) {
                    pdl_wait();
                    waited = true;
                }
                // B buffer bl % BB: wait until the MMAs of its previous fill are done
                const int bb = bl % BB;
                if (bl >= (uint32_t)BB && !mbar_wait(bempty0 + 8 * bb, (bl / BB - 1) & 1)) {
                    if (lane == 0) fail(1);
                    break;
                }
                const int ntok = u.p1 - u.p0;
                if (lane == 0) {
                    const uint32_t bfull = bfull0 + 8 * bb;
                    mbar_arrive_expect_tx(bfull, (uint32_t)(ntok * (Sh::TOKB + Sh::TOKS)));
                    for (int j = 0; j < ntok; j++) {
                        const int pair = pair_at(a, u.p0 + j);
                        const int src = PH == 0 ? pair / kK : pair;
                        const uint8_t *img = a.img_in + (size_t)src * img_bytes(Sh::K);
                        bulk_g2s(bimg0 + (bb * NTOK + j) * Sh::TOKB, img, Sh::TOKB, bfull, pol_img);
                        bulk_g2s(simg0 + (bb * NTOK + j) * Sh::TOKS, img + Sh::TOKB, Sh::TOKS, bfull, pol_img);
                    }
                }
                bl++;
                cur_key = key;
            }
            bool ok = true;
            for (int c = p.lo + 1; c < p.hi && ok; c++) ok = issue_stage(c);
            if (!ok) break;
        }
        // copies still in flight (after a wait gave up) land before the CTA leaves
        if (lane == 0 && (!drain_ring(tfull0, S, su) || !drain_ring(bfull0, BB, bl)))
            report_status(a.status, kStatusWaitTimeout, 13);
    } else if (warp == kSfWarp) {
        // -------------------------------------------------- scale loader --
        // A tile's scale rows (128 x G bytes per matrix, contiguous in
        // memory) arrive in one bulk copy per part into one of SBUF buffers:
        // with two, the next part's copy is issued when the current part
        // starts; with one, after its last chunk is transposed.  Lane l turns
        // rows l, l + 32, l + 64, l + 96 into the l-th line of each chunk's
        // two atoms.
        constexpr int SB = Sh::SBUF;
        const uint64_t pol = l2_evict_first_policy();
        auto rows_of = [&](const Part &p, int m) {
            const size_t off = (size_t)(p.item % MT) * 128 * G;
            return (m == 0 ? (PH == 0 ? p.u.ex.s1 : p.u.ex.s2) : p.u.ex.s3) + off;
        };
        uint32_t ni = 0;                   // parts whose scale rows were issued
        auto issue = [&](const Part &p, int buf) {
            // every lane's earlier reads of this buffer are done (their
            // values were stored) before the copy may overwrite it
            ni++;
            __syncwarp();
            fence_async_smem();
            if (lane == 0) {
                mbar_arrive_expect_tx(sfull0 + 8 * buf, Sh::SRAW);
#pragma unroll
                for (int m = 0; m < NMAT; m++)
                    bulk_g2s(sraw0 + buf * Sh::SRAW + m * 128 * G, rows_of(p, m), 128 * G, sfull0 + 8 * buf, pol);
            }
        };
        uint32_t su = 0, np = 0;           // stage uses, parts taken
        long long q = q0;
        Part cur, nxt;
        bool have = next_part(q, cur);
        if (have) issue(cur, 0);
        while (have && !*abort_flag) {
            const int buf = np % SB;
            long long qn = q;
            const bool more = next_part(qn, nxt);
            if (more && SB == 2) issue(nxt, (np + 1) % SB);
            if (!mbar_wait(sfull0 + 8 * buf, (np / SB) & 1)) {
                if (lane == 0) fail(3);
                break;
            }
            const uint32_t sraw = sraw0 + buf * Sh::SRAW;
            bool ok = true;
            for (int c = cur.lo; c < cur.hi; c++, su++) {
                const int s = su % S;
                if (!mbar_wait(empty0 + 8 * s, ((su / S) & 1) ^ 1)) {
                    if (lane == 0) fail(9);
                    ok = false;
                    break;
                }
                uint2 w[NMAT][4];
#pragma unroll
                for (int m = 0; m < NMAT; m++)
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                                     : "=r"(w[m][j].x), "=r"(w[m][j].y)
                                     : "r"(sraw + m * 128 * G + (lane + 32 * j) * G + c * 8));
                const uint32_t stg = st0 + s * Sh::STAGE, at0 = stg + NMAT * kTileBytes;
                // groups with scale 255 contribute nothing: once the stage's
                // weight tiles landed, their codes are zeroed (rare; most
                // stages skip this)
                uint32_t nan = 0;
#pragma unroll
                for (int m = 0; m < NMAT; m++)
#pragma unroll
                    for (int j = 0; j < 4; j++) nan |= nan_scale_mask(w[m][j].x) | nan_scale_mask(w[m][j].y);
                if (__any_sync(0xffffffffu, nan != 0)) {
                    if (!mbar_wait(tfull0 + 8 * s, (su / S) & 1)) {
                        if (lane == 0) fail(12);
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int m = 0; m < NMAT; m++)
#pragma unroll
                        for (int j = 0; j < 4; j++) zero_nan_groups_sw128(stg + m * kTileBytes, lane + 32 * j, w[m][j]);
                }
#pragma unroll
                for (int m = 0; m < NMAT; m++) {
                    sts128(at0 + (2 * m) * kAtomBytes + 16 * lane, drop_nan_scales(w[m][0].x),
                           drop_nan_scales(w[m][1].x), drop_nan_scales(w[m][2].x), drop_nan_scales(w[m][3].x));
                    sts128(at0 + (2 * m + 1) * kAtomBytes + 16 * lane, drop_nan_scales(w[m][0].y),
                           drop_nan_scales(w[m][1].y), drop_nan_scales(w[m][2].y), drop_nan_scales(w[m][3].y));
                }
                fence_async_smem();
                if (SB == 1 && c == cur.hi - 1 && more) issue(nxt, 0);
                mbar_arrive(full0 + 8 * s);
            }
            if (!ok) break;
            np++;
            q = qn;
            cur = nxt;
            have = more;
        }
        if (lane == 0 && !drain_ring(sfull0, SB, ni)) report_status(a.status, kStatusWaitTimeout, 14);
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------- MMA issuer --
        if (lane == 0) {
            uint32_t su = 0, bu = 0, it = 0, bcur = 0;
            long long cur_key = -1, q = q0;
            bool run = true;
            Part p;
            while (run && !*abort_flag && next_part(q, p)) {
                const Unit &u = p.u;
                const long long key = unit_key(u);
                const int ntok = u.p1 - u.p0;
                const int n = ntok <= 1 ? 8 : (ntok == 2 ? 16 : 32);
                if (key != cur_key) {
                    bcur = bu % BB;
                    if (!mbar_wait(bfull0 + 8 * bcur, (bu / BB) & 1)) {
                        fail(4);
                        break;
                    }
                    bu++;
                    tc_fence_after();
                    // one token: the atom's four 8-line groups all read its lines
                    // (rows 8-31 are never used with N = 8)
                    const uint32_t simg = simg0 + bcur * NTOK * Sh::TOKS;
                    for (int at = 0; at < Sh::K / 128; at++)
                        tmem_cp_atom(tmem + Sh::SFB_COL + 4 * at,
                                     desc_atom(simg + at * 128, NTOK == 1 ? 0 : Sh::TOKS));
                    cur_key = key;
                }
                const int b = it & 1;
                if (!mbar_wait(acce0 + 8 * b, ((it >> 1) & 1) ^ 1)) {
                    fail(5);
                    break;
                }
                tc_fence_after();
                for (int c = p.lo; c < p.hi; c++, su++) {
                    const int s = su % S;
                    if (!mbar_wait(tfull0 + 8 * s, (su / S) & 1) || !mbar_wait(full0 + 8 * s, (su / S) & 1)) {
                        fail(6);
                        run = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t stg = st0 + s * Sh::STAGE;
                    const uint32_t sfa = tmem + Sh::SFA_COL + s * NMAT * 8;
#pragma unroll
                    for (int m = 0; m < NMAT; m++)
#pragma unroll
                        for (int at = 0; at < 2; at++)
                            tmem_cp_atom(sfa + m * 8 + at * 4,
                                         desc_atom(stg + NMAT * kTileBytes + (2 * m + at) * kAtomBytes, 128));
#pragma unroll
                    for (int m = 0; m < NMAT; m++)
#pragma unroll
                        for (int ks = 0; ks < 4; ks++) {
                            const int id = 2 * (ks & 1);
                            mma_mxf4(tmem + (b * NMAT + m) * NCOL, desc_sw128(stg + m * kTileBytes + 32 * ks, 1024),
                                     desc_sw128(bimg0 + bcur * NTOK * Sh::TOKB + c * 1024 + 32 * ks, Sh::TOKB),
                                     idesc_mxf4(n, id),
                                     sfa + m * 8 + (ks >> 1) * 4, tmem + Sh::SFB_COL + (c * 2 + (ks >> 1)) * 4,
                                     (c != p.lo || ks != 0) ? 1u : 0u);
                        }
                    umma_commit(empty0 + 8 * s);
                }
                if (!run) break;
                umma_commit(accf0 + 8 * b);
                it++;
                // release the unit's B images once its last MMA is done
                long long qn = q;
                Part nx;
                if (!next_part(qn, nx) || unit_key(nx.u) != key) umma_commit(bempty0 + 8 * bcur);
            }
            umma_commit(done);
        }
    } else {
        // ------------------------------------------------------- epilogue --
        const int q4 = warp & 3;
        const int row_in_tile = 32 * q4 + lane;
        uint32_t it = 0;
        long long q = q0;
        Part p;
        while (!*abort_flag && next_part(q, p)) {
            const Unit &u = p.u;
            const int mt = (int)(p.item % MT);
            const int b = it & 1;
            if (!mbar_wait(accf0 + 8 * b, (it >> 1) & 1)) {
                if (lane == 0) fail(7);
                break;
            }
            tc_fence_after();
            uint32_t v[NMAT][NCOL];
#pragma unroll
            for (int m = 0; m < NMAT; m++)
                tmem_ld<NCOL>(tmem + ((uint32_t)(32 * q4) << 16) + (b * NMAT + m) * NCOL, v[m]);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(acce0 + 8 * b);
            it++;
            const int row = mt * 128 + row_in_tile;
            const int ntok = u.p1 - u.p0;
#pragma unroll
            for (int j = 0; j < NTOK; j++) {
                if (j < ntok) {
                    float acc[NMAT];
#pragma unroll
                    for (int m = 0; m < NMAT; m++) {
                        acc[m] = 0.f;
#pragma unroll
                        for (int pc = 0; pc < kPieces; pc++) acc[m] += __uint_as_float(v[m][8 * j + pc]);
                    }
                    const int pair = pair_at(a, u.p0 + j);
                    if (PH == 0) {
                        float *gu = a.gu + (size_t)pair * 2 * kF;
                        gu[row] = acc[0];
                        gu[kF + row] = acc[NMAT - 1];
                        const float h = situ_glu(acc[0], acc[NMAT - 1]);
                        uint8_t *ib = a.img_out + (size_t)pair * img_bytes(kF);
                        store_pieces(h, ib, ib + img_b(kF), mt * 4 + q4);
                    } else {
                        a.out[(size_t)pair * kD + row] = acc[0];
                    }
                }
            }
        }
    }

    __syncthreads();
    if (warp == kMmaWarp) {
        // no MMA may still be running when TMEM is released
        if (!mbar_wait_drain(done, 0) && lane == 0) report_status(a.status, kStatusWaitTimeout, 8);
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}


// ----------------------------------------------- fused single-token pass --
//
// One token (a batch of one, or one expert): gate/up, down and the weighted
// sum of the token's expert outputs in one persistent launch, so no pass
// waits for another to drain and the weight stream does not pause between
// them.  Stages are 32 KB: a gate/up stage is one 256-column chunk of W1
// and of W3, a down stage two consecutive 256-column chunks of W2.  The
// sequence of stages (every gate/up item, then every down item, in four
// segments) is cut in ranges over the CTAs (stream-K); an item split between two CTAs
// is finished by the one holding its first stage, which adds the other's
// summed pieces in a fixed order.  A down item starts its MMAs once every
// gate/up item of its pair has written its block of h (a per-pair count);
// the last down item of a 128-row tile of y (a per-tile count) adds the
// 16 pairs' rows with their routing weights in slot order.

namespace f1 {
constexpr int KCG = kD / kChunk;                 // 14 gate/up stages per item
constexpr int KCD = kF / (2 * kChunk);           // 6 down stages per item
constexpr int MTG = kF / 128, MTD = kD / 128;    // 24 gate/up, 28 down items per unit
constexpr int GG = kD / 32, GD = kF / 32;        // scale bytes per weight row: 112, 96
constexpr int STAGE = 2 * kTileBytes + 4 * kAtomBytes;
constexpr int XB = img_b(kD), XS = img_s(kD);    // the token's x pieces
constexpr int HB = img_b(kF), HS = img_s(kF);    // a pair's h pieces
constexpr int SOFF = 2 * HB;                     // scale parts after the two h B parts
constexpr int BREG = 2 * HB + 2 * HS;            // x's image overlaps both h buffers
constexpr int SRAW = 2 * 128 * GG;               // a gate/up tile's scale rows (the larger)
constexpr int FIXED = 1024 + BREG + 2 * SRAW;
constexpr int S = (kSmemLimit - 1024 - FIXED) / STAGE;
constexpr int SMEM = 1024 + FIXED + S * STAGE;
constexpr int SFA_COL = 2 * 2 * 8;               // accumulators [2][2][8] first
constexpr int SFB_COL = SFA_COL + S * 16;
constexpr int TMEM_COLS = 256;
constexpr int NSEG = 4;                          // work segments: gate/up A, gate/up B, down A, down B
constexpr int PARTIAL = 2 * 128;                 // floats per hand-over slot: the summed pieces
constexpr int SYNC_HDONE = NSEG * kMaxGrid, SYNC_TILE = SYNC_HDONE + kK;   // after the segments' flags
constexpr int SYNC_INTS = SYNC_TILE + 64;
static_assert(MTD <= 64, "tile counts");
constexpr int MAX_UNITS = kK;                    // one token: at most 16 units
static_assert(XB <= 2 * HB && XS <= 2 * HS, "x image must fit the h buffers");
static_assert(S >= 3 && S <= 10, "pipeline depth");
static_assert(SFB_COL + (kD / 128) * 4 <= TMEM_COLS, "TMEM budget");
static_assert(SMEM <= kSmemLimit, "shared memory budget");
static_assert(kE * (int)sizeof(k3mx_expert) <= S * STAGE, "the expert table is staged in the ring");
}  // namespace f1

__global__ void __launch_bounds__(kThreads, 1) k_mx1(const MxArgs a) {
    using namespace f1;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Hdr *hd = reinterpret_cast<Hdr *>(smem);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t st0 = sbase + 1024;
    const uint32_t breg = st0 + S * STAGE;
    const uint32_t sraw0 = breg + BREG;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t full0 = smem_addr(hd->full), empty0 = smem_addr(hd->empty);
    const uint32_t tfull0 = smem_addr(hd->tfull);
    const uint32_t accf0 = smem_addr(hd->accf), acce0 = smem_addr(hd->acce);
    const uint32_t bfull0 = smem_addr(hd->bfull), bempty0 = smem_addr(hd->bempty);
    const uint32_t sfull0 = smem_addr(hd->sfull), done = smem_addr(&hd->done);
    const uint32_t tbar = smem_addr(&hd->table);
    if (tid == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(full0 + 8 * i, 32);
            mbar_init(tfull0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        mbar_init(tbar, 1);
        for (int i = 0; i < 2; i++) {
            mbar_init(accf0 + 8 * i, 1);
            mbar_init(acce0 + 8 * i, 128);
            mbar_init(bfull0 + 8 * i, 1);
            mbar_init(bempty0 + 8 * i, 1);
            mbar_init(sfull0 + 8 * i, 1);
        }
        mbar_init(done, 1);
        hd->abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(smem_addr(&hd->tmem), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = hd->tmem;
    volatile int *abort_flag = &hd->abort;

    // Four work segments: the gate/up stages of the first half of the
    // units (A), of the second half (B), then the down stages of A and of B,
    // each cut in equal stage ranges over the CTAs (stream-K) when there is
    // enough work, else in whole items.  Every CTA runs its share of each
    // segment in that order, so the h of A is complete while the CTAs
    // stream gate/up B, and the down parts of A start without waiting; by
    // the time they reach down B, B's h is complete too.
    struct Sched {
        int gu, r0[NSEG], r1[NSEG], cum[NSEG + 1];
        bool sk;
    };
    auto plan = [&](int nu) {
        Sched sc;
        const int GU = nu * MTG * KCG, GDn = nu * MTD * KCD;
        const int G = gridDim.x, B = blockIdx.x;
        sc.gu = GU;
        const int nA = (nu + 1) / 2;
        const int GA = nA * MTG * KCG, DA = nA * MTD * KCD;
        sc.sk = a.partials != nullptr && GA >= G * (KCG + 1) && DA >= G * (KCD + 1);
        const int st[NSEG] = {0, GA, GU, GU + DA}, len[NSEG] = {GA, GU - GA, DA, GDn - DA};
        const int kc[NSEG] = {KCG, KCG, KCD, KCD};
        // stream-K cuts: CTA B's stages before segment i's range, taken from
        // cuts of the running totals (GA, GU, GU + DA, all stages) so that
        // the CTAs' totals over the four segments differ by at most one
        // stage (cutting each segment alone, a CTA could draw the shorter
        // share in all four)
        auto before = [&](int i, int b) -> int {
            const long long cA = (long long)GA * b / G, cU = (long long)GU * b / G, cD = (long long)DA * b / G;
            const long long cT = (long long)(GU + GDn) * b / G;
            return (int)(i == 0 ? cA : i == 1 ? cU - cA : i == 2 ? cD : cT - cU - cD);
        };
        sc.cum[0] = 0;
#pragma unroll
        for (int i = 0; i < NSEG; i++) {
            if (sc.sk) {
                sc.r0[i] = st[i] + before(i, B);
                sc.r1[i] = st[i] + before(i, B + 1);
            } else {
                const int items = len[i] / kc[i];
                sc.r0[i] = st[i] + items * B / G * kc[i];
                sc.r1[i] = st[i] + items * (B + 1) / G * kc[i];
            }
            sc.cum[i + 1] = sc.cum[i] + (sc.r1[i] - sc.r0[i]);
        }
        return sc;
    };
    // A token keeps all 16 experts unless top-p drops some: the partition
    // for 16 units is made while the routing kernel runs.  The expert table
    // is an input of the call that no kernel of the step writes, so it is
    // staged now in the stage ring (unused until the first weight copy),
    // and a unit's pointers become a shared-memory lookup.
    // One bulk copy, waited for only where the producer first looks a unit
    // up: a CTA that starts late (its SM still held by blocks of the
    // kernel before) does not spend its start on the copy.
    Sched sc = plan(MAX_UNITS);
    const uint2 *tab = reinterpret_cast<const uint2 *>(smem + 1024);
    constexpr uint32_t kTableBytes = kE * (uint32_t)sizeof(k3mx_expert);
    static_assert(kTableBytes % 16 == 0, "bulk copy size");
    if (a.experts != nullptr && tid == 0) {
        mbar_arrive_expect_tx(tbar, kTableBytes);
        bulk_g2s(st0, a.experts, kTableBytes, tbar, l2_evict_last_policy());   // 16-byte aligned (checked)
    }
    pdl_wait();
    pdl_launch_dependents();
    __syncthreads();

    // the token's work units (at most 16): the unit count, the unit list
    // and perm in one round of loads (all 16 entries lie in the workspace)
    __shared__ Unit s_unit[MAX_UNITS];
    __shared__ int s_pair[MAX_UNITS];
    __shared__ int s_nunits;
    if (warp == kProdWarp) {
        if (a.experts == nullptr) {
            if (lane == 0) {
                s_unit[0] = unit_at(a, 0);
                s_pair[0] = 0;
                s_nunits = 1;
            }
        } else {
            const int n_raw = __ldg(a.n_units);
            int e = 0, p0 = 0, p1 = 0, pr = 0;
            if (lane < MAX_UNITS) {
                e = __ldg(a.units + 3 * lane);
                p0 = __ldg(a.units + 3 * lane + 1);
                p1 = __ldg(a.units + 3 * lane + 2);
                pr = __ldg(a.perm + lane);
            }
            if (!mbar_wait(tbar, 0)) {
                if (lane == 0) report_status(a.status, kStatusWaitTimeout, 15);
                *abort_flag = 1;
            }
            const int nu = min(max(n_raw, 0), MAX_UNITS);
            const int pair = __shfl_sync(0xffffffffu, pr, p0 & (MAX_UNITS - 1));
            if (lane < nu) {
                Unit u;
                u.e = e;
                u.p0 = p0;
                u.p1 = p1;
                const bool in = (unsigned)e < (unsigned)kE;
                const uint2 *t = tab + 6 * (in ? e : 0);
                uint64_t w[6], orp = 0;
#pragma unroll
                for (int i = 0; i < 6; i++) {
                    w[i] = (uint64_t)t[i].y << 32 | t[i].x;
                    orp |= w[i];
                }
                u.ex.w1 = reinterpret_cast<const uint8_t *>(w[0]);
                u.ex.s1 = reinterpret_cast<const uint8_t *>(w[1]);
                u.ex.w3 = reinterpret_cast<const uint8_t *>(w[2]);
                u.ex.s3 = reinterpret_cast<const uint8_t *>(w[3]);
                u.ex.w2 = reinterpret_cast<const uint8_t *>(w[4]);
                u.ex.s2 = reinterpret_cast<const uint8_t *>(w[5]);
                u.ok = in && (orp & 15u) == 0;
                s_unit[lane] = u;
                s_pair[lane] = pair;
            }
            if (lane == 0) s_nunits = nu;
        }
    }
    // the table reads before the ring's first asynchronous writes
    fence_async_smem();
    __syncthreads();
    const int n_units = s_nunits;
    if (n_units != MAX_UNITS) sc = plan(n_units);
    const int nseg = NSEG;
    auto fail = [&](int detail) {
        report_status(a.status, kStatusWaitTimeout, detail);
        *abort_flag = 1;
    };
    struct Part {
        int ph;          // 0 gate/up, 1 down
        int seg;         // work segment
        int item;        // within the phase
        int lo, hi;      // stages of the item
        int mt;          // 128-row tile
        int pair;        // the unit's pair
        Unit u;
    };
    // parts in order: `t` walks this CTA's stages, segment after segment
    auto next_part = [&](int &t, Part &p) -> bool {
        for (;;) {
            int sg = 0;
#pragma unroll
            for (int i = 1; i < NSEG; i++) sg += (i < nseg && t >= sc.cum[i]) ? 1 : 0;
            if (t >= sc.cum[nseg]) return false;
            int q0s = sc.r0[0], q1s = sc.r1[0], c0 = sc.cum[0];
#pragma unroll
            for (int i = 1; i < NSEG; i++)
                if (sg == i) q0s = sc.r0[i], q1s = sc.r1[i], c0 = sc.cum[i];
            const int q = q0s + (t - c0);
            const bool up = q < sc.gu;
            const int kc = up ? KCG : KCD;
            const int r = q - (up ? 0 : sc.gu);
            p.ph = up ? 0 : 1;
            p.seg = sg;
            p.item = r / kc;
            p.lo = r % kc;
            p.hi = min(kc, p.lo + (q1s - q));
            t += p.hi - p.lo;
            const int mts = up ? MTG : MTD;
            p.mt = p.item % mts;
            const int ui = p.item / mts;
            p.u = s_unit[ui];
            p.pair = s_pair[ui];
            if (p.u.ok) return true;
            if (warp == kProdWarp && lane == 0 && p.lo == 0 && p.mt == 0)
                report_status(a.status, kStatusBadPointer, p.u.e);
        }
    };
    // B epoch of a part: the token's x for gate/up, the pair's h for down
    auto b_key = [&](const Part &p) -> long long {
        return p.ph == 0 ? -1 : (long long)p.pair;
    };
    // B buffer of epoch n: epoch 0 is x (overlapping both h buffers)
    auto b_off = [&](uint32_t n) { return (uint32_t)((n & 1) * HB); };
    auto s_off = [&](uint32_t n) { return (uint32_t)(SOFF + (n & 1) * HS); };

    if (warp == kProdWarp) {
        // ---------------------------------------------------- TMA producer --
        const uint64_t pol = l2_evict_first_policy();
        const uint64_t pol_img = l2_evict_last_policy();
        int cur_e = -1, cur_ph = -1;
        const uint8_t *map0 = nullptr, *map1 = nullptr;
        long long cur_key = -2;
        int q = 0;
        uint32_t su = 0, bl = 0;
        bool x_first = false;            // epoch 0 held x (which overlaps both h buffers)
        Part p;
        while (!*abort_flag && next_part(q, p)) {
            const Unit &u = p.u;
            if (u.e != cur_e || p.ph != cur_ph) {
                const uint8_t *em = a.maps + (size_t)u.e * kMapsPerExpert * kMapBytes;
                map0 = em + (p.ph == 0 ? 0 : 2) * kMapBytes;
                map1 = em + (p.ph == 0 ? 1 : 2) * kMapBytes;
                acquire_map(map0);
                if (p.ph == 0) acquire_map(map1);
                cur_e = u.e;
                cur_ph = p.ph;
            }
            auto issue_stage = [&](int c) -> bool {
                const int s = su % S;
                if (!mbar_wait(empty0 + 8 * s, ((su / S) & 1) ^ 1)) {
                    if (lane == 0) fail(2);
                    return false;
                }
                if (lane == 0) {
                    const uint32_t dst = st0 + s * STAGE;
                    const uint32_t tf = tfull0 + 8 * s;
                    mbar_arrive_expect_tx(tf, 2 * kTileBytes);
                    if (p.ph == 0) {
                        tma_2d(dst, map0, c * 128, p.mt * 128, tf, pol);
                        tma_2d(dst + kTileBytes, map1, c * 128, p.mt * 128, tf, pol);
                    } else {
                        tma_2d(dst, map0, (2 * c) * 128, p.mt * 128, tf, pol);
                        tma_2d(dst + kTileBytes, map0, (2 * c + 1) * 128, p.mt * 128, tf, pol);
                    }
                }
                __syncwarp();
                su++;
                return true;
            };
            // A new B image: the token's x is ready, so it goes out before
            // the part's weight tiles (which would queue ahead of it); a
            // pair's h waits for the gate/up pass, so up to a ring of weight
            // tiles (which need nothing) goes out first.
            const long long key = b_key(p);
            const int pre = key != cur_key && p.ph == 0 ? 0 : min(S, p.hi - p.lo);
            bool ok = true;
            for (int c = p.lo; c < p.lo + pre && ok; c++) ok = issue_stage(c);
            if (!ok) break;
            if (key != cur_key) {
                // epoch bl: x (bl = 0) or a pair's h; wait for the epoch that
                // used its buffer (x overlaps both h buffers)
                if (bl >= 2 || (bl == 1 && x_first)) {
                    const uint32_t wb = bl == 1 ? 0 : (bl & 1), par = bl == 1 ? 0 : ((bl / 2 - 1) & 1);
                    if (!mbar_wait(bempty0 + 8 * wb, par)) {
                        if (lane == 0) fail(1);
                        break;
                    }
                }
                if (bl == 0) x_first = p.ph == 0;
                const uint8_t *src;
                uint32_t nb, ns;
                if (p.ph == 0) {
                    src = a.img_in + (size_t)(p.pair / kK) * img_bytes(kD);
                    nb = XB;
                    ns = XS;
                } else {
                    // the pair's h: every gate/up item of the pair has written its block
                    const int pair = (int)key;
                    const int *cnt = a.sync + SYNC_HDONE + (a.experts == nullptr ? 0 : pair % kK);
                    int f = 0;
                    const uint32_t lim = wait_polls();
                    for (uint32_t i = 0; i < lim && f < MTG; i++) {
                        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(f) : "l"(cnt) : "memory");
                        if (f < MTG) __nanosleep(128);
                    }
                    if (f < MTG) {
                        if (lane == 0) fail(11);
                        break;
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    src = a.img_out + (size_t)pair * img_bytes(kF);
                    nb = HB;
                    ns = HS;
                }
                if (lane == 0) {
                    const uint32_t bf = bfull0 + 8 * (bl & 1);
                    mbar_arrive_expect_tx(bf, nb + ns);
                    bulk_g2s(breg + b_off(bl), src, nb, bf, pol_img);
                    bulk_g2s(breg + s_off(bl), src + nb, ns, bf, pol_img);
                }
                __syncwarp();
                bl++;
                cur_key = key;
            }
            for (int c = p.lo + pre; c < p.hi && ok; c++) ok = issue_stage(c);
            if (!ok) break;
        }
        // copies still in flight (after a wait gave up) land before the CTA leaves
        if (lane == 0 && (!drain_ring(tfull0, S, su) || !drain_ring(bfull0, 2, bl)))
            report_status(a.status, kStatusWaitTimeout, 13);
    } else if (warp == kSfWarp) {
        // -------------------------------------------------- scale loader --
        // a part's tile scale rows in one bulk copy into one of two buffers
        // (the next part's copy goes out when the current part starts);
        // per stage, the 4 atoms: gate/up W1 and W3 of the chunk, down the
        // two chunks of W2
        const uint64_t pol = l2_evict_first_policy();
        uint32_t ni = 0;                   // parts whose scale rows were issued
        auto issue = [&](const Part &p, int buf) {
            ni++;
            __syncwarp();
            fence_async_smem();
            if (lane == 0) {
                const int G = p.ph == 0 ? GG : GD;
                const size_t off = (size_t)p.mt * 128 * G;
                const uint32_t dst = sraw0 + buf * SRAW;
                mbar_arrive_expect_tx(sfull0 + 8 * buf, (p.ph == 0 ? 2 : 1) * 128 * G);
                if (p.ph == 0) {
                    bulk_g2s(dst, p.u.ex.s1 + off, 128 * G, sfull0 + 8 * buf, pol);
                    bulk_g2s(dst + 128 * G, p.u.ex.s3 + off, 128 * G, sfull0 + 8 * buf, pol);
                } else {
                    bulk_g2s(dst, p.u.ex.s2 + off, 128 * G, sfull0 + 8 * buf, pol);
                }
            }
        };
        uint32_t su = 0, np = 0;
        int q = 0;
        Part cur, nxt;
        bool have = next_part(q, cur);
        if (have) issue(cur, 0);
        while (have && !*abort_flag) {
            const int buf = np & 1;
            int qn = q;
            const bool more = next_part(qn, nxt);
            if (more) issue(nxt, (np + 1) & 1);
            if (!mbar_wait(sfull0 + 8 * buf, (np / 2) & 1)) {
                if (lane == 0) fail(3);
                break;
            }
            const uint32_t sraw = sraw0 + buf * SRAW;
            const int G = cur.ph == 0 ? GG : GD;
            bool ok = true;
            for (int c = cur.lo; c < cur.hi; c++, su++) {
                const int s = su % S;
                if (!mbar_wait(empty0 + 8 * s, ((su / S) & 1) ^ 1)) {
                    if (lane == 0) fail(9);
                    ok = false;
                    break;
                }
                uint2 wv[2][4];
#pragma unroll
                for (int t = 0; t < 2; t++) {
                    // sub-tile t: gate/up matrix t of chunk c; down chunk 2c + t
                    const uint32_t base = cur.ph == 0 ? sraw + t * 128 * G + c * 8 : sraw + (2 * c + t) * 8;
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                                     : "=r"(wv[t][j].x), "=r"(wv[t][j].y)
                                     : "r"(base + (lane + 32 * j) * G));
                }
                const uint32_t stg = st0 + s * STAGE, at0 = stg + 2 * kTileBytes;
                // groups with scale 255 contribute nothing: once the stage's
                // weight tiles landed, their codes are zeroed (rare)
                uint32_t nan = 0;
#pragma unroll
                for (int t = 0; t < 2; t++)
#pragma unroll
                    for (int j = 0; j < 4; j++) nan |= nan_scale_mask(wv[t][j].x) | nan_scale_mask(wv[t][j].y);
                if (__any_sync(0xffffffffu, nan != 0)) {
                    if (!mbar_wait(tfull0 + 8 * s, (su / S) & 1)) {
                        if (lane == 0) fail(12);
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int t = 0; t < 2; t++)
#pragma unroll
                        for (int j = 0; j < 4; j++) zero_nan_groups_sw128(stg + t * kTileBytes, lane + 32 * j, wv[t][j]);
                }
#pragma unroll
                for (int t = 0; t < 2; t++) {
                    sts128(at0 + (2 * t) * kAtomBytes + 16 * lane, drop_nan_scales(wv[t][0].x),
                           drop_nan_scales(wv[t][1].x), drop_nan_scales(wv[t][2].x), drop_nan_scales(wv[t][3].x));
                    sts128(at0 + (2 * t + 1) * kAtomBytes + 16 * lane, drop_nan_scales(wv[t][0].y),
                           drop_nan_scales(wv[t][1].y), drop_nan_scales(wv[t][2].y), drop_nan_scales(wv[t][3].y));
                }
                fence_async_smem();
                mbar_arrive(full0 + 8 * s);
            }
            if (!ok) break;
            np++;
            q = qn;
            cur = nxt;
            have = more;
        }
        if (lane == 0 && !drain_ring(sfull0, 2, ni)) report_status(a.status, kStatusWaitTimeout, 14);
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------- MMA issuer --
        if (lane == 0) {
            uint32_t su = 0, bu = 0, it = 0, bcur = 0;
            long long cur_key = -2;
            int q = 0;
            bool run = true;
            Part p;
            while (run && !*abort_flag && next_part(q, p)) {
                const long long key = b_key(p);
                if (key != cur_key) {
                    bcur = bu;
                    if (!mbar_wait(bfull0 + 8 * (bu & 1), (bu / 2) & 1)) {
                        fail(4);
                        break;
                    }
                    bu++;
                    tc_fence_after();
                    // scale atoms of the epoch's B (one token: the four 8-line
                    // groups all read its lines)
                    const int atoms = p.ph == 0 ? kD / 128 : kF / 128;
                    for (int at = 0; at < atoms; at++)
                        tmem_cp_atom(tmem + SFB_COL + 4 * at, desc_atom(breg + s_off(bcur) + at * 128, 0));
                    cur_key = key;
                }
                const uint32_t bimg = breg + b_off(bcur);
                const int b = it & 1;
                if (!mbar_wait(acce0 + 8 * b, ((it >> 1) & 1) ^ 1)) {
                    fail(5);
                    break;
                }
                tc_fence_after();
                for (int c = p.lo; c < p.hi; c++, su++) {
                    const int s = su % S;
                    if (!mbar_wait(tfull0 + 8 * s, (su / S) & 1) || !mbar_wait(full0 + 8 * s, (su / S) & 1)) {
                        fail(6);
                        run = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t stg = st0 + s * STAGE;
                    const uint32_t sfa = tmem + SFA_COL + s * 16;
#pragma unroll
                    for (int at = 0; at < 4; at++)
                        tmem_cp_atom(sfa + at * 4, desc_atom(stg + 2 * kTileBytes + at * kAtomBytes, 128));
#pragma unroll
                    for (int t = 0; t < 2; t++) {
                        // gate/up: matrix t into accumulator t; down: chunk 2c + t into accumulator 0
                        const int bc = p.ph == 0 ? c : 2 * c + t;          // B's 256-column chunk
                        const uint32_t d = tmem + (b * 2 + (p.ph == 0 ? t : 0)) * 8;
#pragma unroll
                        for (int ks = 0; ks < 4; ks++) {
                            const int id = 2 * (ks & 1);
                            const bool fresh = c == p.lo && ks == 0 && (p.ph == 0 || t == 0);
                            mma_mxf4(d, desc_sw128(stg + t * kTileBytes + 32 * ks, 1024),
                                     desc_sw128(bimg + bc * 1024 + 32 * ks, 1024), idesc_mxf4(8, id),
                                     sfa + t * 8 + (ks >> 1) * 4, tmem + SFB_COL + (bc * 2 + (ks >> 1)) * 4,
                                     fresh ? 0u : 1u);
                        }
                    }
                    umma_commit(empty0 + 8 * s);
                }
                if (!run) break;
                umma_commit(accf0 + 8 * b);
                it++;
                int qn = q;
                Part nx;
                if (!next_part(qn, nx) || b_key(nx) != key) umma_commit(bempty0 + 8 * (bcur & 1));
            }
            umma_commit(done);
        }
    } else {
        // ------------------------------------------------------- epilogue --
        const int q4 = warp & 3;
        const int row_in_tile = 32 * q4 + lane;
        __shared__ int last_tile;
        uint32_t it = 0;
        int q = 0;
        Part p;
        while (!*abort_flag && next_part(q, p)) {
            const int kc = p.ph == 0 ? KCG : KCD;
            const int b = it & 1;
            if (!mbar_wait(accf0 + 8 * b, (it >> 1) & 1)) {
                if (lane == 0) fail(7);
                break;
            }
            tc_fence_after();
            uint32_t v[2][8];
#pragma unroll
            for (int m = 0; m < 2; m++) tmem_ld<8>(tmem + ((uint32_t)(32 * q4) << 16) + (b * 2 + m) * 8, v[m]);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(acce0 + 8 * b);
            it++;
            const int nm = p.ph == 0 ? 2 : 1;
            float acc[2] = {0.f, 0.f};
#pragma unroll
            for (int m = 0; m < 2; m++)
#pragma unroll
                for (int pc = 0; pc < kPieces; pc++) acc[m] += __uint_as_float(v[m][pc]);
            const size_t slot = (size_t)p.seg * kMaxGrid + blockIdx.x;
            if (sc.sk && p.lo > 0) {
                // the tail of an item begun by the previous CTA: hand over
                // the summed pieces and move on
                float *dst = a.partials + slot * PARTIAL;
#pragma unroll
                for (int m = 0; m < 2; m++)
                    if (m < nm) dst[m * 128 + row_in_tile] = acc[m];
                named_sync(1, 128);
                if (q4 == 0 && lane == 0) {
                    __threadfence();
                    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(a.sync + slot), "r"(1) : "memory");
                }
                continue;
            }
            if (sc.sk && p.hi < kc) {
                // the head of an item the next CTA finishes: add its sums
                const int *flag = a.sync + slot + 1;
                int f = 0;
                const uint32_t lim = wait_polls();
                for (uint32_t i = 0; i < lim && f == 0; i++) {
                    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(f) : "l"(flag) : "memory");
                    if (f == 0) __nanosleep(64);
                }
                if (f == 0) fail(10);
                const float *src = a.partials + (slot + 1) * PARTIAL;
#pragma unroll
                for (int m = 0; m < 2; m++)
                    if (m < nm) acc[m] += __ldcg(src + m * 128 + row_in_tile);
            }
            const int pair = p.pair;
            const int row = p.mt * 128 + row_in_tile;
            if (p.ph == 0) {
                float *gu = a.gu + (size_t)pair * 2 * kF;
                gu[row] = acc[0];
                gu[kF + row] = acc[1];
                uint8_t *ib = a.img_out + (size_t)pair * img_bytes(kF);
                store_pieces(situ_glu(acc[0], acc[1]), ib, ib + img_b(kF), p.mt * 4 + q4);
                // this item's block of h is written: count it for the pair
                // (the barrier orders the four warps' writes before one
                // thread's fence and count)
                named_sync(1, 128);
                if (q4 == 0 && lane == 0) {
                    __threadfence();
                    atomicAdd(a.sync + SYNC_HDONE + (a.experts == nullptr ? 0 : pair % kK), 1);
                }
            } else if (a.w == nullptr) {
                a.y[row] = acc[0];                      // one expert: its output is y
            } else {
                a.out[(size_t)pair * kD + row] = acc[0];
                // the last of the token's 16 pairs to finish this tile forms y
                named_sync(1, 128);
                if (q4 == 0 && lane == 0) {
                    __threadfence();
                    const int done_pairs = atomicAdd(a.sync + SYNC_TILE + p.mt, 1) + 1;
                    __threadfence();
                    last_tile = done_pairs == n_units;     // the token's pairs (top-p may keep fewer than 16)
                }
                named_sync(1, 128);
                if (last_tile) {
                    const int t = pair / kK;
                    float yv = 0.f;
#pragma unroll 4
                    for (int k = 0; k < kK; k++) {
                        const float wk = __ldg(a.w + (size_t)t * kK + k);
                        if (wk != 0.f)                     // a slot dropped by top-p has no row
                            yv = fmaf(wk, __ldcg(a.out + ((size_t)t * kK + k) * kD + row), yv);
                    }
                    a.y[(size_t)t * kD + row] = yv;
                }
            }
        }
    }

    __syncthreads();
    if (warp == kMmaWarp) {
        if (!mbar_wait_drain(done, 0) && lane == 0) report_status(a.status, kStatusWaitTimeout, 8);
        tc_fence_after();
        tmem_dealloc(tmem, f1::TMEM_COLS);
    }
}

// ------------------------------------------------------------- launchers --

template <int PH, int NTOK>
cudaError_t launch_mx_t(const Ctx &c, MxArgs a, bool pdl) {
    using Sh = MxShape<PH, NTOK>;
    static std::atomic<uint64_t> configured{0};
    const cudaError_t e = ensure_smem((const void *)k_mx<PH, NTOK>, Sh::SMEM, configured);
    if (e != cudaSuccess) return e;
    a.status = c.status;
    int grid = c.num_sms < kMaxGrid ? c.num_sms : kMaxGrid;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Sh::SMEM;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_mx<PH, NTOK>, a);
}

MxArgs mx_args(const DecodeExperts &d) {
    MxArgs a{};
    if (d.single) {
        a.one = *d.single;
    } else {
        a.experts = d.experts;
        a.units = d.units;
        a.n_units = d.n_units;
        a.perm = d.perm;
    }
    return a;
}

}  // namespace

// The driver entry point, resolved once (a function-local static, so the
// first calls from several threads are safe).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        const bool ok = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                                         &q) == cudaSuccess &&
                        q == cudaDriverEntryPointSuccess;
        return ok ? reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f) : nullptr;
    }();
    return fn;
}

// Tensor-map templates (tmaps.cuh), encoded once per device.  They point at
// the library's own scratch array (larger than one matrix), so a map is
// never left pointing at memory that is not allocated.
bool weight_map_templates(CUtensorMap &w13, CUtensorMap &w2) {
    constexpr int kDevs = 64;
    static std::atomic<int> state[kDevs];  // 0 not tried, 1 ok, 2 failed
    static CUtensorMap t13[kDevs], t2[kDevs];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return false;
    if (state[dev].load(std::memory_order_acquire) == 0) {
        void *base = library_scratch();   // takes the set-up lock itself
        auto enc = tensor_map_encoder();
        std::lock_guard<std::mutex> lock(setup_mutex());
        if (state[dev].load(std::memory_order_relaxed) == 0) {
            bool ok = base != nullptr && enc != nullptr && library_scratch_bytes() >= (size_t)kD / 2 * kF &&
                      library_scratch_bytes() >= (size_t)kF / 2 * kD;
            if (ok) {
                const cuuint32_t box[2] = {128, 128}, es[2] = {1, 1};
                const cuuint64_t d13[2] = {(cuuint64_t)kD / 2, (cuuint64_t)kF}, s13[1] = {(cuuint64_t)kD / 2};
                const cuuint64_t d2[2] = {(cuuint64_t)kF / 2, (cuuint64_t)kD}, s2[1] = {(cuuint64_t)kF / 2};
                ok = enc(&t13[dev], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, d13, s13, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
                     enc(&t2[dev], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, d2, s2, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
            }
            state[dev].store(ok ? 1 : 2, std::memory_order_release);
        }
    }
    if (state[dev].load(std::memory_order_acquire) != 1) return false;
    w13 = t13[dev];
    w2 = t2[dev];
    return true;
}

// stream-K region of the fused single-token pass: the hand-over flags
// [4 segments][kMaxGrid], the per-pair h counts and the per-tile y counts
// (ints), then the hand-over partials [4 segments][kMaxGrid][2][128] fp32
namespace {
constexpr size_t kSkFlagBytes = (size_t)f1::SYNC_INTS * sizeof(int);
constexpr size_t kSkPartBytes = (size_t)f1::NSEG * kMaxGrid * f1::PARTIAL * sizeof(float);
}  // namespace
cudaError_t launch_mx_fused1(const Ctx &c, const DecodeExperts &d, const uint8_t *ximg, uint8_t *himg, float *gu,
                             float *stage, const float *w, float *y, const uint8_t *maps, uint8_t *sk) {
    static std::atomic<uint64_t> configured{0};
    const cudaError_t e = ensure_smem((const void *)k_mx1, f1::SMEM, configured);
    if (e != cudaSuccess) return e;
    MxArgs a = mx_args(d);
    a.img_in = ximg;
    a.img_out = himg;
    a.gu = gu;
    a.out = stage;
    a.maps = maps;
    a.w = w;
    a.y = y;
    a.status = c.status;
    a.sync = reinterpret_cast<int *>(sk);
    a.partials = reinterpret_cast<float *>(sk + kSkFlagBytes);
    const int grid = c.num_sms < kMaxGrid ? c.num_sms : kMaxGrid;
    return launch_pdl(k_mx1, dim3(grid), dim3(kThreads), f1::SMEM, c.stream, a);
}

cudaError_t set_wait_polls_mx(uint32_t polls) { return set_wait_polls_here(polls); }

size_t mx_ximg_bytes(int n_tokens) { return (size_t)n_tokens * img_bytes(kD); }
size_t mx_himg_bytes(int n_pairs) { return (size_t)n_pairs * img_bytes(kF); }
size_t mx_maps_bytes(int n_experts) { return expert_maps_bytes(n_experts); }

size_t mx_streamk_bytes() { return kSkFlagBytes + kSkPartBytes; }
int mx_streamk_flag_count() { return (int)(kSkFlagBytes / sizeof(int)); }

cudaError_t launch_mx_ximg(const Ctx &c, const void *x, int x_bf16, int n_tokens, uint8_t *ximg, uint8_t *sk,
                           uint8_t *maps, const k3mx_expert *table, const k3mx_expert *one) {
    CUtensorMap w13, w2;
    if (!weight_map_templates(w13, w2)) return cudaErrorNotSupported;
    const long long warps = (long long)n_tokens * (kD / 32);
    const int piece_ctas = (int)((warps + 7) / 8);
    const int n_map_experts = one != nullptr ? 1 : kE;
    const int map_ctas = (n_map_experts * kMapsPerExpert + kMapsPerCta - 1) / kMapsPerCta;
    const k3mx_expert single = one != nullptr ? *one : k3mx_expert{};
    k_mx_ximg<<<(unsigned)(piece_ctas + map_ctas), 256, 0, c.stream>>>(
        x, x_bf16, n_tokens, ximg, reinterpret_cast<int *>(sk), sk != nullptr ? mx_streamk_flag_count() : 0, piece_ctas,
        maps, n_map_experts, one != nullptr ? nullptr : table, single, w13, w2);
    return cudaGetLastError();
}

cudaError_t launch_mx_gate_up(const Ctx &c, const DecodeExperts &d, const uint8_t *ximg, uint8_t *himg,
                              float *gu, uint8_t *maps) {
    MxArgs a = mx_args(d);
    a.img_in = ximg;
    a.img_out = himg;
    a.gu = gu;
    a.maps = maps;
    return launch_mx_t<0, kUnitPairs>(c, a, true);
}

cudaError_t launch_mx_down(const Ctx &c, const DecodeExperts &d, const uint8_t *himg, float *out,
                           uint8_t *maps) {
    MxArgs a = mx_args(d);
    a.img_in = himg;
    a.out = out;
    a.maps = maps;
    return launch_mx_t<1, kUnitPairs>(c, a, true);
}

}  // namespace k3mx
