// route_group.cu - router top-16 selection and token-to-expert grouping.
//
// Routing (Kimi K3 engine (c/kimi_k3.c), "Architecture notes", Stable
// LatentMoE; kimi-k3-in-c README, "Three invariants", item 3): the score is
// sigma(logit), the selection key is score + bias, the top 16 keys win, and
// the combining weights are the selected raw scores renormalised.
//   - sigma is evaluated in double and rounded to fp32 once, so the fp32
//     score, key and selection agree bit for bit with a CPU evaluation in the
//     same precision;
//   - equal keys go to the lower expert index: a key is paired with its
//     complemented index and the warp takes the lexicographic maximum;
//   - -0 counts as +0 and a NaN key ranks below every number.
// One warp per token: lane l holds experts l, l+32, ..., 28 keys in
// registers; 16 rounds of a warp maximum (redux.sync) pick the winners in
// key order.
//
// Grouping (Kimi K3 engine (c/kimi_k3.c), "Chunked prefill": every unique
// expert of a chunk is loaded once for all its tokens): counts per expert,
// exclusive offsets, and the pair list sorted by (expert, pair index).  The
// counts come from shared-memory integer atomics (order-free); the placement
// is a stable warp-sequential scatter, so the output is deterministic.
#include "common.cuh"
#include "pieces.cuh"
#include "tmaps.cuh"

namespace k3mx {
namespace {

constexpr float kRoutedScale = 1.0f;     // K3Cfg routed_scale
constexpr int kPer = kE / 32;            // 28 experts per lane
constexpr int kSeg = 1024;               // pairs per grouping segment (one warp scatters one)
constexpr int kRouteWarpMax = 64;        // more tokens: one routing CTA per token

__device__ __forceinline__ uint32_t order_key(float k) {
    if (k != k) k = -INFINITY;           // NaN ranks last
    if (k == 0.0f) k = 0.0f;             // -0 -> +0
    const uint32_t u = __float_as_uint(k);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// sigma(logit) in double, rounded to fp32 once: the score both sides agree on
__device__ __forceinline__ float exact_score(float l) {
    return (float)(1.0 / (1.0 + exp(-(double)l)));
}

// An fp32 estimate of the same score.  expf is within 2 ulp, the add and the
// division round once each, so |approx - exact| < 2^-21 (scores lie in
// [0, 1]); after adding the bias and rounding, two keys differ by less than
// 2^-20 * max(1, |key|).
__device__ __forceinline__ float approx_score(float l) {
    return 1.0f / (1.0f + expf(-l));
}

// A score s in [2^-24, 1] in units of 2^-47: its significand shifted by the
// exponent, integer operations only (exact: s = M 2^(E-150), E >= 103).
__device__ __forceinline__ long long score_fx(float s) {
    const uint32_t u = __float_as_uint(s);
    const uint32_t E = (u >> 23) & 0xFFu, M = (u & 0x7FFFFFu) | 0x800000u;
    return (long long)((unsigned long long)M << (E - 103u));
}

// A sum of at most 16 such values (0 < v < 2^52) times 2^-47 as a double,
// built from its bits: exact, since v has at most 52 significant bits.
__device__ __forceinline__ double fx_to_double(long long v) {
    const unsigned long long x = (unsigned long long)v;
    const int t = 63 - __clzll(x);                    // leading bit, t <= 51
    const unsigned long long frac = (x << (52 - t)) & 0xFFFFFFFFFFFFFull;
    return __longlong_as_double((long long)(((unsigned long long)(1023 + t - 47) << 52) | frac));
}

__device__ __forceinline__ float canon_key(float k) {
    if (k != k) return -INFINITY;        // NaN ranks last
    if (k == 0.0f) return 0.0f;          // -0 -> +0
    return k;
}

__device__ __forceinline__ float key_of_order(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// the lane's best remaining key (strictly greater wins, so among equal keys
// the lower slot, i.e. the lower expert index, is kept) and its slot
__device__ __forceinline__ uint32_t lane_best(const uint32_t (&ok)[kPer], int &slot) {
    uint32_t b = ok[0];
    slot = 0;
#pragma unroll
    for (int i = 1; i < kPer; i++)
        if (ok[i] > b) {
            b = ok[i];
            slot = i;
        }
    return b;
}

__device__ __forceinline__ void clear_slot(uint32_t (&ok)[kPer], int slot) {
#pragma unroll
    for (int i = 0; i < kPer; i++)
        if (i == slot) ok[i] = 0;
}

// The warp's largest (key, complemented index) pair: the largest key first,
// then among its holders the largest complemented index (lowest expert).
// Each lane offers its best (hi, lo); returns both halves.
__device__ __forceinline__ void warp_max_pair(uint32_t hi, uint32_t lo, uint32_t &mhi, uint32_t &mlo) {
    mhi = __reduce_max_sync(0xffffffffu, hi);
    mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
}

// The token's routing result; lane k < 16 holds slot k's expert e and raw
// score s, `sum` is the slot-order double sum of the 16 scores.  With
// top_p > 0 the low-weight tail is dropped (Kimi K3 engine (c/kimi_k3.c),
// "Streaming design", K3_TOPP): in order of decreasing score (ties: lower
// index) an expert is kept while the scores ahead of it sum to less than
// top_p * sum; kept weights are raw scores over the kept sum, a dropped slot
// gets index -1 and weight 0.  The sums are slot-order double sums, or, with
// every score in [2^-24, 1], exact sums in units of 2^-47 (the same values).
// Whole warp.
__device__ __forceinline__ int write_routing(int32_t *idx_t, float *w_t, int lane, int my_e,
                                             float my_s, double sum, double top_p) {
    if (top_p > 0.0) {
        const float s = my_s;
        const int e = my_e;
        const bool fixed = __all_sync(0xffffffffu, lane >= kK || (s >= 0x1p-24f && s <= 1.0f));
        double before = 0.0, kept = 0.0;
        long long bfx = 0, kfx = 0;
#pragma unroll 1
        for (int j = 0; j < kK; j++) {
            const float sj = __shfl_sync(0xffffffffu, s, j);
            const int ej = __shfl_sync(0xffffffffu, e, j);
            if (sj > s || (sj == s && ej < e)) {
                if (fixed) bfx += score_fx(sj);
                else before += (double)sj;
            }
        }
        if (fixed) before = bfx > 0 ? fx_to_double(bfx) : 0.0;
        const bool keep = lane < kK && before < top_p * sum;
#pragma unroll 1
        for (int j = 0; j < kK; j++) {
            const int kj = __shfl_sync(0xffffffffu, keep ? 1 : 0, j);
            const float sj = __shfl_sync(0xffffffffu, s, j);
            if (kj) {
                if (fixed) kfx += score_fx(sj);
                else kept += (double)sj;
            }
        }
        if (fixed) kept = fx_to_double(kfx);
        if (lane < kK) {
            idx_t[lane] = keep ? e : -1;
            w_t[lane] = keep ? (float)((double)s / kept) * kRoutedScale : 0.f;
        }
        return keep ? e : -1;
    }
    if (lane < kK) {
        idx_t[lane] = my_e;
        w_t[lane] = (float)((double)my_s / sum) * kRoutedScale;
    }
    return my_e;
}

// Exact selection over all 896 experts (used when the candidate filter
// below would keep more than 64 experts, e.g. with many equal or NaN keys).
__device__ void route_warp_all(const float *__restrict__ lt, const float *__restrict__ bias,
                               int32_t *__restrict__ idx_t, float *__restrict__ w_t, int lane, double top_p) {
    uint32_t ok[kPer];
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const int e = lane + 32 * i;
        ok[i] = order_key(exact_score(__ldg(lt + e)) + __ldg(bias + e));
    }
    int slot;
    uint32_t best = lane_best(ok, slot);
    float my_s = 0.f;
    int my_e = 0;
    double sum = 0.0;
#pragma unroll 1
    for (int k = 0; k < kK; k++) {
        uint32_t mhi, mlo;
        warp_max_pair(best, 0xFFFFFFFFu - (uint32_t)(lane + 32 * slot), mhi, mlo);
        const int e = (int)(0xFFFFFFFFu - mlo);
        if ((e & 31) == lane) {
            clear_slot(ok, slot);
            best = lane_best(ok, slot);
        }
        const float s_win = exact_score(__ldg(lt + e));
        sum += (double)s_win;                       // slot order, as on the CPU
        if (lane == k) {
            my_s = s_win;
            my_e = e;
        }
    }
    write_routing(idx_t, w_t, lane, my_e, my_s, sum, top_p);
}

// One token on one warp.  (1) fp32 estimates of all 896 keys (28 per lane,
// in registers); (2) the 16th largest estimate a16 by 16 rounds of a warp
// maximum; (3) every expert whose estimate is within 2^-18 * max(1,|a16|)
// of a16 is a candidate: an expert of the exact top 16 cannot lie further
// below (each estimate is within 2^-20 * max(1,|key|) of its exact key, and
// the 16th order statistic moves by no more than that); (4) exact keys for
// the candidates only, and the exact top-16 among them.  `scratch` is 128
// ints of shared memory for this warp.
__device__ void route_warp(const float *__restrict__ lt, const float *__restrict__ bias,
                           int32_t *__restrict__ idx_t, float *__restrict__ w_t, int lane,
                           int *scratch, double top_p) {
    uint32_t ok[kPer];
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const int e = lane + 32 * i;
        ok[i] = order_key(canon_key(approx_score(__ldg(lt + e)) + __ldg(bias + e)));
    }
    // the 16th largest estimate (equal estimates count once each)
    uint32_t cand[kPer];
#pragma unroll
    for (int i = 0; i < kPer; i++) cand[i] = ok[i];
    int slot;
    uint32_t best = lane_best(cand, slot), m16 = 0;
#pragma unroll 1
    for (int k = 0; k < kK; k++) {
        m16 = __reduce_max_sync(0xffffffffu, best);
        const int owner = __ffs(__ballot_sync(0xffffffffu, best == m16)) - 1;
        if (lane == owner) {
            clear_slot(cand, slot);
            best = lane_best(cand, slot);
        }
    }
    const float a16 = key_of_order(m16);
    // a non-finite a16 (infinite biases) keeps every expert: exact path
    const uint32_t tau = isfinite(a16) ? order_key(a16 - 0x1p-18f * fmaxf(1.0f, fabsf(a16))) : 0u;

    // candidates into a compact per-warp list (at most 64)
    const unsigned lt_mask = (1u << lane) - 1u;
    int n = 0;
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const bool c = ok[i] >= tau;
        const unsigned bm = __ballot_sync(0xffffffffu, c);
        const int pos = n + __popc(bm & lt_mask);
        if (c && pos < 64) scratch[pos] = lane + 32 * i;
        n += __popc(bm);
    }
    __syncwarp();
    if (n > 64) {
        route_warp_all(lt, bias, idx_t, w_t, lane, top_p);
        return;
    }
    // exact keys: lane holds candidates lane and lane + 32
    uint32_t khi[2], klo[2];
    float cs[2];
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const int pos = lane + 32 * j;
        khi[j] = 0;
        klo[j] = 0;
        cs[j] = 0.f;
        if (pos < n) {
            const int e = scratch[pos];
            cs[j] = exact_score(__ldg(lt + e));
            khi[j] = order_key(cs[j] + __ldg(bias + e));
            klo[j] = 0xFFFFFFFFu - (uint32_t)e;
        }
    }
    __syncwarp();
    float my_s = 0.f;
    int my_e = 0;
    double sum = 0.0;
#pragma unroll 1
    for (int k = 0; k < kK; k++) {
        const bool first = khi[0] > khi[1] || (khi[0] == khi[1] && klo[0] > klo[1]);
        const uint32_t bh = first ? khi[0] : khi[1], bl = first ? klo[0] : klo[1];
        uint32_t mhi, mlo;
        warp_max_pair(bh, bl, mhi, mlo);
        const int e = (int)(0xFFFFFFFFu - mlo);
        // packed pairs are unique (they carry the index): one lane owns it
        const bool mine = bh == mhi && bl == mlo;
        float s_win = 0.f;
        if (mine) {
            s_win = first ? cs[0] : cs[1];
            if (first) {
                khi[0] = 0;
                klo[0] = 0;
            } else {
                khi[1] = 0;
                klo[1] = 0;
            }
        }
        const int owner = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
        s_win = __shfl_sync(0xffffffffu, s_win, owner);
        sum += (double)s_win;                       // slot order, as on the CPU
        if (lane == k) {
            my_s = s_win;
            my_e = e;
        }
    }
    write_routing(idx_t, w_t, lane, my_e, my_s, sum, top_p);
}

__global__ void __launch_bounds__(256) k_route(int32_t *idx, float *w, const float *logits,
                                               const float *bias, int n_tokens, double top_p) {
    __shared__ int scratch[8][128];
    pdl_wait();                          // the logits, when a router pass writes them
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = blockIdx.x * (blockDim.x / 32) + warp;
    if (t >= n_tokens) return;
    route_warp(logits + (size_t)t * kE, bias, idx + (size_t)t * kK, w + (size_t)t * kK, lane,
               scratch[warp], top_p);
}

// exclusive scan of one int per thread over the block (up to 32 warps);
// *total gets the sum.  `tmp` is 33 ints of shared memory.
__device__ int block_excl_scan(int v, int *tmp, int *total) {
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32, nwarps = blockDim.x / 32;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int ws = lane < nwarps ? tmp[lane] : 0;
        int wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        tmp[lane] = wi - ws;
        if (lane == 31) tmp[32] = wi;
    }
    __syncthreads();
    const int r = incl - v + tmp[warp];
    *total = tmp[32];
    __syncthreads();
    return r;
}

// Counts, offsets and the active-expert list from the per-expert counts in
// cnt_sm.  Thread i owns experts i*EPT .. i*EPT+EPT-1 (EPT = 896 / threads,
// rounded up).  Writes counts/offsets/act/n_active; cnt_sm becomes each
// expert's starting offset.
__device__ void finish_counts(int *cnt_sm, const GroupOut &g, int *tmp) {
    const int ept = (kE + blockDim.x - 1) / blockDim.x;
    const int e0 = threadIdx.x * ept;
    int c[4] = {0, 0, 0, 0};
    int sum = 0, nz = 0;
    for (int j = 0; j < ept; j++) {
        const int e = e0 + j;
        c[j] = e < kE ? cnt_sm[e] : 0;
        sum += c[j];
        nz += c[j] > 0;
    }
    int nu = 0;
    for (int j = 0; j < ept; j++) nu += (c[j] + kUnitPairs - 1) / kUnitPairs;
    int total, n_act, n_un;
    int off = block_excl_scan(sum, tmp, &total);
    int apos = block_excl_scan(nz, tmp, &n_act);
    int upos = block_excl_scan(nu, tmp, &n_un);
    for (int j = 0; j < ept; j++) {
        const int e = e0 + j;
        if (e < kE) {
            g.counts[e] = c[j];
            g.offsets[e] = off;
            cnt_sm[e] = off;
            if (c[j] > 0) g.act[apos++] = e;
            if (g.units != nullptr)
                for (int q = 0; q < c[j]; q += kUnitPairs, upos++) {
                    g.units[3 * upos + 0] = e;
                    g.units[3 * upos + 1] = off + q;
                    g.units[3 * upos + 2] = off + min(q + kUnitPairs, c[j]);
                }
            off += c[j];
        }
    }
    if (threadIdx.x == 0) {
        g.offsets[kE] = total;
        *g.n_active = n_act;
        if (g.n_units != nullptr) *g.n_units = n_un;
    }
    __syncthreads();
}

// Stable placement of pairs [p_begin, p_end) by one warp: running[e] holds
// the next free position of expert e and advances as the warp walks the
// pairs in order, 32 at a time.
__device__ void scatter_warp(const int32_t *idx, int p_begin, int p_end, int *running,
                             int32_t *perm) {
    constexpr int kChunks = kSeg / 32;
    const int lane = threadIdx.x % 32;
    const unsigned lt_mask = (1u << lane) - 1u;
    // the segment's expert indices first (independent loads), then the
    // placement chunk by chunk
    int ev[kChunks];
#pragma unroll
    for (int k = 0; k < kChunks; k++) {
        const int p = p_begin + 32 * k + lane;
        int e = -1;
        if (p < p_end) {
            e = idx[p];
            if (e < 0 || e >= kE) e = -1;
        }
        ev[k] = e;
    }
#pragma unroll
    for (int k = 0; k < kChunks; k++) {
        const int e = ev[k];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt_mask);
        if (e >= 0) perm[running[e] + rank] = p_begin + 32 * k + lane;
        __syncwarp();
        if (e >= 0 && rank == 0) running[e] += __popc(peers);
        __syncwarp();
    }
}

// ------------------------------------------------- one token per CTA --
//
// For a few tokens the warp-per-token router leaves the GPU idle, so each
// token gets a 256-thread CTA: thread t holds experts t, t+256, t+512,
// t+768.  (1) fp32 estimates of the 896 keys; (2) the experts fall into 64
// groups (group g: the experts of threads g, g+64, g+128, g+192), and v,
// the 16th largest of the 64 group maxima, stands in for a16, the 16th
// largest estimate: 16 distinct experts (the maxima of 16 groups) have
// estimates >= v, so v <= a16, and v = a16 unless two of the top 16 share
// a group; (3) candidates within 2^-18 * max(1,|v|) below v (the bound of
// route_warp; the bound grows with v, so it keeps every expert that the
// bound at a16 keeps);
// (4) exact double scores for the candidates, each candidate's rank among
// them by (key, lower index); (5) warp 0 forms the slot-order sum of the 16
// winners' scores and the weights.  Every phase is a few dozen
// instructions: a single token's step waits for this CTA alone.

constexpr int kRT = 256;                 // threads per routing CTA
constexpr int kRS = 4;                   // expert slots per thread

struct RouteSmem {
    uint32_t tmax[kRT];                  // each thread's largest key
    uint32_t tau;
    int n;
    int cand[64];
    unsigned long long ck[64];           // exact key << 32 | complemented expert index
    float cs[64];
    int sel_e[kK];
    float sel_s[kK];
};

__device__ void route_cta(const float *__restrict__ lt, const float *__restrict__ bias,
                          int32_t *__restrict__ idx_t, float *__restrict__ w_t, RouteSmem &sm, double top_p) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float lv[kRS], bv[kRS];
#pragma unroll
    for (int j = 0; j < kRS; j++) {
        const int e = tid + kRT * j;
        lv[j] = e < kE ? __ldg(lt + e) : 0.f;
        bv[j] = e < kE ? __ldg(bias + e) : 0.f;
    }
    if (tid == 0) sm.n = 0;
    uint32_t ok[kRS], mx = 0;
#pragma unroll
    for (int j = 0; j < kRS; j++) {
        ok[j] = tid + kRT * j < kE ? order_key(canon_key(approx_score(lv[j]) + bv[j])) : 0u;
        mx = max(mx, ok[j]);
    }
    sm.tmax[tid] = mx;
    __syncthreads();
    if (warp == 0) {
        // groups lane and lane + 32, then the 16th largest of the 64 maxima
        // (equal maxima count once each)
        uint32_t g0 = 0, g1 = 0;
#pragma unroll
        for (int q = 0; q < kRT / 64; q++) {
            g0 = max(g0, sm.tmax[lane + 64 * q]);
            g1 = max(g1, sm.tmax[lane + 32 + 64 * q]);
        }
        // the 16th largest with multiplicity: the smallest value that fewer
        // than 16 of the 64 exceed (each lane counts, for its two values, the
        // values greater than them: 64 independent comparisons, no chain)
        int c0 = 0, c1 = 0;
#pragma unroll
        for (int u = 0; u < 32; u++) {
            const uint32_t a0 = __shfl_sync(0xffffffffu, g0, u), a1 = __shfl_sync(0xffffffffu, g1, u);
            c0 += (a0 > g0) + (a1 > g0);
            c1 += (a0 > g1) + (a1 > g1);
        }
        const uint32_t m16 = __reduce_min_sync(0xffffffffu, min(c0 < kK ? g0 : 0xFFFFFFFFu, c1 < kK ? g1 : 0xFFFFFFFFu));
        if (lane == 0) {
            // a non-finite v (infinite keys) keeps every expert: exact path
            const float v = key_of_order(m16);
            sm.tau = isfinite(v) ? order_key(v - 0x1p-18f * fmaxf(1.0f, fabsf(v))) : 0u;
        }
    }
    __syncthreads();
    const uint32_t tau = sm.tau;
#pragma unroll
    for (int j = 0; j < kRS; j++) {
        const int e = tid + kRT * j;
        if (e < kE && ok[j] >= tau) {
            const int pos = atomicAdd(&sm.n, 1);       // list order is free: ranks decide
            if (pos < 64) sm.cand[pos] = e;
        }
    }
    __syncthreads();
    const int n = sm.n;
    if (n > 64) {
        if (warp == 0) route_warp_all(lt, bias, idx_t, w_t, lane, top_p);
        __syncthreads();
        if (tid < kK) sm.sel_e[tid] = idx_t[tid];
        __syncthreads();
        return;
    }
    if (tid < n) {
        const int e = sm.cand[tid];
        const float s = exact_score(__ldg(lt + e));
        sm.cs[tid] = s;
        sm.ck[tid] = (unsigned long long)order_key(s + __ldg(bias + e)) << 32 | (0xFFFFFFFFu - (uint32_t)e);
    }
    __syncthreads();
    if (tid < n) {
        // rank = the candidates ahead (larger key, or equal key and lower
        // index); the comparisons are independent, so they are unrolled
        const unsigned long long me = sm.ck[tid];
        int r = 0;
#pragma unroll 16
        for (int u = 0; u < n; u++) r += sm.ck[u] > me;
        if (r < kK) {
            sm.sel_e[r] = (int)(0xFFFFFFFFu - (uint32_t)me);
            sm.sel_s[r] = sm.cs[tid];
        }
    }
    __syncthreads();
    if (warp == 0) {
        // The slot-order double sum.  With every score in [2^-24, 1] each
        // term is a multiple of 2^-47 and the sum stays below 2^5, so every
        // partial sum is exact in double and the sum equals the integer
        // sum of the scores in units of 2^-47, whatever the order of adds.
        const float sr = lane < kK ? sm.sel_s[lane] : 0.f;
        const bool fixed = __all_sync(0xffffffffu, lane >= kK || (sr >= 0x1p-24f && sr <= 1.0f));
        long long acc = lane < kK && fixed ? score_fx(sr) : 0ll;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        double sum = fixed ? fx_to_double(acc) : 0.0;
        if (!fixed) {
            sum = 0.0;
            for (int r = 0; r < kK; r++) sum += (double)sm.sel_s[r];
        }
        const int kept_e = write_routing(idx_t, w_t, lane, lane < kK ? sm.sel_e[lane] : 0, sr, sum, top_p);
        // the grouping of a single token reads the (possibly dropped) slots
        __syncwarp();
        if (lane < kK) sm.sel_e[lane] = kept_e;
    }
}

// Grouping of a single token's 16 pairs (pair p = slot p) inside its
// routing CTA, warp 0: the experts are distinct, so each kept slot (index
// >= 0; top-p may drop some) has one pair and one work unit; units and perm
// follow increasing expert index.  The decode passes read only the units and
// perm; counts, offsets and the active list are not written.
__device__ void group_one_token(const GroupOut &g, const RouteSmem &sm) {
    const int lane = threadIdx.x & 31;
    const int ei = lane < kK ? sm.sel_e[lane] : -1;
    const int e = ei >= 0 ? ei : 0x7FFFFFFF;
    int rank = 0;
#pragma unroll
    for (int u = 0; u < kK; u++) rank += __shfl_sync(0xffffffffu, e, u) < e;
    if (ei >= 0) {
        g.perm[rank] = lane;
        g.units[3 * rank + 0] = e;
        g.units[3 * rank + 1] = rank;
        g.units[3 * rank + 2] = rank + 1;
    }
    const int kept = __popc(__ballot_sync(0xffffffffu, ei >= 0));
    if (lane == 0) *g.n_units = kept;
}

// CTAs 0..n_tokens-1 route one token each (and, for a single token with a
// work-unit list, group it); the CTAs after them (when x is given) write
// the tokens' x piece images, one warp per 32-column block; the rest build
// the weight tensor maps of the expert table.  The last CTA zeroes the
// stream-K flags and pulls the expert table into L2.
__global__ void __launch_bounds__(kRT)
k_route_prep(int32_t *idx, float *w, const float *logits, const float *bias, int n_tokens,
             const void *x, int x_bf16, uint8_t *ximg, GroupOut g, int *flags, int n_flags,
             const k3mx_expert *experts, int piece_ctas, uint8_t *maps, double top_p,
             const __grid_constant__ CUtensorMap w13, const __grid_constant__ CUtensorMap w2) {
    __shared__ RouteSmem sm;
    // the expert passes may launch now: their prologues overlap this kernel
    pdl_launch_dependents();
    pdl_wait();                          // the logits, when a router pass writes them
    if ((int)blockIdx.x < n_tokens) {
        const int t = blockIdx.x;
        route_cta(logits + (size_t)t * kE, bias, idx + (size_t)t * kK, w + (size_t)t * kK, sm, top_p);
        if (n_tokens == 1 && g.units != nullptr) {
            __syncthreads();
            if (threadIdx.x < 32) group_one_token(g, sm);
        }
        return;
    }
    if (blockIdx.x == gridDim.x - 1) {
        for (int i = threadIdx.x; i < n_flags; i += blockDim.x) flags[i] = 0;
        // the expert pointer table into L2 for the passes' first lookups
        if (experts != nullptr)
            for (int i = threadIdx.x; i < (int)(kE * sizeof(k3mx_expert) / 128); i += blockDim.x)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const uint8_t *>(experts) + 128 * i));
    }
    if ((int)blockIdx.x < n_tokens + piece_ctas)
        ximg_block(x, x_bf16, n_tokens, ximg, (blockIdx.x - n_tokens) * (kRT / 32) + (threadIdx.x >> 5));
    else
        build_maps_cta(maps, kE, experts, k3mx_expert{}, w13, w2, blockIdx.x - n_tokens - piece_ctas);
}

// grouping of n_tokens * 16 <= 1024 pairs in one CTA, launched as a
// programmatic dependent of the routing kernel
__global__ void __launch_bounds__(512) k_group_small(const int32_t *idx, int n_tokens, GroupOut g) {
    __shared__ int cnt[kE];
    __shared__ int tmp[33];
    for (int e = threadIdx.x; e < kE; e += blockDim.x) cnt[e] = 0;
    pdl_wait();
    pdl_launch_dependents();
    __syncthreads();
    const int n_pairs = n_tokens * kK;
    for (int p = threadIdx.x; p < n_pairs; p += blockDim.x) {
        const int e = idx[p];
        if (e >= 0 && e < kE) atomicAdd(&cnt[e], 1);     // -1: a slot dropped by top-p
    }
    __syncthreads();
    finish_counts(cnt, g, tmp);
    if (threadIdx.x < 32) scatter_warp(idx, 0, n_pairs, cnt, g.perm);
}

// per-segment histograms: hist[seg][e]
__global__ void __launch_bounds__(256)
k_group_count(const int32_t *idx, int n_pairs, int *hist, int *status) {
    __shared__ int cnt[kE];
    for (int e = threadIdx.x; e < kE; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int p0 = blockIdx.x * kSeg;
    const int p1 = min(p0 + kSeg, n_pairs);
    for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
        const int e = idx[p];
        if (e >= 0 && e < kE)
            atomicAdd(&cnt[e], 1);
        else if (e != -1)                                 // -1: a slot dropped by top-p
            report_status(status, kStatusBadIndex, p);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kE; e += blockDim.x) hist[(size_t)blockIdx.x * kE + e] = cnt[e];
}

// column sums, offsets, active list, and per-segment starting positions
// within each expert (the scatter adds the expert offsets)
__global__ void __launch_bounds__(1024)
k_group_scan(int *hist, int n_seg, GroupOut g) {
    __shared__ int cnt[kE];
    __shared__ int tmp[33];
    const int e = threadIdx.x;
    constexpr int B = 16;                            // segments per batch of independent loads
    if (e < kE) {
        int c = 0;
        for (int s0 = 0; s0 < n_seg; s0 += B) {
            int h[B];
#pragma unroll
            for (int j = 0; j < B; j++) h[j] = s0 + j < n_seg ? hist[(size_t)(s0 + j) * kE + e] : 0;
#pragma unroll
            for (int j = 0; j < B; j++)
                if (s0 + j < n_seg) {
                    hist[(size_t)(s0 + j) * kE + e] = c;   // within-expert start of segment s0 + j
                    c += h[j];
                }
        }
        cnt[e] = c;
    }
    __syncthreads();
    finish_counts(cnt, g, tmp);                      // offsets: the scatter adds them
}

__global__ void __launch_bounds__(32)
k_group_scatter(const int32_t *idx, int n_pairs, const int *base, const int32_t *offsets, int32_t *perm) {
    __shared__ int running[kE];
    for (int e = threadIdx.x; e < kE; e += 32) running[e] = base[(size_t)blockIdx.x * kE + e] + offsets[e];
    __syncwarp();
    const int p0 = blockIdx.x * kSeg;
    scatter_warp(idx, p0, min(p0 + kSeg, n_pairs), running, perm);
}

}  // namespace

cudaError_t launch_route(const Ctx &c, int32_t *idx, float *w, const float *logits,
                         const float *bias, int n_tokens, double top_p, bool pdl) {
    if (n_tokens > kRouteWarpMax) {
        // many tokens: a CTA per token (its phases are a few dozen
        // instructions each; a warp per token runs 16 dependent rounds)
        const dim3 grid(n_tokens);
        const GroupOut g{};
        if (pdl)
            return launch_pdl(k_route_prep, grid, dim3(kRT), 0, c.stream, idx, w, logits, bias, n_tokens,
                              (const void *)nullptr, 0, (uint8_t *)nullptr, g, (int *)nullptr, 0,
                              (const k3mx_expert *)nullptr, 0, (uint8_t *)nullptr, top_p, CUtensorMap{},
                              CUtensorMap{});
        k_route_prep<<<grid, kRT, 0, c.stream>>>(idx, w, logits, bias, n_tokens, nullptr, 0, nullptr, g, nullptr,
                                                 0, nullptr, 0, nullptr, top_p, CUtensorMap{}, CUtensorMap{});
        return cudaGetLastError();
    }
    const int per_block = 8;
    const dim3 grid((n_tokens + per_block - 1) / per_block);
    if (pdl) return launch_pdl(k_route, grid, dim3(32 * per_block), 0, c.stream, idx, w, logits, bias, n_tokens, top_p);
    k_route<<<grid, 32 * per_block, 0, c.stream>>>(idx, w, logits, bias, n_tokens, top_p);
    return cudaGetLastError();
}

cudaError_t launch_route_prep(const Ctx &c, int32_t *idx, float *w, const float *logits,
                              const float *bias, int n_tokens, const void *x, int x_bf16,
                              uint8_t *ximg, const GroupOut *g_one, int *flags, int n_flags,
                              const k3mx_expert *experts, uint8_t *maps, double top_p, bool pdl) {
    const int piece_ctas = x != nullptr ? (n_tokens * (kD / 32) + kRT / 32 - 1) / (kRT / 32) : 0;
    CUtensorMap w13{}, w2{};
    int map_ctas = 0;
    if (maps != nullptr && experts != nullptr) {
        if (!weight_map_templates(w13, w2)) return cudaErrorNotSupported;
        map_ctas = (kE * kMapsPerExpert + kMapsPerCta - 1) / kMapsPerCta;
    }
    GroupOut g{};
    if (g_one != nullptr && n_tokens == 1) g = *g_one;
    static std::atomic<uint64_t> carveout{0};
    const cudaError_t e = ensure_max_carveout((const void *)k_route_prep, carveout);
    if (e != cudaSuccess) return e;
    const dim3 grid(n_tokens + piece_ctas + map_ctas);
    if (pdl)
        return launch_pdl(k_route_prep, grid, dim3(kRT), 0, c.stream, idx, w, logits, bias, n_tokens, x, x_bf16,
                          ximg, g, flags, flags ? n_flags : 0, experts, piece_ctas, maps, top_p, w13, w2);
    k_route_prep<<<grid, kRT, 0, c.stream>>>(idx, w, logits, bias, n_tokens, x, x_bf16, ximg, g, flags,
                                             flags ? n_flags : 0, experts, piece_ctas, maps, top_p, w13, w2);
    return cudaGetLastError();
}

cudaError_t launch_group_small(const Ctx &c, const int32_t *idx, int n_tokens, const GroupOut &g) {
    return launch_pdl(k_group_small, dim3(1), dim3(512), 0, c.stream, idx, n_tokens, g);
}

size_t group_scratch_bytes(int n_tokens) {
    const size_t n_seg = ((size_t)n_tokens * kK + kSeg - 1) / kSeg;
    return n_seg * kE * sizeof(int);
}

cudaError_t launch_group(const Ctx &c, const int32_t *idx, int n_tokens, const GroupOut &g,
                         void *scratch) {
    const int n_pairs = n_tokens * kK;
    const int n_seg = (n_pairs + kSeg - 1) / kSeg;
    int *hist = static_cast<int *>(scratch);
    k_group_count<<<n_seg, 256, 0, c.stream>>>(idx, n_pairs, hist, c.status);
    k_group_scan<<<1, 1024, 0, c.stream>>>(hist, n_seg, g);
    k_group_scatter<<<n_seg, 32, 0, c.stream>>>(idx, n_pairs, hist, g.offsets, g.perm);
    return cudaGetLastError();
}

}  // namespace k3mx
