// route_group.cu - router top-16 selection and token-to-expert grouping.
//
// Routing (Kimi K3 engine (c/kimi_k3.c), "Architecture notes", Stable
// LatentMoE; kimi-k3-in-c README, "Three invariants", item 3): the score is
// sigma(logit), the selection key is score + bias, the top 16 keys win, and
// the combining weights are the selected raw scores renormalised.
//   - sigma is evaluated in double and rounded to fp32 once, so the fp32
//     score, key and selection agree bit for bit with a CPU evaluation in the
//     same precision;
//   - equal keys go to the lower expert index: each key is packed with the
//     complemented index into one 64-bit word and the warp takes maxima;
//   - -0 counts as +0 and a NaN key ranks below every number.
// One warp per token: lane l holds experts l, l+32, ..., 28 keys in
// registers; 16 rounds of a warp max pick the winners in key order.
//
// Grouping (Kimi K3 engine (c/kimi_k3.c), "Chunked prefill": every unique
// expert of a chunk is loaded once for all its tokens): counts per expert,
// exclusive offsets, and the pair list sorted by (expert, pair index).  The
// counts come from shared-memory integer atomics (order-free); the placement
// is a stable warp-sequential scatter, so the output is deterministic.
#include "common.cuh"

namespace k3mx {
namespace {

constexpr float kRoutedScale = 1.0f;     // K3Cfg routed_scale
constexpr int kPer = kE / 32;            // 28 experts per lane
constexpr int kSeg = 4096;               // pairs per grouping segment

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

__device__ __forceinline__ float canon_key(float k) {
    if (k != k) return -INFINITY;        // NaN ranks last
    if (k == 0.0f) return 0.0f;          // -0 -> +0
    return k;
}

__device__ __forceinline__ float key_of_order(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// the lane's best remaining key packed with its complemented expert index
__device__ __forceinline__ unsigned long long lane_best(const uint32_t (&ok)[kPer], int lane) {
    uint32_t b = 0;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        if (ok[i] > b) {            // strict: equal keys keep the lower index
            b = ok[i];
            bi = i;
        }
    }
    return ((unsigned long long)b << 32) | (0xFFFFFFFFu - (uint32_t)(lane + 32 * bi));
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, m, o);
        m = other > m ? other : m;
    }
    return m;
}

__device__ __forceinline__ void write_routing(int32_t *idx_t, float *w_t, int lane, int my_e,
                                              float my_s, double sum) {
    if (lane < kK) {
        idx_t[lane] = my_e;
        w_t[lane] = (float)((double)my_s / sum) * kRoutedScale;
    }
}

// Exact selection over all 896 experts (used when the candidate filter
// below would keep more than 64 experts, e.g. with many equal or NaN keys).
__device__ void route_warp_all(const float *__restrict__ lt, const float *__restrict__ bias,
                               int32_t *__restrict__ idx_t, float *__restrict__ w_t, int lane) {
    uint32_t ok[kPer];
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const int e = lane + 32 * i;
        ok[i] = order_key(exact_score(__ldg(lt + e)) + __ldg(bias + e));
    }
    unsigned long long best = lane_best(ok, lane);
    float my_s = 0.f;
    int my_e = 0;
    double sum = 0.0;
#pragma unroll 1
    for (int k = 0; k < kK; k++) {
        const unsigned long long m = warp_max_u64(best);
        const int e = (int)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFull));
        const int owner = e & 31, slot = e >> 5;
        float s_win = 0.f;
        if (lane == owner) {
#pragma unroll
            for (int i = 0; i < kPer; i++)
                if (i == slot) ok[i] = 0;
            best = lane_best(ok, lane);
            s_win = exact_score(__ldg(lt + e));
        }
        s_win = __shfl_sync(0xffffffffu, s_win, owner);
        sum += (double)s_win;                       // slot order, as on the CPU
        if (lane == k) {
            my_s = s_win;
            my_e = e;
        }
    }
    write_routing(idx_t, w_t, lane, my_e, my_s, sum);
}

// One token on one warp.  (1) fp32 estimates of all 896 keys; (2) the 16th
// largest estimate a16; (3) every expert whose estimate is within
// 2^-18 * max(1,|a16|) of a16 is a candidate: an expert of the exact top 16
// cannot lie further below (each estimate is within 2^-20 * max(1,|key|) of
// its exact key, and the 16th order statistic moves by no more than that);
// (4) exact keys for the candidates only, and the exact top-16 among them.
// `scratch` is 128 ints of shared memory for this warp.
__device__ void route_warp(const float *__restrict__ lt, const float *__restrict__ bias,
                           int32_t *__restrict__ idx_t, float *__restrict__ w_t, int lane,
                           int *scratch) {
    float ak[kPer];
    uint32_t ok[kPer];
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const int e = lane + 32 * i;
        ak[i] = canon_key(approx_score(__ldg(lt + e)) + __ldg(bias + e));
        ok[i] = order_key(ak[i]);
    }
    unsigned long long best = lane_best(ok, lane);
    unsigned long long m16 = 0;
#pragma unroll 1
    for (int k = 0; k < kK; k++) {
        const unsigned long long m = warp_max_u64(best);
        const int e = (int)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFull));
        if (lane == (e & 31)) {
#pragma unroll
            for (int i = 0; i < kPer; i++)
                if (i == (e >> 5)) ok[i] = 0;
            best = lane_best(ok, lane);
        }
        m16 = m;
    }
    const float a16 = key_of_order((uint32_t)(m16 >> 32));
    // a non-finite a16 (infinite biases) keeps every expert: exact path
    const float tau = isfinite(a16) ? a16 - 0x1p-18f * fmaxf(1.0f, fabsf(a16)) : -INFINITY;

    // candidates into a compact per-warp list (at most 64)
    const unsigned lt_mask = (1u << lane) - 1u;
    int n = 0;
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const bool c = ak[i] >= tau;
        const unsigned bm = __ballot_sync(0xffffffffu, c);
        const int pos = n + __popc(bm & lt_mask);
        if (c && pos < 64) scratch[pos] = lane + 32 * i;
        n += __popc(bm);
    }
    __syncwarp();
    if (n > 64) {
        route_warp_all(lt, bias, idx_t, w_t, lane);
        return;
    }
    // exact keys: lane holds candidates lane and lane + 32
    unsigned long long ck[2];
    float cs[2];
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const int pos = lane + 32 * j;
        ck[j] = 0;
        cs[j] = 0.f;
        if (pos < n) {
            const int e = scratch[pos];
            cs[j] = exact_score(__ldg(lt + e));
            ck[j] = ((unsigned long long)order_key(cs[j] + __ldg(bias + e)) << 32) |
                    (0xFFFFFFFFu - (uint32_t)e);
        }
    }
    __syncwarp();
    float my_s = 0.f;
    int my_e = 0;
    double sum = 0.0;
#pragma unroll 1
    for (int k = 0; k < kK; k++) {
        const unsigned long long mine = ck[0] > ck[1] ? ck[0] : ck[1];
        const unsigned long long m = warp_max_u64(mine);
        const int e = (int)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFull));
        float s_win = 0.f;
#pragma unroll
        for (int j = 0; j < 2; j++)
            if (ck[j] == m) {
                s_win = cs[j];
                ck[j] = 0;
            }
        // packed keys are unique (they carry the index): one lane owns m
        const int owner = __ffs(__ballot_sync(0xffffffffu, mine == m)) - 1;
        s_win = __shfl_sync(0xffffffffu, s_win, owner);
        sum += (double)s_win;                       // slot order, as on the CPU
        if (lane == k) {
            my_s = s_win;
            my_e = e;
        }
    }
    write_routing(idx_t, w_t, lane, my_e, my_s, sum);
}

__global__ void __launch_bounds__(256) k_route(int32_t *idx, float *w, const float *logits,
                                               const float *bias, int n_tokens) {
    __shared__ int scratch[8][128];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = blockIdx.x * (blockDim.x / 32) + warp;
    if (t >= n_tokens) return;
    route_warp(logits + (size_t)t * kE, bias, idx + (size_t)t * kK, w + (size_t)t * kK, lane,
               scratch[warp]);
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
    const int lane = threadIdx.x % 32;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = p_begin; base < p_end; base += 32) {
        const int p = base + lane;
        int e = -1;
        if (p < p_end) {
            e = idx[p];
            if (e < 0 || e >= kE) e = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt_mask);
        if (e >= 0) perm[running[e] + rank] = p;
        __syncwarp();
        if (e >= 0 && rank == 0) running[e] += __popc(peers);
        __syncwarp();
    }
}

// route + group for n_tokens * 16 <= 1024 pairs, one 512-thread CTA
__global__ void __launch_bounds__(512)
k_route_group_small(int32_t *idx, float *w, const float *logits, const float *bias,
                    int n_tokens, GroupOut g) {
    __shared__ int cnt[kE];
    __shared__ int tmp[33];
    __shared__ int scratch[16][128];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = blockDim.x / 32;
    for (int t = warp; t < n_tokens; t += nwarps)
        route_warp(logits + (size_t)t * kE, bias, idx + (size_t)t * kK, w + (size_t)t * kK, lane,
                   scratch[warp]);
    for (int e = threadIdx.x; e < kE; e += blockDim.x) cnt[e] = 0;
    __syncthreads();                         // idx written by this block is visible
    const int n_pairs = n_tokens * kK;
    for (int p = threadIdx.x; p < n_pairs; p += blockDim.x) atomicAdd(&cnt[idx[p]], 1);
    __syncthreads();
    finish_counts(cnt, g, tmp);
    if (warp == 0) scatter_warp(idx, 0, n_pairs, cnt, g.perm);
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
        else
            report_status(status, kStatusBadIndex, p);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kE; e += blockDim.x) hist[(size_t)blockIdx.x * kE + e] = cnt[e];
}

// column sums, offsets, active list, and per-segment starting positions
__global__ void __launch_bounds__(1024)
k_group_scan(int *hist, int n_seg, GroupOut g) {
    __shared__ int cnt[kE];
    __shared__ int tmp[33];
    const int e = threadIdx.x;
    if (e < kE) {
        int c = 0;
        for (int s = 0; s < n_seg; s++) {
            const int h = hist[(size_t)s * kE + e];
            hist[(size_t)s * kE + e] = c;            // within-expert start of segment s
            c += h;
        }
        cnt[e] = c;
    }
    __syncthreads();
    finish_counts(cnt, g, tmp);
    if (e < kE)
        for (int s = 0; s < n_seg; s++) hist[(size_t)s * kE + e] += cnt[e];
}

__global__ void __launch_bounds__(32)
k_group_scatter(const int32_t *idx, int n_pairs, const int *base, int32_t *perm) {
    __shared__ int running[kE];
    for (int e = threadIdx.x; e < kE; e += 32) running[e] = base[(size_t)blockIdx.x * kE + e];
    __syncwarp();
    const int p0 = blockIdx.x * kSeg;
    scatter_warp(idx, p0, min(p0 + kSeg, n_pairs), running, perm);
}

}  // namespace

cudaError_t launch_route(const Ctx &c, int32_t *idx, float *w, const float *logits,
                         const float *bias, int n_tokens) {
    const int per_block = 8;
    k_route<<<(n_tokens + per_block - 1) / per_block, 32 * per_block, 0, c.stream>>>(
        idx, w, logits, bias, n_tokens);
    return cudaGetLastError();
}

cudaError_t launch_route_group_small(const Ctx &c, int32_t *idx, float *w, const float *logits,
                                     const float *bias, int n_tokens, const GroupOut &g) {
    k_route_group_small<<<1, 512, 0, c.stream>>>(idx, w, logits, bias, n_tokens, g);
    return cudaGetLastError();
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
    k_group_scatter<<<n_seg, 32, 0, c.stream>>>(idx, n_pairs, hist, g.perm);
    return cudaGetLastError();
}

}  // namespace k3mx
