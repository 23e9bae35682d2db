/*
 * k3mx.h - C ABI of the MXFP4 routed-expert layer on GB300 (sm_103a).
 *
 * One library, libk3mx.so, computes the Kimi-K3 Stable LatentMoE routed-expert
 * layer straight out of packed MXFP4 weights on one GPU.  Plain pointers and
 * sizes only: every array argument is DEVICE memory owned by the caller unless
 * the function name ends in _host.  Nothing here allocates device memory;
 * scratch comes from a caller-provided workspace whose size the *_workspace_size
 * functions return.
 *
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 * default stream).  The return value reports argument validation and launch
 * errors only.  On any error no kernel has been enqueued and the outputs are
 * untouched.  Device-side bounded waits that give up are reported later by
 * k3mx_device_status().  Arguments are refused, never defaulted: a size or
 * pointer outside what a function documents returns an error code.
 *
 * Kernels are launched as programmatic dependents of the kernel before them
 * on the stream: each may start while that kernel finishes and waits for its
 * results before it reads an input.  The bf16 weight matrices of
 * k3mx_router and k3mx_latent_moe are read before that wait (the first
 * weight tiles go out while the kernel before ends), so they must not be
 * written by the kernel launched immediately before the call on the same
 * stream: put an event wait, a copy or another kernel between.  Every other
 * argument may come from the kernel right before.
 *
 * Co-residency: the one-token decode pass (the routed layer at one token,
 * k3mx_expert_ffn, k3mx_latent_moe at one token) runs one block per SM, and
 * its blocks wait (bounded) for one another's partial results.  If a kernel
 * of another stream holds SMs until those waits give up, the call reports
 * K3MX_ETIMEOUT through k3mx_device_status() instead of a result; nothing
 * faults and the next call is unaffected.  Run it where no other stream's
 * kernels occupy SMs for long (milliseconds), or on its own stream order.
 *
 * Host threads: the library's one-time set-up per device (device
 * properties, kernel attributes, tensor-map templates) is serialised
 * internally, so first calls may come from several threads at once.  Calls
 * that share a workspace, or the fixed array of k3mx_moe_decode_noalloc,
 * must be ordered by the caller (one stream, or events between streams).
 *
 * Weight format (Kimi K3 engine (c/kimi_k3.c), "Weights"): a matrix of
 * `rows` x `in` weights is two arrays, both row-major:
 *   packed [rows][in/2] bytes: e2m1 codes, two per byte, the LOW nibble is
 *          the EVEN column; bit 3 of a code is its sign, bits 2..0 index the
 *          magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6};
 *   scales [rows][in/32] bytes: one ue8m0 byte s per 32 consecutive columns,
 *          weight = code value * 2^(s - 127); s = 255 (NaN) means the group
 *          contributes nothing.
 */
#ifndef K3MX_H_
#define K3MX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Fixed shapes of the routed-expert layer (kimi-k3-in-c README, "2. The
 * config reader that refuses to guess", K3Cfg: n_experts, topk, latent,
 * moe_inter; "Part II" shard census for the byte count). */
#define K3MX_GROUP          32
#define K3MX_N_EXPERTS      896
#define K3MX_TOPK           16
#define K3MX_LATENT         3584        /* D: expert input and output width */
#define K3MX_INTER          3072        /* F: expert intermediate width    */
#define K3MX_EXPERT_BYTES   17547264    /* w1 + w3 + w2, packed + scales    */

/* a cudaStream_t without including CUDA headers */
typedef struct CUstream_st *k3mx_stream_t;

typedef enum k3mx_status {
    K3MX_OK = 0,
    K3MX_EINVAL = 1,      /* NULL pointer, unknown enum value              */
    K3MX_EALIGN = 2,      /* a pointer is not aligned as required          */
    K3MX_ESHAPE = 3,      /* a size outside the documented range           */
    K3MX_EWORKSPACE = 4,  /* workspace NULL or smaller than required       */
    K3MX_ECUDA = 5,       /* a CUDA runtime call or a launch failed        */
    K3MX_ETIMEOUT = 6,    /* a bounded device-side wait gave up            */
    K3MX_EDEVICE = 7      /* the current device is not sm_103              */
} k3mx_status;

/* activation element type */
enum { K3MX_F32 = 0, K3MX_BF16 = 1 };

/* execution path of k3mx_moe_routed */
enum {
    K3MX_PATH_AUTO = 0,       /* PREFILL_MX when x is bf16 and n_tokens >= K3MX_PREFILL_MIN_TOKENS, else DECODE */
    K3MX_PATH_DECODE = 1,     /* fp32 activations; x and h as 8 MXFP4 pieces, kind::mxf4 MMAs   */
    K3MX_PATH_PREFILL = 2,    /* bf16 activations; weights dequantised to f16, kind::f16 MMAs   */
    K3MX_PATH_PREFILL_MX = 3  /* bf16 activations; x, h as 2 MXFP8 pieces, kind::mxf8f6f4 MMAs */
};
#define K3MX_PREFILL_MIN_TOKENS 256
#define K3MX_MAX_TOKENS         65536

/*
 * One routed expert: six device pointers (Kimi K3 engine (c/kimi_k3.c),
 * "Streaming design": the six tensors of an expert; "Architecture notes":
 * GLU experts, inter 3072, in the 3584 latent).  w1 (gate) and w3 (up) are
 * [F x D] = [3072 x 3584]; w2 (down) is [D x F] = [3584 x 3072].  Each
 * pointer must be 16-byte aligned; the PREFILL_MX path of k3mx_moe_routed
 * (and AUTO from K3MX_PREFILL_MIN_TOKENS bf16 tokens) also needs w1, w3
 * and w2 32-byte aligned.  The table lives in device memory, so a violation
 * is found there: the expert's pairs are skipped and k3mx_device_status
 * reports K3MX_EALIGN with the expert's index.
 */
typedef struct k3mx_expert {
    const uint8_t *w1, *s1;     /* gate: packed [F][D/2], scales [F][D/32] */
    const uint8_t *w3, *s3;     /* up:   packed [F][D/2], scales [F][D/32] */
    const uint8_t *w2, *s2;     /* down: packed [D][F/2], scales [D][F/32] */
} k3mx_expert;

/*
 * y[r] = sum_g 2^(s_rg - 127) * sum_{i<32} v(r, 32g+i) * x[32g+i]
 * (kimi-k3-in-c: 2.78 trillion parameters, one CPU, 8 GB of RAM,
 * "Reduction one: the experts already ship at half a byte").
 *   y      [rows] fp32, written (not accumulated)
 *   x      [in] fp32
 *   packed [rows][in/2], scales [rows][in/32] as described above
 *   in     multiple of 32, 32 <= in <= 16384;  1 <= rows <= 2^24
 * y, x, packed must be 16-byte aligned; scales needs no alignment.
 * fp32 products, per-group fp32 sums, fp32 row sums: |error| is within
 * 1e-5 * sum_c |w_rc| |x_c| of the double-accumulated result.
 */
k3mx_status k3mx_gemv(float *y, const float *x, const uint8_t *packed,
                      const uint8_t *scales, int in, int rows,
                      k3mx_stream_t stream);

/*
 * One routed expert, one token (Kimi K3 engine (c/kimi_k3.c), "Architecture
 * notes": SiTU-GLU 4 tanh(g/4) sigma(g) 25 tanh(u/25)):
 *   g = W1 x, u = W3 x, h = SiTU(g, u), y = W2 h.
 *   y [3584] fp32 (written), x [3584] fp32, *expert a HOST struct of device
 *   pointers.  workspace: device, >= k3mx_expert_ffn_workspace_size() bytes,
 *   256-byte aligned; it begins with g and u ([2][3072] fp32, written),
 *   followed by the pieces of x and h and per-CTA tensor-map slots.
 * The multiplies run on the tensor cores with MXFP4 operands (kind::mxf4):
 * x and h are each split exactly into eight MXFP4 vectors plus a residual
 * of at most 4^-8 of the largest magnitude of its 32-column block, and the
 * tensor cores accumulate in fp32: g, u within 1e-5 * sum_c |w_rc| |x_c|.
 */
size_t k3mx_expert_ffn_workspace_size(void);
k3mx_status k3mx_expert_ffn(float *y, const float *x, const k3mx_expert *expert,
                            void *workspace, size_t ws_bytes,
                            k3mx_stream_t stream);

/*
 * Router selection (Kimi K3 engine (c/kimi_k3.c), "Architecture notes",
 * Stable LatentMoE; kimi-k3-in-c README, "Three invariants", item 3), per
 * token t:  s_e = sigma(logit_e) (double, rounded to fp32 once);
 * key_e = s_e + bias_e (fp32); idx = the 16 largest keys, ties to the lower
 * expert index, in key-descending order; w_k = s_{idx_k} / sum_j s_{idx_j}
 * (double, rounded to fp32) * routed_scale (1.0).
 *   idx [n_tokens][16] int32, w [n_tokens][16] fp32 (written)
 *   logits [n_tokens][896] fp32, bias [896] fp32
 *   1 <= n_tokens <= K3MX_MAX_TOKENS
 * Index results are bit-identical to a CPU evaluation in the same precision.
 */
k3mx_status k3mx_route_topk(int32_t *idx, float *w, const float *logits,
                            const float *bias, int n_tokens,
                            k3mx_stream_t stream);

/*
 * k3mx_route_topk followed by the top-p truncation (Kimi K3 engine
 * (c/kimi_k3.c), "Streaming design": K3_TOPP keeps the routed experts up to
 * a cumulative weight p, dropping the low-weight tail of the top-16 and
 * renormalising the rest).  Per token, the 16 selected experts are taken in
 * order of decreasing raw score s (ties: lower expert index); an expert is
 * kept while the scores ahead of it sum to less than top_p times the sum of
 * all 16 (the shortest prefix reaching top_p); a kept slot's weight is
 * s / (sum of the kept scores) (double, rounded to fp32) * routed_scale; a
 * dropped slot gets index -1 and weight 0 and keeps its place.  The sums
 * are exact (scores in [2^-24, 1]) or slot-order double sums.
 *   top_p: finite; top_p <= 0 keeps all 16 (the same result as
 *          k3mx_route_topk), top_p >= 1 keeps all 16; NaN or Inf is
 *          refused (K3MX_EINVAL).  Other arguments as k3mx_route_topk.
 * Index results are bit-identical to a CPU evaluation in the same precision.
 */
k3mx_status k3mx_route_topp(int32_t *idx, float *w, const float *logits,
                            const float *bias, int n_tokens, float top_p,
                            k3mx_stream_t stream);

/*
 * The router and its top-16 (Kimi K3 engine (c/kimi_k3.c), "Architecture
 * notes", Stable LatentMoE: a sigmoid router [896, 7168] over the hidden
 * state; the trunk, router included, is bf16):
 *   logits[t][e] = sum_c router_w[e][c] * hidden[t][c]        (fp32 sums)
 * followed by the routing of k3mx_route_topk (top_p > 0: k3mx_route_topp)
 * on those logits.
 *   logits [n_tokens][896] fp32 (written)
 *   idx [n_tokens][16] int32, w [n_tokens][16] fp32 (written)
 *   hidden [n_tokens][7168], h_dtype K3MX_F32 or K3MX_BF16
 *   router_w [896][7168] bf16 bit patterns, row-major; bias [896] fp32
 *   top_p: finite (<= 0: off); 1 <= n_tokens <= K3MX_MAX_TOKENS
 * All pointers device, 16-byte aligned.  Each logit is within
 * 1e-5 * sum_c |router_w[e][c] hidden[t][c]| of the exact sum; idx and w
 * are exactly the routing of the logits written.
 */
k3mx_status k3mx_router(float *logits, int32_t *idx, float *w, const void *hidden, int h_dtype,
                        const uint16_t *router_w, const float *bias, int n_tokens, float top_p,
                        k3mx_stream_t stream);

/*
 * The Stable LatentMoE block around the routed experts (Kimi K3 engine
 * (c/kimi_k3.c), "Architecture notes"; K3Cfg n_shared 2 "full width, added
 * UNWEIGHTED", latent_norm 1 "RMSNorm on the AGGREGATE", rms_eps 1e-5):
 *   logits = router h                          (k3mx_router's product)
 *   x      = w_dn h                            (7168 -> 3584)
 *   r      = sum_k w_k expert_k(x)             (k3mx_moe_routed on x, logits)
 *   y      = w_up (RMSNorm(r) * g_norm) + w2s SiTU-GLU(w1s h, w3s h)
 * All matrices bf16 (bit patterns), row-major; the structure holds device
 * pointers and lives on the host.
 */
typedef struct {
    const uint16_t *router_w;    /* [896][7168] */
    const float *bias;           /* [896] score-correction bias */
    const uint16_t *w_dn;        /* [3584][7168] */
    const uint16_t *w_up;        /* [7168][3584] */
    const uint16_t *g_norm;      /* [3584] RMSNorm weight of the routed sum */
    const uint16_t *w1s, *w3s;   /* [6144][7168] fused shared experts: gate, up */
    const uint16_t *w2s;         /* [7168][6144] fused shared experts: down */
} k3mx_latent_block;

/*
 *   y [n_tokens][7168] fp32 (written); hidden [n_tokens][7168], h_dtype
 *   K3MX_F32 or K3MX_BF16; experts as for k3mx_moe_routed; top_p as for
 *   k3mx_route_topp (<= 0: off); idx_out, w_out optional [n_tokens][16].
 * fp32 states or up to 16 bf16 ones run in fp32 on CUDA cores (the routed
 * part on the DECODE path); from 17 bf16 states the products run on the
 * tensor cores with bf16 operands (x, SiTU(g, u) and the normalised sum
 * rounded to bf16) and the routed part takes its bf16 default path.
 * Numerics: per token, |y - exact| / |exact| (L2) is at most 1e-4 with fp32
 * states (measured ~5e-7) and 1e-2 with bf16 batches (measured ~7e-3, the
 * bf16 rounding of the intermediates).  workspace: device,
 * 256-byte aligned, >= k3mx_latent_moe_workspace_size(n_tokens, h_dtype).
 */
size_t k3mx_latent_moe_workspace_size(int n_tokens, int h_dtype);
k3mx_status k3mx_latent_moe(float *y, const void *hidden, int h_dtype, int n_tokens,
                            const k3mx_latent_block *blk, const k3mx_expert *experts, float top_p,
                            int32_t *idx_out, float *w_out, void *workspace, size_t ws_bytes,
                            k3mx_stream_t stream);

/*
 * Token-to-expert grouping (Kimi K3 engine (c/kimi_k3.c), "Chunked prefill":
 * each unique expert of a chunk is loaded once for all its tokens):
 *   counts [896]          pairs routed to each expert
 *   offsets [897]         exclusive prefix sum of counts, offsets[896] = 16 T
 *   perm [16 T]           pair indices p = t*16 + k sorted by (expert, p)
 *   idx [n_tokens][16]    int32 expert ids in 0..895, or -1 for a slot
 *                         dropped by top-p (not grouped); other entries are
 *                         clamped out: they are not counted and the device
 *                         status reports K3MX_EINVAL
 * Bit-exact and deterministic.  workspace: device, 16-byte aligned,
 * >= k3mx_group_workspace_size(n_tokens) bytes.
 */
size_t k3mx_group_workspace_size(int n_tokens);
k3mx_status k3mx_group(int32_t *counts, int32_t *offsets, int32_t *perm,
                       const int32_t *idx, int n_tokens,
                       void *workspace, size_t ws_bytes,
                       k3mx_stream_t stream);

/*
 * The routed-expert layer: route, group, run the selected experts, and form
 * y_t = sum_k w_tk * expert_{idx_tk}(x_t) (Kimi K3 engine (c/kimi_k3.c),
 * "Architecture notes", Stable LatentMoE).
 *   y        [n_tokens][3584] fp32 (written)
 *   x        [n_tokens][3584], fp32 (x_dtype K3MX_F32) or bf16 bits (K3MX_BF16)
 *   experts  DEVICE array of 896 k3mx_expert
 *   logits   [n_tokens][896] fp32, bias [896] fp32
 *   path     K3MX_PATH_*; PREFILL and PREFILL_MX require bf16 x
 *   idx_out, w_out: optional DEVICE arrays [n_tokens][16] (NULL to skip)
 *            receiving the routing result
 *   workspace: device, 256-byte aligned, >= k3mx_moe_workspace_size(...)
 * DECODE runs the tensor-core multiplies of k3mx_expert_ffn (x and h as
 * eight exact MXFP4 pieces, fp32 accumulation): |error| within 1e-5 of the
 * abs-weighted sums.
 * PREFILL converts x (bf16) to f16, dequantises the
 * weights to f16, rounds h to f16 and multiplies f16 x f16 on the tensor
 * cores with fp32 accumulation: per-token relative L2 error within 1e-2.
 * PREFILL_MX splits x and h (h from a hardware-tanh SiTU, staged as f16
 * under a power-of-two scale per 32-column block) into two MXFP8 (e4m3)
 * pieces per 32-column block (two pieces reproduce a bf16 x exactly, and h
 * to about 2^-9 of each value) and multiplies them with the weights as
 * stored (e2m1 codes and ue8m0 scales, kind::mxf8f6f4) with fp32
 * accumulation: per-token relative L2
 * error within 1e-2 (about 3e-4 on the synthetic workload).  DECODE is
 * deterministic; both prefill paths add the 16 expert contributions of a
 * token with fp32 atomics, so the order of those adds, and the last bits
 * of y, may vary between runs.
 */
size_t k3mx_moe_workspace_size(int n_tokens, int x_dtype, int path);
k3mx_status k3mx_moe_routed(float *y, const void *x, int x_dtype, int n_tokens,
                            const k3mx_expert *experts, const float *logits,
                            const float *bias, int path,
                            int32_t *idx_out, float *w_out,
                            void *workspace, size_t ws_bytes,
                            k3mx_stream_t stream);

/*
 * k3mx_moe_routed with the top-p routing of k3mx_route_topp: dropped slots
 * run no expert (idx_out -1, w_out 0).  top_p <= 0 or >= 1: the same result
 * as k3mx_moe_routed.  Workspace: k3mx_moe_workspace_size(...).
 */
k3mx_status k3mx_moe_routed_topp(float *y, const void *x, int x_dtype, int n_tokens,
                                 const k3mx_expert *experts, const float *logits,
                                 const float *bias, int path, float top_p,
                                 int32_t *idx_out, float *w_out,
                                 void *workspace, size_t ws_bytes,
                                 k3mx_stream_t stream);

/*
 * k3mx_moe_routed with HOST activations, logits, bias and output: copies
 * x, logits and bias to the workspace, runs the layer, copies y back, and
 * waits for the stream.  Weights (experts) stay DEVICE-resident.  Host
 * buffers may be pageable.  On the DECODE path, when all four buffers are
 * page-locked, mapped into the device's address space and 16-byte aligned,
 * the kernels read x, logits and bias and write y in place instead (no
 * copies; the same results).
 *   workspace: >= k3mx_moe_host_workspace_size(...) bytes.
 */
size_t k3mx_moe_host_workspace_size(int n_tokens, int x_dtype, int path);
k3mx_status k3mx_moe_routed_host(float *y_host, const void *x_host, int x_dtype,
                                 int n_tokens, const k3mx_expert *experts,
                                 const float *logits_host, const float *bias_host,
                                 int path, void *workspace, size_t ws_bytes,
                                 k3mx_stream_t stream);

/*
 * The DECODE path of k3mx_moe_routed without a caller workspace: the pages
 * have no counterpart; it serves callers that cannot allocate device memory
 * at the point of the call: a runtime that owns the whole device memory
 * budget and hands the library no scratch, or a latency-critical loop that
 * must not take the synchronisation an allocation can imply.  Its scratch is
 * one fixed array in
 * the library's device memory, 8 MiB, enough for K3MX_NOALLOC_MAX_TOKENS
 * tokens.  Arguments as for k3mx_moe_routed with path DECODE.
 *   1 <= n_tokens <= K3MX_NOALLOC_MAX_TOKENS, else K3MX_ESHAPE.
 * The first call on each device looks up that array's address (with the
 * device current); make that first call before any stream capture.
 * Calls that overlap on the GPU (concurrent streams, or several host
 * threads) share the one array and race: serialise them on one stream.
 * Results are bit-identical to k3mx_moe_routed with path DECODE.
 */
#define K3MX_NOALLOC_MAX_TOKENS 8
k3mx_status k3mx_moe_decode_noalloc(float *y, const void *x, int x_dtype,
                                    int n_tokens, const k3mx_expert *experts,
                                    const float *logits, const float *bias,
                                    int32_t *idx_out, float *w_out,
                                    k3mx_stream_t stream);

/*
 * Waits for `stream`, then reports and clears the device status word: K3MX_OK,
 * K3MX_ETIMEOUT when a bounded device-side wait gave up since the last call,
 * K3MX_EINVAL when a device-side range check rejected an index, K3MX_EALIGN
 * when a weight pointer read from a device expert table is not 16-byte
 * aligned (that expert's work is skipped), or K3MX_ECUDA
 * when the stream reports a CUDA error.  `detail` (may be NULL) receives a
 * kernel-specific code of the first failure.
 */
k3mx_status k3mx_device_status(k3mx_stream_t stream, int *detail);

/*
 * The limit of the library's bounded device-side waits, a diagnostic aid
 * with no counterpart on the pages.  Every kernel's waits for work (on a
 * pipeline barrier, or on a flag another CTA sets) give up after `polls`
 * polls (each at most a few microseconds) and report K3MX_ETIMEOUT through
 * k3mx_device_status; the CTA then waits for its own copies in flight and
 * its MMAs with the default limit, frees its tensor memory and returns, so
 * the context stays usable and the next call runs normally.  polls = 0
 * restores the default (2^22 polls, seconds); larger values are clamped to
 * it.  Applies to the current device, from the next launch on; outputs of a
 * call whose wait gave up are unspecified.  Waits for the device.
 */
k3mx_status k3mx_set_wait_limit(unsigned int polls);

/*
 * Launch tracing, a measurement aid with no counterpart on the pages.  While
 * enabled, every kernel launch group the library issues is bracketed by a
 * pair of CUDA events recorded on the caller's stream, so durations are
 * those of the kernels themselves.  k3mx_trace_read waits for the recorded
 * events, writes one entry per kernel name (launch count and summed
 * milliseconds, at most max_entries), clears the record and returns the
 * number of entries.  Not for streams under graph capture; not thread-safe.
 * Events come from a fixed pool of 8192 pairs: launches beyond it are not
 * traced.
 */
typedef struct k3mx_trace_entry {
    char name[32];
    int launches;
    double total_ms;
} k3mx_trace_entry;
k3mx_status k3mx_trace_enable(int on);
int k3mx_trace_read(k3mx_trace_entry *out, int max_entries);

/* a static string naming a status code */
const char *k3mx_status_str(k3mx_status status);

/* the name of the last CUDA error that a call made on this host thread
 * reported as K3MX_ECUDA ("cudaSuccess" if none); a static string */
const char *k3mx_last_cuda_error(void);

/* version of this ABI, (major << 16) | minor */
int k3mx_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* K3MX_H_ */
