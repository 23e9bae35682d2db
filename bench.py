"""Benchmark of the MXFP4 routed-expert layer on GB300.

One JSON line on rank 0.  A step is one pass of the layer over one batch of
synthetic tokens through the public C ABI (k3mx_moe_routed): routing,
grouping, the selected experts and the weighted sum.  The headline workload
is the batch-1 decode step: all 896 experts (15.72 GB of packed MXFP4)
resident in HBM, one fp32 token per step with fresh seeded router logits, so
every step streams 16 different experts (280.8 MB).  `value` is expert bytes
streamed per second (GB/s); the line also carries the batch-64 decode and
4096-token prefill workloads under "secondary".

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
  python bench.py --profile-case decode|prefill|router|latent --tokens T [--resident R]
                  [--confine] [--mx] [--iters I]

The --profile-case form runs a small case of one path for Nsight Compute
captures (a few GB on the device): R experts (default 64, 1.1 GB, larger
than L2) behind the full 896-entry table (entry e -> expert e mod R), I
calls with fresh logits, then prints the device status.  With --confine the
bias keeps routing on the R resident experts, so each expert a launch
touches is a distinct one, as in the full workload.

Timing: one CUDA event pair on the launching stream around the K timed
steps, with a few milliseconds of device work queued ahead of them so that
the host's launches run ahead of the device and the events time device
work, not host launch latency (which the end-to-end figure "e2e" includes).  The inputs
of every step are larger than L2 (129 MB): a decode step streams 16 experts
it has not just used (280.8 MB; 10.7 GB at batch 64), a prefill step all
15.7 GB, so L2 is not flushed between timed steps; the batch-1 line also
reports the same steps with L2 flushed by a 256 MB write between them
("l2_flushed"), which adds the write-back of that buffer's dirty lines and
cold instruction and table fetches to every step.
N > 1 runs independent replicas, one per GPU (weak scaling), timed between
barriers; rank 0 reports the maximum over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP4 expert GB/s (% HBM peak) at decode; prefill tokens/s per MoE layer"
EXPERT_BYTES = 17547264
GATE_UP_BYTES = 2 * (5505024 + 344064)          # w1 + w3 of one expert, packed + scales
D, F, E, K = 3584, 3072, 896, 16
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# kernels per traced launch group
KERNELS_PER_GROUP = {"router": 1, "hidden_products": 1, "latent_out": 1, "latent_down": 1, "shared_gate_up": 1, "shared_down": 2, "latent_up": 2,
                     "route": 1, "group_small": 1, "group": 3, "mx_pieces": 1,
                     "decode_expert": 1, "decode_gate_up": 1, "decode_down": 1, "combine": 1,
                     "prefill_prep": 3, "prefill_gate_up": 1, "prefill_down": 1}
PARAMS_PER_EXPERT = 33030144
X_IMAGE_BYTES = 8 * 3584 // 2 + 3584          # 8 MXFP4 pieces of x and their scale lines
H_IMAGE_BYTES = 8 * 3072 // 2 + 3072
GATE_UP_PARAMS = 2 * 3072 * 3584


# the sources of each profiled kernel: a committed DRAM-traffic figure is
# reported only while these are unchanged
DECODE_SOURCES = ["mx.cu", "common.cuh", "pieces.cuh", "tc.cuh", "tmaps.cuh"]
PREFILL_SOURCES = ["prefill.cu", "prefill.cuh", "common.cuh"]
PREFILL_MX_SOURCES = ["px.cu", "prefill.cuh", "tc.cuh", "pieces.cuh", "common.cuh", "tmaps.cuh"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", FALLBACK_HBM_GBS), d.get("bf16_tflops", FALLBACK_BF16_TFLOPS), \
            d.get("bf16_tflops_sustained"), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "mxfp4_routed_expert_k3mx_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload, src_hash):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(f"{kernel}/{workload}")
    if not rec or rec.get("source_hash") != src_hash:
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock and throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ oracle --

def oracle_decode_sample(steps_inputs, budget_s, max_tokens, seed=0):
    """The CPU oracle on decode tokens of the workload until `budget_s`
    seconds of oracle work: returns (expert bytes, seconds, tokens, cores).
    Expert bytes are drawn on the host first, outside the timed part."""
    import numpy as np
    import oracle
    import synth
    total_s, nbytes, tokens = 0.0, 0, 0
    for x, logits, bias in steps_inputs:
        if total_s >= budget_s or tokens >= max_tokens:
            break
        idx, w = oracle.route(logits, bias)
        experts = {int(e): synth.split_expert(synth.expert(int(e), seed=seed)) for e in np.unique(idx)}
        t0 = time.perf_counter()
        oracle.moe(x, idx, w, experts)
        total_s += time.perf_counter() - t0
        nbytes += len(experts) * EXPERT_BYTES
        tokens += x.shape[0]
    return nbytes, total_s, tokens, oracle.num_threads()


def decode_inputs(step, T, seed_base=1000):
    """Token activations and router logits of one step.  Batch 1 carries the
    score-correction bias N(0, 0.1); batched workloads route flat (no bias)."""
    import numpy as np
    import synth
    x = synth.token_inputs(T, seed=seed_base + step)
    logits, _ = synth.router_inputs(T, seed=seed_base + step)
    if T == 1:
        _, bias = synth.router_inputs(1, seed=0)
    else:
        bias = np.zeros(E, np.float32)
    return x, logits, bias


def reduce_over_ranks(dist, total_ms, nbytes, device=None):
    """Whole-job figures of a timed region: the slowest rank's time and the
    bytes all ranks streamed.  `dist` is torch.distributed (or None for one
    rank)."""
    if dist is None:
        return float(total_ms), float(nbytes)
    import torch
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    b = torch.tensor([float(nbytes)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t[0]), float(b[0])


def run_reference(args):
    """--impl reference: the CPU oracle, as it stands, on the machine's host cores."""
    steps = [decode_inputs(i, 1) for i in range(args.warmup + args.steps)]
    # warm-up steps: one token each, untimed
    oracle_decode_sample(steps[:args.warmup], 1e9, args.warmup)
    nbytes, secs, tokens, cores = oracle_decode_sample(steps[args.warmup:], 1e9, args.steps)
    v = nbytes / secs / 1e9
    line = {
        "metric": METRIC, "value": round(v, 3), "unit": "GB/s", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "moe_decode_b1", "tokens_per_step": 1, "n_experts": E, "topk": K,
                   "latent": D, "inter": F},
        "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{tokens} decode tokens x 16 experts (one token per step)"},
        "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- GPU steps --

class Workload:
    def __init__(self, name, T, x_bf16, path):
        self.name, self.T, self.x_bf16, self.path = name, T, x_bf16, path


def prepare(wl, n_steps, dev):
    import numpy as np
    import torch
    import synth
    xs, lgs = [], []
    for i in range(n_steps):
        x, logits, bias = decode_inputs(i, wl.T)
        if wl.x_bf16:
            xb = synth.f32_to_bf16(x)
            xs.append(torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev))
        else:
            xs.append(torch.from_numpy(x).to(dev))
        lgs.append(torch.from_numpy(logits).to(dev))
    return xs, lgs, torch.from_numpy(bias).to(dev)


def device_ahead(torch, n_steps, host_ms_per_step=0.25):
    """Queue a spin kernel of a few milliseconds (outside the events) so that
    the host enqueues the following steps while the device is still busy:
    the events then time the steps' device work back to back rather than the
    pace of the host's launches."""
    ms = max(2.0, n_steps * host_ms_per_step)
    torch.cuda._sleep(int(ms * 1e-3 * 2.1e9))


def time_workload(k3mx, wl, table, dev, steps, warmup, dist, flush):
    """Device-timed steps: returns dict of timings and trace."""
    import torch
    xs, lgs, bias = prepare(wl, warmup + steps, dev)
    T = wl.T
    dt = k3mx.K3MX_BF16 if wl.x_bf16 else k3mx.K3MX_F32
    ws = torch.empty(k3mx.k3mx_moe_workspace_size(T, dt, wl.path), dtype=torch.uint8, device=dev)
    y = torch.empty((T, D), dtype=torch.float32, device=dev)
    idx = torch.empty((steps, T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(warmup):
        k3mx.k3mx_moe_routed(y, xs[i], table, lgs[i], bias, ws, path=wl.path, idx_out=idx[0], w_out=w)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # timed steps: one event pair around all of them, so consecutive steps
    # follow each other as they would in a run (the library chains its
    # kernels as programmatic dependents, which an event between steps
    # would serialise); with an L2 flush between steps (outside the events)
    # an event pair around each step instead
    device_ahead(torch, steps)
    if flush is None:
        ev[0][0].record(stream)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
            ev[i][0].record(stream)
        k3mx.k3mx_moe_routed(y, xs[warmup + i], table, lgs[warmup + i], bias, ws, path=wl.path,
                             idx_out=idx[i], w_out=w)
        if flush is not None:
            ev[i][1].record(stream)
    if flush is None:
        ev[0][1].record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    # the same steps again with an event pair around every kernel launch:
    # per-kernel durations
    k3mx.k3mx_trace_read()
    device_ahead(torch, steps)
    k3mx.k3mx_trace_enable(True)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        k3mx.k3mx_moe_routed(y, xs[warmup + i], table, lgs[warmup + i], bias, ws, path=wl.path,
                             idx_out=idx[i], w_out=w)
    torch.cuda.synchronize(dev)
    k3mx.k3mx_trace_enable(False)
    trace = k3mx.k3mx_trace_read()
    st, det = k3mx.k3mx_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({det})")
    ms = [a.elapsed_time(b) for a, b in ev] if flush is not None else [ev[0][0].elapsed_time(ev[0][1]) / steps] * steps
    distinct = [int(torch.unique(idx[i]).numel()) for i in range(steps)]
    return {"ms": ms, "trace": trace, "distinct": distinct}


def time_e2e(k3mx, wl, table, dev, steps, warmup, flush):
    """Steps through the C-ABI entry k3mx_moe_routed_host with pinned host
    buffers: the host->device transfers of x, logits and bias and the
    device->host transfer of y are inside the timed region.  The call is made
    through ctypes with its arguments prepared beforehand, as a C caller
    makes it (the Python binding's argument checks are not the library's
    work)."""
    import numpy as np
    import torch
    import synth
    T = wl.T
    dt = k3mx.K3MX_BF16 if wl.x_bf16 else k3mx.K3MX_F32
    ws = torch.empty(k3mx.k3mx_moe_host_workspace_size(T, dt, wl.path), dtype=torch.uint8, device=dev)
    y = torch.empty((T, D), dtype=torch.float32).pin_memory()
    hx, hl = [], []
    for i in range(warmup + steps):
        x, logits, bias = decode_inputs(i, T)
        bias_h = torch.from_numpy(bias).pin_memory()
        if wl.x_bf16:
            hx.append(torch.from_numpy(synth.f32_to_bf16(x).view(np.int16)).view(torch.bfloat16).pin_memory())
        else:
            hx.append(torch.from_numpy(x).pin_memory())
        hl.append(torch.from_numpy(logits).pin_memory())
    stream = torch.cuda.current_stream(dev)
    # the binding once, for its checks, then the C entry with the same arguments
    k3mx.k3mx_moe_routed_host(y, hx[0], table, hl[0], bias_h, ws, path=wl.path)
    L = k3mx.lib()
    args = [(y.data_ptr(), hx[i].data_ptr(), dt, T, table.data_ptr(), hl[i].data_ptr(), bias_h.data_ptr(),
             wl.path, ws.data_ptr(), ws.numel(), stream.cuda_stream) for i in range(warmup + steps)]
    for i in range(warmup):
        if L.k3mx_moe_routed_host(*args[i]) != 0:
            raise RuntimeError("k3mx_moe_routed_host failed")
    ms = []
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        rc = L.k3mx_moe_routed_host(*args[warmup + i])
        b.record(stream)
        b.synchronize()
        if rc != 0:
            raise RuntimeError(f"k3mx_moe_routed_host failed: {rc}")
        ms.append(a.elapsed_time(b))
    h2d = hx[0].numel() * hx[0].element_size() + hl[0].numel() * 4 + bias_h.numel() * 4
    d2h = y.numel() * 4
    return ms, h2d, d2h


GEMV_ROWS, GEMV_IN = 3072, 3584
GEMV_W_BYTES = GEMV_ROWS * GEMV_IN // 2 + GEMV_ROWS * GEMV_IN // 32      # 5,849,088
GEMV_BYTES = GEMV_W_BYTES + GEMV_IN * 4 + GEMV_ROWS * 4                  # + x + y: 5,875,712


def graph_of(k3mx, dev, calls):
    """A CUDA graph of the given library calls (each a no-argument function
    issuing its launches on the current stream)."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for c in calls:
                c()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    return g


def time_graph(g, dev, reps, warmup):
    import torch
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    return ms


def time_gemv(k3mx, dev, flush, steps, warmup, hbm_peak, cpu_budget_s):
    """The single MXFP4 GEMV, W [3072 x 3584] (scales U{120..130}, 1% set to
    255), x fp32 N(0,1): 64 calls over 64 distinct copies of W (374 MB, 2.9x
    L2) in one CUDA graph, replayed; GB/s = 64 x 5,875,712 B / graph time.
    Also one call alone after an L2 flush (latency), the kernel's own
    duration from the launch trace, and the oracle on the host cores."""
    import numpy as np
    import torch
    import synth
    p, s, x = synth.gemv_inputs(seed=0)
    n_copies = 64
    P = torch.from_numpy(p).to(dev)
    S = torch.from_numpy(s).to(dev)
    Ps = [P.clone() for _ in range(n_copies)]
    Ss = [S.clone() for _ in range(n_copies)]
    xd = torch.from_numpy(x).to(dev)
    ys = torch.empty((n_copies, GEMV_ROWS), dtype=torch.float32, device=dev)
    for i in range(n_copies):
        k3mx.k3mx_gemv(ys[i], xd, Ps[i], Ss[i])
    torch.cuda.synchronize(dev)
    calls = [lambda i=i: k3mx.k3mx_gemv(ys[i], xd, Ps[i], Ss[i]) for i in range(n_copies)]
    g = graph_of(k3mx, dev, calls)
    ms = time_graph(g, dev, max(3, steps // 2), warmup)
    per_call_ms = statistics.median(ms) / n_copies
    gbs = GEMV_BYTES / (per_call_ms / 1e3) / 1e9
    # one call after an L2 flush (write outside the events), and the trace
    stream = torch.cuda.current_stream(dev)
    lat = []
    for i in range(max(5, steps // 2)):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        k3mx.k3mx_gemv(ys[i % n_copies], xd, Ps[i % n_copies], Ss[i % n_copies])
        b.record(stream)
        b.synchronize()
        lat.append(a.elapsed_time(b))
    k3mx.k3mx_trace_read()
    k3mx.k3mx_trace_enable(True)
    for i in range(n_copies):
        k3mx.k3mx_gemv(ys[i], xd, Ps[i], Ss[i])
    torch.cuda.synchronize(dev)
    k3mx.k3mx_trace_enable(False)
    tr = k3mx.k3mx_trace_read()
    kus = 1e3 * tr["gemv"][1] / tr["gemv"][0] if "gemv" in tr else None
    out = {"GB_s": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
           "us_per_gemv": round(1e3 * per_call_ms, 3),
           "timing": f"{n_copies} GEMVs over distinct weight copies ({n_copies * GEMV_W_BYTES / 1e6:.0f} MB) "
                     "in one CUDA graph, median of replays",
           "single_call_us_l2_flushed": round(1e3 * statistics.median(lat), 2),
           "roofline": {"kernel": "gemv", "bound": "hbm", "unit": "GB/s", "peak": hbm_peak,
                        "algorithmic_bytes_per_launch": GEMV_BYTES,
                        "achieved": round(GEMV_BYTES / (kus / 1e6) / 1e9, 1) if kus else None,
                        "frac": round(GEMV_BYTES / (kus / 1e6) / 1e9 / hbm_peak, 4) if kus else None,
                        "kernel_us": round(kus, 3) if kus else None}}
    # the oracle on the host cores: the same GEMV, repeated for ~1/4 of the budget
    import oracle
    oracle.gemv(x, p, s)
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < cpu_budget_s / 4 or n < 2:
        oracle.gemv(x, p, s)
        n += 1
    secs = time.perf_counter() - t0
    out["cpu_baseline"] = {"value": round(n * GEMV_W_BYTES / secs / 1e9, 3), "unit": "GB/s",
                           "cores": oracle.num_threads(), "kind": "oracle",
                           "sample": f"{n} GEMVs of the same 3072 x 3584 matrix"}
    del Ps, Ss, g
    torch.cuda.empty_cache()
    return out


def time_expert(k3mx, dev, arena, steps, warmup, hbm_peak, cpu_budget_s):
    """One full routed expert at one token (k3mx_expert_ffn): 32 calls over
    32 distinct experts of the arena (561 MB, 4.4x L2), x fp32 N(0,1), in
    one CUDA graph, replayed; GB/s = 32 x 17,547,264 B / graph time.  Also
    the fused kernel's own duration and the oracle on the host cores."""
    import torch
    import synth
    n_exp = 32
    offs = k3mx.expert_offsets()
    exs = [k3mx.expert_struct(*[arena.data_ptr() + e * EXPERT_BYTES + o for o in offs]) for e in range(n_exp)]
    xs = torch.from_numpy(synth.token_inputs(n_exp, seed=77)).to(dev)
    ys = torch.empty((n_exp, D), dtype=torch.float32, device=dev)
    ws = torch.empty(k3mx.k3mx_expert_ffn_workspace_size(), dtype=torch.uint8, device=dev)
    for e in range(n_exp):
        k3mx.k3mx_expert_ffn(ys[e], xs[e], exs[e], ws)
    torch.cuda.synchronize(dev)
    calls = [lambda e=e: k3mx.k3mx_expert_ffn(ys[e], xs[e], exs[e], ws) for e in range(n_exp)]
    g = graph_of(k3mx, dev, calls)
    ms = time_graph(g, dev, max(3, steps // 2), warmup)
    per_call_ms = statistics.median(ms) / n_exp
    gbs = EXPERT_BYTES / (per_call_ms / 1e3) / 1e9
    k3mx.k3mx_trace_read()
    k3mx.k3mx_trace_enable(True)
    for e in range(n_exp):
        k3mx.k3mx_expert_ffn(ys[e], xs[e], exs[e], ws)
    torch.cuda.synchronize(dev)
    k3mx.k3mx_trace_enable(False)
    tr = k3mx.k3mx_trace_read()
    # the fused kernel's bytes: the expert's weights, the x pieces, g and u
    # written, h pieces written and read, y written
    kbytes = EXPERT_BYTES + X_IMAGE_BYTES + 2 * F * 4 + 2 * H_IMAGE_BYTES + D * 4
    kus = 1e3 * tr["decode_expert"][1] / tr["decode_expert"][0] if "decode_expert" in tr else None
    out = {"GB_s": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
           "us_per_expert": round(1e3 * per_call_ms, 3),
           "timing": f"{n_exp} calls over distinct experts ({n_exp * EXPERT_BYTES / 1e6:.0f} MB) in one CUDA "
                     "graph, median of replays",
           "kernels": {k: {"launches": v[0], "avg_us": round(1e3 * v[1] / max(1, v[0]), 2)} for k, v in tr.items()},
           "roofline": {"kernel": "decode_expert", "bound": "hbm", "unit": "GB/s", "peak": hbm_peak,
                        "algorithmic_bytes_per_launch": kbytes,
                        "achieved": round(kbytes / (kus / 1e6) / 1e9, 1) if kus else None,
                        "frac": round(kbytes / (kus / 1e6) / 1e9 / hbm_peak, 4) if kus else None}}
    import oracle
    w = synth.split_expert(synth.expert(0, seed=0))
    x0 = synth.token_inputs(1, seed=77)[0]
    oracle.expert(x0, *w)
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < cpu_budget_s / 4 or n < 2:
        oracle.expert(x0, *w)
        n += 1
    secs = time.perf_counter() - t0
    out["cpu_baseline"] = {"value": round(n * EXPERT_BYTES / secs / 1e9, 3), "unit": "GB/s",
                           "cores": oracle.num_threads(), "kind": "oracle",
                           "sample": f"{n} evaluations of one expert at one token"}
    del g
    return out


def oracle_batch_sample(T, budget_s, seed_base=1000, flops=False):
    """The oracle on tokens of a batched workload (T tokens per step, flat
    routing), token after token until ~budget_s: tokens/s, expert GB/s
    (each selected expert's bytes once per token) and GFLOP/s (2 x 33,030,144
    per token and expert)."""
    import numpy as np
    import oracle
    import synth
    x, logits, bias = decode_inputs(0, T, seed_base)
    if T > 64:
        x = synth.bf16_to_f32(synth.f32_to_bf16(x))
    idx, w = oracle.route(logits, bias)
    total_s, toks, pairs = 0.0, 0, 0
    cache = {}
    for t in range(T):
        if total_s >= budget_s:
            break
        ids = [int(e) for e in idx[t]]
        ex = {}
        for e in ids:
            if e not in cache:
                if len(cache) > 64:
                    cache.clear()
                cache[e] = synth.split_expert(synth.expert(e, seed=0))
            ex[e] = cache[e]
        t0 = time.perf_counter()
        oracle.moe(x[t:t + 1], idx[t:t + 1], w[t:t + 1], ex)
        total_s += time.perf_counter() - t0
        toks += 1
        pairs += len(ids)
    return {"tokens_per_s": round(toks / total_s, 3),
            "GB_s": round(pairs * EXPERT_BYTES / total_s / 1e9, 3),
            "GFLOP_s": round(2.0 * PARAMS_PER_EXPERT * pairs / total_s / 1e9, 2),
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{toks} of the {T} tokens of one step, token by token (16 experts each)"}


def time_router(k3mx, dev, flush, steps, warmup, bf16_peak, hbm_peak):
    """The router (logits of the bf16 [896, 7168] router, then the top-16)
    at one fp32 decode token and at 4096 bf16 prefill tokens.  Its inputs fit
    in L2, so L2 is flushed (256 MB write) before every timed call."""
    import numpy as np
    import torch
    import synth
    W = torch.from_numpy(synth.router_weights(seed=0).view(np.int16)).to(dev)
    _, bias_np = synth.router_inputs(1, seed=0)
    bias = torch.from_numpy(bias_np).to(dev)
    out = {}
    stream = torch.cuda.current_stream(dev)
    for name, T, bf16 in (("router_b1", 1, False), ("router_4096", 4096, True)):
        h = synth.hidden_inputs(T, seed=1)
        ht = (torch.from_numpy(synth.f32_to_bf16(h).view(np.int16)).view(torch.bfloat16) if bf16
              else torch.from_numpy(h)).to(dev)
        lg = torch.empty((T, E), dtype=torch.float32, device=dev)
        idx = torch.empty((T, K), dtype=torch.int32, device=dev)
        w = torch.empty((T, K), dtype=torch.float32, device=dev)
        for _ in range(warmup):
            k3mx.k3mx_router(lg, idx, w, ht, W, bias)
        ms = []
        k3mx.k3mx_trace_read()
        k3mx.k3mx_trace_enable(True)
        for _ in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            k3mx.k3mx_router(lg, idx, w, ht, W, bias)
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        k3mx.k3mx_trace_enable(False)
        tr = k3mx.k3mx_trace_read()
        m = statistics.median(ms)
        wbytes = E * 7168 * 2
        flops = 2.0 * T * E * 7168
        r = {"us_per_call": round(1e3 * m, 2), "tokens_per_s": round(T / (m / 1e3), 1),
             "kernels": {k: {"launches": v[0], "avg_us": round(1e3 * v[1] / max(1, v[0]), 2)} for k, v in tr.items()},
             "l2": "flushed before every call (256 MB write, outside the events)"}
        if "router" in tr:
            kus = 1e3 * tr["router"][1] / tr["router"][0]
            if T == 1:
                gbs = (wbytes + T * 7168 * 4 + T * E * 4) / (kus / 1e6) / 1e9
                r["logits_kernel"] = {"us": round(kus, 2), "GB_s": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4)}
            else:
                tf = flops / (kus / 1e6) / 1e12
                r["logits_kernel"] = {"us": round(kus, 2), "TFLOP_s": round(tf, 1),
                                      "frac_bf16_peak": round(tf / bf16_peak, 4)}
        out[name] = r
    return out


def time_latent_block(k3mx, dev, table, steps, warmup, bf16_peak, hbm_peak):
    """The whole Stable LatentMoE block (router, latent projections, routed
    experts, RMSNorm, fused shared experts) at one fp32 decode token and at
    4096 bf16 prefill tokens.  Its inputs exceed L2 (the block's 379 MB of
    bf16 matrices plus 280.8 MB of experts per decode token), so L2 is not
    flushed."""
    import numpy as np
    import torch
    import synth
    host = synth.latent_block_weights(seed=0)
    host["router_w"] = synth.router_weights(seed=0)
    dblk = {k: torch.from_numpy(v.view(np.int16)).to(dev) for k, v in host.items()}
    _, bias = synth.router_inputs(1, seed=0)
    dblk["bias"] = torch.from_numpy(bias).to(dev)
    blk = k3mx.latent_block(dblk)
    dense_bytes = sum(v.size * 2 for k, v in host.items())
    out = {}
    stream = torch.cuda.current_stream(dev)
    for name, T, bf16 in (("latent_block_b1", 1, False), ("latent_block_4096", 4096, True)):
        hs = [synth.hidden_inputs(T, seed=200 + i) for i in range(warmup + steps)]
        dt = k3mx.K3MX_BF16 if bf16 else k3mx.K3MX_F32
        hts = [(torch.from_numpy(synth.f32_to_bf16(h).view(np.int16)).view(torch.bfloat16) if bf16
                else torch.from_numpy(h)).to(dev) for h in hs]
        y = torch.empty((T, 7168), dtype=torch.float32, device=dev)
        idx = torch.empty((T, K), dtype=torch.int32, device=dev)
        ws = torch.empty(k3mx.k3mx_latent_moe_workspace_size(T, dt), dtype=torch.uint8, device=dev)
        for i in range(warmup):
            k3mx.k3mx_latent_moe(y, hts[i], blk, table, ws, idx_out=idx)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        distinct = []
        device_ahead(torch, steps)
        ev[0][0].record(stream)
        for i in range(steps):
            k3mx.k3mx_latent_moe(y, hts[warmup + i], blk, table, ws, idx_out=idx)
            if T == 1:
                distinct.append(16)
        ev[0][1].record(stream)
        torch.cuda.synchronize(dev)
        k3mx.k3mx_trace_read()
        device_ahead(torch, 1)
        k3mx.k3mx_trace_enable(True)
        k3mx.k3mx_latent_moe(y, hts[-1], blk, table, ws, idx_out=idx)
        torch.cuda.synchronize(dev)
        k3mx.k3mx_trace_enable(False)
        tr = k3mx.k3mx_trace_read()
        ms = ev[0][0].elapsed_time(ev[0][1]) / steps
        r = {"us_per_call": round(1e3 * ms, 2), "tokens_per_s": round(T / (ms / 1e3), 1),
             "kernels": {k: {"launches": v[0], "avg_us": round(1e3 * v[1] / max(1, v[0]), 2)} for k, v in tr.items()},
             "l2": "not flushed (inputs exceed L2)"}
        if T == 1:
            gbs = (dense_bytes + 16 * EXPERT_BYTES) / (ms / 1e3) / 1e9
            r["weight_GB_s"] = round(gbs, 1)
            r["hbm_frac"] = round(gbs / hbm_peak, 4)
        else:
            flops = 2.0 * T * (dense_bytes / 2 - 3584) + 2.0 * PARAMS_PER_EXPERT * T * K
            r["TFLOP_s"] = round(flops / (ms / 1e3) / 1e12, 1)
            r["frac_bf16_peak"] = round(flops / (ms / 1e3) / 1e12 / bf16_peak, 4)
        out[name] = r
    return out


def run_ours(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()
    import mxfp4_routed_expert_k3mx_gb300 as k3mx
    import synth

    hbm_peak, bf16_peak, bf16_sust, peak_src = load_peaks()
    t0 = time.time()
    arena = synth.expert_arena_device(dev, seed=0, lo=118, hi=128)
    table = k3mx.expert_table(arena)
    arena_s = time.time() - t0
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    primary = Workload("moe_decode_b1", 1, False, k3mx.K3MX_PATH_DECODE)
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    clocks.start()
    res = time_workload(k3mx, primary, table, dev, args.steps, args.warmup, dist, None)
    clk = clocks.stop()
    # the same workload with L2 flushed between steps (reported beside it)
    res_fl = time_workload(k3mx, primary, table, dev, args.steps, args.warmup, dist, flush)
    fl_ms = sum(res_fl["ms"])
    fl_bytes = sum(d * EXPERT_BYTES for d in res_fl["distinct"])

    total_ms = sum(res["ms"])
    bytes_total = sum(d * EXPERT_BYTES for d in res["distinct"])
    total_ms_max, bytes_all = reduce_over_ranks(dist, total_ms, bytes_total, dev)
    value = bytes_all / (total_ms_max / 1e3) / 1e9

    # dominant kernel: one token per step runs gate/up, down and the weighted
    # sum in one persistent launch (decode_expert); batches run the fused
    # gate/up + SiTU pass (decode_gate_up, two thirds of the bytes)
    tr = res["trace"]
    avg_distinct = sum(res["distinct"]) / max(1, len(res["distinct"]))
    pairs = primary.T * K
    if "decode_expert" in tr:
        dom = "decode_expert"
        # weights of every selected expert, the x pieces, per pair g and u
        # written, h pieces written and read, the pair's output row written
        # and read, y written
        dom_bytes = (avg_distinct * EXPERT_BYTES + primary.T * X_IMAGE_BYTES
                     + pairs * (2 * F * 4 + 2 * H_IMAGE_BYTES + 2 * D * 4) + primary.T * D * 4)
    else:
        dom = "decode_gate_up"
        # w1, w3 of every selected expert, the x pieces, per pair g and u
        # (fp32) and the h pieces written
        dom_bytes = (avg_distinct * GATE_UP_BYTES + primary.T * X_IMAGE_BYTES
                     + pairs * (H_IMAGE_BYTES + 2 * F * 4))
    n_launch, ms_dom = tr.get(dom, (0, 0.0))
    achieved = dom_bytes / (ms_dom / max(1, n_launch) / 1e3) / 1e9 if n_launch else None
    src_hash = kernel_source_hash(DECODE_SOURCES)
    traffic = profiled_traffic(dom, primary.name, src_hash)
    launches = sum(KERNELS_PER_GROUP.get(k, 1) * v[0] for k, v in tr.items())

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "moe_decode_b1", "tokens_per_step": 1, "n_experts": E, "topk": K,
                   "latent": D, "inter": F, "arena_gb": round(E * EXPERT_BYTES / 1e9, 2),
                   "expert_bytes_per_step": 16 * EXPERT_BYTES, "x": "fp32 N(0,1)",
                   "logits": "fresh seeded N(0,1) per step", "bias": "N(0,0.1)",
                   "l2": "not flushed: every step streams 280.8 MB of experts it has not just used "
                         "(2.2x the 129 MB L2)",
                   "parallelism": f"replicas x{world}",
                   "timing": "one event pair around the timed steps; a spin kernel queued ahead of them keeps "
                             "the host's launches ahead of the device"},
        "l2_flushed": {"value": round(fl_bytes / (fl_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                       "ms_per_step": round(fl_ms / len(res_fl["ms"]), 4),
                       "flush": "256 MB write between timed steps, outside the events"},
        "hbm_frac": round(value / world / hbm_peak, 4),
        "hbm_frac_nominal_8tbs": round(value / world / 8000.0, 4),
        "roofline": {"kernel": dom, "bound": "hbm",
                     "achieved": round(achieved, 1) if achieved else None, "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4) if achieved else None,
                     "traffic": traffic, "algorithmic_bytes_per_launch": int(dom_bytes),
                     "peak_source": f"{peak_src} HBM copy"},
        "kernels": {k: {"launches": v[0], "avg_us": round(1e3 * v[1] / max(1, v[0]), 2)} for k, v in tr.items()},
        "gpu_launches": launches,
        "clocks": clk,
        "setup_s": {"arena": round(arena_s, 1)},
    }

    if rank == 0:
        # end to end through the host-buffer entry point
        e2e_ms, h2d, d2h = time_e2e(k3mx, primary, table, dev, args.steps, args.warmup, None)
        e2e_gbs = 16 * EXPERT_BYTES * len(e2e_ms) / (sum(e2e_ms) / 1e3) / 1e9 * world
        line["e2e"] = {"value": round(e2e_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": round(sum(e2e_ms) / len(e2e_ms), 4)}
        # secondary workloads: batch 64 decode (bf16 -> fp32)
        sec = {}
        if not args.primary_only:
            cb = 0.0 if args.no_cpu_baseline else args.cpu_budget_s
            sec["gemv_3072x3584"] = time_gemv(k3mx, dev, flush, args.steps, args.warmup, hbm_peak, cb)
            sec["expert_ffn_1tok"] = time_expert(k3mx, dev, arena, args.steps, args.warmup, hbm_peak, cb)
            if args.no_cpu_baseline:
                for k in ("gemv_3072x3584", "expert_ffn_1tok"):
                    sec[k].pop("cpu_baseline", None)
            wl = Workload("moe_decode_b64", 64, True, k3mx.K3MX_PATH_DECODE)
            r = time_workload(k3mx, wl, table, dev, max(3, args.steps // 2), args.warmup, None, None)
            ms = sum(r["ms"])
            b = sum(d * EXPERT_BYTES for d in r["distinct"])
            sec["moe_decode_b64"] = {"GB_s": round(b / (ms / 1e3) / 1e9, 2),
                                     "tokens_per_s": round(64 * len(r["ms"]) / (ms / 1e3), 1),
                                     "ms_per_step": round(ms / len(r["ms"]), 4),
                                     "distinct_experts_per_step": round(sum(r["distinct"]) / len(r["distinct"]), 1),
                                     "hbm_frac": round(b / (ms / 1e3) / 1e9 / hbm_peak, 4),
                                     "kernels": {k: {"launches": v[0], "avg_us": round(1e3 * v[1] / max(1, v[0]), 2)}
                                                 for k, v in r["trace"].items()}}
            if not args.no_cpu_baseline:
                sec["moe_decode_b64"]["cpu_baseline"] = oracle_batch_sample(64, args.cpu_budget_s / 2)
            # prefill, 4096 bf16 tokens, flat routing: tcgen05 grouped GEMMs,
            # weights dequantised to f16 (PREFILL) or fed as stored to the
            # block-scaled MMAs with x and h as MXFP4 pieces (PREFILL_MX)
            for wname, wpath, srcs in (("moe_prefill_4096", k3mx.K3MX_PATH_PREFILL, PREFILL_SOURCES),
                                       ("moe_prefill_4096_mx", k3mx.K3MX_PATH_PREFILL_MX, PREFILL_MX_SOURCES)):
                wl = Workload(wname, 4096, True, wpath)
                r = time_workload(k3mx, wl, table, dev, max(3, args.steps // 4), args.warmup, None, None)
                ms = sum(r["ms"]) / len(r["ms"])
                pairs = 4096 * K
                flops = 2.0 * PARAMS_PER_EXPERT * pairs
                tr = r["trace"]
                kern = {}
                pf_hash = kernel_source_hash(srcs)
                for name, params in (("prefill_gate_up", GATE_UP_PARAMS),
                                     ("prefill_down", PARAMS_PER_EXPERT - GATE_UP_PARAMS)):
                    if name in tr:
                        kms = tr[name][1] / tr[name][0]
                        tf = 2.0 * params * pairs / (kms / 1e3) / 1e12
                        kern[name] = {"avg_ms": round(kms, 4), "TFLOP_s": round(tf, 1),
                                      "frac_bf16_peak": round(tf / bf16_peak, 4),
                                      "traffic": profiled_traffic(name, wl.name, pf_hash)}
                sec[wname] = {
                    "tokens_per_s": round(4096 / (ms / 1e3), 1), "ms_per_step": round(ms, 4),
                    "TFLOP_s": round(flops / (ms / 1e3) / 1e12, 1),
                    "frac_bf16_peak": round(flops / (ms / 1e3) / 1e12 / bf16_peak, 4),
                    "expert_GB_s": round(E * EXPERT_BYTES / (ms / 1e3) / 1e9, 1),
                    "peak_source": f"{peak_src} bf16 burst {bf16_peak} TFLOP/s (algorithmic FLOPs)",
                    "tensor_kernels": kern,
                    "kernels": {k: {"launches": v[0], "avg_us": round(1e3 * v[1] / max(1, v[0]), 2)}
                                for k, v in tr.items()}}
            if not args.no_cpu_baseline:
                sec["moe_prefill_4096_mx"]["cpu_baseline"] = oracle_batch_sample(4096, args.cpu_budget_s / 2)
            sec.update(time_router(k3mx, dev, flush, max(5, args.steps // 2), args.warmup, bf16_peak, hbm_peak))
            sec.update(time_latent_block(k3mx, dev, table, max(3, args.steps // 4), args.warmup, bf16_peak, hbm_peak))
        line["secondary"] = sec
        if not args.no_cpu_baseline:
            steps_in = [decode_inputs(i, 1) for i in range(64)]
            nb, secs, toks, cores = oracle_decode_sample(steps_in, args.cpu_budget_s, 64)
            line["cpu_baseline"] = {"value": round(nb / secs / 1e9, 3), "unit": "GB/s", "cores": cores,
                                    "kind": "oracle",
                                    "sample": f"{toks} decode tokens of the same workload, 16 experts each"}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def run_profile_case(args):
    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import mxfp4_routed_expert_k3mx_gb300 as k3mx
    import synth
    dev = torch.device("cuda:0")
    if args.profile_case == "latent":
        # the whole LatentMoE block over R resident experts (entry e -> e mod R)
        T, R = args.tokens, args.resident
        arena = synth.expert_arena_device(dev, seed=0, lo=118, hi=128, n_experts=R)
        table = k3mx.expert_table(arena, n_experts=R)[torch.arange(E, device=dev) % R].contiguous()
        host = synth.latent_block_weights(seed=0)
        host["router_w"] = synth.router_weights(seed=0)
        dblk = {k: torch.from_numpy(v.view(np.int16)).to(dev) for k, v in host.items()}
        _, bias = synth.router_inputs(1, seed=0)
        dblk["bias"] = torch.from_numpy(bias).to(dev)
        blk = k3mx.latent_block(dblk)
        h = synth.hidden_inputs(T, seed=1)
        bf16 = T > 16
        ht = (torch.from_numpy(synth.f32_to_bf16(h).view(np.int16)).view(torch.bfloat16) if bf16
              else torch.from_numpy(h)).to(dev)
        dt = k3mx.K3MX_BF16 if bf16 else k3mx.K3MX_F32
        y = torch.empty((T, 7168), dtype=torch.float32, device=dev)
        ws = torch.empty(k3mx.k3mx_latent_moe_workspace_size(T, dt), dtype=torch.uint8, device=dev)
        for _ in range(args.iters):
            k3mx.k3mx_latent_moe(y, ht, blk, table, ws)
        torch.cuda.synchronize(dev)
        st = k3mx.k3mx_device_status()
        print(json.dumps({"profile_case": "latent", "tokens": T, "resident": R, "iters": args.iters, "status": st}),
              flush=True)
        if st[0] != 0:
            sys.exit(1)
        return
    if args.profile_case == "gemv":
        # `iters` graph replays of 64 GEMVs over distinct copies of the
        # 3072 x 3584 matrix (374 MB)
        p, s, x = synth.gemv_inputs(seed=0)
        P, S = torch.from_numpy(p).to(dev), torch.from_numpy(s).to(dev)
        Ps, Ss = [P.clone() for _ in range(64)], [S.clone() for _ in range(64)]
        xd = torch.from_numpy(x).to(dev)
        ys = torch.empty((64, GEMV_ROWS), dtype=torch.float32, device=dev)
        for i in range(64):
            k3mx.k3mx_gemv(ys[i], xd, Ps[i], Ss[i])
        g = graph_of(k3mx, dev, [lambda i=i: k3mx.k3mx_gemv(ys[i], xd, Ps[i], Ss[i]) for i in range(64)])
        for _ in range(args.iters):
            g.replay()
        torch.cuda.synchronize(dev)
        st = k3mx.k3mx_device_status()
        print(json.dumps({"profile_case": "gemv", "iters": args.iters, "status": st}), flush=True)
        if st[0] != 0:
            sys.exit(1)
        return
    if args.profile_case == "expert":
        # `iters` rounds of k3mx_expert_ffn over R resident experts, one token each
        R = args.resident
        arena = synth.expert_arena_device(dev, seed=0, lo=118, hi=128, n_experts=R)
        offs = k3mx.expert_offsets()
        exs = [k3mx.expert_struct(*[arena.data_ptr() + e * EXPERT_BYTES + o for o in offs]) for e in range(R)]
        xs = torch.from_numpy(synth.token_inputs(R, seed=77)).to(dev)
        ys = torch.empty((R, D), dtype=torch.float32, device=dev)
        ws = torch.empty(k3mx.k3mx_expert_ffn_workspace_size(), dtype=torch.uint8, device=dev)
        for _ in range(args.iters):
            for e in range(R):
                k3mx.k3mx_expert_ffn(ys[e], xs[e], exs[e], ws)
        torch.cuda.synchronize(dev)
        st = k3mx.k3mx_device_status()
        print(json.dumps({"profile_case": "expert", "resident": R, "iters": args.iters, "status": st}), flush=True)
        if st[0] != 0:
            sys.exit(1)
        return
    if args.profile_case == "router":
        # the router alone: fp32 states up to 16 tokens, bf16 beyond
        T = args.tokens
        W = torch.from_numpy(synth.router_weights(seed=0).view(np.int16)).to(dev)
        _, bias = synth.router_inputs(1, seed=0)
        h = synth.hidden_inputs(T, seed=1)
        ht = (torch.from_numpy(h) if T <= 16 else
              torch.from_numpy(synth.f32_to_bf16(h).view(np.int16)).view(torch.bfloat16)).to(dev)
        lg = torch.empty((T, E), dtype=torch.float32, device=dev)
        idx = torch.empty((T, K), dtype=torch.int32, device=dev)
        w = torch.empty((T, K), dtype=torch.float32, device=dev)
        for _ in range(args.iters):
            k3mx.k3mx_router(lg, idx, w, ht, W, torch.from_numpy(bias).to(dev))
        torch.cuda.synchronize(dev)
        st = k3mx.k3mx_device_status()
        print(json.dumps({"profile_case": "router", "tokens": T, "iters": args.iters, "status": st}), flush=True)
        if st[0] != 0:
            sys.exit(1)
        return
    T, R = args.tokens, args.resident
    arena = synth.expert_arena_device(dev, seed=0, lo=118, hi=128, n_experts=R)
    table = k3mx.expert_table(arena, n_experts=R)[torch.arange(E, device=dev) % R].contiguous()
    bias = torch.zeros(E, dtype=torch.float32, device=dev)
    if args.confine:
        bias[R:] = -100.0
    prefill = args.profile_case == "prefill"
    path = (k3mx.K3MX_PATH_PREFILL_MX if args.mx else k3mx.K3MX_PATH_PREFILL) if prefill else k3mx.K3MX_PATH_DECODE
    dt = k3mx.K3MX_BF16 if prefill else k3mx.K3MX_F32
    ws = torch.empty(k3mx.k3mx_moe_workspace_size(T, dt, path), dtype=torch.uint8, device=dev)
    y = torch.empty((T, D), dtype=torch.float32, device=dev)
    for i in range(args.iters):
        x, logits, _ = decode_inputs(i, T)
        if prefill:
            xt = torch.from_numpy(synth.f32_to_bf16(x).view(np.int16)).view(torch.bfloat16).to(dev)
        else:
            xt = torch.from_numpy(x).to(dev)
        k3mx.k3mx_moe_routed(y, xt, table, torch.from_numpy(logits).to(dev), bias, ws, path=path)
    torch.cuda.synchronize(dev)
    st = k3mx.k3mx_device_status()
    print(json.dumps({"profile_case": args.profile_case, "mx": args.mx, "tokens": T, "resident": R,
                      "confine": args.confine, "iters": args.iters, "status": st,
                      "y_abs_sum": float(y.abs().sum())}), flush=True)
    if st[0] != 0:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--primary-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--profile-case", choices=["decode", "prefill", "router", "latent", "gemv", "expert"])
    ap.add_argument("--tokens", type=int, default=1)
    ap.add_argument("--resident", type=int, default=64)
    ap.add_argument("--confine", action="store_true")
    ap.add_argument("--mx", action="store_true", help="prefill profile case on the block-scaled path")
    ap.add_argument("--iters", type=int, default=4)
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    args.warmup = max(args.warmup, 3)            # at least 3 untimed warm-up steps
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
