"""First calls from several host threads at once.

The library sets up each device lazily (device properties, kernel shared
memory attributes, tensor-map templates, the fixed scratch array).  A fresh
process (so nothing is set up yet) starts four threads together, each on its
own stream and workspace: DECODE, PREFILL_MX and PREFILL of the routed layer
and the router.  Afterwards the same calls run again one after another; the
threaded results must match them (bit for bit where the path is
deterministic, to fp32 summation order where prefill adds with atomics)."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N_DISTINCT = 8          # experts in the arena; the table repeats them


def _child():
    import threading

    import torch

    sys.path.insert(0, ROOT)
    import synth
    import mxfp4_routed_expert_k3mx_gb300 as k3mx

    dev = torch.device("cuda:0")
    torch.cuda.init()
    n = synth.expert_nbytes()
    host = np.empty(N_DISTINCT * n, dtype=np.uint8)
    for e in range(N_DISTINCT):
        synth.expert(e, seed=3, out=host[e * n:(e + 1) * n])
    arena = torch.from_numpy(host).to(dev)
    offs = torch.tensor(k3mx.expert_offsets(), dtype=torch.int64)
    rows = torch.arange(k3mx.K3MX_N_EXPERTS, dtype=torch.int64) % N_DISTINCT
    table = (arena.data_ptr() + rows[:, None] * n + offs[None, :]).to(dev)

    def moe_case(T, bf16, path, seed):
        x = synth.token_inputs(T, seed=seed)
        logits, _ = synth.router_inputs(T, seed=seed)
        if bf16:
            xt = torch.from_numpy(synth.f32_to_bf16(x).view(np.int16)).view(torch.bfloat16).to(dev)
            dt = k3mx.K3MX_BF16
        else:
            xt = torch.from_numpy(x).to(dev)
            dt = k3mx.K3MX_F32
        lg = torch.from_numpy(logits).to(dev)
        bias = torch.zeros(896, dtype=torch.float32, device=dev)
        ws = torch.empty(k3mx.k3mx_moe_workspace_size(T, dt, path), dtype=torch.uint8, device=dev)

        def run(stream):
            y = torch.full((T, 3584), float("nan"), dtype=torch.float32, device=dev)
            idx = torch.full((T, 16), -1, dtype=torch.int32, device=dev)
            with torch.cuda.stream(stream):
                k3mx.k3mx_moe_routed(y, xt, table, lg, bias, ws, path=path, idx_out=idx, stream=stream)
            return y, idx
        return run

    def router_case(T, seed):
        hid = torch.from_numpy(synth.hidden_inputs(T, seed=seed)).to(dev)
        rw = torch.from_numpy(synth.router_weights(seed=seed).view(np.int16)).to(dev)
        bias = torch.zeros(896, dtype=torch.float32, device=dev)

        def run(stream):
            lg = torch.empty((T, 896), dtype=torch.float32, device=dev)
            idx = torch.empty((T, 16), dtype=torch.int32, device=dev)
            w = torch.empty((T, 16), dtype=torch.float32, device=dev)
            k3mx.k3mx_router(lg, idx, w, hid, rw, bias, stream=stream)
            return lg, idx
        return run

    cases = {
        "decode": moe_case(4, False, k3mx.K3MX_PATH_DECODE, 11),
        "prefill_mx": moe_case(256, True, k3mx.K3MX_PATH_PREFILL_MX, 12),
        "prefill": moe_case(256, True, k3mx.K3MX_PATH_PREFILL, 13),
        "router": router_case(32, 14),
    }
    torch.cuda.synchronize(dev)
    start = threading.Barrier(len(cases))
    got, errors = {}, []

    def worker(name, run):
        try:
            torch.cuda.set_device(dev)
            stream = torch.cuda.Stream(device=dev)
            start.wait()
            got[name] = run(stream)
            stream.synchronize()
        except Exception as e:          # reported by the parent
            errors.append(f"{name}: {e!r}")

    threads = [threading.Thread(target=worker, args=item) for item in cases.items()]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize(dev)
    assert k3mx.k3mx_device_status() == (0, 0)

    s = torch.cuda.current_stream(dev)
    for name, run in cases.items():
        ref = run(s)
        torch.cuda.synchronize(dev)
        a, b = got[name], ref
        assert torch.equal(a[1], b[1]), f"{name}: indices differ"
        assert torch.isfinite(a[0]).all(), f"{name}: non-finite output"
        if name in ("decode", "router"):
            assert torch.equal(a[0].view(torch.int32), b[0].view(torch.int32)), f"{name}: not bit-identical"
        else:
            d = (a[0] - b[0]).norm(dim=1) / b[0].norm(dim=1).clamp_min(1e-30)
            assert float(d.max()) < 1e-5, f"{name}: {float(d.max())}"
    print("threads ok")


def test_first_calls_from_four_threads(cuda_dev):
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "child"], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]


if __name__ == "__main__" and sys.argv[1:] == ["child"]:
    _child()
