"""The Stable LatentMoE block (Kimi K3 engine (c/kimi_k3.c), "Architecture
notes": router, latent projections 7168 -> 3584 -> 7168, the routed experts
in the latent, RMSNorm on their sum, the fused shared experts added
unweighted) against the oracle.  The routing is checked bit-exact against
the oracle's routing of the GPU's own router logits; y per token within
relative L2 1e-4 (fp32 states, CUDA cores) or 1e-2 (bf16 batches, tensor
cores)."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx
import oracle
import synth
from helpers import arena_expert

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def block(cuda_dev):
    host = synth.latent_block_weights(seed=0)
    host["router_w"] = synth.router_weights(seed=0)
    _, bias = synth.router_inputs(1, seed=0)
    dev = {k: torch.from_numpy(v.view(np.int16)).to(cuda_dev) for k, v in host.items()}
    dev["bias"] = torch.from_numpy(bias).to(cuda_dev)
    host["bias"] = bias
    return host, dev, k3mx.latent_block(dev)


def run_block(dev, table, blk, h, top_p=0.0):
    T = h.shape[0]
    if h.dtype == np.uint16:
        ht = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)
        dt = k3mx.K3MX_BF16
    else:
        ht = torch.from_numpy(h).to(dev)
        dt = k3mx.K3MX_F32
    y = torch.full((T, 7168), float("nan"), dtype=torch.float32, device=dev)
    idx = torch.empty((T, 16), dtype=torch.int32, device=dev)
    w = torch.empty((T, 16), dtype=torch.float32, device=dev)
    ws = torch.empty(k3mx.k3mx_latent_moe_workspace_size(T, dt), dtype=torch.uint8, device=dev)
    k3mx.k3mx_latent_moe(y, ht, blk, table, ws, top_p=top_p, idx_out=idx, w_out=w)
    st, det = k3mx.k3mx_device_status()
    assert st == 0, (st, det)
    return y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), ht


def gpu_logits(dev, dblk, ht):
    """The router logits of the same kernel the block runs (deterministic)."""
    T = ht.shape[0]
    lg = torch.empty((T, 896), dtype=torch.float32, device=dev)
    idx = torch.empty((T, 16), dtype=torch.int32, device=dev)
    w = torch.empty((T, 16), dtype=torch.float32, device=dev)
    k3mx.k3mx_router(lg, idx, w, ht, dblk["router_w"], dblk["bias"])
    return lg.cpu().numpy()


def check(host, h, y, idx, w, lg, tokens, tol, top_p=0.0):
    bias = host["bias"]
    ir, wr = oracle.route_topp(lg, bias, float(np.float32(top_p))) if top_p > 0 else oracle.route(lg, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w.view(np.uint32), wr.view(np.uint32))
    experts = {int(e): arena_expert(int(e)) for e in np.unique(ir[tokens]) if e >= 0}
    yr, _ = oracle.latent_block(h, host, ir, wr, experts, tokens=tokens)
    worst = 0.0
    for i, t in enumerate(tokens):
        rel = np.linalg.norm(y[t].astype(np.float64) - yr[i]) / np.linalg.norm(yr[i])
        assert rel <= tol, f"token {t}: relative L2 error {rel:.3e}"
        worst = max(worst, rel)
    return worst


@pytest.mark.parametrize("T", [1, 3, 5])
def test_latent_block_fp32(arena, cuda_dev, block, T):
    """5 states: two input chunks (3 + 2) through every CUDA-core product."""
    host, dblk, blk = block
    _, table = arena
    h = synth.hidden_inputs(T, seed=90 + T)
    y, idx, w, ht = run_block(cuda_dev, table, blk, h)
    assert np.all(np.isfinite(y))
    worst = check(host, h, y, idx, w, gpu_logits(cuda_dev, dblk, ht), list(range(T)), 1e-4)
    assert worst < 1e-5


def test_latent_block_fp32_top_p(arena, cuda_dev, block):
    host, dblk, blk = block
    _, table = arena
    h = synth.hidden_inputs(2, seed=95)
    y, idx, w, ht = run_block(cuda_dev, table, blk, h, top_p=0.8)
    assert np.any(idx < 0)
    check(host, h, y, idx, w, gpu_logits(cuda_dev, dblk, ht), [0, 1], 1e-4, top_p=0.8)


def test_latent_block_bf16_small(arena, cuda_dev, block):
    """16 bf16 states stay on the CUDA cores (fp32 intermediates)."""
    host, dblk, blk = block
    _, table = arena
    hb = synth.f32_to_bf16(synth.hidden_inputs(16, seed=116))
    y, idx, w, ht = run_block(cuda_dev, table, blk, hb)
    check(host, hb, y, idx, w, gpu_logits(cuda_dev, dblk, ht), [0, 7, 15], 1e-4)


@pytest.mark.parametrize("T", [20, 300])
def test_latent_block_bf16_batch(arena, cuda_dev, block, T):
    """Tensor-core products with bf16 operands; 20 tokens take the routed
    DECODE path, 300 the block-scaled prefill."""
    host, dblk, blk = block
    _, table = arena
    hb = synth.f32_to_bf16(synth.hidden_inputs(T, seed=100 + T))
    y, idx, w, ht = run_block(cuda_dev, table, blk, hb)
    assert np.all(np.isfinite(y))
    check(host, hb, y, idx, w, gpu_logits(cuda_dev, dblk, ht), [0, T // 2, T - 1], 1e-2)
