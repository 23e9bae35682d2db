"""Device-side waits that give up, made to happen without any fault: the
library's wait limit is cut to one poll (k3mx_set_wait_limit), so the
pipeline waits of the next call run out long before the data they wait for
arrives.  Each case checks that the device status reports K3MX_ETIMEOUT with
a detail code, that the context stays usable, and that once the limit is
restored the same call gives the result of a clean run (the refuse-never-
guess discipline of kimi-k3-in-c README, "2. The config reader that refuses
to guess": a wait that cannot complete is reported, never papered over)."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx
import synth

pytestmark = pytest.mark.gpu

K3MX_ETIMEOUT = 6


def run_layer(dev, table, x_t, logits, bias, path):
    T = x_t.shape[0]
    y = torch.full((T, 3584), float("nan"), dtype=torch.float32, device=dev)
    dt = k3mx.K3MX_BF16 if x_t.dtype == torch.bfloat16 else k3mx.K3MX_F32
    ws = torch.empty(k3mx.k3mx_moe_workspace_size(T, dt, path), dtype=torch.uint8, device=dev)
    k3mx.k3mx_moe_routed(y, x_t, table, logits, bias, ws, path=path)
    return y


def timed_out_then_clean(dev, call):
    """call() once clean, once with a one-poll limit, once clean again."""
    ref = call()
    st, det = k3mx.k3mx_device_status()
    assert st == 0, (st, det)
    k3mx.k3mx_set_wait_limit(1)
    try:
        call()
        st, det = k3mx.k3mx_device_status()
    finally:
        k3mx.k3mx_set_wait_limit(0)
    assert st == K3MX_ETIMEOUT, (st, det)
    assert det != 0
    again = call()
    st2, det2 = k3mx.k3mx_device_status()
    assert st2 == 0, (st2, det2)
    return ref.cpu().numpy(), again.cpu().numpy(), det


@pytest.mark.parametrize("T", [1, 5])
def test_decode_wait_timeout(arena, cuda_dev, T):
    """The decode path: one token (the fused persistent pass, whose down
    parts wait on a count other CTAs raise) and five (the batched passes)."""
    _, table = arena
    x = torch.from_numpy(synth.token_inputs(T, seed=61)).to(cuda_dev)
    lg, bias = synth.router_inputs(T, seed=61)
    lg, bias = torch.from_numpy(lg).to(cuda_dev), torch.from_numpy(bias).to(cuda_dev)
    ref, again, det = timed_out_then_clean(
        cuda_dev, lambda: run_layer(cuda_dev, table, x, lg, bias, k3mx.K3MX_PATH_DECODE))
    assert np.array_equal(ref, again), det                   # deterministic path: bit-identical


def test_prefill_mx_wait_timeout(arena, cuda_dev):
    """The block-scaled prefill (its y is summed with atomics, so the clean
    runs agree to rounding)."""
    _, table = arena
    T = 300
    xb = synth.f32_to_bf16(synth.token_inputs(T, seed=62))
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(cuda_dev)
    lg, bias = synth.router_inputs(T, seed=62)
    lg, bias = torch.from_numpy(lg).to(cuda_dev), torch.from_numpy(bias).to(cuda_dev)
    ref, again, det = timed_out_then_clean(
        cuda_dev, lambda: run_layer(cuda_dev, table, x, lg, bias, k3mx.K3MX_PATH_PREFILL_MX))
    rel = np.linalg.norm(ref - again, axis=1) / np.linalg.norm(ref, axis=1)
    assert rel.max() <= 1e-5, (rel.max(), det)


def test_latent_block_wait_timeout(arena, cuda_dev):
    """The LatentMoE block at one token: its CUDA-core products wait on ring
    slots filled by a producer warp."""
    _, table = arena
    host = synth.latent_block_weights(seed=0)
    host["router_w"] = synth.router_weights(seed=0)
    dblk = {k: torch.from_numpy(v.view(np.int16)).to(cuda_dev) for k, v in host.items()}
    _, bias = synth.router_inputs(1, seed=0)
    dblk["bias"] = torch.from_numpy(bias).to(cuda_dev)
    blk = k3mx.latent_block(dblk)
    h = torch.from_numpy(synth.hidden_inputs(1, seed=63)).to(cuda_dev)
    y = torch.empty((1, 7168), dtype=torch.float32, device=cuda_dev)
    ws = torch.empty(k3mx.k3mx_latent_moe_workspace_size(1, k3mx.K3MX_F32), dtype=torch.uint8, device=cuda_dev)

    def call():
        y.fill_(float("nan"))
        k3mx.k3mx_latent_moe(y, h, blk, table, ws)
        return y.clone()
    ref, again, det = timed_out_then_clean(cuda_dev, call)
    assert np.array_equal(ref, again), det
