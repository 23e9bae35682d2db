"""The allocation-free decode entry point against k3mx_moe_routed (DECODE)
on the same inputs, two calls in a row, through the C ABI.  The scratch of
the no-alloc entry is a fixed device array; the second call checks that
what the first left behind in it does not leak into the result."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _inputs(T, seed, dev, bf16):
    x = synth.token_inputs(T, seed=seed)
    logits, _ = synth.router_inputs(T, seed=seed)
    if bf16:
        xt = torch.from_numpy(synth.f32_to_bf16(x).view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        xt = torch.from_numpy(x).to(dev)
    return xt, torch.from_numpy(logits).to(dev), torch.zeros(896, dtype=torch.float32, device=dev)


@pytest.mark.parametrize("T,bf16", [(1, False), (8, True), (3, False)])
def test_noalloc_matches_workspace_entry(cuda_dev, arena, T, bf16):
    import mxfp4_routed_expert_k3mx_gb300 as k3mx
    dev = cuda_dev
    _, table = arena
    dt = k3mx.K3MX_BF16 if bf16 else k3mx.K3MX_F32
    ws = torch.empty(k3mx.k3mx_moe_workspace_size(T, dt, k3mx.K3MX_PATH_DECODE),
                     dtype=torch.uint8, device=dev)
    for call, seed in enumerate((71 + T, 72 + T)):
        x, lg, bias = _inputs(T, seed, dev, bf16)
        y_ref = torch.empty((T, 3584), dtype=torch.float32, device=dev)
        idx_ref = torch.empty((T, 16), dtype=torch.int32, device=dev)
        w_ref = torch.empty((T, 16), dtype=torch.float32, device=dev)
        k3mx.k3mx_moe_routed(y_ref, x, table, lg, bias, ws, path=k3mx.K3MX_PATH_DECODE,
                             idx_out=idx_ref, w_out=w_ref)
        y = torch.full((T, 3584), float("nan"), dtype=torch.float32, device=dev)
        idx = torch.full((T, 16), -1, dtype=torch.int32, device=dev)
        w = torch.full((T, 16), float("nan"), dtype=torch.float32, device=dev)
        k3mx.k3mx_moe_decode_noalloc(y, x, table, lg, bias, idx_out=idx, w_out=w)
        torch.cuda.synchronize(dev)
        assert k3mx.k3mx_device_status() == (0, 0)
        assert torch.equal(idx, idx_ref), f"call {call}"
        assert torch.equal(w.view(torch.int32), w_ref.view(torch.int32)), f"call {call}"
        # same kernels on the same inputs: identical, well inside the decode tolerance
        assert torch.isfinite(y).all()
        assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32)), f"call {call}"


def test_noalloc_rejects_too_many_tokens(cuda_dev, arena):
    import mxfp4_routed_expert_k3mx_gb300 as k3mx
    dev = cuda_dev
    _, table = arena
    T = k3mx.K3MX_NOALLOC_MAX_TOKENS + 1
    x, lg, bias = _inputs(T, 5, dev, False)
    y = torch.empty((T, 3584), dtype=torch.float32, device=dev)
    with pytest.raises(k3mx.K3mxError):
        k3mx.k3mx_moe_decode_noalloc(y, x, table, lg, bias)
