"""The routed-expert layer on the two prefill paths (bf16 activations,
grouped tcgen05 GEMMs: weights dequantised to f16, or x and h as two MXFP8
pieces each against the weights as stored on the block-scaled MMAs) against
the oracle.  Routing bit-exact;
per sampled token the relative L2 error of y is at most 1e-2 (the
bf16-activation tolerance)."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx
import oracle
import synth
from helpers import arena_expert_bytes, moe_oracle, moe_oracle_rows

pytestmark = pytest.mark.gpu


PATHS = [pytest.param(k3mx.K3MX_PATH_PREFILL, id="f16"), pytest.param(k3mx.K3MX_PATH_PREFILL_MX, id="mx")]


def run_prefill(dev, table, xb, logits, bias, path):
    T = xb.shape[0]
    x_t = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev)
    y = torch.full((T, 3584), float("nan"), dtype=torch.float32, device=dev)
    idx = torch.empty((T, 16), dtype=torch.int32, device=dev)
    w = torch.empty((T, 16), dtype=torch.float32, device=dev)
    ws = torch.empty(k3mx.k3mx_moe_workspace_size(T, k3mx.K3MX_BF16, path), dtype=torch.uint8, device=dev)
    k3mx.k3mx_moe_routed(y, x_t, table, torch.from_numpy(logits).to(dev), torch.from_numpy(bias).to(dev),
                         ws, path=path, idx_out=idx, w_out=w)
    st, det = k3mx.k3mx_device_status()
    assert st == 0, (st, det)
    return y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def check_tokens(y, x, ir, wr, tokens, what):
    yr, _ = moe_oracle(x, ir, wr, tokens)
    for i, t in enumerate(tokens):
        rel = np.linalg.norm(y[t].astype(np.float64) - yr[i]) / np.linalg.norm(yr[i])
        assert rel <= 1e-2, f"{what}: token {t} relative L2 error {rel:.3e}"
    return max(np.linalg.norm(y[t].astype(np.float64) - yr[i]) / np.linalg.norm(yr[i])
               for i, t in enumerate(tokens))


@pytest.mark.parametrize("path", PATHS)
def test_prefill_4096_tokens(arena, cuda_dev, path):
    """x bf16 [4096 x 3584] ~ N(0,1), top-16 of 896 with flat routing
    (about 73 tokens per expert)."""
    _, table = arena
    T = 4096
    xb = synth.f32_to_bf16(synth.token_inputs(T, seed=0))
    x = synth.bf16_to_f32(xb)
    logits, _ = synth.router_inputs(T, seed=0)
    bias = np.zeros(896, np.float32)
    y, idx, w = run_prefill(cuda_dev, table, xb, logits, bias, path)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w, wr)
    counts = np.bincount(ir.ravel(), minlength=896)
    assert counts.min() > 0 and 60 < counts.mean() < 90
    assert np.all(np.isfinite(y))
    # a seeded 512-token subset (the first and last tokens included)
    rng = np.random.default_rng(4096)
    tokens = sorted(set([0, 1, 4095] + rng.choice(T, 509, replace=False).tolist()))
    yr = moe_oracle_rows(x, ir, wr, tokens, arena_expert_bytes)
    rel = [np.linalg.norm(y[t].astype(np.float64) - yr[i].astype(np.float64)) / np.linalg.norm(yr[i].astype(np.float64))
           for i, t in enumerate(tokens)]
    assert max(rel) <= 1e-2, f"prefill 4096: worst token {tokens[int(np.argmax(rel))]} relative L2 {max(rel):.3e}"
    assert max(rel) < 5e-3


@pytest.mark.parametrize("path", PATHS)
def test_prefill_small_batch_and_padding(arena, cuda_dev, path):
    """300 tokens: about 5 tokens per expert, so every tile pads N to 16."""
    _, table = arena
    T = 300
    xb = synth.f32_to_bf16(synth.token_inputs(T, seed=4))
    x = synth.bf16_to_f32(xb)
    logits, bias = synth.router_inputs(T, seed=4)
    y, idx, w = run_prefill(cuda_dev, table, xb, logits, bias, path)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir)
    check_tokens(y, x, ir, wr, [0, 150, 299], "prefill 300")


@pytest.mark.parametrize("path", PATHS)
def test_prefill_expert_with_more_than_128_tokens(arena, cuda_dev, path):
    """200 tokens on the same 16 experts: each expert's list splits into
    several work units (128 + 72 pairs on the f16 path, 3 x 66-67 on the
    block-scaled path)."""
    _, table = arena
    T = 200
    xb = synth.f32_to_bf16(synth.token_inputs(T, seed=8))
    x = synth.bf16_to_f32(xb)
    logits, _ = synth.router_inputs(T, seed=8)
    bias = np.zeros(896, np.float32)
    logits[:, 300:316] += 8.0
    y, idx, w = run_prefill(cuda_dev, table, xb, logits, bias, path)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir)
    assert np.all(np.bincount(ir.ravel(), minlength=896)[300:316] == T)
    check_tokens(y, x, ir, wr, [0, 127, 128, 199], "prefill skewed")


def test_prefill_paths_agree(arena, cuda_dev):
    """The two prefill paths on the same 1024 tokens: every token's outputs
    agree to the sum of their error bounds (relative L2 within 2e-2), and
    the default path for bf16 batches is the block-scaled one."""
    _, table = arena
    T = 1024
    xb = synth.f32_to_bf16(synth.token_inputs(T, seed=12))
    logits, bias = synth.router_inputs(T, seed=12)
    a, _, _ = run_prefill(cuda_dev, table, xb, logits, bias, k3mx.K3MX_PATH_PREFILL)
    b, _, _ = run_prefill(cuda_dev, table, xb, logits, bias, k3mx.K3MX_PATH_PREFILL_MX)
    c, _, _ = run_prefill(cuda_dev, table, xb, logits, bias, k3mx.K3MX_PATH_AUTO)
    rel = np.linalg.norm(a - b, axis=1) / np.linalg.norm(a, axis=1)
    assert rel.max() <= 2e-2, rel.max()
    relc = np.linalg.norm(c - b, axis=1) / np.linalg.norm(b, axis=1)
    assert relc.max() <= 1e-5, relc.max()                 # same kernels; only the atomic order differs
