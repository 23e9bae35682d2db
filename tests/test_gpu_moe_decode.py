"""The routed-expert layer on the decode path (fp32 activations) against the
oracle, on the full 896-expert arena:
  - batch 1, x fp32 ~ N(0,1), logits ~ N(0,1), bias ~ N(0, 0.1);
  - batch 64, x bf16 -> fp32, each token routed independently with flat
    routing (no score-correction bias), so about 610 distinct experts run.
Routing bit-exact; y within sum_k w_k * (per-expert decode bound)."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx
import oracle
import synth
from helpers import assert_within, moe_oracle

pytestmark = pytest.mark.gpu


def run_moe(dev, table, x_t, logits, bias, path):
    T = x_t.shape[0]
    y = torch.full((T, 3584), float("nan"), dtype=torch.float32, device=dev)
    idx = torch.empty((T, 16), dtype=torch.int32, device=dev)
    w = torch.empty((T, 16), dtype=torch.float32, device=dev)
    dt = k3mx.K3MX_BF16 if x_t.dtype == torch.bfloat16 else k3mx.K3MX_F32
    ws = torch.empty(k3mx.k3mx_moe_workspace_size(T, dt, path), dtype=torch.uint8, device=dev)
    k3mx.k3mx_moe_routed(y, x_t.to(dev), table, torch.from_numpy(logits).to(dev),
                         torch.from_numpy(bias).to(dev), ws, path=path, idx_out=idx, w_out=w)
    st, det = k3mx.k3mx_device_status()
    assert st == 0, (st, det)
    return y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def test_decode_batch1(arena, cuda_dev):
    _, table = arena
    x = synth.token_inputs(1, seed=0)
    logits, bias = synth.router_inputs(1, seed=0)
    y, idx, w = run_moe(cuda_dev, table, torch.from_numpy(x), logits, bias, k3mx.K3MX_PATH_DECODE)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w, wr)
    yr, bound = moe_oracle(x, ir, wr, [0])
    r = assert_within(y, yr, 1e-5 * bound, "decode batch 1")
    assert r < 0.1


def test_decode_batch64_bf16(arena, cuda_dev):
    _, table = arena
    T = 64
    xb = synth.f32_to_bf16(synth.token_inputs(T, seed=0))
    x = synth.bf16_to_f32(xb)                         # exact widening, as the layer sees it
    logits, _ = synth.router_inputs(T, seed=0)
    bias = np.zeros(896, np.float32)                  # flat routing
    x_t = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    y, idx, w = run_moe(cuda_dev, table, x_t, logits, bias, k3mx.K3MX_PATH_DECODE)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w, wr)
    assert len(np.unique(ir)) > 500                   # ~610 distinct experts expected
    tokens = list(range(T))
    yr, bound = moe_oracle(x, ir, wr, tokens)
    assert_within(y[tokens], yr, 1e-5 * bound, "decode batch 64")


def test_decode_host_entry_matches_device_entry(arena, cuda_dev):
    _, table = arena
    T = 3
    x = synth.token_inputs(T, seed=7)
    logits, bias = synth.router_inputs(T, seed=7)
    y_dev, _, _ = run_moe(cuda_dev, table, torch.from_numpy(x), logits, bias, k3mx.K3MX_PATH_DECODE)
    ws = torch.empty(k3mx.k3mx_moe_host_workspace_size(T, 0, 1), dtype=torch.uint8, device=cuda_dev)
    y_host = torch.full((T, 3584), float("nan"), dtype=torch.float32).pin_memory()
    k3mx.k3mx_moe_routed_host(y_host, torch.from_numpy(x).pin_memory(), table,
                              torch.from_numpy(logits), torch.from_numpy(bias), ws,
                              path=k3mx.K3MX_PATH_DECODE)
    assert np.array_equal(y_host.numpy(), y_dev)      # same kernels, deterministic


@pytest.mark.parametrize("T", [1, 3])
def test_decode_host_entry_in_place_buffers(arena, cuda_dev, T):
    """All four host buffers page-locked (the kernels may use them in place)
    and one of them pageable (copies): both equal the device entry bit for
    bit."""
    _, table = arena
    x = synth.token_inputs(T, seed=17)
    logits, bias = synth.router_inputs(T, seed=17)
    y_dev, _, _ = run_moe(cuda_dev, table, torch.from_numpy(x), logits, bias, k3mx.K3MX_PATH_DECODE)
    ws = torch.empty(k3mx.k3mx_moe_host_workspace_size(T, 0, 1), dtype=torch.uint8, device=cuda_dev)
    for pageable_bias in (False, True):
        y_host = torch.full((T, 3584), float("nan"), dtype=torch.float32).pin_memory()
        b = torch.from_numpy(bias)
        k3mx.k3mx_moe_routed_host(y_host, torch.from_numpy(x).pin_memory(), table,
                                  torch.from_numpy(logits).pin_memory(), b if pageable_bias else b.pin_memory(),
                                  ws, path=k3mx.K3MX_PATH_DECODE)
        assert np.array_equal(y_host.numpy(), y_dev), pageable_bias


def test_decode_is_deterministic(arena, cuda_dev):
    _, table = arena
    x = synth.token_inputs(5, seed=9)
    logits, bias = synth.router_inputs(5, seed=9)
    a, _, _ = run_moe(cuda_dev, table, torch.from_numpy(x), logits, bias, k3mx.K3MX_PATH_DECODE)
    b, _, _ = run_moe(cuda_dev, table, torch.from_numpy(x), logits, bias, k3mx.K3MX_PATH_DECODE)
    assert np.array_equal(a, b)


def test_decode_experts_shared_by_many_tokens(arena, cuda_dev):
    """Nine tokens routed to the same 16 experts: every expert runs for nine
    tokens (three work units of at most four), the grouping's longest lists."""
    _, table = arena
    T = 9
    x = synth.token_inputs(T, seed=21)
    logits, _ = synth.router_inputs(T, seed=21)
    bias = np.zeros(896, np.float32)
    logits[:, 100:116] += 8.0                         # the same 16 winners for every token
    y, idx, w = run_moe(cuda_dev, table, torch.from_numpy(x), logits, bias, k3mx.K3MX_PATH_DECODE)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w, wr)
    assert sorted(set(ir.ravel().tolist())) == list(range(100, 116))
    yr, bound = moe_oracle(x, ir, wr, list(range(T)))
    assert_within(y, yr, 1e-5 * bound, "shared experts")


def test_decode_routing_ties_and_crowded_keys(arena, cuda_dev):
    """The layer's one-CTA-per-token router on hard key sets, bit-exact
    against the oracle: every key equal (more than 64 candidates, the exact
    fallback), 40 equal keys around the 16th place, keys one ulp apart, and
    a bias that lifts a block of experts to the top."""
    _, table = arena
    T = 4
    x = synth.token_inputs(T, seed=31)
    logits, bias = synth.router_inputs(T, seed=31)
    logits[0, :] = 0.25                                   # all 896 keys tie
    logits[1, 300:340] = 3.0                              # 40-way tie for the top 16
    base = np.float32(1.5)
    logits[2, 500:540] = np.nextafter(base, np.float32(10), dtype=np.float32) * 0 + base
    logits[2, 500:540:2] = np.nextafter(base, np.float32(10), dtype=np.float32)
    bias = bias.copy()
    bias[700:716] = 2.0                                   # token 3's winners come from the bias
    y, idx, w = run_moe(cuda_dev, table, torch.from_numpy(x), logits, bias, k3mx.K3MX_PATH_DECODE)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w, wr)
    yr, bound = moe_oracle(x, ir, wr, list(range(T)))
    assert_within(y, yr, 1e-5 * bound, "routing ties")
