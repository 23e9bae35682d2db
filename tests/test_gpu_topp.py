"""Top-p routing (Kimi K3 engine (c/kimi_k3.c), "Streaming design": K3_TOPP)
on the GPU against the oracle: the kept experts, their order and the dropped
slots (-1) bit-exact; weights bit-equal (both sides take the same exact or
double-precision sums); grouping skips the dropped slots; the layer runs only
the kept experts on every path.  top_p goes to the oracle rounded to fp32,
the precision the C ABI takes it in."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx
import oracle
import synth
from helpers import assert_within, moe_oracle

pytestmark = pytest.mark.gpu


def f32(p):
    return float(np.float32(p))


def gpu_route_topp(dev, logits, bias, p):
    T = logits.shape[0]
    idx = torch.full((T, 16), 7, dtype=torch.int32, device=dev)
    w = torch.full((T, 16), float("nan"), dtype=torch.float32, device=dev)
    k3mx.k3mx_route_topp(idx, w, torch.from_numpy(logits).to(dev), torch.from_numpy(bias).to(dev), p)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def check_kept(idx, w):
    """The kept slots form a prefix in score order, weights sum to one."""
    kept = idx >= 0
    assert np.all(kept.sum(1) >= 1)
    assert np.all(w[~kept] == 0)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1) <= 16 * 2.0 ** -24)


@pytest.mark.parametrize("T", [1, 3, 64, 300, 4096])
@pytest.mark.parametrize("p", [0.3, 0.8, 0.95])
def test_route_topp_matches_oracle(cuda_dev, T, p):
    logits, bias = synth.router_inputs(T, seed=3)
    idx, w = gpu_route_topp(cuda_dev, logits, bias, p)
    ir, wr = oracle.route_topp(logits, bias, f32(p))
    assert np.array_equal(idx, ir), f"{np.sum(np.any(idx != ir, 1))} tokens differ"
    assert np.array_equal(w.view(np.uint32), wr.view(np.uint32))
    check_kept(idx, w)
    if T >= 64:                                       # the tail is really dropped
        assert 0 < np.mean(idx < 0) < 1


@pytest.mark.parametrize("p", [0.0, -2.0, 1.0, 3.5])
def test_route_topp_keeps_all_outside_the_unit_interval(cuda_dev, p):
    logits, bias = synth.router_inputs(64, seed=4)
    idx, w = gpu_route_topp(cuda_dev, logits, bias, p)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir)
    assert np.array_equal(w.view(np.uint32), wr.view(np.uint32))


def test_route_topp_tiny_p_keeps_the_heaviest(cuda_dev):
    """p just above zero keeps one expert per token, with weight 1."""
    logits, bias = synth.router_inputs(64, seed=5)
    idx, w = gpu_route_topp(cuda_dev, logits, bias, 1e-6)
    ir, wr = oracle.route_topp(logits, bias, f32(1e-6))
    assert np.array_equal(idx, ir)
    assert np.all((idx >= 0).sum(1) == 1) and np.all(w.max(1) == 1.0)


@pytest.mark.parametrize("case", ["all_equal", "inf_bias", "clustered", "nan_inf"])
def test_route_topp_ties_and_exact_fallbacks(cuda_dev, case):
    """Equal scores (the kept prefix is decided on exact sums and ties go to
    the lower expert index), infinite keys and crowded candidates."""
    E, T = 896, 4
    logits, bias = synth.router_inputs(T, seed=11)
    if case == "all_equal":
        logits[:] = 0.25
        bias[:] = 0.0
    elif case == "inf_bias":
        bias[100:120] = np.inf
        bias[7] = -np.inf
    elif case == "clustered":
        logits[:, :200] = 3.0
        logits[:, :200] += np.linspace(0, 1e-6, 200, dtype=np.float32)
        bias[:] = 0.0
    else:
        logits[1, 300] = np.inf                       # sigma = 1
        logits[2, :] = -np.inf                        # 4 scores of 1/2, 12 zero scores
        logits[2, 40:44] = 0.0
    for p in (0.25, 0.5, 0.75):
        idx, w = gpu_route_topp(cuda_dev, logits, bias, p)
        ir, wr = oracle.route_topp(logits, bias, f32(p))
        assert np.array_equal(idx, ir), (case, p)
        assert np.array_equal(w.view(np.uint32), wr.view(np.uint32)), (case, p)
    if case == "all_equal":                           # 16 equal scores: keep ceil(16 p)
        assert np.all((idx >= 0).sum(1) == 12)


@pytest.mark.parametrize("T", [1, 300, 4096])
def test_group_skips_dropped_slots(cuda_dev, T):
    logits, bias = synth.router_inputs(T, seed=6)
    ir, _ = oracle.route_topp(logits, bias, f32(0.7))
    counts = torch.full((896,), -1, dtype=torch.int32, device=cuda_dev)
    offsets = torch.full((897,), -1, dtype=torch.int32, device=cuda_dev)
    perm = torch.full((T * 16,), -1, dtype=torch.int32, device=cuda_dev)
    ws = torch.empty(k3mx.k3mx_group_workspace_size(T), dtype=torch.uint8, device=cuda_dev)
    k3mx.k3mx_group(counts, offsets, perm, torch.from_numpy(ir).to(cuda_dev), ws)
    st, det = k3mx.k3mx_device_status()
    assert st == 0, (st, det)                         # -1 is not an out-of-range index
    c, o, p = counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy()
    cr, orr, pr = oracle.group(ir)
    assert np.array_equal(c, cr) and np.array_equal(o, orr)
    assert o[-1] == np.sum(ir >= 0) < 16 * T
    assert np.array_equal(p[:o[-1]], pr)


def run_moe_topp(dev, table, x_t, logits, bias, path, p):
    T = x_t.shape[0]
    y = torch.full((T, 3584), float("nan"), dtype=torch.float32, device=dev)
    idx = torch.empty((T, 16), dtype=torch.int32, device=dev)
    w = torch.empty((T, 16), dtype=torch.float32, device=dev)
    dt = k3mx.K3MX_BF16 if x_t.dtype == torch.bfloat16 else k3mx.K3MX_F32
    ws = torch.empty(k3mx.k3mx_moe_workspace_size(T, dt, path), dtype=torch.uint8, device=dev)
    k3mx.k3mx_moe_routed_topp(y, x_t.to(dev), table, torch.from_numpy(logits).to(dev),
                              torch.from_numpy(bias).to(dev), ws, p, path=path, idx_out=idx, w_out=w)
    st, det = k3mx.k3mx_device_status()
    assert st == 0, (st, det)
    return y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T", [1, 5, 64])
def test_decode_topp(arena, cuda_dev, T):
    """fp32 activations on the decode path; y within sum_k w_k * (per-expert
    decode bound) of the oracle over the kept experts only."""
    _, table = arena
    p = 0.8
    x = synth.token_inputs(T, seed=8)
    logits, bias = synth.router_inputs(T, seed=8)
    y, idx, w = run_moe_topp(cuda_dev, table, torch.from_numpy(x), logits, bias, k3mx.K3MX_PATH_DECODE, p)
    ir, wr = oracle.route_topp(logits, bias, f32(p))
    assert np.array_equal(idx, ir) and np.array_equal(w.view(np.uint32), wr.view(np.uint32))
    assert np.any(ir < 0)
    tokens = list(range(T))
    yr, bound = moe_oracle(x, ir, wr, tokens)
    assert_within(y, yr, 1e-5 * bound, f"decode top-p batch {T}")


@pytest.mark.parametrize("path", [pytest.param(k3mx.K3MX_PATH_PREFILL, id="f16"),
                                  pytest.param(k3mx.K3MX_PATH_PREFILL_MX, id="mx")])
def test_prefill_topp(arena, cuda_dev, path):
    """bf16 activations, 512 tokens, p = 0.9: per sampled token the relative
    L2 error of y is at most 1e-2 (the bf16-activation tolerance)."""
    _, table = arena
    T, p = 512, 0.9
    xb = synth.f32_to_bf16(synth.token_inputs(T, seed=9))
    x = synth.bf16_to_f32(xb)
    logits, _ = synth.router_inputs(T, seed=9)
    bias = np.zeros(896, np.float32)
    x_t = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    y, idx, w = run_moe_topp(cuda_dev, table, x_t, logits, bias, path, p)
    ir, wr = oracle.route_topp(logits, bias, f32(p))
    assert np.array_equal(idx, ir) and np.array_equal(w.view(np.uint32), wr.view(np.uint32))
    assert 0 < np.mean(ir < 0) < 0.5
    assert np.all(np.isfinite(y))
    tokens = [0, 1, 100, 255, 256, 511]
    yr, _ = moe_oracle(x, ir, wr, tokens)
    for i, t in enumerate(tokens):
        rel = np.linalg.norm(y[t].astype(np.float64) - yr[i]) / np.linalg.norm(yr[i])
        assert rel <= 1e-2, f"prefill top-p: token {t} relative L2 error {rel:.3e}"
