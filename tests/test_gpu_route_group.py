"""Routing and grouping against the oracle: indices, counts, offsets and the
pair order bit-exact; weights within 1e-6 (and expected bit-equal, since both
sides take the same double-precision steps)."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx
import oracle
import synth

pytestmark = pytest.mark.gpu


def gpu_route(dev, logits, bias):
    T = logits.shape[0]
    idx = torch.full((T, 16), -1, dtype=torch.int32, device=dev)
    w = torch.full((T, 16), float("nan"), dtype=torch.float32, device=dev)
    k3mx.k3mx_route_topk(idx, w, torch.from_numpy(logits).to(dev), torch.from_numpy(bias).to(dev))
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def gpu_group(dev, idx):
    T = idx.shape[0]
    counts = torch.full((896,), -1, dtype=torch.int32, device=dev)
    offsets = torch.full((897,), -1, dtype=torch.int32, device=dev)
    perm = torch.full((T * 16,), -1, dtype=torch.int32, device=dev)
    ws = torch.empty(k3mx.k3mx_group_workspace_size(T), dtype=torch.uint8, device=dev)
    k3mx.k3mx_group(counts, offsets, perm, torch.from_numpy(np.ascontiguousarray(idx)).to(dev), ws)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy()


@pytest.mark.parametrize("T", [1, 3, 64, 4096])
def test_route_matches_oracle(cuda_dev, T):
    logits, bias = synth.router_inputs(T, seed=0)
    idx, w = gpu_route(cuda_dev, logits, bias)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir), f"{np.sum(np.any(idx != ir, 1))} tokens differ"
    assert np.max(np.abs(w - wr)) <= 1e-6
    assert np.array_equal(w.view(np.uint32), wr.view(np.uint32))
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1) <= 16 * 2.0 ** -24)


def test_route_ties_bias_and_special_keys(cuda_dev):
    E = 896
    logits = np.zeros((6, E), np.float32)
    bias = np.zeros(E, np.float32)
    bias[16:32] = 0.5                    # row 1..5: biased experts win; weights stay raw
    logits[0, 16:32] = -12.0
    for t in range(1, 6):
        logits[t, 16:32] = np.linspace(0.2 + 0.1 * t, 1.6, 16)
    logits[2, 100] = np.nan              # a NaN score ranks last
    logits[3, 200] = np.inf              # sigma = 1: a clear winner
    logits[4, 300] = -np.inf             # sigma = 0
    bias[5] = -0.0
    idx, w = gpu_route(cuda_dev, logits, bias)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir)
    assert np.array_equal(w.view(np.uint32), wr.view(np.uint32))
    # row 0: sigma(-12) + 0.5 > sigma(0) + 0, so the bias lifts experts 16..31
    assert sorted(idx[0]) == list(range(16, 32))


@pytest.mark.parametrize("T", [1, 64, 300, 4096])
def test_group_matches_oracle(cuda_dev, T):
    logits, bias = synth.router_inputs(T, seed=1)
    ir, _ = oracle.route(logits, bias)
    c, o, p = gpu_group(cuda_dev, ir)
    cr, orr, pr = oracle.group(ir)
    assert np.array_equal(c, cr) and np.array_equal(o, orr) and np.array_equal(p, pr)


def test_group_skewed_routing(cuda_dev):
    """Every token on the same 16 experts, one expert per slot: the longest
    per-expert lists, and a stable order within each."""
    T = 2048
    idx = np.tile(np.arange(880, 896, dtype=np.int32), (T, 1))
    idx[::7] = idx[::7, ::-1]
    c, o, p = gpu_group(cuda_dev, idx)
    cr, orr, pr = oracle.group(idx)
    assert np.array_equal(c, cr) and np.array_equal(o, orr) and np.array_equal(p, pr)


@pytest.mark.parametrize("case", ["all_equal", "inf_bias", "clustered"])
def test_route_exact_fallbacks(cuda_dev, case):
    """Cases where the fp32 candidate filter keeps more than 64 experts or
    meets infinite keys, so the exact all-expert path decides."""
    E, T = 896, 4
    logits, bias = synth.router_inputs(T, seed=11)
    if case == "all_equal":
        logits[:] = 0.25
        bias[:] = 0.0
    elif case == "inf_bias":
        bias[100:120] = np.inf
        bias[7] = -np.inf
    else:
        logits[:, :200] = 3.0                    # 200 experts within float rounding of each other
        logits[:, :200] += np.linspace(0, 1e-6, 200, dtype=np.float32)
        bias[:] = 0.0
    idx, w = gpu_route(cuda_dev, logits, bias)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir)
    assert np.array_equal(w.view(np.uint32), wr.view(np.uint32))
