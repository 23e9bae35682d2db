"""The router (Kimi K3 engine (c/kimi_k3.c), "Architecture notes": the
sigmoid router [896, 7168] over the hidden state, bf16 weights) and its
top-16 against the oracle: every logit within 1e-5 * sum_c |W[e,c] h[t,c]|
of the oracle's double sum; the routing bit-exact against the oracle's
routing of the logits the GPU wrote."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def router_w(cuda_dev):
    W = synth.router_weights(seed=0)
    return W, torch.from_numpy(W.view(np.int16)).to(cuda_dev)


def run_router(dev, Wt, h, bias, top_p=0.0):
    T = h.shape[0]
    if h.dtype == np.uint16:
        ht = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        ht = torch.from_numpy(h).to(dev)
    logits = torch.full((T, 896), float("nan"), dtype=torch.float32, device=dev)
    idx = torch.full((T, 16), 7, dtype=torch.int32, device=dev)
    w = torch.full((T, 16), float("nan"), dtype=torch.float32, device=dev)
    k3mx.k3mx_router(logits, idx, w, ht, Wt, torch.from_numpy(bias).to(dev), top_p)
    torch.cuda.synchronize()
    st, det = k3mx.k3mx_device_status()
    assert st == 0, (st, det)
    return logits.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def check(W, h, lg, idx, w, bias, top_p=0.0):
    ref = oracle.router_logits(W, h)
    scale = oracle.router_absdot(W, h)
    err = np.abs(lg.astype(np.float64) - ref)
    assert np.all(err <= 1e-5 * scale), f"max err/scale {np.max(err / scale):.3e}"
    ir, wr = oracle.route_topp(lg, bias, float(np.float32(top_p))) if top_p > 0 else oracle.route(lg, bias)
    assert np.array_equal(idx, ir)
    assert np.array_equal(w.view(np.uint32), wr.view(np.uint32))
    return np.max(err / scale)


@pytest.mark.parametrize("T", [1, 3, 16, 64, 100])
def test_router_fp32_hidden(cuda_dev, router_w, T):
    W, Wt = router_w
    h = synth.hidden_inputs(T, seed=T)
    _, bias = synth.router_inputs(1, seed=T)
    lg, idx, w = run_router(cuda_dev, Wt, h, bias)
    r = check(W, h, lg, idx, w, bias)
    assert r < 2e-6
    assert 0.8 < lg.std() < 1.2                      # unit-variance logits by construction


@pytest.mark.parametrize("T", [1, 5, 16, 17, 300])
def test_router_bf16_hidden(cuda_dev, router_w, T):
    """bf16 states: CUDA cores up to 16 tokens, tensor cores from 17 (a
    ragged last tile of 256 tokens)."""
    W, Wt = router_w
    hb = synth.f32_to_bf16(synth.hidden_inputs(T, seed=40 + T))
    _, bias = synth.router_inputs(1, seed=40 + T)
    lg, idx, w = run_router(cuda_dev, Wt, hb, bias)
    check(W, hb, lg, idx, w, bias)


def test_router_bf16_prefill_4096(cuda_dev, router_w):
    """The prefill batch (16 token tiles x 7 router-row tiles): sampled
    tokens against the oracle, the routing of every token bit-exact."""
    W, Wt = router_w
    T = 4096
    hb = synth.f32_to_bf16(synth.hidden_inputs(T, seed=4096))
    _, bias = synth.router_inputs(1, seed=4096)
    lg, idx, w = run_router(cuda_dev, Wt, hb, bias)
    tokens = np.array([0, 1, 255, 256, 1000, 2047, 3840, 4095])
    ref = oracle.router_logits(W, hb[tokens])
    scale = oracle.router_absdot(W, hb[tokens])
    assert np.all(np.abs(lg[tokens].astype(np.float64) - ref) <= 1e-5 * scale)
    ir, wr = oracle.route(lg, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w.view(np.uint32), wr.view(np.uint32))


def test_router_top_p(cuda_dev, router_w):
    W, Wt = router_w
    h = synth.hidden_inputs(8, seed=77)
    _, bias = synth.router_inputs(1, seed=77)
    lg, idx, w = run_router(cuda_dev, Wt, h, bias, top_p=0.7)
    check(W, h, lg, idx, w, bias, top_p=0.7)
    assert np.any(idx < 0)


def test_router_one_hot_columns(cuda_dev, router_w):
    """One-hot hidden states read columns of W exactly."""
    W, Wt = router_w
    cols = [0, 1, 4095, 7167]
    h = np.zeros((len(cols), 7168), np.float32)
    for t, c in enumerate(cols):
        h[t, c] = 1.0
    bias = np.zeros(896, np.float32)
    lg, _, _ = run_router(cuda_dev, Wt, h, bias)
    for t, c in enumerate(cols):
        assert np.array_equal(lg[t], synth.bf16_to_f32(W[:, c]))
