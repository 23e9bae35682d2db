"""Parity at the edges of the MXFP4 format and of the activations, on every
tensor-core path, against the oracle:
  - experts whose groups take scale 255 ("NaN: contributes nothing"), 0, 1
    and 254 (helpers.edge_expert_bytes) through k3mx_expert_ffn, the decode
    path at 1 and 64 tokens and both prefill paths;
  - activations with one large value per 32-column block, blocks of mixed
    magnitudes, all-zero blocks and scaled tokens, through the same paths.
Decode outputs hold the per-output bound sum_k w_k * 1e-5 * expert_bound;
prefill outputs hold relative L2 <= 1e-2 per token.  A row of only NaN
groups gives exactly 0."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx
import oracle
import synth
from helpers import (EDGE_ROWS, arena_expert, arena_expert_bytes, assert_within, edge_expert_bytes, moe_oracle,
                     moe_oracle_rows)

pytestmark = pytest.mark.gpu

N_EDGE = 32                 # distinct edge experts; table entry e uses edge expert e % 32
EXPERT_BYTES = synth.expert_nbytes()


@pytest.fixture(scope="module")
def edge_table(cuda_dev):
    buf = torch.empty(N_EDGE * EXPERT_BYTES, dtype=torch.uint8, device=cuda_dev)
    for i in range(N_EDGE):
        buf[i * EXPERT_BYTES:(i + 1) * EXPERT_BYTES].copy_(torch.from_numpy(edge_expert_bytes(i)))
    base = buf.data_ptr()
    offs = torch.tensor(k3mx.expert_offsets(), dtype=torch.int64)
    ent = torch.arange(896, dtype=torch.int64) % N_EDGE
    table = (base + ent[:, None] * EXPERT_BYTES + offs[None, :]).to(cuda_dev)
    torch.cuda.synchronize()
    yield buf, table
    del buf, table
    torch.cuda.empty_cache()


def edge_bytes_of_entry(e):
    return edge_expert_bytes(e % N_EDGE)


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


def decode_bound(x, idx, w, tokens, expert_bytes):
    """sum_k w_tk * 1e-5 * expert_bound per output of each listed token."""
    out = []
    for t in tokens:
        b = np.zeros(x.shape[1])
        for k in range(idx.shape[1]):
            e = int(idx[t, k])
            if e < 0:
                continue
            ex = synth.split_expert(expert_bytes(e))
            _, _, _, h = oracle.expert(x[t], *ex, intermediates=True)
            b += float(w[t, k]) * 1e-5 * oracle.expert_bound(x[t], h, *ex)
        out.append(b)
    return np.array(out)


# ---------------------------------------------------------- activations --

def activation_cases(T, seed):
    """fp32 [T, 3584] rows cycling through five recipes:
    0 one value per 32-column block scaled by 1e3 (outliers);
    1 every value scaled by 10^U(-3, 3) (mixed magnitudes in every block);
    2 30% of the blocks all zero;
    3 the token scaled by 1e2;
    4 the token scaled by 1e-6."""
    x = synth.token_inputs(T, seed=seed).astype(np.float64)
    rng = np.random.default_rng(seed)
    for t in range(T):
        kind = t % 5
        if kind == 0:
            j = rng.integers(0, 32, 112) + np.arange(0, 3584, 32)
            x[t, j] *= 1e3
        elif kind == 1:
            x[t] *= 10.0 ** rng.uniform(-3, 3, 3584)
        elif kind == 2:
            blocks = rng.random(112) < 0.3
            x[t].reshape(112, 32)[blocks] = 0.0
        elif kind == 3:
            x[t] *= 1e2
        else:
            x[t] *= 1e-6
    return x.astype(np.float32)


# -------------------------------------------------------------- one expert --

def test_expert_ffn_edge_scales(cuda_dev):
    """k3mx_expert_ffn on an edge expert: g, u within the GEMV bound, y within
    the expert bound, and the all-NaN rows exactly 0."""
    buf = edge_expert_bytes(0)
    w = synth.split_expert(buf)
    x = synth.token_inputs(1, seed=41)[0]
    d = torch.from_numpy(buf).to(cuda_dev)
    ex = k3mx.expert_struct(*[d.data_ptr() + o for o in k3mx.expert_offsets()])
    y = torch.full((3584,), float("nan"), dtype=torch.float32, device=cuda_dev)
    ws = torch.empty(k3mx.k3mx_expert_ffn_workspace_size(), dtype=torch.uint8, device=cuda_dev)
    k3mx.k3mx_expert_ffn(y, torch.from_numpy(x).to(cuda_dev), ex, ws)
    st, det = k3mx.k3mx_device_status()
    assert st == 0, (st, det)
    y = y.cpu().numpy()
    gu = ws[:2 * 3072 * 4].view(torch.float32).cpu().numpy()
    yr, g, u, h = oracle.expert(x, *w, intermediates=True)
    assert_within(gu[:3072], g, 1e-5 * oracle.gemv_absdot(x, w[0], w[1]), "g")
    assert_within(gu[3072:], u, 1e-5 * oracle.gemv_absdot(x, w[2], w[3]), "u")
    assert_within(y, yr, 1e-5 * oracle.expert_bound(x, h, *w), "y")
    r = EDGE_ROWS["nan"]
    assert gu[r] == 0.0 and gu[3072 + r] == 0.0 and y[r] == 0.0
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(gu))


@pytest.mark.parametrize("kind", [0, 1, 2, 3, 4])
def test_expert_ffn_activation_cases(arena, cuda_dev, kind):
    """One expert, one token from each activation recipe."""
    x = activation_cases(5, seed=43)[kind]
    w = arena_expert(17)
    buf, _ = arena
    base = buf.data_ptr() + 17 * EXPERT_BYTES
    ex = k3mx.expert_struct(*[base + o for o in k3mx.expert_offsets()])
    y = torch.full((3584,), float("nan"), dtype=torch.float32, device=cuda_dev)
    ws = torch.empty(k3mx.k3mx_expert_ffn_workspace_size(), dtype=torch.uint8, device=cuda_dev)
    k3mx.k3mx_expert_ffn(y, torch.from_numpy(x).to(cuda_dev), ex, ws)
    st, det = k3mx.k3mx_device_status()
    assert st == 0, (st, det)
    yr, g, u, h = oracle.expert(x, *w, intermediates=True)
    gu = ws[:2 * 3072 * 4].view(torch.float32).cpu().numpy()
    assert_within(gu[:3072], g, 1e-5 * oracle.gemv_absdot(x, w[0], w[1]), f"g, recipe {kind}")
    assert_within(gu[3072:], u, 1e-5 * oracle.gemv_absdot(x, w[2], w[3]), f"u, recipe {kind}")
    assert_within(y.cpu().numpy(), yr, 1e-5 * oracle.expert_bound(x, h, *w), f"y, recipe {kind}")


# ---------------------------------------------------------------- decode --

def test_decode_batch1_edge_experts(edge_table, cuda_dev):
    _, table = edge_table
    x = synth.token_inputs(1, seed=45)
    logits, bias = synth.router_inputs(1, seed=45)
    y, idx, w = run_moe(cuda_dev, table, torch.from_numpy(x), logits, bias, k3mx.K3MX_PATH_DECODE)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w, wr)
    yr = moe_oracle_rows(x, ir, wr, [0], edge_bytes_of_entry)
    assert_within(y, yr, decode_bound(x, ir, wr, [0], edge_bytes_of_entry), "decode batch 1, edge experts")
    assert y[0, EDGE_ROWS["nan"]] == 0.0


def test_decode_batch64_edge_experts(edge_table, cuda_dev):
    _, table = edge_table
    T = 64
    xb = synth.f32_to_bf16(synth.token_inputs(T, seed=46))
    x = synth.bf16_to_f32(xb)
    logits, _ = synth.router_inputs(T, seed=46)
    bias = np.zeros(896, np.float32)
    x_t = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    y, idx, w = run_moe(cuda_dev, table, x_t, logits, bias, k3mx.K3MX_PATH_DECODE)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w, wr)
    tokens = list(range(0, T, 3))
    yr = moe_oracle_rows(x, ir, wr, tokens, edge_bytes_of_entry)
    assert_within(y[tokens], yr, decode_bound(x, ir, wr, tokens, edge_bytes_of_entry), "decode batch 64, edge")
    assert np.all(y[:, EDGE_ROWS["nan"]] == 0.0)


@pytest.mark.parametrize("T", [1, 10])
def test_decode_activation_cases(arena, cuda_dev, T):
    """The decode path (one token: the fused pass; ten: the batched pass) on
    the activation recipes, fp32."""
    _, table = arena
    x = activation_cases(T, seed=47 + T)
    if T == 1:
        x = activation_cases(5, seed=48)[0:1]           # the outlier recipe
    logits, bias = synth.router_inputs(T, seed=47)
    y, idx, w = run_moe(cuda_dev, table, torch.from_numpy(x), logits, bias, k3mx.K3MX_PATH_DECODE)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w, wr)
    tokens = list(range(T))
    yr, bound = moe_oracle(x, ir, wr, tokens)
    assert_within(y, yr, 1e-5 * bound, f"decode activation recipes, T={T}")


# --------------------------------------------------------------- prefill --

PATHS = [pytest.param(k3mx.K3MX_PATH_PREFILL, id="f16"), pytest.param(k3mx.K3MX_PATH_PREFILL_MX, id="mx")]


def run_prefill(dev, table, x, logits, bias, path):
    xb = synth.f32_to_bf16(x)
    x_t = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    y, idx, w = run_moe(dev, table, x_t, logits, bias, path)
    return y, idx, w, synth.bf16_to_f32(xb)


def check_rel(y, yr, tokens, what):
    worst = 0.0
    for i, t in enumerate(tokens):
        rel = np.linalg.norm(y[t].astype(np.float64) - yr[i]) / np.linalg.norm(yr[i].astype(np.float64))
        assert rel <= 1e-2, f"{what}: token {t} relative L2 error {rel:.3e}"
        worst = max(worst, rel)
    return worst


@pytest.mark.parametrize("path", PATHS)
def test_prefill_edge_experts(edge_table, cuda_dev, path):
    """400 tokens through the 32 edge experts (about 200 pairs each, split
    over the 896 table entries), flat routing."""
    _, table = edge_table
    T = 400
    x = synth.token_inputs(T, seed=51)
    logits, _ = synth.router_inputs(T, seed=51)
    bias = np.zeros(896, np.float32)
    y, idx, w, xw = run_prefill(cuda_dev, table, x, logits, bias, path)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir) and np.array_equal(w, wr)
    assert np.all(np.isfinite(y))
    tokens = list(range(0, T, 25))
    yr = moe_oracle_rows(xw, ir, wr, tokens, edge_bytes_of_entry)
    check_rel(y, yr, tokens, "prefill, edge experts")
    assert np.all(y[:, EDGE_ROWS["nan"]] == 0.0)


@pytest.mark.parametrize("path", PATHS)
def test_prefill_activation_cases(arena, cuda_dev, path):
    """500 bf16 tokens cycling through the five activation recipes.  The
    f16-dequant path keeps h in f16 (the operand type of its kind::f16 MMAs),
    whose normal range ends at 2^-14; recipe 4 (x scaled by 1e-6, so
    |h| ~ 1e-12) lies below it and is checked on the block-scaled path
    only, which stages h scaled per 32-feature block."""
    _, table = arena
    T = 500
    x = activation_cases(T, seed=53)
    logits, _ = synth.router_inputs(T, seed=53)
    bias = np.zeros(896, np.float32)
    y, idx, w, xw = run_prefill(cuda_dev, table, x, logits, bias, path)
    ir, wr = oracle.route(logits, bias)
    assert np.array_equal(idx, ir)
    assert np.all(np.isfinite(y))
    tokens = [t for t in range(0, T, 7)][:40]
    if path == k3mx.K3MX_PATH_PREFILL:
        tokens = [t for t in tokens if t % 5 != 4]
    yr = moe_oracle_rows(xw, ir, wr, tokens, arena_expert_bytes)
    check_rel(y, yr, tokens, "prefill activation recipes")
