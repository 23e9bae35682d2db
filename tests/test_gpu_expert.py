"""k3mx_expert_ffn (one full routed expert, one token) against the oracle.
Tolerance per output i: 1e-5 * sum_j |w2_ij| (|h_j| + 30 E_j), the decode
bound carried through SiTU-GLU (see the oracle's expert_bound)."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx
import oracle
import synth
from helpers import assert_within

pytestmark = pytest.mark.gpu


def run_expert(dev, buf, x):
    d = torch.from_numpy(buf).to(dev)
    ex = k3mx.expert_struct(*[d.data_ptr() + o for o in k3mx.expert_offsets()])
    y = torch.full((k3mx.K3MX_LATENT,), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(k3mx.k3mx_expert_ffn_workspace_size(), dtype=torch.uint8, device=dev)
    k3mx.k3mx_expert_ffn(y, torch.from_numpy(x).to(dev), ex, ws)
    torch.cuda.synchronize()
    # the workspace begins with g and u, [2][3072] fp32
    return y.cpu().numpy(), ws[:2 * 3072 * 4].view(torch.float32).cpu().numpy()


@pytest.mark.parametrize("expert_id,seed", [(0, 0), (511, 3)])
def test_one_routed_expert(cuda_dev, expert_id, seed):
    """x fp32 [3584] ~ N(0,1); w1, w3 [3072 x 3584], w2 [3584 x 3072], scales U{118..128}."""
    buf = synth.expert(expert_id, seed=seed, lo=118, hi=128)
    w = synth.split_expert(buf)
    x = synth.token_inputs(1, seed=seed)[0]
    y, gu = run_expert(cuda_dev, buf, x)
    yr, g, u, h = oracle.expert(x, *w, intermediates=True)
    # g = W1 x and u = W3 x between the phases, each within the GEMV bound
    assert_within(gu[:3072], g, 1e-5 * oracle.gemv_absdot(x, w[0], w[1]), "g")
    assert_within(gu[3072:], u, 1e-5 * oracle.gemv_absdot(x, w[2], w[3]), "u")
    r = assert_within(y, yr, 1e-5 * oracle.expert_bound(x, h, *w), "expert y")
    assert r < 0.1
