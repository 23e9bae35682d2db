"""k3mx_gemv against the oracle: |y - y_oracle| <= 1e-5 * sum_c |w_rc| |x_c|
per row (the decode tolerance of the routed-expert layer)."""
import numpy as np
import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx
import oracle
import synth
from helpers import assert_within

pytestmark = pytest.mark.gpu


def run_gemv(dev, p, s, x):
    y = torch.full((p.shape[0],), float("nan"), dtype=torch.float32, device=dev)
    k3mx.k3mx_gemv(y, torch.from_numpy(x).to(dev), torch.from_numpy(p).to(dev), torch.from_numpy(s).to(dev))
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("rows,cols", [(1, 32), (7, 64), (61, 512), (3, 3584), (129, 3072),
                                       (1000, 3584), (33, 16384)])
def test_gemv_shapes_and_ragged_tails(cuda_dev, rows, cols):
    p, s, x = synth.gemv_inputs(seed=rows + cols, rows=rows, cols=cols)
    y = run_gemv(cuda_dev, p, s, x)
    assert_within(y, oracle.gemv(x, p, s), 1e-5 * oracle.gemv_absdot(x, p, s), f"gemv {rows}x{cols}")


def test_gemv_full_single_matrix_workload(cuda_dev):
    """W 3072 x 3584, scales U{120..130} with 1% NaN, x ~ N(0,1), seed 0."""
    p, s, x = synth.gemv_inputs(seed=0)
    y = run_gemv(cuda_dev, p, s, x)
    r = assert_within(y, oracle.gemv(x, p, s), 1e-5 * oracle.gemv_absdot(x, p, s), "gemv 3072x3584")
    assert r < 0.1           # observed error is far inside the bound


def test_gemv_nibble_order_sign_and_scale(cuda_dev):
    packed = np.zeros((2, 16), np.uint8)
    packed[0, 0] = 0x72                 # col 0: +1.0, col 1: +6.0
    packed[0, 1] = 0xA9                 # col 2: -0.5, col 3: -1.0
    packed[1, :] = 0x8F                 # col even: -6 (code 15), col odd: -0 (code 8); x 2^-1
    scales = np.array([[128], [126]], np.uint8)
    for c, expect in enumerate([(2.0, -3.0), (12.0, -0.0), (-1.0, -3.0), (-2.0, -0.0)]):
        x = np.zeros(32, np.float32)
        x[c] = 1.0
        y = run_gemv(cuda_dev, packed, scales, x)
        assert y[0] == expect[0] and y[1] == expect[1], (c, y)


def test_gemv_scale_edges_and_nan_groups(cuda_dev):
    rng = np.random.default_rng(5)
    rows, cols = 6, 128
    p = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    s = np.array([[0] * 4, [1] * 4, [127] * 4, [254] * 4, [255] * 4, [255, 127, 255, 0]], np.uint8)
    x = rng.standard_normal(cols).astype(np.float32) * 1e-3
    x[0] = np.inf                       # only under NaN groups of rows 4 and 5
    s[:4, 0] = 255
    y = run_gemv(cuda_dev, p, s, x)
    ref = oracle.gemv(x, p, s)
    assert y[4] == 0.0 and np.all(np.isfinite(y))
    assert_within(y, ref, 1e-5 * oracle.gemv_absdot(np.where(np.isinf(x), 0, x), p, s) + 1e-45, "scale edges")
