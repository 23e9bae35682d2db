"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: values the
pages print (tests/golden), the e2m1 bit definition, brute force on tiny
shapes through numpy, closed forms, a full sort, invariants.  A plausible
mistake in the oracle (a swapped nibble, a wrong sign or scale offset, a
transposed matrix, g and u exchanged, bias used as a weight, an unstable
grouping) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from conftest import read_golden


# ---------------------------------------------------------------- decoding --

def e2m1_from_bits(code):
    """e2m1 from its bit fields: 1 sign (bit 3), 2 exponent bits (bias 1),
    1 mantissa bit; exponent 0 is subnormal (0.5 * mantissa)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else (2.0 ** (e - 1)) * (1.0 + 0.5 * m)
    return -mag if s else mag


def test_e2m1_table_matches_bit_definition_and_pages():
    gold = read_golden("e2m1_magnitudes.txt")
    for code in range(16):
        v = oracle.e2m1(code)
        assert v == e2m1_from_bits(code)
        assert abs(v) == float(gold[str(code & 7)])
        assert math.copysign(1.0, v) == (-1.0 if code & 8 else 1.0)   # -0 for code 8


def test_e8m0_scale():
    assert oracle.e8m0(127) == 1.0
    assert oracle.e8m0(128) == 2.0
    assert oracle.e8m0(118) == 2.0 ** -9
    assert oracle.e8m0(0) == 2.0 ** -127
    assert oracle.e8m0(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0(255))


def dequant(packed, scales):
    """Brute-force dequantisation to a float64 matrix (NaN groups -> 0),
    written from the layout: byte j of a row holds columns 2j (low nibble)
    and 2j+1 (high nibble); one scale byte per 32 columns."""
    rows, half = packed.shape
    lo = packed & 15
    hi = packed >> 4
    codes = np.empty((rows, 2 * half), np.int64)
    codes[:, 0::2] = lo
    codes[:, 1::2] = hi
    lut = np.array([e2m1_from_bits(c) for c in range(16)])
    W = lut[codes]
    sc = np.repeat(scales.astype(np.int64), 32, axis=1)
    mult = np.where(sc == 255, 0.0, np.ldexp(1.0, sc - 127))
    return W * mult


# ---------------------------------------------------------------- sizes --

def test_expert_census_from_dimensions():
    gold = read_golden("expert_census.txt")
    cfg = read_golden("k3cfg_moe.txt")
    D, F, G = int(cfg["latent"]), int(cfg["moe_inter"]), int(cfg["mxfp4_group"])
    params = 3 * F * D                                  # w1, w3 [F x D]; w2 [D x F]
    nbytes = params // 2 + params // G                  # nibbles + one scale byte per 32
    assert params == int(gold["params_per_expert"])
    assert nbytes == int(gold["bytes_per_expert"])
    assert nbytes / params == float(gold["bytes_per_param"])
    assert int(gold["routed_experts_per_layer"]) * int(gold["moe_layers"]) == int(gold["experts_total"])
    # 82,432 x 17,547,264 B = 1.44645 TB; the page prints 1.447 (its last digit
    # rounds up), so the pin allows one unit in the printed last place
    assert abs(int(gold["experts_total"]) * nbytes / 1e12 - float(gold["routed_expert_set_bytes_tb"])) <= 1e-3
    per_tok = int(gold["moe_layers"]) * int(cfg["topk"])
    assert per_tok == int(gold["experts_per_token"])
    assert round(per_tok * nbytes / 1e9, 2) == float(gold["packed_bytes_per_token_gb"])
    # the generator lays out exactly that many bytes per expert
    assert synth.expert_nbytes(D, F) == nbytes
    assert (D, F) == (synth.D_LATENT, synth.F_INTER)
    assert int(cfg["n_experts"]) == synth.N_EXPERTS and int(cfg["topk"]) == synth.TOP_K


# ---------------------------------------------------------------- gemv --

@pytest.mark.parametrize("rows,n_in", [(1, 32), (3, 64), (4, 96), (2, 160)])
def test_gemv_brute_force_tiny(rows, n_in):
    rng = np.random.default_rng(rows * 1000 + n_in)
    packed = rng.integers(0, 256, (rows, n_in // 2), dtype=np.uint8)
    scales = rng.integers(110, 140, (rows, n_in // 32), dtype=np.uint8)
    scales[0, 0] = 255
    x = rng.standard_normal(n_in).astype(np.float32)
    W = dequant(packed, scales)
    ref = W @ x.astype(np.float64)
    y = oracle.gemv(x, packed, scales)
    absdot = np.abs(W) @ np.abs(x.astype(np.float64))
    # group-wise vs whole-row double order: ~1e-16 relative; then one fp32 rounding
    assert np.all(np.abs(y - ref) <= 2.0 ** -24 * np.abs(ref) + 1e-12 * absdot)


def test_gemv_exact_on_integer_inputs():
    """Scale 127 and small integer x: every value is exact, so y is exact."""
    rng = np.random.default_rng(7)
    rows, n_in = 4, 96
    packed = rng.integers(0, 256, (rows, n_in // 2), dtype=np.uint8)
    scales = np.full((rows, n_in // 32), 127, np.uint8)
    x = rng.integers(-8, 9, n_in).astype(np.float32)
    ref = dequant(packed, scales) @ x.astype(np.float64)
    assert np.array_equal(oracle.gemv(x, packed, scales).astype(np.float64), ref)


def test_gemv_nibble_order_and_sign():
    """Byte 0x72: low nibble 2 (1.0) is column 0, high nibble 7 (6.0) column 1.
    Byte 0xA9: low nibble 9 (-0.5) column 2, high nibble 10 (-1.0) column 3."""
    packed = np.zeros((1, 16), np.uint8)
    packed[0, 0] = 0x72
    packed[0, 1] = 0xA9
    scales = np.full((1, 1), 128, np.uint8)           # x2
    expect = [2.0, 12.0, -1.0, -2.0]
    for c, e in enumerate(expect):
        x = np.zeros(32, np.float32)
        x[c] = 1.0
        assert oracle.gemv(x, packed, scales)[0] == e


def test_gemv_one_hot_is_a_column():
    p, s, _ = synth.gemv_inputs(seed=3, rows=8, cols=128, nan_frac=0.0)
    W = dequant(p, s)
    for c in (0, 1, 31, 32, 127):
        x = np.zeros(128, np.float32)
        x[c] = 1.0
        assert np.array_equal(oracle.gemv(x, p, s).astype(np.float64), W[:, c].astype(np.float32))


def test_gemv_nan_scale_groups_contribute_nothing():
    rng = np.random.default_rng(11)
    rows, n_in = 3, 128
    packed = rng.integers(0, 256, (rows, n_in // 2), dtype=np.uint8)
    scales = rng.integers(120, 131, (rows, n_in // 32), dtype=np.uint8)
    x = rng.standard_normal(n_in).astype(np.float32) * 1e3
    scales[0, :] = 255                                   # a row of NaN groups is exactly 0
    y = oracle.gemv(x, packed, scales)
    assert y[0] == 0.0
    # turning group 2 of row 1 into NaN removes exactly that group's sub-sum
    before = dequant(packed, scales)[1] @ x.astype(np.float64)
    s2 = scales.copy()
    s2[1, 2] = 255
    sub = dequant(packed, scales)[1, 64:96] @ x[64:96].astype(np.float64)
    after = oracle.gemv(x, packed, s2)[1]
    assert abs(after - (before - sub)) <= 2.0 ** -23 * abs(before - sub) + 1e-9
    # NaN / inf in x under a NaN group stays out of the sum
    x2 = x.copy()
    x2[0] = np.inf
    assert oracle.gemv(x2, packed, scales)[0] == 0.0


def test_gemv_reassociation_bound_full_size():
    """Group-wise double sums against dequantise-then-multiply on the full
    3072 x 3584 workload: the pages bound the reordering at about 1e-16
    relative and gate at 1e-6 (kimi-k3-in-c article, "A floating-point
    contract, not a convention")."""
    p, s, x = synth.gemv_inputs(seed=0)
    W = dequant(p, s)
    ref = W @ x.astype(np.float64)
    absdot = np.abs(W) @ np.abs(x.astype(np.float64))
    y = oracle.gemv(x, p, s).astype(np.float64)
    assert np.all(np.abs(y - ref) <= 2.0 ** -24 * np.abs(ref) + 1e-12 * absdot)
    b = oracle.gemv_absdot(x, p, s)
    assert np.allclose(b, absdot, rtol=1e-12, atol=0)


# ---------------------------------------------------------------- SiTU --

def test_situ_closed_forms():
    # either factor zero -> zero
    for u in (-50.0, -1.0, 0.3, 80.0):
        assert oracle.situ(0.0, u) == 0.0
    for g in (-7.0, 0.1, 9.0):
        assert oracle.situ(g, 0.0) == 0.0
    # g -> +inf: 4 tanh(g/4) sigma(g) -> 4, so h -> 100 tanh(u/25)
    for u in (-30.0, 2.0, 25.0):
        assert oracle.situ(80.0, u) == pytest.approx(100.0 * math.tanh(u / 25.0), rel=1e-12)
    # g -> -inf: sigma(g) -> 0 faster than tanh saturates
    assert abs(oracle.situ(-80.0, 10.0)) < 1e-30
    # u -> +inf: 25 tanh(u/25) -> 25, so h -> 100 tanh(g/4) sigma(g);
    # at g = 2: tanh(0.5) = 0.46211715726000974, sigma(2) = 0.8807970779778823
    assert oracle.situ(2.0, 2000.0) == pytest.approx(100 * 0.46211715726000974 * 0.8807970779778823, rel=1e-12)
    # first order at the origin: h ~ (g/2) * u
    g, u = 1e-5, 3e-5
    assert oracle.situ(g, u) == pytest.approx(0.5 * g * u, rel=1e-4)
    # sign structure: odd in u, not in g
    assert oracle.situ(1.5, -4.0) == -oracle.situ(1.5, 4.0)
    assert oracle.situ(-1.5, 4.0) != -oracle.situ(1.5, 4.0)
    # sigma itself
    assert oracle.sigmoid(0.0) == 0.5
    for z in (-3.0, 0.7, 12.0):
        assert oracle.sigmoid(z) + oracle.sigmoid(-z) == pytest.approx(1.0, abs=4e-16)


def brute_expert(x, w1p, w1s, w3p, w3s, w2p, w2s):
    """numpy expert on dequantised matrices (tiny shapes only)."""
    xd = x.astype(np.float64)
    g = (dequant(w1p, w1s) @ xd).astype(np.float32)
    u = (dequant(w3p, w3s) @ xd).astype(np.float32)
    return g, u, dequant(w2p, w2s)


def test_expert_composition_tiny():
    """g = W1 x, u = W3 x, y = W2 h on a D=96, F=64 expert."""
    D, F = 96, 64
    buf = synth.expert(5, seed=9, D=D, F=F)
    w = synth.split_expert(buf, D=D, F=F)
    x = synth.token_inputs(1, seed=9, D=D)[0]
    y, g, u, h = oracle.expert(x, *w, intermediates=True)
    g_ref, u_ref, W2 = brute_expert(x, *w)
    assert np.array_equal(g, g_ref) or np.allclose(g, g_ref, rtol=2 ** -23, atol=0)
    assert np.allclose(u, u_ref, rtol=2 ** -23, atol=0)
    # h is SiTU of (g, u) with g from W1: at saturation limits the roles differ
    big = np.abs(g) > 60
    if big.any():
        expect = np.where(g[big] > 0, 100 * np.tanh(u[big].astype(np.float64) / 25), 0.0)
        assert np.allclose(h[big], expect, rtol=1e-6, atol=1e-6)
    y_ref = W2 @ h.astype(np.float64)
    absdot = np.abs(W2) @ np.abs(h.astype(np.float64))
    assert np.all(np.abs(y - y_ref) <= 2.0 ** -24 * np.abs(y_ref) + 1e-12 * absdot)


def test_expert_bound_brute_force_tiny():
    """The decode tolerance helper, brute force on a D=96, F=64 expert with
    NaN groups: bound_i = sum_j |w2_ij| (|h_j| + 30 E_j) with
    E_j = sum_c (|w1_jc| + |w3_jc|) |x_c|, NaN groups excluded, from the
    dequantised matrices.  A wrong factor, a dropped term or a NaN group
    counted changes the result by far more than rounding."""
    D, F = 96, 64
    buf = synth.expert(6, seed=10, D=D, F=F, nan_frac=0.05)
    w = synth.split_expert(buf, D=D, F=F)
    x = synth.token_inputs(1, seed=10, D=D)[0]
    _, _, _, h = oracle.expert(x, *w, intermediates=True)
    b = oracle.expert_bound(x, h, *w)
    W1, W3, W2 = dequant(w[0], w[1]), dequant(w[2], w[3]), dequant(w[4], w[5])
    E = (np.abs(W1) + np.abs(W3)) @ np.abs(x.astype(np.float64))
    ref = np.abs(W2) @ (np.abs(h.astype(np.float64)) + 30.0 * E)
    assert np.allclose(b, ref, rtol=1e-12, atol=0)
    assert (w[1] == 255).any() and (w[5] == 255).any()


def test_expert_bound_covers_admissible_errors():
    """What the bound is for: if g and u each move by at most 1e-5 of their
    GEMV bound (sum_c |w_jc| |x_c|) and h by at most 1e-5 |h|, y moves by at
    most 1e-5 * bound.  Checked in double on a tiny expert with the signs of
    the moves set against each output row (the worst case of a linear
    model) and with random moves, through the exact SiTU-GLU."""
    D, F = 96, 64
    buf = synth.expert(7, seed=11, D=D, F=F, nan_frac=0.02)
    w = synth.split_expert(buf, D=D, F=F)
    rng = np.random.default_rng(11)
    W1, W3, W2 = dequant(w[0], w[1]), dequant(w[2], w[3]), dequant(w[4], w[5])
    situ = np.vectorize(oracle.situ)
    for scale in (0.05, 1.0, 20.0):
        x = (synth.token_inputs(1, seed=12, D=D)[0] * scale).astype(np.float32)
        xd = x.astype(np.float64)
        g, u = W1 @ xd, W3 @ xd
        h = situ(g, u)
        b = oracle.expert_bound(x, h.astype(np.float32), *w)
        e1 = 1e-5 * (np.abs(W1) @ np.abs(xd))
        e3 = 1e-5 * (np.abs(W3) @ np.abs(xd))
        for trial in range(6):
            if trial < 2:
                sg = np.sign(W2[trial]) if trial == 0 else -np.sign(W2[trial])
                dg, du = sg * e1, sg * e3
            else:
                dg, du = rng.uniform(-1, 1, F) * e1, rng.uniform(-1, 1, F) * e3
            h2 = situ(g + dg, u + du)
            h2 = h2 + rng.uniform(-1, 1, F) * 1e-5 * np.abs(h2)
            dy = np.abs(W2 @ h2 - W2 @ h)
            assert np.all(dy <= 1e-5 * b * (1 + 1e-9)), (scale, trial, np.max(dy / (1e-5 * b)))


def test_expert_w1_is_gate():
    """Zeroing W3 (u = 0) zeroes h; zeroing W1 (g = 0) zeroes h too, but a
    large positive W1 row saturates the gate so h = 100 tanh(u/25)."""
    D, F = 64, 32
    w1p, w1s, w3p, w3s, w2p, w2s = [a.copy() for a in synth.split_expert(synth.expert(1, seed=2, D=D, F=F), D=D, F=F)]
    x = np.ones(D, np.float32)
    w1p[:] = 0x77                                         # every weight +6
    w1s[:] = 127                                          # g = 6 * 64 = 384
    _, g, u, h = oracle.expert(x, w1p, w1s, w3p, w3s, w2p, w2s, intermediates=True)
    assert np.all(g == 384.0)
    assert np.allclose(h, 100 * np.tanh(u.astype(np.float64) / 25), rtol=1e-7, atol=1e-6)
    w3p[:] = 0
    _, g, u, h = oracle.expert(x, w1p, w1s, w3p, w3s, w2p, w2s, intermediates=True)
    assert np.all(u == 0.0) and np.all(h == 0.0)


# ---------------------------------------------------------------- routing --

def brute_route(s, bias, k):
    """full sort of (key, e) with key = fp32(s + bias); -0 -> +0; NaN last."""
    key = (s.astype(np.float32) + bias.astype(np.float32)).astype(np.float32)
    order = sorted(range(len(s)), key=lambda e: (-(float(key[e]) if key[e] == key[e] else -math.inf), e))
    return np.array(order[:k], np.int32)


def test_route_matches_full_sort_and_library_sigmoid():
    logits, bias = synth.router_inputs(24, seed=4)
    idx, w, s = oracle.route(logits, bias, return_scores=True)
    s_lib = (1.0 / (1.0 + np.exp(-logits.astype(np.float64)))).astype(np.float32)
    assert np.array_equal(s, s_lib)
    for t in range(24):
        assert np.array_equal(idx[t], brute_route(s[t], bias, 16))
        sel = s[t, idx[t]].astype(np.float64)
        assert np.allclose(w[t], sel / sel.sum(), rtol=2 ** -23, atol=0)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 16 * 2.0 ** -24)


def test_route_bias_selects_raw_scores_weight():
    """Invariant 3 of the kimi-k3-in-c README ("Three invariants"): the bias
    steers selection only; the weights are the unbiased scores renormalised.
    A fixture whose bias reorders the top-16 on five of its six rows."""
    E, K, T = 896, 16, 6
    logits = np.full((T, E), -6.0, np.float32)
    bias = np.zeros(E, np.float32)
    logits[:, 0:16] = 2.0                       # unbiased winners
    bias[16:32] = 0.5                           # biased experts 16..31
    logits[0, 16:32] = -12.0                    # row 0: bias cannot lift them
    for t in range(1, T):
        logits[t, 16:32] = np.linspace(0.2 + 0.1 * t, 1.6, 16)   # sigma + 0.5 > sigma(2)
    idx, w, s = oracle.route(logits, bias, return_scores=True)
    assert sorted(idx[0]) == list(range(16))
    for t in range(1, T):
        assert sorted(idx[t]) == list(range(16, 32))
        raw = s[t, idx[t]].astype(np.float64)
        assert np.allclose(w[t], raw / raw.sum(), rtol=2 ** -23, atol=0)
        biased = raw + 0.5
        assert not np.allclose(w[t], biased / biased.sum(), rtol=1e-3)
        # selection order: key descending, i.e. expert 31 (largest logit) first
        assert idx[t][0] == 31 and idx[t][-1] == 16
    unbiased, _ = oracle.route(logits, np.zeros(E, np.float32))
    changed = [t for t in range(T) if set(unbiased[t]) != set(idx[t])]
    assert changed == [1, 2, 3, 4, 5]


def test_route_ties_go_to_lower_index():
    logits = np.zeros((2, 896), np.float32)
    bias = np.zeros(896, np.float32)
    idx, w = oracle.route(logits, bias)
    assert list(idx[0]) == list(range(16))
    assert np.all(w == np.float32(1 / 16))
    # -0 and +0 keys compare equal: lower index first
    bias[5] = -0.0
    logits[1, 40] = 0.0
    idx, _ = oracle.route(logits, bias)
    assert list(idx[1]) == list(range(16))


def test_route_zero_bias_is_top_logits():
    logits, _ = synth.router_inputs(8, seed=12)
    idx, _ = oracle.route(logits, np.zeros(896, np.float32))
    for t in range(8):
        order = sorted(range(896), key=lambda e: (-float(logits[t, e]), e))[:16]
        assert list(idx[t]) == order


# ---------------------------------------------------------------- grouping --

@pytest.mark.parametrize("T", [1, 3, 64])
def test_group_invariants_and_stable_sort(T):
    logits, bias = synth.router_inputs(T, seed=T)
    idx, _ = oracle.route(logits, bias)
    counts, offsets, perm = oracle.group(idx)
    n = T * 16
    assert counts.sum() == n and offsets[0] == 0 and offsets[-1] == n
    assert np.all(np.diff(offsets) == counts)
    assert sorted(perm.tolist()) == list(range(n))
    flat = idx.ravel()
    expect = sorted(range(n), key=lambda p: (int(flat[p]), p))
    assert perm.tolist() == expect
    for e in np.nonzero(counts)[0]:
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


def test_group_rejects_out_of_range():
    idx = np.zeros((1, 16), np.int32)
    idx[0, 3] = 896
    with pytest.raises(ValueError):
        oracle.group(idx)


# ---------------------------------------------------------------- routed sum --

def test_moe_is_weighted_sum_of_experts_tiny():
    D, F = 64, 32
    experts = {e: synth.split_expert(synth.expert(e, seed=1, D=D, F=F), D=D, F=F) for e in range(6)}
    x = synth.token_inputs(2, seed=5, D=D)
    idx = np.array([[4, 1, 0], [2, 2, 5]], np.int32)
    w = np.array([[0.5, 0.25, 0.25], [0.125, 0.375, 0.5]], np.float32)
    y = oracle.moe(x, idx, w, experts)
    for t in range(2):
        acc = np.zeros(D)
        for k in range(3):
            g, u, W2 = brute_expert(x[t], *experts[int(idx[t, k])])
            h = np.array([oracle.situ(a, b) for a, b in zip(g, u)], np.float32)
            acc += float(w[t, k]) * (W2 @ h.astype(np.float64)).astype(np.float32)
        assert np.allclose(y[t], acc, rtol=1e-6, atol=1e-6 * np.abs(acc).max())
    # all the weight on one expert: y is that expert's output, bit for bit
    w1 = np.array([[1.0, 0.0, 0.0]] * 2, np.float32)
    y1 = oracle.moe(x, idx, w1, experts)
    assert np.array_equal(y1[0], oracle.expert(x[0], *experts[4]))
    assert np.array_equal(y1[1], oracle.expert(x[1], *experts[2]))


# ------------------------------------------------------------ top-p routing --
# K3_TOPP (Kimi K3 engine (c/kimi_k3.c), "Streaming design"; environment
# table): keep the routed experts up to cumulative weight p, drop the
# low-weight tail of the top-16 and renormalise the rest.

def _topp_brute(logits, bias, p):
    """The truncation from its definition on the full-precision route result:
    sort the 16 by raw score (ties: lower index), keep the shortest prefix
    whose scores reach p of their total, renormalise over the kept."""
    idx, w, s = oracle.route(logits, bias, return_scores=True)
    out_i, out_w = idx.copy(), w.copy()
    for t in range(idx.shape[0]):
        sc = [(float(s[t, e]), int(e)) for e in idx[t]]
        order = sorted(range(16), key=lambda k: (-sc[k][0], sc[k][1]))
        total = sum(v for v, _ in sc)
        kept, cum = set(), 0.0
        for k in order:
            if cum < p * total:
                kept.add(k)
            cum += sc[k][0]
        ks = sum(sc[k][0] for k in kept)
        for k in range(16):
            if k in kept:
                out_w[t, k] = np.float32(sc[k][0] / ks)
            else:
                out_i[t, k], out_w[t, k] = -1, 0.0
    return out_i, out_w


def test_topp_matches_its_definition():
    logits, bias = synth.router_inputs(40, seed=51)
    for p in (0.3, 0.5, 0.8, 0.9, 0.99):
        i1, w1 = oracle.route_topp(logits, bias, p)
        i2, w2 = _topp_brute(logits, bias, p)
        assert np.array_equal(i1, i2) and np.array_equal(w1, w2), p


def test_topp_special_cases():
    logits, bias = synth.router_inputs(12, seed=52)
    i0, w0 = oracle.route(logits, bias)
    for p in (0.0, -1.0, 1.0, 2.0):                   # off, and p >= 1 keeps everything
        i, w = oracle.route_topp(logits, bias, p)
        assert np.array_equal(i, i0) and np.array_equal(w, w0), p
    i, w = oracle.route_topp(logits, bias, 1e-9)      # only the heaviest expert survives
    assert np.all((i >= 0).sum(1) == 1)
    assert np.all(w[i >= 0] == 1.0)
    _, _, s = oracle.route(logits, bias, return_scores=True)
    for t in range(12):                               # ... and it is the largest raw score
        e = i[t][i[t] >= 0][0]
        assert s[t, e] == s[t, i0[t]].max()


def test_topp_invariants():
    logits, bias = synth.router_inputs(64, seed=53)
    for p in (0.4, 0.7, 0.95):
        i, w = oracle.route_topp(logits, bias, p)
        i0, _, s = oracle.route(logits, bias, return_scores=True)
        kept = i >= 0
        assert np.all(kept.sum(1) >= 1)
        assert np.all(np.abs(w.sum(1, dtype=np.float64) - 1.0) <= 16 * 2.0 ** -24)
        assert np.all(w[~kept] == 0.0)
        assert np.array_equal(i[kept], i0[kept])      # kept slots keep their expert and place
        for t in range(64):
            ks = s[t, i[t][kept[t]]].astype(np.float64)
            ds = s[t, i0[t][~kept[t]]].astype(np.float64)
            tot = s[t, i0[t]].astype(np.float64).sum()
            assert ks.sum() >= p * tot                        # the kept part reaches p
            assert ks.sum() - ks.min() < p * tot              # and no kept expert is spare
            if ds.size:
                assert ds.max() <= ks.min()                   # only the lightest are dropped
        counts, offsets, perm = oracle.group(i)
        assert offsets[-1] == kept.sum() and len(perm) == kept.sum()


def test_topp_equal_scores_keep_the_lowest_indices():
    """16 equal scores: each carries 1/16, so the shortest prefix reaching p
    has ceil(16 p) experts, and ties rank the lower expert index first."""
    logits = np.full((3, 896), 0.25, np.float32)
    bias = np.zeros(896, np.float32)
    for p, n in ((0.25, 4), (0.26, 5), (0.75, 12), (0.999, 16)):
        i, w = oracle.route_topp(logits, bias, p)
        assert np.all((i >= 0).sum(1) == n), p
        assert sorted(i[0][i[0] >= 0]) == list(range(n))
        assert np.all(w[i >= 0] == np.float32(1.0 / n))


# ---- router logits (Kimi K3 engine (c/kimi_k3.c), "Architecture notes":
# the sigmoid router [896, 7168] over the hidden state; bf16 trunk)

def test_bf16_patterns():
    """bf16 = the upper half of an fp32: sign, 8 exponent bits, 7 fraction bits."""
    assert oracle.bf16(0x3F80) == 1.0
    assert oracle.bf16(0xC000) == -2.0
    assert oracle.bf16(0x3F81) == 1.0 + 2.0 ** -7
    assert oracle.bf16(0x0001) == 2.0 ** -133            # smallest subnormal
    assert oracle.bf16(0x7F80) == float("inf")
    z = oracle.bf16(0x8000)
    assert z == 0.0 and np.copysign(1.0, z) == -1.0


def test_router_logits_one_hot_and_integers():
    """A one-hot hidden state reads one column of W exactly; integer weights
    and states give exact integer logits."""
    rng = np.random.default_rng(61)
    E, C = 5, 96
    W = synth.f32_to_bf16(rng.standard_normal((E, C)).astype(np.float32))
    for c in (0, 17, 95):
        h = np.zeros((1, C), np.float32)
        h[0, c] = 1.0
        lg = oracle.router_logits(W, h)
        assert [lg[0, e] for e in range(E)] == [oracle.bf16(W[e, c]) for e in range(E)]
    Wi = rng.integers(-8, 9, (E, C)).astype(np.float32)       # small integers: exact in bf16
    hi = rng.integers(-100, 101, (3, C)).astype(np.float32)
    lg = oracle.router_logits(synth.f32_to_bf16(Wi), hi)
    exact = hi.astype(np.int64) @ Wi.astype(np.int64).T        # integer arithmetic
    assert np.array_equal(lg.astype(np.int64), exact) and np.all(lg == exact)


def test_router_logits_linear_and_dtype_paths():
    """Linear in h up to one fp32 rounding per logit; a bf16 hidden state
    gives the same logits as its exact fp32 widening."""
    W = synth.router_weights(seed=62, E=32, C=7168)
    h1 = synth.hidden_inputs(2, seed=63)
    h2 = synth.hidden_inputs(2, seed=64)
    l1, l2, l12 = (oracle.router_logits(W, h) for h in (h1, h2, (h1 + h2).astype(np.float32)))
    scale = oracle.router_absdot(W, h1) + oracle.router_absdot(W, h2)
    assert np.all(np.abs(l12.astype(np.float64) - l1 - l2) <= 1e-6 * scale)
    hb = synth.f32_to_bf16(h1)
    assert np.array_equal(oracle.router_logits(W, hb), oracle.router_logits(W, synth.bf16_to_f32(hb)))


def test_router_logits_brute_force_small():
    """Against a numpy dot in float64 on tiny shapes (a different summation
    order): equal within 1e-12 of sum |w h|, and the workload's scale gives
    unit-variance logits."""
    rng = np.random.default_rng(65)
    for E, C in ((3, 32), (7, 100), (2, 7168)):
        W = synth.f32_to_bf16(rng.standard_normal((E, C)).astype(np.float32))
        h = rng.standard_normal((4, C)).astype(np.float32)
        Wd = (W.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ref = h.astype(np.float64) @ Wd.T
        lg = oracle.router_logits(W, h)
        assert np.all(np.abs(lg - ref) <= 1e-12 * (np.abs(h) @ np.abs(Wd).T) + np.abs(ref) * 2.0 ** -24)
    lg = oracle.router_logits(synth.router_weights(seed=0, E=64), synth.hidden_inputs(8, seed=0))
    assert 0.8 < lg.std() < 1.2


# ---- the LatentMoE block around the routed experts (Kimi K3 engine
# (c/kimi_k3.c), "Architecture notes": latent projections, RMSNorm on the
# aggregate, fused shared experts added unweighted)

def test_rmsnorm_closed_forms():
    D = 3584
    one = np.full(D, 0x3F80, np.uint16)                     # g = 1
    for c in (0.5, -3.0, 1e3):
        y = oracle.rmsnorm(np.full((1, D), c, np.float32), one)
        assert np.allclose(y, np.sign(c) * abs(c) / np.sqrt(c * c + 1e-5), rtol=1e-7)
    assert np.all(oracle.rmsnorm(np.zeros((1, D), np.float32), one) == 0.0)
    x = synth.token_inputs(3, seed=71)
    y1 = oracle.rmsnorm(x, one, eps=0.0)
    assert np.array_equal(y1, oracle.rmsnorm(4.0 * x, one, eps=0.0))   # scale-free without eps
    assert np.all(np.abs(np.sqrt(np.mean(y1.astype(np.float64) ** 2, axis=1)) - 1.0) < 1e-6)
    g = synth.f32_to_bf16(np.linspace(0.5, 2.0, D).astype(np.float32))
    assert np.allclose(oracle.rmsnorm(x, g, eps=0.0), y1 * synth.bf16_to_f32(g), rtol=1e-6)


def test_situ_vec_is_the_activation():
    g = np.array([0.0, 1.5, -2.0, 40.0], np.float32)
    u = np.array([3.0, 0.0, -1.0, 2.0], np.float32)
    a = oracle.situ_vec(g, u)
    assert a[0] == 0.0 and a[1] == 0.0
    assert a[2] == np.float32(oracle.situ(-2.0, -1.0)) and a[3] == np.float32(oracle.situ(40.0, 2.0))


def _identity_bf16(rows, cols):
    W = np.zeros((rows, cols), np.uint16)
    n = min(rows, cols)
    W[np.arange(n), np.arange(n)] = 0x3F80
    return W


def test_latent_block_wiring():
    """Identity projections and a silent shared expert expose each stage:
    x = h[:3584], the routed sum of x, its RMSNorm, the shared expert's
    unweighted add."""
    from helpers import arena_expert
    H, D, FS = 7168, 3584, 64
    h = synth.hidden_inputs(1, seed=72)
    logits, bias = synth.router_inputs(1, seed=72)
    idx, w = oracle.route(logits, bias)
    experts = {int(e): arena_expert(int(e)) for e in idx[0]}
    g_norm = synth.f32_to_bf16(np.full(D, 2.0, np.float32))
    blk = {"w_dn": _identity_bf16(D, H), "w_up": _identity_bf16(H, D), "g_norm": g_norm,
           "w1s": np.zeros((FS, H), np.uint16), "w3s": synth.router_weights(seed=73, E=FS, C=H),
           "w2s": synth.router_weights(seed=74, E=H, C=FS)}
    y, (x, yr, z, a) = oracle.latent_block(h, blk, idx, w, experts)
    assert np.array_equal(x, h[:, :D])                     # W_dn = [I 0]
    assert np.array_equal(yr, oracle.moe(h[:, :D], idx, w, experts))
    assert np.array_equal(z, oracle.rmsnorm(yr, g_norm))
    assert np.all(a == 0.0)                                # W1s = 0: SiTU(0, u) = 0
    assert np.array_equal(y[:, :D], z) and np.all(y[:, D:] == 0.0)
    blk["w1s"] = synth.router_weights(seed=75, E=FS, C=H)    # the shared expert on
    y2, (_, _, _, a2) = oracle.latent_block(h, blk, idx, w, experts)
    ysh = oracle.bf16_matvec(blk["w2s"], a2)
    assert np.any(a2 != 0.0)
    assert np.array_equal(y2, (z.astype(np.float64) @ np.eye(D, H) + ysh.astype(np.float64)).astype(np.float32))
