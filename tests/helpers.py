"""Shared helpers of the GPU parity tests (oracle-side expected values)."""
import numpy as np

import oracle
import synth
from conftest import ARENA_SEED, ARENA_SCALE_LO, ARENA_SCALE_HI


def arena_expert_bytes(e):
    """Bytes of routed expert e of the test arena (arena order)."""
    return synth.expert(e, seed=ARENA_SEED, lo=ARENA_SCALE_LO, hi=ARENA_SCALE_HI)


def arena_expert(e):
    """Host copy of routed expert e of the test arena, split in six arrays."""
    return synth.split_expert(arena_expert_bytes(e))


def moe_oracle(x, idx, w, tokens):
    """Oracle output rows and tolerance bounds for the given token ids.
    bound_t[i] = sum_k w_tk * expert_bound_k[i] (the composite of the
    per-expert bound, weighted by the routing weights)."""
    ys, bounds = [], []
    for t in tokens:
        ex = {}
        bnd = np.zeros(x.shape[1])
        for k in range(idx.shape[1]):
            e = int(idx[t, k])
            if e < 0:                                     # dropped by top-p
                continue
            if e not in ex:
                ex[e] = arena_expert(e)
            _, _, _, h = oracle.expert(x[t], *ex[e], intermediates=True)
            bnd += float(w[t, k]) * oracle.expert_bound(x[t], h, *ex[e])
        ys.append(oracle.moe(x[t:t + 1], idx[t:t + 1], w[t:t + 1], ex)[0])
        bounds.append(bnd)
    return np.array(ys), np.array(bounds)


def assert_within(got, ref, bound, what):
    err = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    ratio = err / np.maximum(bound, 1e-300)
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert np.all(err <= bound), (f"{what}: {np.sum(err > bound)} outputs out of tolerance; worst "
                                  f"{worst}: got {got[worst]}, oracle {ref[worst]}, bound {bound[worst]}")
    return float(np.max(ratio))


# ------------------------------------------------ edges of the MXFP4 format --
#
# Experts whose scales reach the ends of the ue8m0 range.  Each of an edge
# expert's three matrices (W1, W3: 3072 rows; W2: 3584 rows) is the seeded
# expert with 1% of its groups at scale 255 ("NaN: contributes nothing"),
# plus rows set on purpose:
#   row   3  every group 255: the row contributes exactly nothing
#   row 130  every group at scale 0 (2^-127, the smallest)
#   row 131  every group at scale 1 (2^-126)
#   row 259  every fourth group at scale 254 (2^127) with codes +0 / -0
#            (zero weights at the largest scale), the rest as drawn
#   row 260  groups alternating 255 and 0
#   row 261  every group 255 except group 5 at 127 (one group left)
# Rows 3, 130-131 and 259-261 lie in the first three 128-row tiles.
EDGE_SEED = 5
EDGE_ROWS = {"nan": 3, "s0": 130, "s1": 131, "s254_zero": 259, "alt": 260, "one_group": 261}


def edge_expert_bytes(i):
    """Bytes of edge expert i (arena order w1p w1s w3p w3s w2p w2s)."""
    buf = synth.expert(i, seed=EDGE_SEED, lo=ARENA_SCALE_LO, hi=ARENA_SCALE_HI, nan_frac=0.01)
    for packed, scales in (synth.split_expert(buf)[0:2], synth.split_expert(buf)[2:4], synth.split_expert(buf)[4:6]):
        G = scales.shape[1]
        scales[EDGE_ROWS["nan"], :] = 255
        scales[EDGE_ROWS["s0"], :] = 0
        scales[EDGE_ROWS["s1"], :] = 1
        r = EDGE_ROWS["s254_zero"]
        for g in range(0, G, 4):
            scales[r, g] = 254
            packed[r, 16 * g:16 * g + 16] = 0x00 if (g // 4) % 2 == 0 else 0x88
        scales[EDGE_ROWS["alt"], 0::2] = 255
        scales[EDGE_ROWS["alt"], 1::2] = 0
        scales[EDGE_ROWS["one_group"], :] = 255
        scales[EDGE_ROWS["one_group"], 5] = 127
    return buf


def moe_oracle_rows(x, idx, w, tokens, expert_bytes):
    """Oracle output rows for the given tokens, expert by expert: each
    selected expert's bytes are drawn once (expert_bytes(e)), its output for
    every (token, slot) that selects it comes from oracle.expert, and each
    token's weighted sum is taken in slot order in double and rounded once,
    as the oracle's routed sum does."""
    tokens = list(tokens)
    K = idx.shape[1]
    outs = {}
    by_e = {}
    for i, t in enumerate(tokens):
        for k in range(K):
            e = int(idx[t, k])
            if e >= 0:
                by_e.setdefault(e, []).append((i, k))
    for e, uses in by_e.items():
        ex = synth.split_expert(expert_bytes(e))
        for i, k in uses:
            outs[(i, k)] = oracle.expert(x[tokens[i]], *ex)
    ys = np.zeros((len(tokens), x.shape[1]), np.float64)
    for i, t in enumerate(tokens):
        for k in range(K):
            if (i, k) in outs:
                ys[i] += np.float64(w[t, k]) * outs[(i, k)].astype(np.float64)
    return ys.astype(np.float32)
