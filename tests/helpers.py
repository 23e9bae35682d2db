"""Shared helpers of the GPU parity tests (oracle-side expected values)."""
import numpy as np

import oracle
import synth
from conftest import ARENA_SEED, ARENA_SCALE_LO, ARENA_SCALE_HI


def arena_expert(e):
    """Host copy of routed expert e of the test arena, split in six arrays."""
    return synth.split_expert(synth.expert(e, seed=ARENA_SEED, lo=ARENA_SCALE_LO, hi=ARENA_SCALE_HI))


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
