"""CPU oracle of the MXFP4 routed-expert layer (ctypes binding of k3mx_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(the package ``mxfp4_routed_expert_k3mx_gb300`` and its CUDA library) never
does.  It shares no code with the CUDA kernels.

Pinned by ``tests/test_oracle_pins.py`` against what the pages fix (the e2m1
table, the expert byte count, NaN-scale groups, brute-force dot products on
tiny shapes, closed forms of SiTU-GLU, a brute-force sort for the router,
invariants of the grouping, linearity of the routed sum).  Parity unpinned:
the last bits of tanh and exp (libm against CUDA) are covered by tolerance
only.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3mx_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

E2M1_MAGNITUDES = None  # filled from the C table by e2m1()


def build(force=False):
    """Compile liboracle.so next to its source.  -ffp-contract=off keeps every
    multiply and add rounding as written (aarch64 gcc contracts by default)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp = ctypes.c_void_p
            i = ctypes.c_int
            lib.orc_e2m1.argtypes = [i]
            lib.orc_e2m1.restype = ctypes.c_double
            lib.orc_e8m0.argtypes = [i]
            lib.orc_e8m0.restype = ctypes.c_double
            lib.orc_sigmoid.argtypes = [ctypes.c_double]
            lib.orc_sigmoid.restype = ctypes.c_double
            lib.orc_situ.argtypes = [ctypes.c_double, ctypes.c_double]
            lib.orc_situ.restype = ctypes.c_double
            lib.orc_gemv.argtypes = [vp, vp, vp, vp, i, i]
            lib.orc_gemv_absdot.argtypes = [vp, vp, vp, vp, i, i]
            lib.orc_expert.argtypes = [vp] * 5 + [vp] + [vp] * 6 + [i, i]
            lib.orc_expert_bound.argtypes = [vp, vp, vp, vp] + [vp] * 6 + [i, i]
            lib.orc_route.argtypes = [vp, vp, vp, vp, vp, i, i, i, ctypes.c_float]
            lib.orc_topp.argtypes = [vp, vp, vp, i, i, i, ctypes.c_float, ctypes.c_double]
            lib.orc_group.argtypes = [vp, vp, vp, vp, i, i, i]
            lib.orc_bf16.restype = ctypes.c_double
            lib.orc_bf16.argtypes = [ctypes.c_uint16]
            lib.orc_router_logits.argtypes = [vp, vp, vp, i, i, i, i]
            lib.orc_router_absdot.argtypes = [vp, vp, vp, i, i, i, i]
            lib.orc_rmsnorm.argtypes = [vp, vp, vp, i, i, ctypes.c_double]
            lib.orc_situ_vec.argtypes = [vp, vp, vp, ctypes.c_longlong]
            lib.orc_group.restype = i
            lib.orc_moe.argtypes = [vp, vp, i, vp, vp, vp, i, i, i, vp]
            lib.orc_num_threads.restype = i
            _lib = lib
    return _lib


def _p(a):
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "contiguous numpy array expected"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads():
    return int(_load().orc_num_threads())


def e2m1(code):
    return float(_load().orc_e2m1(int(code)))


def e8m0(s):
    return float(_load().orc_e8m0(int(s)))


def sigmoid(z):
    return float(_load().orc_sigmoid(float(z)))


def situ(g, u):
    return float(_load().orc_situ(float(g), float(u)))


def gemv(x, packed, scales):
    """y = W x, W read from packed MXFP4 (packed [rows, in/2], scales [rows, in/32])."""
    x = np.ascontiguousarray(x, np.float32)
    packed = np.ascontiguousarray(packed, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    rows, half = packed.shape
    n_in = 2 * half
    assert x.shape == (n_in,) and scales.shape == (rows, n_in // 32) and n_in % 32 == 0
    y = np.empty(rows, np.float32)
    _load().orc_gemv(_p(y), _p(x), _p(packed), _p(scales), n_in, rows)
    return y


def gemv_absdot(xabs, packed, scales):
    """sum_c |w_rc| |x_c| per row (non-NaN groups), double."""
    xabs = np.ascontiguousarray(np.abs(xabs), np.float64)
    rows, half = packed.shape
    b = np.empty(rows, np.float64)
    _load().orc_gemv_absdot(_p(b), _p(xabs), _p(np.ascontiguousarray(packed)),
                            _p(np.ascontiguousarray(scales)), 2 * half, rows)
    return b


def expert(x, w1p, w1s, w3p, w3s, w2p, w2s, intermediates=False):
    """One routed expert: returns y, or (y, g, u, h) with intermediates=True."""
    x = np.ascontiguousarray(x, np.float32)
    F, half = w1p.shape
    D = 2 * half
    y = np.empty(D, np.float32)
    g = np.empty(F, np.float32)
    u = np.empty(F, np.float32)
    h = np.empty(F, np.float32)
    tmp = np.empty(3 * F, np.float32)
    arrs = [np.ascontiguousarray(a, np.uint8) for a in (w1p, w1s, w3p, w3s, w2p, w2s)]
    _load().orc_expert(_p(y), _p(g), _p(u), _p(h), _p(tmp), _p(x), *[_p(a) for a in arrs], D, F)
    return (y, g, u, h) if intermediates else y


def expert_bound(x, h, w1p, w1s, w3p, w3s, w2p, w2s):
    """Per-output tolerance scale of one expert (see k3mx_oracle.c)."""
    F, half = w1p.shape
    D = 2 * half
    b = np.empty(D, np.float64)
    work = np.empty(2 * D + 3 * F, np.float64)
    arrs = [np.ascontiguousarray(a, np.uint8) for a in (w1p, w1s, w3p, w3s, w2p, w2s)]
    _load().orc_expert_bound(_p(b), _p(work), _p(np.ascontiguousarray(x, np.float32)),
                             _p(np.ascontiguousarray(h, np.float32)), *[_p(a) for a in arrs], D, F)
    return b


def route(logits, bias, k=16, routed_scale=1.0, return_scores=False):
    """Top-k of sigmoid(logit) + bias; weights = renormalised raw scores."""
    logits = np.ascontiguousarray(logits, np.float32)
    if logits.ndim == 1:
        logits = logits[None, :]
    T, E = logits.shape
    assert E <= 1024 and k <= E
    bias = np.ascontiguousarray(bias, np.float32)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    s = np.empty((T, E), np.float32)
    _load().orc_route(_p(idx), _p(w), _p(s), _p(logits), _p(bias), T, E, k, routed_scale)
    return (idx, w, s) if return_scores else (idx, w)


def route_topp(logits, bias, p, k=16, routed_scale=1.0):
    """route(), then the top-p truncation: of the k experts in order of
    decreasing raw score (ties: lower index), keep the shortest prefix whose
    scores reach p times their total; kept weights renormalised over the
    kept scores; dropped slots get index -1 and weight 0 (p <= 0: all kept)."""
    idx, w, s = route(logits, bias, k, routed_scale, return_scores=True)
    T, E = s.shape
    _load().orc_topp(_p(idx), _p(w), _p(s), T, E, k, routed_scale, float(p))
    return idx, w


def bf16(bits):
    """A bf16 bit pattern as a float."""
    return float(_load().orc_bf16(int(bits)))


def _router_args(W, h):
    W = np.ascontiguousarray(W, np.uint16)
    if h.dtype == np.uint16:
        hb, h = 1, np.ascontiguousarray(h, np.uint16)
    else:
        hb, h = 0, np.ascontiguousarray(h, np.float32)
    E, C = W.shape
    T = h.shape[0]
    assert h.shape == (T, C)
    return W, h, hb, T, E, C


def router_logits(W, h):
    """Router logits [T, E] fp32 from bf16 router weights W [E, C] (uint16
    bit patterns) and the hidden state h [T, C] (fp32, or uint16 bf16)."""
    W, h, hb, T, E, C = _router_args(W, h)
    out = np.empty((T, E), np.float32)
    _load().orc_router_logits(_p(out), _p(W), _p(h), hb, T, E, C)
    return out


def router_absdot(W, h):
    """sum_c |W[e,c] h[t,c]| [T, E] in double: the scale of a logit's tolerance."""
    W, h, hb, T, E, C = _router_args(W, h)
    out = np.empty((T, E), np.float64)
    _load().orc_router_absdot(_p(out), _p(W), _p(h), hb, T, E, C)
    return out


def bf16_matvec(W, x):
    """y [T, R] fp32 = bf16 W [R, C] times x [T, C] (fp32 or bf16), double
    sums in ascending column order, one rounding (the router's product)."""
    return router_logits(W, x)


def rmsnorm(x, g, eps=1e-5):
    """x [T, D] fp32 / sqrt(mean(x^2) + eps) * g (bf16 [D]), in double."""
    x = np.ascontiguousarray(x, np.float32)
    g = np.ascontiguousarray(g, np.uint16)
    T, D = x.shape
    out = np.empty_like(x)
    _load().orc_rmsnorm(_p(out), _p(x), _p(g), T, D, float(eps))
    return out


def situ_vec(g, u):
    """SiTU-GLU elementwise, fp32 in, double inside, fp32 out."""
    g = np.ascontiguousarray(g, np.float32)
    u = np.ascontiguousarray(u, np.float32)
    out = np.empty_like(g)
    _load().orc_situ_vec(_p(out), _p(g), _p(u), g.size)
    return out


def latent_block(h, blk, idx, w, experts, tokens=None):
    """The Stable LatentMoE block [LM] for hidden states h [T, 7168] (fp32
    or bf16) given the routing (idx, w) of the router logits:
        x  = W_dn h                            (7168 -> 3584)
        yr = sum_k w_k expert_k(x)             (the routed experts)
        y  = W_up rmsnorm(yr) + W2s situ(W1s h, W3s h)
    `blk` maps "w_dn", "w_up", "g_norm", "w1s", "w3s", "w2s" to bf16 arrays;
    `experts` is the list of per-expert (w1p, w1s, w3p, w3s, w2p, w2s).
    Every product step returns fp32; the final sum is taken in double and
    rounded once.  `tokens` restricts the work to those rows of h.  Returns
    y [T', 7168] and the intermediates (x, yr, z, a)."""
    if tokens is not None:
        h, idx, w = h[tokens], idx[tokens], w[tokens]
    x = bf16_matvec(blk["w_dn"], h)
    yr = moe(x, idx, w, experts)
    z = rmsnorm(yr, blk["g_norm"])
    y_up = bf16_matvec(blk["w_up"], z)
    a = situ_vec(bf16_matvec(blk["w1s"], h), bf16_matvec(blk["w3s"], h))
    y_sh = bf16_matvec(blk["w2s"], a)
    y = (y_up.astype(np.float64) + y_sh.astype(np.float64)).astype(np.float32)
    return y, (x, yr, z, a)


def group(idx, n_experts=896):
    """counts [E], offsets [E+1], perm [sum(counts)] (stable by pair index
    t*K+k); index -1 (a slot dropped by top-p) is not grouped."""
    idx = np.ascontiguousarray(idx, np.int32)
    T, K = idx.shape
    counts = np.empty(n_experts, np.int32)
    offsets = np.empty(n_experts + 1, np.int32)
    perm = np.empty(T * K, np.int32)
    rc = _load().orc_group(_p(counts), _p(offsets), _p(perm), _p(idx), T, n_experts, K)
    if rc != 0:
        raise ValueError("expert index out of range")
    return counts, offsets, perm[:int(offsets[-1])]


def moe(x, idx, w, experts):
    """Routed weighted sum.  ``experts`` maps expert id -> (w1p, w1s, w3p, w3s,
    w2p, w2s) numpy arrays; only the selected ids need to be present."""
    x = np.ascontiguousarray(x, np.float32)
    idx = np.ascontiguousarray(idx, np.int32)
    w = np.ascontiguousarray(w, np.float32)
    T, D = x.shape
    K = idx.shape[1]
    assert D <= 8192
    ids = sorted(set(int(e) for e in idx.ravel() if e >= 0))     # -1: a slot dropped by top-p
    some = experts[ids[0]]
    F = some[0].shape[0]
    E = int(idx.max()) + 1
    keep = []
    table = (ctypes.c_void_p * (6 * E))()
    for e in ids:
        arrs = [np.ascontiguousarray(a, np.uint8) for a in experts[e]]
        keep.append(arrs)
        for j, a in enumerate(arrs):
            table[6 * e + j] = a.ctypes.data
    y = np.empty((T, D), np.float32)
    tmp = np.empty(3 * F + D, np.float32)
    _load().orc_moe(_p(y), _p(x), T, ctypes.cast(table, ctypes.c_void_p), _p(idx), _p(w), D, F, K, _p(tmp))
    return y
