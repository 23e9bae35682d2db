"""Seeded synthetic inputs for the MXFP4 routed-expert layer.

A module of its own: it draws numbers and holds none of the layer's
arithmetic.  The oracle side and the CUDA side both take their inputs from
here.  The generator itself is ``synth.c`` (counter-based SplitMix64, see its
header); this file builds it with gcc on first use and wraps it with ctypes.

Stream numbering (seed is the workload seed, 0 unless stated):
  STREAM_W_PACKED / STREAM_W_SCALES : the single GEMV matrix W
  STREAM_X                          : token activations
  STREAM_LOGITS / STREAM_BIAS       : router logits and score-correction bias
  STREAM_ROUTER_W / STREAM_HIDDEN   : router weights and the hidden state
  expert e, tensor t                : 0x100000 + 8 e + t  (inside synth_expert)
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

STREAM_W_PACKED = 1
STREAM_W_SCALES = 2
STREAM_X = 10
STREAM_LOGITS = 11
STREAM_BIAS = 12
STREAM_ROUTER_W = 13
STREAM_HIDDEN = 14
STREAM_BLOCK = 20       # + 0..5: the LatentMoE block's bf16 matrices and norm weight

# Kimi-K3 routed-expert shape: latent width D, expert inter width F.
D_LATENT = 3584
F_INTER = 3072
N_EXPERTS = 896
TOP_K = 16
H_MODEL = 7168          # hidden width the router reads
F_SHARED = 6144         # inter width of the fused shared experts


def build(force=False):
    """Compile libsynth.so next to its source (gcc, OpenMP, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            f32p = ctypes.POINTER(ctypes.c_float)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            sz, u64 = ctypes.c_size_t, ctypes.c_uint64
            lib.synth_bytes.argtypes = [u8p, sz, u64, u64]
            lib.synth_scale_bytes.argtypes = [u8p, sz, u64, u64, ctypes.c_int, ctypes.c_int, ctypes.c_double]
            lib.synth_normal_f32.argtypes = [f32p, sz, u64, u64, ctypes.c_double, ctypes.c_double]
            lib.synth_f32_to_bf16.argtypes = [u16p, f32p, sz]
            lib.synth_bf16_to_f32.argtypes = [f32p, u16p, sz]
            lib.synth_expert_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
            lib.synth_expert_bytes.restype = sz
            lib.synth_expert.argtypes = [u8p, u64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_double]
            lib.synth_mix64.argtypes = [u64]
            lib.synth_mix64.restype = u64
            _lib = lib
    return _lib


def _ptr(a, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def uniform_bytes(n, seed, stream, out=None):
    out = np.empty(n, np.uint8) if out is None else out
    _load().synth_bytes(_ptr(out, ctypes.c_uint8), out.size, seed, stream)
    return out


def scale_bytes(n, seed, stream, lo, hi, nan_frac=0.0, out=None):
    out = np.empty(n, np.uint8) if out is None else out
    _load().synth_scale_bytes(_ptr(out, ctypes.c_uint8), out.size, seed, stream, lo, hi, nan_frac)
    return out


def normal_f32(n, seed, stream, mean=0.0, std=1.0, out=None):
    out = np.empty(n, np.float32) if out is None else out
    _load().synth_normal_f32(_ptr(out, ctypes.c_float), out.size, seed, stream, mean, std)
    return out


def f32_to_bf16(a):
    a = np.ascontiguousarray(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().synth_f32_to_bf16(_ptr(out, ctypes.c_uint16), _ptr(a, ctypes.c_float), a.size)
    return out


def bf16_to_f32(a):
    a = np.ascontiguousarray(a, np.uint16)
    out = np.empty(a.shape, np.float32)
    _load().synth_bf16_to_f32(_ptr(out, ctypes.c_float), _ptr(a, ctypes.c_uint16), a.size)
    return out


def expert_nbytes(D=D_LATENT, F=F_INTER):
    return int(_load().synth_expert_bytes(D, F))


def expert_offsets(D=D_LATENT, F=F_INTER):
    """Byte offsets of (w1p, w1s, w3p, w3s, w2p, w2s) inside one expert's bytes."""
    a, s = F * D // 2, F * D // 32
    return [0, a, a + s, 2 * a + s, 2 * (a + s), 2 * (a + s) + a]


def expert(e, seed=0, lo=118, hi=128, nan_frac=0.0, D=D_LATENT, F=F_INTER, out=None):
    """Bytes of routed expert ``e`` in arena order (w1p w1s w3p w3s w2p w2s)."""
    n = expert_nbytes(D, F)
    out = np.empty(n, np.uint8) if out is None else out
    assert out.size == n
    _load().synth_expert(_ptr(out, ctypes.c_uint8), seed, e, D, F, lo, hi, nan_frac)
    return out


def split_expert(buf, D=D_LATENT, F=F_INTER):
    """Views (w1p, w1s, w3p, w3s, w2p, w2s) into one expert's bytes, 2-D shaped."""
    o = expert_offsets(D, F)
    a, s = F * D // 2, F * D // 32
    w1p = buf[o[0]:o[0] + a].reshape(F, D // 2)
    w1s = buf[o[1]:o[1] + s].reshape(F, D // 32)
    w3p = buf[o[2]:o[2] + a].reshape(F, D // 2)
    w3s = buf[o[3]:o[3] + s].reshape(F, D // 32)
    w2p = buf[o[4]:o[4] + a].reshape(D, F // 2)
    w2s = buf[o[5]:o[5] + s].reshape(D, F // 32)
    return w1p, w1s, w3p, w3s, w2p, w2s


# ---- the five routed-expert workloads -------------------------------------

def gemv_inputs(seed=0, rows=3072, cols=3584, lo=120, hi=130, nan_frac=0.01):
    """Single MXFP4 GEMV: W [rows x cols] packed, scales U{lo..hi} with
    nan_frac set to 255, x ~ N(0,1) fp32."""
    packed = uniform_bytes(rows * cols // 2, seed, STREAM_W_PACKED).reshape(rows, cols // 2)
    scales = scale_bytes(rows * cols // 32, seed, STREAM_W_SCALES, lo, hi, nan_frac).reshape(rows, cols // 32)
    x = normal_f32(cols, seed, STREAM_X)
    return packed, scales, x


def token_inputs(n_tokens, seed=0, D=D_LATENT):
    """Token activations ~ N(0,1): fp32 [T, D]."""
    return normal_f32(n_tokens * D, seed, STREAM_X).reshape(n_tokens, D)


def router_inputs(n_tokens, seed=0, E=N_EXPERTS, bias_std=0.1):
    """Router logits ~ N(0,1) [T, E] and score-correction bias ~ N(0, bias_std) [E]."""
    logits = normal_f32(n_tokens * E, seed, STREAM_LOGITS).reshape(n_tokens, E)
    bias = normal_f32(E, seed, STREAM_BIAS, 0.0, bias_std)
    return logits, bias


def router_weights(seed=0, E=N_EXPERTS, C=H_MODEL):
    """Router weights ~ N(0, 1/C) rounded to bf16: uint16 bit patterns [E, C]
    (with unit-variance hidden states the logits come out about N(0, 1))."""
    w = normal_f32(E * C, seed, STREAM_ROUTER_W, 0.0, float(C) ** -0.5)
    return f32_to_bf16(w).reshape(E, C)


def hidden_inputs(n_tokens, seed=0, C=H_MODEL):
    """Hidden states ~ N(0,1): fp32 [T, C]."""
    return normal_f32(n_tokens * C, seed, STREAM_HIDDEN).reshape(n_tokens, C)


def latent_block_weights(seed=0, H=H_MODEL, D=D_LATENT, FS=F_SHARED):
    """The LatentMoE block's bf16 tensors (uint16 bit patterns): the latent
    projections w_dn [D, H] ~ N(0, 1/H) and w_up [H, D] ~ N(0, 1/D), the
    aggregate's RMSNorm weight g_norm [D] ~ N(1, 0.1^2), and the fused shared
    experts w1s, w3s [FS, H] ~ N(0, 1/H), w2s [H, FS] ~ N(0, 1/FS): unit-scale
    activations in, unit-scale activations out."""
    def mat(k, rows, cols):
        return f32_to_bf16(normal_f32(rows * cols, seed, STREAM_BLOCK + k, 0.0, float(cols) ** -0.5)).reshape(rows, cols)
    return {"w_dn": mat(0, D, H), "w_up": mat(1, H, D),
            "g_norm": f32_to_bf16(normal_f32(D, seed, STREAM_BLOCK + 2, 1.0, 0.1)),
            "w1s": mat(3, FS, H), "w3s": mat(4, FS, H), "w2s": mat(5, H, FS)}


def expert_arena_device(device, seed=0, lo=118, hi=128, n_experts=N_EXPERTS, chunk=16):
    """All routed experts drawn with `seed`, back to back in one device buffer
    (896 x 17,547,264 B = 15.72 GB), copied through two pinned staging
    buffers.  Returns a torch uint8 tensor on `device`."""
    import torch
    n = expert_nbytes()
    buf = torch.empty(n_experts * n, dtype=torch.uint8, device=device)
    stage = [torch.empty(chunk * n, dtype=torch.uint8).pin_memory() for _ in range(2)]
    events = [None, None]
    stream = torch.cuda.current_stream(device)
    for i, e0 in enumerate(range(0, n_experts, chunk)):
        m = min(chunk, n_experts - e0)
        s = stage[i % 2]
        if events[i % 2] is not None:
            events[i % 2].synchronize()
        host = s.numpy()
        for j in range(m):
            expert(e0 + j, seed=seed, lo=lo, hi=hi, out=host[j * n:(j + 1) * n])
        with torch.cuda.stream(stream):
            buf[e0 * n:(e0 + m) * n].copy_(s[:m * n], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(stream)
        events[i % 2] = ev
    torch.cuda.synchronize(device)
    return buf
