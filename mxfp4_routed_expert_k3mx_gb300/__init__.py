"""Python binding of libk3mx.so, the C ABI declared in include/k3mx.h.

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  The functions carry the C names; tensors are passed as their
device pointers.  PyTorch provides device memory and streams.  There is no
CPU fallback: importing this package without a built library raises.
"""
import ctypes
import os
import re

import torch

from . import _build

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = _build.LIB

K3MX_GROUP = 32
K3MX_N_EXPERTS = 896
K3MX_TOPK = 16
K3MX_LATENT = 3584
K3MX_INTER = 3072
K3MX_EXPERT_BYTES = 17547264
K3MX_F32, K3MX_BF16 = 0, 1
K3MX_PATH_AUTO, K3MX_PATH_DECODE, K3MX_PATH_PREFILL, K3MX_PATH_PREFILL_MX = 0, 1, 2, 3
K3MX_PREFILL_MIN_TOKENS = 256
K3MX_MAX_TOKENS = 65536
K3MX_NOALLOC_MAX_TOKENS = 8

STATUS = {0: "K3MX_OK", 1: "K3MX_EINVAL", 2: "K3MX_EALIGN", 3: "K3MX_ESHAPE",
          4: "K3MX_EWORKSPACE", 5: "K3MX_ECUDA", 6: "K3MX_ETIMEOUT", 7: "K3MX_EDEVICE"}


class K3mxError(RuntimeError):
    def __init__(self, func, status):
        self.status = status
        msg = f"{func} failed: {STATUS.get(status, status)} ({lib().k3mx_status_str(status).decode()})"
        if status == 5:
            msg += f": {lib().k3mx_last_cuda_error().decode()}"
        super().__init__(msg)


class Expert(ctypes.Structure):
    """k3mx_expert: six device pointers w1, s1, w3, s3, w2, s2."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("w1", "s1", "w3", "s3", "w2", "s2")]


class LatentBlock(ctypes.Structure):
    """k3mx_latent_block: device pointers of the LatentMoE block's tensors."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("router_w", "bias", "w_dn", "w_up", "g_norm", "w1s", "w3s", "w2s")]


class TraceEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


_lib = None


def lib():
    """The loaded libk3mx.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build(); "
                               "this package has no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sig = {
            "k3mx_gemv": ([vp, vp, vp, vp, i, i, vp], i),
            "k3mx_expert_ffn_workspace_size": ([], sz),
            "k3mx_expert_ffn": ([vp, vp, ctypes.POINTER(Expert), vp, sz, vp], i),
            "k3mx_route_topk": ([vp, vp, vp, vp, i, vp], i),
            "k3mx_route_topp": ([vp, vp, vp, vp, i, ctypes.c_float, vp], i),
            "k3mx_router": ([vp, vp, vp, vp, i, vp, vp, i, ctypes.c_float, vp], i),
            "k3mx_latent_moe_workspace_size": ([i, i], sz),
            "k3mx_latent_moe": ([vp, vp, i, i, ctypes.POINTER(LatentBlock), vp, ctypes.c_float, vp, vp, vp, sz, vp], i),
            "k3mx_group_workspace_size": ([i], sz),
            "k3mx_group": ([vp, vp, vp, vp, i, vp, sz, vp], i),
            "k3mx_moe_workspace_size": ([i, i, i], sz),
            "k3mx_moe_routed": ([vp, vp, i, i, vp, vp, vp, i, vp, vp, vp, sz, vp], i),
            "k3mx_moe_routed_topp": ([vp, vp, i, i, vp, vp, vp, i, ctypes.c_float, vp, vp, vp, sz, vp], i),
            "k3mx_moe_host_workspace_size": ([i, i, i], sz),
            "k3mx_moe_routed_host": ([vp, vp, i, i, vp, vp, vp, i, vp, sz, vp], i),
            "k3mx_moe_decode_noalloc": ([vp, vp, i, i, vp, vp, vp, vp, vp, vp], i),
            "k3mx_device_status": ([vp, ctypes.POINTER(ctypes.c_int)], i),
            "k3mx_set_wait_limit": ([ctypes.c_uint], i),
            "k3mx_status_str": ([i], ctypes.c_char_p),
            "k3mx_last_cuda_error": ([], ctypes.c_char_p),
            "k3mx_abi_version": ([], i),
            "k3mx_trace_enable": ([i], i),
            "k3mx_trace_read": ([ctypes.POINTER(TraceEntry), i], i),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def declared_symbols(header=None):
    """Function names declared in include/k3mx.h."""
    header = header or os.path.join(os.path.dirname(_HERE), "include", "k3mx.h")
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(k3mx_\w+)\s*\(", text)))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(func, status):
    if status != 0:
        raise K3mxError(func, status)


def _dev(t, dtype, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous() and t.dtype == dtype):
        raise TypeError(f"{name}: contiguous CUDA tensor of {dtype} expected")


def _elems(t):
    return t.numel()


# Shape checks run before any device check or library call: the C ABI gets
# raw pointers and sizes only, so a tensor smaller than the sizes passed
# would let a kernel read or write past its end.

def _tokens(x, width, name):
    """Token count of a [T, width] activation tensor."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2 or x.shape[1] != width or x.shape[0] < 1:
        shape = tuple(x.shape) if isinstance(x, torch.Tensor) else type(x).__name__
        raise TypeError(f"{name}: shape [T, {width}] with T >= 1 expected, got {shape}")
    return int(x.shape[0])


def _numel(t, n, name, optional=False):
    if t is None and optional:
        return
    if not isinstance(t, torch.Tensor) or t.numel() != n:
        got = t.numel() if isinstance(t, torch.Tensor) else type(t).__name__
        raise TypeError(f"{name}: {n} elements expected (shape), got {got}")


def _table(experts, name="experts"):
    if not isinstance(experts, torch.Tensor) or experts.dtype != torch.int64 or \
            tuple(experts.shape) != (K3MX_N_EXPERTS, 6):
        got = (tuple(experts.shape), experts.dtype) if isinstance(experts, torch.Tensor) else type(experts).__name__
        raise TypeError(f"{name}: int64 table of shape [{K3MX_N_EXPERTS}, 6] expected, got {got}")


# ------------------------------------------------------------------ calls --

def k3mx_gemv(y, x, packed, scales, stream=None):
    """y[rows] = W x with W given as packed [rows, in/2] uint8 and scales [rows, in/32] uint8."""
    if not isinstance(packed, torch.Tensor) or packed.dim() != 2:
        raise TypeError("packed: shape [rows, in/2] expected")
    rows, half = packed.shape
    if not isinstance(scales, torch.Tensor) or tuple(scales.shape) != (rows, 2 * half // 32):
        raise TypeError(f"scales: shape [{rows}, {2 * half // 32}] expected")
    _numel(x, 2 * half, "x")
    _numel(y, rows, "y")
    _dev(y, torch.float32, "y")
    _dev(x, torch.float32, "x")
    _dev(packed, torch.uint8, "packed")
    _dev(scales, torch.uint8, "scales")
    rows, half = packed.shape
    _check("k3mx_gemv", lib().k3mx_gemv(_ptr(y), _ptr(x), _ptr(packed), _ptr(scales),
                                         2 * half, rows, _stream(stream)))
    return y


def expert_struct(w1, s1, w3, s3, w2, s2):
    """A k3mx_expert from six device tensors or raw device addresses."""
    return Expert(*[_ptr(a) for a in (w1, s1, w3, s3, w2, s2)])


def k3mx_expert_ffn_workspace_size():
    return int(lib().k3mx_expert_ffn_workspace_size())


def k3mx_expert_ffn(y, x, expert, workspace, stream=None):
    """y = W2 SiTU(W1 x, W3 x) for one expert (an Expert struct) and one token."""
    _numel(x, K3MX_LATENT, "x")
    _numel(y, K3MX_LATENT, "y")
    _dev(y, torch.float32, "y")
    _dev(x, torch.float32, "x")
    _check("k3mx_expert_ffn", lib().k3mx_expert_ffn(
        _ptr(y), _ptr(x), ctypes.byref(expert), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return y


def k3mx_route_topk(idx, w, logits, bias, stream=None):
    T = _tokens(logits, K3MX_N_EXPERTS, "logits")
    _numel(idx, T * K3MX_TOPK, "idx")
    _numel(w, T * K3MX_TOPK, "w")
    _numel(bias, K3MX_N_EXPERTS, "bias")
    _dev(idx, torch.int32, "idx")
    _dev(w, torch.float32, "w")
    _dev(logits, torch.float32, "logits")
    _dev(bias, torch.float32, "bias")
    T = logits.shape[0]
    _check("k3mx_route_topk", lib().k3mx_route_topk(_ptr(idx), _ptr(w), _ptr(logits), _ptr(bias), T,
                                                     _stream(stream)))
    return idx, w


def k3mx_router(logits, idx, w, hidden, router_w, bias, top_p=0.0, stream=None):
    """Router logits from the hidden state (fp32 or bf16 [T, 7168]) and the
    bf16 router weights (int16 or uint16-viewed [896, 7168]), then the top-16."""
    T = _tokens(hidden, 7168, "hidden")
    _numel(logits, T * K3MX_N_EXPERTS, "logits")
    _numel(idx, T * K3MX_TOPK, "idx")
    _numel(w, T * K3MX_TOPK, "w")
    _numel(bias, K3MX_N_EXPERTS, "bias")
    _numel(router_w, K3MX_N_EXPERTS * 7168, "router_w")
    _dev(logits, torch.float32, "logits")
    _dev(idx, torch.int32, "idx")
    _dev(w, torch.float32, "w")
    _dev(bias, torch.float32, "bias")
    if not (router_w.is_cuda and router_w.is_contiguous() and router_w.element_size() == 2):
        raise ValueError("router_w: contiguous 16-bit device tensor expected")
    if not (hidden.is_cuda and hidden.is_contiguous()):
        raise ValueError("hidden: contiguous device tensor expected")
    T = hidden.shape[0]
    _check("k3mx_router", lib().k3mx_router(_ptr(logits), _ptr(idx), _ptr(w), _ptr(hidden), _x_dtype(hidden),
                                            _ptr(router_w), _ptr(bias), T, float(top_p), _stream(stream)))
    return logits, idx, w


LATENT_BLOCK_FIELDS = ("router_w", "bias", "w_dn", "w_up", "g_norm", "w1s", "w3s", "w2s")


def latent_block(tensors):
    """A k3mx_latent_block from a dict of contiguous device tensors (bf16
    matrices as int16/uint16/bfloat16, the bias fp32)."""
    for n in LATENT_BLOCK_FIELDS:
        t = tensors[n]
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError(f"{n}: contiguous device tensor expected")
    return LatentBlock(*[tensors[n].data_ptr() for n in LATENT_BLOCK_FIELDS])


def k3mx_latent_moe_workspace_size(n_tokens, h_dtype):
    return int(lib().k3mx_latent_moe_workspace_size(n_tokens, h_dtype))


def k3mx_latent_moe(y, hidden, block, experts, workspace, top_p=0.0, idx_out=None, w_out=None, stream=None):
    """The LatentMoE block: y [T, 7168] fp32 from hidden [T, 7168] (fp32 or
    bf16).  `block` is a LatentBlock (see latent_block), `experts` the
    device expert table."""
    T = _tokens(hidden, 7168, "hidden")
    _numel(y, T * 7168, "y")
    _numel(idx_out, T * K3MX_TOPK, "idx_out", optional=True)
    _numel(w_out, T * K3MX_TOPK, "w_out", optional=True)
    _table(experts)
    _dev(y, torch.float32, "y")
    if not (hidden.is_cuda and hidden.is_contiguous()):
        raise ValueError("hidden: contiguous device tensor expected")
    _check("k3mx_latent_moe", lib().k3mx_latent_moe(
        _ptr(y), _ptr(hidden), _x_dtype(hidden), T, ctypes.byref(block), _ptr(experts), float(top_p),
        _ptr(idx_out), _ptr(w_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return y


def k3mx_route_topp(idx, w, logits, bias, top_p, stream=None):
    """k3mx_route_topk with the top-p truncation (dropped slots: -1, 0)."""
    T = _tokens(logits, K3MX_N_EXPERTS, "logits")
    _numel(idx, T * K3MX_TOPK, "idx")
    _numel(w, T * K3MX_TOPK, "w")
    _numel(bias, K3MX_N_EXPERTS, "bias")
    _dev(idx, torch.int32, "idx")
    _dev(w, torch.float32, "w")
    _dev(logits, torch.float32, "logits")
    _dev(bias, torch.float32, "bias")
    T = logits.shape[0]
    _check("k3mx_route_topp", lib().k3mx_route_topp(_ptr(idx), _ptr(w), _ptr(logits), _ptr(bias), T,
                                                     float(top_p), _stream(stream)))
    return idx, w


def k3mx_group_workspace_size(n_tokens):
    return int(lib().k3mx_group_workspace_size(n_tokens))


def k3mx_group(counts, offsets, perm, idx, workspace, stream=None):
    T = _tokens(idx, K3MX_TOPK, "idx")
    _numel(counts, K3MX_N_EXPERTS, "counts")
    _numel(offsets, K3MX_N_EXPERTS + 1, "offsets")
    _numel(perm, T * K3MX_TOPK, "perm")
    for t, n in ((counts, "counts"), (offsets, "offsets"), (perm, "perm"), (idx, "idx")):
        _dev(t, torch.int32, n)
    T = idx.shape[0]
    _check("k3mx_group", lib().k3mx_group(_ptr(counts), _ptr(offsets), _ptr(perm), _ptr(idx), T,
                                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream)))
    return counts, offsets, perm


def k3mx_moe_workspace_size(n_tokens, x_dtype, path=K3MX_PATH_AUTO):
    return int(lib().k3mx_moe_workspace_size(n_tokens, x_dtype, path))


def k3mx_moe_host_workspace_size(n_tokens, x_dtype, path=K3MX_PATH_AUTO):
    return int(lib().k3mx_moe_host_workspace_size(n_tokens, x_dtype, path))


def _x_dtype(x):
    if x.dtype == torch.float32:
        return K3MX_F32
    if x.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        return K3MX_BF16
    raise TypeError("x must be float32 or bfloat16")


def _moe_shapes(y, x, experts, logits, bias, idx_out, w_out):
    """The routed layer's tensors against the token count of x [T, 3584]."""
    T = _tokens(x, K3MX_LATENT, "x")
    _numel(y, T * K3MX_LATENT, "y")
    _numel(logits, T * K3MX_N_EXPERTS, "logits")
    _numel(bias, K3MX_N_EXPERTS, "bias")
    _numel(idx_out, T * K3MX_TOPK, "idx_out", optional=True)
    _numel(w_out, T * K3MX_TOPK, "w_out", optional=True)
    _table(experts)
    return T


def _dev_opt(t, dtype, name):
    if t is not None:
        _dev(t, dtype, name)


def k3mx_moe_routed(y, x, experts, logits, bias, workspace, path=K3MX_PATH_AUTO,
                    idx_out=None, w_out=None, stream=None):
    """The routed-expert layer on device tensors.  experts: device int64 [896, 6]
    table of pointers (see expert_table)."""
    _moe_shapes(y, x, experts, logits, bias, idx_out, w_out)
    _dev(y, torch.float32, "y")
    if not (x.is_cuda and x.is_contiguous()):
        raise TypeError("x: contiguous CUDA tensor expected")
    _dev(logits, torch.float32, "logits")
    _dev(bias, torch.float32, "bias")
    _dev(experts, torch.int64, "experts")
    _dev_opt(idx_out, torch.int32, "idx_out")
    _dev_opt(w_out, torch.float32, "w_out")
    T = x.shape[0]
    _check("k3mx_moe_routed", lib().k3mx_moe_routed(
        _ptr(y), _ptr(x), _x_dtype(x), T, _ptr(experts), _ptr(logits), _ptr(bias), path,
        _ptr(idx_out), _ptr(w_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return y


def k3mx_moe_routed_topp(y, x, experts, logits, bias, workspace, top_p, path=K3MX_PATH_AUTO,
                         idx_out=None, w_out=None, stream=None):
    """k3mx_moe_routed with top-p routing: the low-weight tail of each
    token's 16 experts is dropped and runs no expert."""
    _moe_shapes(y, x, experts, logits, bias, idx_out, w_out)
    _dev(y, torch.float32, "y")
    if not (x.is_cuda and x.is_contiguous()):
        raise TypeError("x: contiguous CUDA tensor expected")
    _dev(logits, torch.float32, "logits")
    _dev(bias, torch.float32, "bias")
    _dev(experts, torch.int64, "experts")
    _dev_opt(idx_out, torch.int32, "idx_out")
    _dev_opt(w_out, torch.float32, "w_out")
    T = x.shape[0]
    _check("k3mx_moe_routed_topp", lib().k3mx_moe_routed_topp(
        _ptr(y), _ptr(x), _x_dtype(x), T, _ptr(experts), _ptr(logits), _ptr(bias), path, float(top_p),
        _ptr(idx_out), _ptr(w_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return y


def k3mx_moe_decode_noalloc(y, x, experts, logits, bias, idx_out=None, w_out=None, stream=None):
    """The decode path on device tensors with the library's fixed scratch
    instead of a workspace (at most K3MX_NOALLOC_MAX_TOKENS tokens)."""
    _moe_shapes(y, x, experts, logits, bias, idx_out, w_out)
    _dev(y, torch.float32, "y")
    if not (x.is_cuda and x.is_contiguous()):
        raise TypeError("x: contiguous CUDA tensor expected")
    _dev(logits, torch.float32, "logits")
    _dev(bias, torch.float32, "bias")
    _dev(experts, torch.int64, "experts")
    _dev_opt(idx_out, torch.int32, "idx_out")
    _dev_opt(w_out, torch.float32, "w_out")
    _check("k3mx_moe_decode_noalloc", lib().k3mx_moe_decode_noalloc(
        _ptr(y), _ptr(x), _x_dtype(x), x.shape[0], _ptr(experts), _ptr(logits), _ptr(bias),
        _ptr(idx_out), _ptr(w_out), _stream(stream)))
    return y


def k3mx_moe_routed_host(y_host, x_host, experts, logits_host, bias_host, workspace,
                         path=K3MX_PATH_AUTO, stream=None):
    """The layer with host (CPU tensor) activations, logits, bias and output;
    weights and workspace on the device.  Returns after y_host is written."""
    _moe_shapes(y_host, x_host, experts, logits_host, bias_host, None, None)
    for t, n in ((y_host, "y"), (x_host, "x"), (logits_host, "logits"), (bias_host, "bias")):
        if t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{n}: contiguous host tensor expected")
    T = x_host.shape[0]
    _check("k3mx_moe_routed_host", lib().k3mx_moe_routed_host(
        _ptr(y_host), _ptr(x_host), _x_dtype(x_host), T, _ptr(experts), _ptr(logits_host),
        _ptr(bias_host), path, _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return y_host


def k3mx_device_status(stream=None):
    """(status, detail) of the device status word; waits for the stream, clears it."""
    d = ctypes.c_int(0)
    st = lib().k3mx_device_status(_stream(stream), ctypes.byref(d))
    return st, d.value


def k3mx_set_wait_limit(polls):
    """Polls after which a device-side wait gives up (0: the default)."""
    _check("k3mx_set_wait_limit", lib().k3mx_set_wait_limit(int(polls)))


def k3mx_trace_enable(on):
    _check("k3mx_trace_enable", lib().k3mx_trace_enable(1 if on else 0))


def k3mx_trace_read(max_entries=64):
    """{kernel name: (launches, total milliseconds)} of the traced launches; clears them."""
    buf = (TraceEntry * max_entries)()
    n = lib().k3mx_trace_read(buf, max_entries)
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(n)}


def k3mx_status_str(status):
    return lib().k3mx_status_str(status).decode()


def k3mx_abi_version():
    return int(lib().k3mx_abi_version())


# ---------------------------------------------------------- marshalling --

EXPERT_OFFSETS = None


def expert_offsets(D=K3MX_LATENT, F=K3MX_INTER):
    """Byte offsets of w1, s1, w3, s3, w2, s2 inside one expert stored back to back."""
    a, s = F * D // 2, F * D // 32
    return [0, a, a + s, 2 * a + s, 2 * (a + s), 2 * (a + s) + a]


def expert_table(arena, n_experts=K3MX_N_EXPERTS, stride=K3MX_EXPERT_BYTES):
    """Device int64 [n_experts, 6] pointer table (the k3mx_expert array) for an
    arena holding the experts back to back, each in w1 s1 w3 s3 w2 s2 order."""
    base = arena.data_ptr()
    offs = torch.tensor(expert_offsets(), dtype=torch.int64)
    table = base + torch.arange(n_experts, dtype=torch.int64)[:, None] * stride + offs[None, :]
    return table.to(arena.device)
