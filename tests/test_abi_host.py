"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/k3mx.h declares, and refuses bad arguments before it
touches the device."""
import ctypes
import re
import subprocess

import pytest
import torch

import mxfp4_routed_expert_k3mx_gb300 as k3mx

FAKE = 0x10000          # an aligned, non-null address that is never dereferenced


def test_library_exports_every_declared_symbol():
    L = k3mx.lib()
    declared = k3mx.declared_symbols()
    assert len(declared) == 23
    out = subprocess.run(["nm", "-D", "--defined-only", k3mx.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(k3mx_\w+)", out))
    assert set(declared) <= exported, set(declared) - exported
    for name in declared:
        assert hasattr(L, name)


def test_status_strings_and_version():
    assert k3mx.k3mx_abi_version() >> 16 == 1
    for code in range(8):
        assert k3mx.k3mx_status_str(code)
    assert k3mx.k3mx_status_str(99) == "unknown status"
    assert k3mx.lib().k3mx_last_cuda_error() in (b"cudaSuccess", b"cudaErrorNoDevice", b"cudaErrorInsufficientDriver")


def test_gemv_refuses_bad_arguments():
    L = k3mx.lib()
    assert L.k3mx_gemv(None, FAKE, FAKE, FAKE, 64, 4, None) == 1            # NULL
    assert L.k3mx_gemv(FAKE, FAKE, FAKE, FAKE, 33, 4, None) == 3            # in % 32
    assert L.k3mx_gemv(FAKE, FAKE, FAKE, FAKE, 0, 4, None) == 3
    assert L.k3mx_gemv(FAKE, FAKE, FAKE, FAKE, 16384 + 32, 4, None) == 3    # in too large
    assert L.k3mx_gemv(FAKE, FAKE, FAKE, FAKE, 64, 0, None) == 3            # rows < 1
    assert L.k3mx_gemv(FAKE + 4, FAKE, FAKE, FAKE, 64, 4, None) == 2        # y misaligned
    assert L.k3mx_gemv(FAKE, FAKE, FAKE + 8, FAKE, 64, 4, None) == 2        # packed misaligned


def test_route_group_refuse_bad_arguments():
    L = k3mx.lib()
    assert L.k3mx_route_topk(FAKE, FAKE, FAKE, None, 1, None) == 1
    assert L.k3mx_route_topk(FAKE, FAKE, FAKE, FAKE, 0, None) == 3
    assert L.k3mx_route_topk(FAKE, FAKE, FAKE, FAKE, 65537, None) == 3
    assert L.k3mx_route_topk(FAKE, FAKE + 4, FAKE, FAKE, 1, None) == 2
    for p in (float("nan"), float("inf"), float("-inf")):                 # top_p not finite
        assert L.k3mx_route_topp(FAKE, FAKE, FAKE, FAKE, 1, p, None) == 1
    assert L.k3mx_route_topp(FAKE, FAKE, FAKE, None, 1, 0.5, None) == 1
    assert L.k3mx_route_topp(FAKE, FAKE, FAKE, FAKE, 0, 0.5, None) == 3
    assert L.k3mx_route_topp(FAKE, FAKE + 4, FAKE, FAKE, 1, 0.5, None) == 2
    ws = k3mx.k3mx_group_workspace_size(64)
    assert ws > 0 and k3mx.k3mx_group_workspace_size(0) == 0
    assert L.k3mx_group(FAKE, FAKE, FAKE, FAKE, 64, FAKE, ws - 1, None) == 4
    assert L.k3mx_group(FAKE, FAKE, FAKE, FAKE, 64, None, ws, None) == 4


def test_router_refuses_bad_arguments():
    L = k3mx.lib()
    ok = dict(lg=FAKE, idx=FAKE, w=FAKE, h=FAKE, dt=0, W=FAKE, b=FAKE, T=1, p=0.0)
    call = lambda **kw: L.k3mx_router(*(dict(ok, **kw)[k] for k in ("lg", "idx", "w", "h", "dt", "W", "b", "T", "p")),
                                      None)
    assert call(W=None) == 1
    assert call(dt=2) == 1                           # unknown hidden dtype
    assert call(p=float("nan")) == 1
    assert call(T=0) == 3 and call(T=65537) == 3
    assert call(h=FAKE + 4) == 2 and call(W=FAKE + 8) == 2


def test_latent_block_refuses_bad_arguments():
    L = k3mx.lib()
    blk = k3mx.LatentBlock(*([FAKE] * 8))
    ws = k3mx.k3mx_latent_moe_workspace_size(1, k3mx.K3MX_F32)
    assert ws > k3mx.k3mx_moe_workspace_size(1, k3mx.K3MX_F32, k3mx.K3MX_PATH_DECODE)
    assert k3mx.k3mx_latent_moe_workspace_size(0, 0) == 0 and k3mx.k3mx_latent_moe_workspace_size(1, 2) == 0
    # bf16 batches keep bf16 intermediates: a 4096-token workspace holds the
    # shared experts' g | u in fp32 and their activation in bf16
    assert k3mx.k3mx_latent_moe_workspace_size(4096, 1) >= 4096 * (2 * 6144 * 4 + 6144 * 2)
    call = lambda **kw: L.k3mx_latent_moe(*(dict(dict(y=FAKE, h=FAKE, dt=0, T=1, b=ctypes.byref(blk), ex=FAKE, p=0.0,
                                                      io=None, wo=None, ws=FAKE, wsb=ws), **kw)[k]
                                            for k in ("y", "h", "dt", "T", "b", "ex", "p", "io", "wo", "ws", "wsb")),
                                          None)
    assert call(b=None) == 1 and call(ex=None) == 1
    assert call(dt=2) == 1 and call(p=float("nan")) == 1
    assert call(T=0) == 3
    assert call(h=FAKE + 4) == 2
    assert call(wsb=ws - 1) == 4
    bad = k3mx.LatentBlock(*([FAKE] * 7 + [None]))
    assert call(b=ctypes.byref(bad)) == 1                      # every tensor of the block is required
    bad = k3mx.LatentBlock(*([FAKE] * 4 + [FAKE + 2] + [FAKE] * 3))
    assert call(b=ctypes.byref(bad)) == 2                      # g_norm misaligned


def test_moe_refuses_bad_arguments():
    L = k3mx.lib()
    ws = k3mx.k3mx_moe_workspace_size(1, k3mx.K3MX_F32, k3mx.K3MX_PATH_DECODE)
    args = lambda **kw: dict(dict(y=FAKE, x=FAKE, dt=0, T=1, ex=FAKE, lg=FAKE, b=FAKE, path=1,
                                  io=None, wo=None, ws=FAKE, wsb=ws), **kw)
    call = lambda a: L.k3mx_moe_routed(a["y"], a["x"], a["dt"], a["T"], a["ex"], a["lg"], a["b"],
                                       a["path"], a["io"], a["wo"], a["ws"], a["wsb"], None)
    assert call(args(ex=None)) == 1
    assert call(args(dt=2)) == 1                     # unknown dtype
    assert call(args(path=4)) == 1                   # unknown path
    assert call(args(path=2)) == 1                   # prefill needs bf16 x
    assert call(args(path=3)) == 1                   # so does the block-scaled prefill
    assert call(args(T=0)) == 3
    assert call(args(x=FAKE + 2)) == 2
    assert call(args(wsb=ws - 1)) == 4
    assert call(args(ws=FAKE + 16)) == 2             # workspace must be 256-byte aligned


def test_workspace_sizes():
    d = [k3mx.k3mx_moe_workspace_size(t, 0, 1) for t in (1, 2, 64, 1000)]
    # grows with the batch (one token also holds the split-item hand-over region)
    assert all(a < b for a, b in zip(d[1:], d[2:])) and d[0] > 0
    # the decode path keeps h and the per-pair outputs in fp32
    assert k3mx.k3mx_moe_workspace_size(64, 0, 1) >= 64 * 16 * (2 * 3072 + 3584) * 4
    # AUTO picks prefill for bf16 and many tokens; its h is f16
    assert k3mx.k3mx_moe_workspace_size(4096, 1, 0) == k3mx.k3mx_moe_workspace_size(4096, 1, 3)
    assert k3mx.k3mx_moe_workspace_size(4096, 1, 2) >= 4096 * 16 * 3072 * 2
    assert k3mx.k3mx_moe_host_workspace_size(64, 1, 1) > k3mx.k3mx_moe_workspace_size(64, 1, 1)
    # g and u, then the MXFP4 pieces of x and h and the tensor-map slots
    assert k3mx.k3mx_expert_ffn_workspace_size() >= 2 * 3072 * 4 + 8 * (3584 + 3072) // 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour only")
def test_valid_call_without_gpu_fails_loudly():
    """With no device the library reports a CUDA error; it has no CPU path."""
    L = k3mx.lib()
    assert L.k3mx_gemv(FAKE, FAKE, FAKE, FAKE, 64, 4, None) in (5, 7)


def test_noalloc_refuses_bad_arguments():
    L = k3mx.lib()
    call = lambda T, dt=0, x=FAKE, io=None: L.k3mx_moe_decode_noalloc(
        FAKE, x, dt, T, FAKE, FAKE, FAKE, io, None, None)
    assert call(k3mx.K3MX_NOALLOC_MAX_TOKENS + 1) == 3       # above the fixed scratch
    assert call(0) == 3
    assert call(1, dt=2) == 1
    assert call(1, x=FAKE + 2) == 2
    assert call(1, io=FAKE + 4) == 2
    # the fixed 8 MiB array holds the decode layout of the largest batch, either dtype
    for dt in (0, 1):
        assert k3mx.k3mx_moe_workspace_size(k3mx.K3MX_NOALLOC_MAX_TOKENS, dt, 1) <= 8 << 20


def test_binding_refuses_mismatched_shapes():
    """The Python binding checks every tensor against the token count before
    any device check or library call (the C ABI sees raw pointers only, so a
    short output would be written past its end)."""
    f32 = lambda *s: torch.zeros(*s, dtype=torch.float32)
    table = torch.zeros(896, 6, dtype=torch.int64)
    ws = torch.zeros(16, dtype=torch.uint8)
    bad = [
        # x must be [T, 3584]: a 1-D x would read as 3584 tokens
        lambda: k3mx.k3mx_moe_routed(f32(3584), f32(3584), table, f32(896), f32(896), ws),
        # y shorter than the batch
        lambda: k3mx.k3mx_moe_routed(f32(1, 3584), f32(8, 3584), table, f32(8, 896), f32(896), ws),
        # logits of another batch
        lambda: k3mx.k3mx_moe_routed(f32(8, 3584), f32(8, 3584), table, f32(4, 896), f32(896), ws),
        # routing outputs too short
        lambda: k3mx.k3mx_moe_routed(f32(8, 3584), f32(8, 3584), table, f32(8, 896), f32(896), ws,
                                     idx_out=torch.zeros(16, dtype=torch.int32)),
        # expert table of the wrong shape or type
        lambda: k3mx.k3mx_moe_routed(f32(2, 3584), f32(2, 3584), table[:100], f32(2, 896), f32(896), ws),
        lambda: k3mx.k3mx_moe_routed(f32(2, 3584), f32(2, 3584), table.int(), f32(2, 896), f32(896), ws),
        lambda: k3mx.k3mx_moe_routed_topp(f32(2, 3584), f32(2, 3584), table, f32(2, 896), f32(895), ws, 0.5),
        lambda: k3mx.k3mx_moe_decode_noalloc(f32(3, 3584), f32(2, 3584), table, f32(2, 896), f32(896)),
        lambda: k3mx.k3mx_moe_routed_host(f32(2, 3584), f32(2, 3583), table, f32(2, 896), f32(896), ws),
        lambda: k3mx.k3mx_route_topk(torch.zeros(2, 16, dtype=torch.int32), f32(2, 8), f32(2, 896), f32(896)),
        lambda: k3mx.k3mx_route_topp(torch.zeros(2, 16, dtype=torch.int32), f32(2, 16), f32(896), f32(896), 0.5),
        lambda: k3mx.k3mx_group(torch.zeros(896, dtype=torch.int32), torch.zeros(896, dtype=torch.int32),
                                torch.zeros(32, dtype=torch.int32), torch.zeros(2, 16, dtype=torch.int32), ws),
        lambda: k3mx.k3mx_router(f32(2, 896), torch.zeros(2, 16, dtype=torch.int32), f32(2, 16), f32(2, 7000),
                                 torch.zeros(896, 7168, dtype=torch.int16), f32(896)),
        lambda: k3mx.k3mx_latent_moe(f32(2, 3584), f32(2, 7168), None, table, ws),
        lambda: k3mx.k3mx_expert_ffn(f32(3584), f32(3072), None, ws),
        lambda: k3mx.k3mx_gemv(f32(64), f32(128), torch.zeros(64, 64, dtype=torch.uint8),
                               torch.zeros(64, 3, dtype=torch.uint8)),
        lambda: k3mx.k3mx_gemv(f32(63), f32(128), torch.zeros(64, 64, dtype=torch.uint8),
                               torch.zeros(64, 4, dtype=torch.uint8)),
    ]
    for i, call in enumerate(bad):
        with pytest.raises(TypeError) as err:
            call()
        assert "CUDA" not in str(err.value), (i, str(err.value))    # refused for its shape, not its device
    # well-shaped host tensors pass the shape checks and stop at the device check
    with pytest.raises(TypeError, match="CUDA"):
        k3mx.k3mx_moe_routed(f32(2, 3584), f32(2, 3584), table, f32(2, 896), f32(896), ws)
