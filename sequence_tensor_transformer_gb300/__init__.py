"""GB300 (sm_103a) SP-TP FFN boundary and Delayed-TP stack.

Thin ctypes binding over libsptp.so: every function here marshals torch
tensors (device memory) and the current CUDA stream into the C ABI declared
in include/sptp.h and raises on a non-zero status.  All computation runs in
the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "SPTP_BF16", "SPTP_FP32", "SPTP_WS_HEADER_BYTES", "SptpError", "lib", "load_library",
    "sptp_ffn_workspace_size", "sptp_ffn_forward", "dtp_ffn_stack_workspace_size",
    "dtp_ffn_stack_forward", "sptp_prologue", "sptp_gateup_swiglu", "sptp_down_proj",
    "sptp_read_device_status", "sptp_wait_selftest", "sptp_status_string", "EXPORTED_SYMBOLS",
    "sptp_ffn_forward_noalloc", "SPTP_NOALLOC_SCRATCH_BYTES", "sptp_permute_ffn_neurons",
    "sptp_attn_qkv_workspace_size", "sptp_attn_qkv_forward", "sptp_quantize_rows_e4m3",
    "quantize_ffn_weights_e4m3", "sptp_ffn_fp8_workspace_size", "sptp_ffn_forward_fp8",
    "sptp_gateup_swiglu_e4m3", "sptp_down_proj_e4m3", "sptp_prologue_e4m3", "VARIANTS", "STATUS",
    "sptp_noalloc_read_device_status", "sptp_noalloc_wait_selftest", "CHECKED_LIB_PATH", "set_library",
]

SPTP_BF16 = 0
SPTP_FP32 = 1
SPTP_WS_HEADER_BYTES = 4096
SPTP_NOALLOC_SCRATCH_BYTES = 64 << 20
# sptp_variant: how a boundary call is split into launches (include/sptp.h)
VARIANTS = {"auto": 0, "pair": 1, "chain": 2, "fused": 3, "layers": 4}
# sptp_status codes
STATUS = {"ok": 0, "null": -1, "shape": -2, "dtype": -3, "workspace": -4, "cuda": -5, "timeout": -6,
          "unimplemented": -7, "alias": -8, "too_large": -9, "device": -10, "bounds": -11}
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsptp.so")

EXPORTED_SYMBOLS = (
    "sptp_ffn_workspace_size", "sptp_ffn_forward", "dtp_ffn_stack_workspace_size",
    "dtp_ffn_stack_forward", "sptp_prologue", "sptp_gateup_swiglu", "sptp_down_proj",
    "sptp_read_device_status", "sptp_wait_selftest", "sptp_status_string", "sptp_ffn_forward_noalloc",
    "sptp_permute_ffn_neurons", "sptp_attn_qkv_workspace_size", "sptp_attn_qkv_forward",
    "sptp_quantize_rows_e4m3", "sptp_ffn_fp8_workspace_size", "sptp_ffn_forward_fp8", "sptp_gateup_swiglu_e4m3",
    "sptp_down_proj_e4m3", "sptp_prologue_e4m3", "sptp_ffn_forward_ex", "dtp_ffn_stack_forward_ex",
    "sptp_attn_qkv_forward_ex", "sptp_noalloc_read_device_status", "sptp_noalloc_wait_selftest",
)

_lib = None

_P, _I, _F, _Z, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_ulonglong
_LL = ctypes.c_longlong
_SIGS = {
    "sptp_ffn_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "sptp_ffn_forward": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _Z, _P]),
    "dtp_ffn_stack_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "dtp_ffn_stack_forward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "sptp_prologue": (_I, [_P, _P, _P, _I, _I, _I, _F, _I, _P, _P, _P]),
    "sptp_gateup_swiglu": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "sptp_down_proj": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "sptp_read_device_status": (_I, [_P, _P]),
    "sptp_wait_selftest": (_I, [_P, _Z, _U64, _I, _P]),
    "sptp_status_string": (ctypes.c_char_p, [_I]),
    "sptp_ffn_forward_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P]),
    "sptp_permute_ffn_neurons": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "sptp_attn_qkv_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "sptp_attn_qkv_forward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _Z, _P]),
    "sptp_quantize_rows_e4m3": (_I, [_P, _LL, _I, _P, _P, _P]),
    "sptp_ffn_fp8_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "sptp_ffn_forward_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _Z,
                                  _P]),
    "sptp_gateup_swiglu_e4m3": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "sptp_down_proj_e4m3": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "sptp_prologue_e4m3": (_I, [_P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _P, _P]),
    "sptp_ffn_forward_ex": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _Z, _P, _I]),
    "dtp_ffn_stack_forward_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P, _I]),
    "sptp_attn_qkv_forward_ex": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _Z, _P, _I]),
    "sptp_noalloc_read_device_status": (_I, [_P]),
    "sptp_noalloc_wait_selftest": (_I, [_U64, _I, _P]),
}


class SptpError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({sptp_status_string(code)})")
        self.code = code


CHECKED_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsptp_check.so")


def load_library(path: str = LIB_PATH, replace: bool = False):
    """Loads libsptp.so (built by sequence_tensor_transformer_gb300.build) on
    first use.  replace=True makes `path` the library every later call uses:
    for example CHECKED_LIB_PATH, the bounds-checked build (build(checked=True))."""
    global _lib
    if _lib is None or replace:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib_ = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib_, name)
            f.restype = res
            f.argtypes = args
        _lib = lib_
    return _lib


def set_library(handle):
    """Makes a handle returned by load_library the one every call uses."""
    global _lib
    _lib = handle


def lib():
    return load_library()


def sptp_status_string(code: int) -> str:
    return lib().sptp_status_string(int(code)).decode()


# ------------------------------------------------------------------ helpers

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPTP_BF16
    if t.dtype == torch.float32:
        return SPTP_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensors only")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _expect(name, t, shape, dtype, optional=False):
    """Shape and dtype of a tensor argument, checked before any pointer is
    passed: the C ABI takes pointers and sizes only, so a tensor of the wrong
    shape would otherwise be read or written past its end."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")


def _same_device(*ts):
    """Every tensor argument on one CUDA device, the current one: the library
    launches on the current device and takes its stream, scratch and device
    properties from it, so a tensor elsewhere would be handed to kernels of
    another device.  Checked before any pointer reaches the C ABI."""
    ts = [t for t in ts if t is not None]
    for t in ts[1:]:
        if t.device != ts[0].device:
            raise ValueError(f"tensors on {ts[0].device} and {t.device}: one device expected")
    if ts and ts[0].device.type != "cuda":
        raise ValueError("device tensors only")
    if ts:
        cur = torch.cuda.current_device()
        if ts[0].device.index != cur:
            raise ValueError(f"tensors on {ts[0].device} but the current device is cuda:{cur}: "
                             f"call torch.cuda.set_device({ts[0].device.index}) first")


def _variant(v) -> int:
    if isinstance(v, str):
        if v not in VARIANTS:
            raise ValueError(f"unknown variant {v!r}; one of {sorted(VARIANTS)}")
        return VARIANTS[v]
    return int(v)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if stream.device.index != torch.cuda.current_device():
        raise ValueError(f"stream on {stream.device} but the current device is cuda:{torch.cuda.current_device()}")
    return stream.cuda_stream


def _check(fn: str, code: int):
    if code != 0:
        raise SptpError(fn, code)


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, SPTP_WS_HEADER_BYTES), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ entry points

def sptp_ffn_workspace_size(M, d, F, P, chunks, dtype=SPTP_BF16) -> int:
    return int(lib().sptp_ffn_workspace_size(M, d, F, P, chunks, dtype))


def dtp_ffn_stack_workspace_size(M, d, F, P, L, delta, dtype=SPTP_BF16) -> int:
    return int(lib().dtp_ffn_stack_workspace_size(M, d, F, P, L, delta, dtype))


def _check_ffn_args(x, partials, gamma, W1g, W1u, W2, P, out, resid_out, dtype=None):
    M, d = x.shape
    F = W1g.shape[0]
    dt = x.dtype if dtype is None else dtype
    _expect("partials", partials, (P, M, d), dt)
    _expect("gamma", gamma, (d,), dt)
    _expect("W1g", W1g, (F, d), dt)
    _expect("W1u", W1u, (F, d), dt)
    _expect("W2", W2, (d, F), dt)
    _expect("out", out, (P, M, d), dt, optional=True)
    _expect("resid_out", resid_out, (M, d), dt, optional=True)
    _same_device(x, partials, gamma, W1g, W1u, W2, out, resid_out)


def sptp_ffn_forward(x, partials, gamma, W1g, W1u, W2, P, chunks, eps, out=None, resid_out=None,
                     workspace=None, stream=None, write_resid=True, variant="auto"):
    """SP-TP FFN boundary.  Returns (out [P,M,d], resid_out [M,d] or None).
    variant: "auto" (the library's default), "pair", "chain" or "fused"."""
    M, d = x.shape
    F = W1g.shape[0]
    dt = _dtype_code(x)
    _check_ffn_args(x, partials, gamma, W1g, W1u, W2, P, out, resid_out)
    if out is None:
        out = torch.empty((P, M, d), dtype=x.dtype, device=x.device)
    if resid_out is None and write_resid:
        resid_out = torch.empty_like(x)
    if workspace is None:
        workspace = _workspace(sptp_ffn_workspace_size(M, d, F, P, chunks, dt), x.device)
    _same_device(x, workspace)
    code = lib().sptp_ffn_forward_ex(
        _ptr(x), _ptr(partials), _ptr(gamma), _ptr(W1g), _ptr(W1u), _ptr(W2), M, d, F, P, chunks,
        float(eps), dt, _ptr(out), _ptr(resid_out), _ptr(workspace), _nbytes(workspace), _stream(stream),
        _variant(variant))
    _check("sptp_ffn_forward", code)
    return out, resid_out


def dtp_ffn_stack_forward(x_shards, gamma, W1g, W1u, W2, P, L, delta, flush, eps, workspace=None,
                          stream=None, variant="auto"):
    """Delayed-TP stack; updates x_shards [P,M,d] in place and returns it.
    variant: "auto" (the library's default), "fused" or "layers"."""
    _, M, d = x_shards.shape
    F = W1g.shape[1]
    dt = _dtype_code(x_shards)
    _expect("x_shards", x_shards, (P, M, d), x_shards.dtype)
    _expect("gamma", gamma, (L, d), x_shards.dtype)
    _expect("W1g", W1g, (L, F, d), x_shards.dtype)
    _expect("W1u", W1u, (L, F, d), x_shards.dtype)
    _expect("W2", W2, (L, d, F), x_shards.dtype)
    if workspace is None:
        workspace = _workspace(dtp_ffn_stack_workspace_size(M, d, F, P, L, delta, dt), x_shards.device)
    _same_device(x_shards, gamma, W1g, W1u, W2, workspace)
    code = lib().dtp_ffn_stack_forward_ex(
        _ptr(x_shards), _ptr(gamma), _ptr(W1g), _ptr(W1u), _ptr(W2), M, d, F, P, L, delta, int(flush),
        float(eps), dt, _ptr(workspace), _nbytes(workspace), _stream(stream), _variant(variant))
    _check("dtp_ffn_stack_forward", code)
    return x_shards


def sptp_prologue(x, partials, gamma, eps, h_out=None, y_out=None, stream=None, write_h=True):
    M, d = x.shape
    P = partials.shape[0]
    _expect("partials", partials, (P, M, d), x.dtype)
    _expect("gamma", gamma, (d,), x.dtype)
    _expect("h_out", h_out, (M, d), x.dtype, optional=True)
    _expect("y_out", y_out, (M, d), x.dtype, optional=True)
    _same_device(x, partials, gamma, h_out, y_out)
    if y_out is None:
        y_out = torch.empty_like(x)
    if h_out is None and write_h:
        h_out = torch.empty_like(x)
    code = lib().sptp_prologue(_ptr(x), _ptr(partials), _ptr(gamma), M, d, P, float(eps), _dtype_code(x),
                               _ptr(h_out), _ptr(y_out), _stream(stream))
    _check("sptp_prologue", code)
    return h_out, y_out


def sptp_gateup_swiglu(y, W1g, W1u, P, s_out=None, workspace=None, stream=None):
    M, d = y.shape
    F = W1g.shape[0]
    _expect("W1g", W1g, (F, d), y.dtype)
    _expect("W1u", W1u, (F, d), y.dtype)
    _expect("s_out", s_out, (P, M, F // P), y.dtype, optional=True)
    if s_out is None:
        s_out = torch.empty((P, M, F // P), dtype=y.dtype, device=y.device)
    if workspace is None:
        workspace = _workspace(SPTP_WS_HEADER_BYTES, y.device)
    _same_device(y, W1g, W1u, s_out, workspace)
    code = lib().sptp_gateup_swiglu(_ptr(y), _ptr(W1g), _ptr(W1u), M, d, F, P, _dtype_code(y), _ptr(s_out),
                                    _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check("sptp_gateup_swiglu", code)
    return s_out


def sptp_down_proj(s, W2, P, out=None, workspace=None, stream=None):
    _, M, f = s.shape
    d, F = W2.shape
    _expect("s", s, (P, M, F // P), s.dtype)
    _expect("out", out, (P, M, d), s.dtype, optional=True)
    _expect("W2", W2, (d, F), s.dtype)
    if out is None:
        out = torch.empty((P, M, d), dtype=s.dtype, device=s.device)
    if workspace is None:
        workspace = _workspace(SPTP_WS_HEADER_BYTES, s.device)
    _same_device(s, W2, out, workspace)
    code = lib().sptp_down_proj(_ptr(s), _ptr(W2), M, d, F, P, _dtype_code(s), _ptr(out), _ptr(workspace),
                                _nbytes(workspace), _stream(stream))
    _check("sptp_down_proj", code)
    return out


def sptp_ffn_forward_noalloc(x, partials, gamma, W1g, W1u, W2, P, chunks, eps, out, resid_out=None,
                             stream=None):
    """SP-TP FFN boundary on the library's static scratch (no workspace and no
    device allocation inside the call; the caller passes out/resid_out)."""
    M, d = x.shape
    F = W1g.shape[0]
    _expect("out", out, (P, M, d), x.dtype)
    _check_ffn_args(x, partials, gamma, W1g, W1u, W2, P, out, resid_out)
    code = lib().sptp_ffn_forward_noalloc(
        _ptr(x), _ptr(partials), _ptr(gamma), _ptr(W1g), _ptr(W1u), _ptr(W2), M, d, F, P, chunks, float(eps),
        _dtype_code(x), _ptr(out), _ptr(resid_out), _stream(stream))
    _check("sptp_ffn_forward_noalloc", code)
    return out, resid_out


def sptp_noalloc_read_device_status(stream=None) -> int:
    """Status words of the last no-allocation forward on the current device."""
    return int(lib().sptp_noalloc_read_device_status(_stream(stream)))


def sptp_noalloc_wait_selftest(limit_ns: int, preset_flag: bool, stream=None) -> int:
    return int(lib().sptp_noalloc_wait_selftest(int(limit_ns), int(preset_flag), _stream(stream)))


def sptp_attn_qkv_workspace_size(M, d, N, P, chunks, dtype=SPTP_BF16) -> int:
    return int(lib().sptp_attn_qkv_workspace_size(M, d, N, P, chunks, dtype))


def sptp_attn_qkv_forward(x, partials, gamma, Wqkv, P, chunks, eps, qkv_out=None, resid_out=None,
                          workspace=None, stream=None, write_resid=True, variant="auto"):
    """Boundary in front of attention: returns (qkv [P,M,N/P], resid_out).
    variant: "auto" (the library's default), "pair" or "fused"."""
    M, d = x.shape
    N = Wqkv.shape[0]
    dt = _dtype_code(x)
    _expect("partials", partials, (P, M, d), x.dtype)
    _expect("gamma", gamma, (d,), x.dtype)
    _expect("Wqkv", Wqkv, (N, d), x.dtype)
    _expect("qkv_out", qkv_out, (P, M, N // P), x.dtype, optional=True)
    _expect("resid_out", resid_out, (M, d), x.dtype, optional=True)
    _same_device(x, partials, gamma, Wqkv, qkv_out, resid_out, workspace)
    if qkv_out is None:
        qkv_out = torch.empty((P, M, N // P), dtype=x.dtype, device=x.device)
    if resid_out is None and write_resid:
        resid_out = torch.empty_like(x)
    if workspace is None:
        workspace = _workspace(sptp_attn_qkv_workspace_size(M, d, N, P, chunks, dt), x.device)
    code = lib().sptp_attn_qkv_forward_ex(_ptr(x), _ptr(partials), _ptr(gamma), _ptr(Wqkv), M, d, N, P, chunks,
                                          float(eps), dt, _ptr(qkv_out), _ptr(resid_out), _ptr(workspace),
                                          _nbytes(workspace), _stream(stream), _variant(variant))
    _check("sptp_attn_qkv_forward", code)
    return qkv_out, resid_out


def sptp_permute_ffn_neurons(W1g, W1u, W2, perm, workspace=None, stream=None):
    """Renumbers every module's neurons (W1g/W1u [L,F,d] rows, W2 [L,d,F]
    columns) by perm [L,F] (int32, device); returns the permuted copies."""
    L, F, d = W1g.shape
    _expect("W1u", W1u, (L, F, d), W1g.dtype)
    _expect("W2", W2, (L, d, F), W1g.dtype)
    _expect("perm", perm, (L, F), torch.int32)
    if workspace is None:
        workspace = _workspace(SPTP_WS_HEADER_BYTES, W1g.device)
    _same_device(W1g, W1u, W2, perm, workspace)
    outs = [torch.empty_like(W1g), torch.empty_like(W1u), torch.empty_like(W2)]
    code = lib().sptp_permute_ffn_neurons(_ptr(W1g), _ptr(W1u), _ptr(W2), _ptr(perm), L, d, F, _dtype_code(W1g),
                                          _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _ptr(workspace),
                                          _nbytes(workspace), _stream(stream))
    _check("sptp_permute_ffn_neurons", code)
    return tuple(outs)


def sptp_read_device_status(workspace, stream=None) -> int:
    _same_device(workspace)
    return int(lib().sptp_read_device_status(_ptr(workspace), _stream(stream)))


def sptp_wait_selftest(workspace, limit_ns: int, preset_flag: bool, stream=None) -> int:
    _same_device(workspace)
    return int(lib().sptp_wait_selftest(_ptr(workspace), _nbytes(workspace), int(limit_ns), int(preset_flag),
                                        _stream(stream)))


# ------------------------------------------------------------------ fp8 (E4M3)

def sptp_quantize_rows_e4m3(a, q=None, scale=None, stream=None):
    """Row-wise E4M3 quantisation of a bf16 tensor viewed as [R][K] (K = the
    last dimension).  Returns (q uint8 [..., K], scale float32 [...]):
    a ~= q * scale[..., None] with scale a power of two per row."""
    if a.dtype != torch.bfloat16:
        raise TypeError("bf16 input expected")
    K = a.shape[-1]
    R = a.numel() // K if K else 0
    _expect("q", q, tuple(a.shape), torch.uint8, optional=True)
    _expect("scale", scale, tuple(a.shape[:-1]), torch.float32, optional=True)
    _same_device(a, q, scale)
    if q is None:
        q = torch.empty(a.shape, dtype=torch.uint8, device=a.device)
    if scale is None:
        scale = torch.empty(a.shape[:-1], dtype=torch.float32, device=a.device)
    code = lib().sptp_quantize_rows_e4m3(_ptr(a), R, K, _ptr(q), _ptr(scale), _stream(stream))
    _check("sptp_quantize_rows_e4m3", code)
    return q, scale


def quantize_ffn_weights_e4m3(W1g, W1u, W2, P, stream=None):
    """The fp8 weights of one FFN in the layout sptp_ffn_forward_fp8 takes:
    (qW1g, sW1g [F], qW1u, sW1u [F], qW2 [d,F], sW2 [d,P]); W2 is quantised as
    [d*P][F/P] rows, one scale per output feature and shard."""
    d, F = W2.shape
    _expect("W1g", W1g, (F, d), torch.bfloat16)
    _expect("W1u", W1u, (F, d), torch.bfloat16)
    if F % P != 0:
        raise ValueError(f"F = {F} is not a multiple of P = {P}")
    qg, sg = sptp_quantize_rows_e4m3(W1g, stream=stream)
    qu, su = sptp_quantize_rows_e4m3(W1u, stream=stream)
    q2, s2 = sptp_quantize_rows_e4m3(W2.view(d, P, F // P), stream=stream)
    return qg, sg, qu, su, q2.view(d, F), s2


def sptp_ffn_fp8_workspace_size(M, d, F, P, chunks) -> int:
    return int(lib().sptp_ffn_fp8_workspace_size(M, d, F, P, chunks))


def sptp_ffn_forward_fp8(x, partials, gamma, qweights, P, chunks, eps, out=None, resid_out=None, workspace=None,
                         stream=None, write_resid=True):
    """SP-TP FFN boundary with E4M3 linear layers; qweights as returned by
    quantize_ffn_weights_e4m3.  Returns (out [P,M,d], resid_out [M,d] or None)."""
    qg, sg, qu, su, q2, s2 = qweights
    M, d = x.shape
    F = qg.shape[0]
    bf = torch.bfloat16
    _expect("x", x, (M, d), bf)
    _expect("partials", partials, (P, M, d), bf)
    _expect("gamma", gamma, (d,), bf)
    for name, t, shape, dt in (("qW1g", qg, (F, d), torch.uint8), ("sW1g", sg, (F,), torch.float32),
                               ("qW1u", qu, (F, d), torch.uint8), ("sW1u", su, (F,), torch.float32),
                               ("qW2", q2, (d, F), torch.uint8), ("sW2", s2, (d, P), torch.float32)):
        _expect(name, t, shape, dt)
    _expect("out", out, (P, M, d), bf, optional=True)
    _expect("resid_out", resid_out, (M, d), bf, optional=True)
    _same_device(x, partials, gamma, qg, sg, qu, su, q2, s2, out, resid_out, workspace)
    if out is None:
        out = torch.empty((P, M, d), dtype=x.dtype, device=x.device)
    if resid_out is None and write_resid:
        resid_out = torch.empty_like(x)
    if workspace is None:
        workspace = _workspace(sptp_ffn_fp8_workspace_size(M, d, F, P, chunks), x.device)
    code = lib().sptp_ffn_forward_fp8(
        _ptr(x), _ptr(partials), _ptr(gamma), _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su), _ptr(q2), _ptr(s2), M, d, F,
        P, chunks, float(eps), _ptr(out), _ptr(resid_out), _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check("sptp_ffn_forward_fp8", code)
    return out, resid_out


def sptp_prologue_e4m3(x, partials, gamma, eps, h_out=None, y_work=None, q_out=None, scale_out=None, stream=None,
                       write_h=True):
    """Partial sum + residual + RMSNorm with y quantised to E4M3 in the same
    launch.  Returns (h or None, q uint8 [M,d], scale float32 [M])."""
    M, d = x.shape
    P = partials.shape[0]
    bf = torch.bfloat16
    _expect("x", x, (M, d), bf)
    _expect("partials", partials, (P, M, d), bf)
    _expect("gamma", gamma, (d,), bf)
    _expect("h_out", h_out, (M, d), bf, optional=True)
    _expect("y_work", y_work, (M, d), bf, optional=True)
    _expect("q_out", q_out, (M, d), torch.uint8, optional=True)
    _expect("scale_out", scale_out, (M,), torch.float32, optional=True)
    _same_device(x, partials, gamma, h_out, y_work, q_out, scale_out)
    if h_out is None and write_h:
        h_out = torch.empty_like(x)
    if y_work is None:
        y_work = torch.empty_like(x)
    if q_out is None:
        q_out = torch.empty((M, d), dtype=torch.uint8, device=x.device)
    if scale_out is None:
        scale_out = torch.empty((M,), dtype=torch.float32, device=x.device)
    code = lib().sptp_prologue_e4m3(_ptr(x), _ptr(partials), _ptr(gamma), M, d, P, float(eps), _ptr(h_out),
                                    _ptr(y_work), _ptr(q_out), _ptr(scale_out), _stream(stream))
    _check("sptp_prologue_e4m3", code)
    return h_out, q_out, scale_out


def sptp_gateup_swiglu_e4m3(qy, sy, qW1g, sW1g, qW1u, sW1u, P, s_out=None, workspace=None, stream=None):
    M, d = qy.shape
    F = qW1g.shape[0]
    for name, t, shape, dt in (("qy", qy, (M, d), torch.uint8), ("sy", sy, (M,), torch.float32),
                               ("qW1g", qW1g, (F, d), torch.uint8), ("sW1g", sW1g, (F,), torch.float32),
                               ("qW1u", qW1u, (F, d), torch.uint8), ("sW1u", sW1u, (F,), torch.float32)):
        _expect(name, t, shape, dt)
    _expect("s_out", s_out, (P, M, F // P), torch.bfloat16, optional=True)
    _same_device(qy, sy, qW1g, sW1g, qW1u, sW1u, s_out, workspace)
    if s_out is None:
        s_out = torch.empty((P, M, F // P), dtype=torch.bfloat16, device=qy.device)
    if workspace is None:
        workspace = _workspace(SPTP_WS_HEADER_BYTES, qy.device)
    code = lib().sptp_gateup_swiglu_e4m3(_ptr(qy), _ptr(sy), _ptr(qW1g), _ptr(sW1g), _ptr(qW1u), _ptr(sW1u), M, d,
                                         F, P, _ptr(s_out), _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check("sptp_gateup_swiglu_e4m3", code)
    return s_out


def sptp_down_proj_e4m3(qs, ss, qW2, sW2, P, out=None, workspace=None, stream=None):
    _, M, f = qs.shape
    d, F = qW2.shape
    for name, t, shape, dt in (("qs", qs, (P, M, F // P), torch.uint8), ("ss", ss, (P, M), torch.float32),
                               ("qW2", qW2, (d, F), torch.uint8), ("sW2", sW2, (d, P), torch.float32)):
        _expect(name, t, shape, dt)
    _expect("out", out, (P, M, d), torch.bfloat16, optional=True)
    _same_device(qs, ss, qW2, sW2, out, workspace)
    if out is None:
        out = torch.empty((P, M, d), dtype=torch.bfloat16, device=qs.device)
    if workspace is None:
        workspace = _workspace(SPTP_WS_HEADER_BYTES, qs.device)
    code = lib().sptp_down_proj_e4m3(_ptr(qs), _ptr(ss), _ptr(qW2), _ptr(sW2), M, d, F, P, _ptr(out),
                                     _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check("sptp_down_proj_e4m3", code)
    return out
