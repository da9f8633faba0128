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
    "sptp_gateup_swiglu_e4m3", "sptp_down_proj_e4m3", "sptp_prologue_e4m3",
]

SPTP_BF16 = 0
SPTP_FP32 = 1
SPTP_WS_HEADER_BYTES = 4096
SPTP_NOALLOC_SCRATCH_BYTES = 64 << 20
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsptp.so")

EXPORTED_SYMBOLS = (
    "sptp_ffn_workspace_size", "sptp_ffn_forward", "dtp_ffn_stack_workspace_size",
    "dtp_ffn_stack_forward", "sptp_prologue", "sptp_gateup_swiglu", "sptp_down_proj",
    "sptp_read_device_status", "sptp_wait_selftest", "sptp_status_string", "sptp_ffn_forward_noalloc",
    "sptp_permute_ffn_neurons", "sptp_attn_qkv_workspace_size", "sptp_attn_qkv_forward",
    "sptp_quantize_rows_e4m3", "sptp_ffn_fp8_workspace_size", "sptp_ffn_forward_fp8", "sptp_gateup_swiglu_e4m3",
    "sptp_down_proj_e4m3", "sptp_prologue_e4m3",
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
}


class SptpError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({sptp_status_string(code)})")
        self.code = code


def load_library(path: str = LIB_PATH):
    """Loads libsptp.so (built by sequence_tensor_transformer_gb300.build)."""
    global _lib
    if _lib is None:
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


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


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


def sptp_ffn_forward(x, partials, gamma, W1g, W1u, W2, P, chunks, eps, out=None, resid_out=None,
                     workspace=None, stream=None, write_resid=True):
    """SP-TP FFN boundary.  Returns (out [P,M,d], resid_out [M,d] or None)."""
    M, d = x.shape
    F = W1g.shape[0]
    dt = _dtype_code(x)
    if out is None:
        out = torch.empty((P, M, d), dtype=x.dtype, device=x.device)
    if resid_out is None and write_resid:
        resid_out = torch.empty_like(x)
    if workspace is None:
        workspace = _workspace(sptp_ffn_workspace_size(M, d, F, P, chunks, dt), x.device)
    code = lib().sptp_ffn_forward(
        _ptr(x), _ptr(partials), _ptr(gamma), _ptr(W1g), _ptr(W1u), _ptr(W2), M, d, F, P, chunks,
        float(eps), dt, _ptr(out), _ptr(resid_out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("sptp_ffn_forward", code)
    return out, resid_out


def dtp_ffn_stack_forward(x_shards, gamma, W1g, W1u, W2, P, L, delta, flush, eps, workspace=None,
                          stream=None):
    """Delayed-TP stack; updates x_shards [P,M,d] in place and returns it."""
    _, M, d = x_shards.shape
    F = W1g.shape[1]
    dt = _dtype_code(x_shards)
    if workspace is None:
        workspace = _workspace(dtp_ffn_stack_workspace_size(M, d, F, P, L, delta, dt), x_shards.device)
    code = lib().dtp_ffn_stack_forward(
        _ptr(x_shards), _ptr(gamma), _ptr(W1g), _ptr(W1u), _ptr(W2), M, d, F, P, L, delta, int(flush),
        float(eps), dt, _ptr(workspace), workspace.numel(), _stream(stream))
    _check("dtp_ffn_stack_forward", code)
    return x_shards


def sptp_prologue(x, partials, gamma, eps, h_out=None, y_out=None, stream=None, write_h=True):
    M, d = x.shape
    P = partials.shape[0]
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
    if s_out is None:
        s_out = torch.empty((P, M, F // P), dtype=y.dtype, device=y.device)
    if workspace is None:
        workspace = _workspace(SPTP_WS_HEADER_BYTES, y.device)
    code = lib().sptp_gateup_swiglu(_ptr(y), _ptr(W1g), _ptr(W1u), M, d, F, P, _dtype_code(y), _ptr(s_out),
                                    _ptr(workspace), workspace.numel(), _stream(stream))
    _check("sptp_gateup_swiglu", code)
    return s_out


def sptp_down_proj(s, W2, P, out=None, workspace=None, stream=None):
    _, M, f = s.shape
    d, F = W2.shape
    if out is None:
        out = torch.empty((P, M, d), dtype=s.dtype, device=s.device)
    if workspace is None:
        workspace = _workspace(SPTP_WS_HEADER_BYTES, s.device)
    code = lib().sptp_down_proj(_ptr(s), _ptr(W2), M, d, F, P, _dtype_code(s), _ptr(out), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    _check("sptp_down_proj", code)
    return out


def sptp_ffn_forward_noalloc(x, partials, gamma, W1g, W1u, W2, P, chunks, eps, out, resid_out=None,
                             stream=None):
    """SP-TP FFN boundary on the library's static scratch (no workspace and no
    device allocation inside the call; the caller passes out/resid_out)."""
    M, d = x.shape
    F = W1g.shape[0]
    code = lib().sptp_ffn_forward_noalloc(
        _ptr(x), _ptr(partials), _ptr(gamma), _ptr(W1g), _ptr(W1u), _ptr(W2), M, d, F, P, chunks, float(eps),
        _dtype_code(x), _ptr(out), _ptr(resid_out), _stream(stream))
    _check("sptp_ffn_forward_noalloc", code)
    return out, resid_out


def sptp_attn_qkv_workspace_size(M, d, N, P, chunks, dtype=SPTP_BF16) -> int:
    return int(lib().sptp_attn_qkv_workspace_size(M, d, N, P, chunks, dtype))


def sptp_attn_qkv_forward(x, partials, gamma, Wqkv, P, chunks, eps, qkv_out=None, resid_out=None,
                          workspace=None, stream=None, write_resid=True):
    """Boundary in front of attention: returns (qkv [P,M,N/P], resid_out)."""
    M, d = x.shape
    N = Wqkv.shape[0]
    dt = _dtype_code(x)
    if qkv_out is None:
        qkv_out = torch.empty((P, M, N // P), dtype=x.dtype, device=x.device)
    if resid_out is None and write_resid:
        resid_out = torch.empty_like(x)
    if workspace is None:
        workspace = _workspace(sptp_attn_qkv_workspace_size(M, d, N, P, chunks, dt), x.device)
    code = lib().sptp_attn_qkv_forward(_ptr(x), _ptr(partials), _ptr(gamma), _ptr(Wqkv), M, d, N, P, chunks,
                                       float(eps), dt, _ptr(qkv_out), _ptr(resid_out), _ptr(workspace),
                                       workspace.numel(), _stream(stream))
    _check("sptp_attn_qkv_forward", code)
    return qkv_out, resid_out


def sptp_permute_ffn_neurons(W1g, W1u, W2, perm, workspace=None, stream=None):
    """Renumbers every module's neurons (W1g/W1u [L,F,d] rows, W2 [L,d,F]
    columns) by perm [L,F] (int32, device); returns the permuted copies."""
    L, F, d = W1g.shape
    outs = [torch.empty_like(W1g), torch.empty_like(W1u), torch.empty_like(W2)]
    if workspace is None:
        workspace = _workspace(SPTP_WS_HEADER_BYTES, W1g.device)
    if perm.dtype != torch.int32:
        raise TypeError("perm must be int32")
    code = lib().sptp_permute_ffn_neurons(_ptr(W1g), _ptr(W1u), _ptr(W2), _ptr(perm), L, d, F, _dtype_code(W1g),
                                          _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _ptr(workspace),
                                          workspace.numel(), _stream(stream))
    _check("sptp_permute_ffn_neurons", code)
    return tuple(outs)


def sptp_read_device_status(workspace, stream=None) -> int:
    return int(lib().sptp_read_device_status(_ptr(workspace), _stream(stream)))


def sptp_wait_selftest(workspace, limit_ns: int, preset_flag: bool, stream=None) -> int:
    return int(lib().sptp_wait_selftest(_ptr(workspace), workspace.numel(), int(limit_ns), int(preset_flag),
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
    if out is None:
        out = torch.empty((P, M, d), dtype=x.dtype, device=x.device)
    if resid_out is None and write_resid:
        resid_out = torch.empty_like(x)
    if workspace is None:
        workspace = _workspace(sptp_ffn_fp8_workspace_size(M, d, F, P, chunks), x.device)
    code = lib().sptp_ffn_forward_fp8(
        _ptr(x), _ptr(partials), _ptr(gamma), _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su), _ptr(q2), _ptr(s2), M, d, F,
        P, chunks, float(eps), _ptr(out), _ptr(resid_out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("sptp_ffn_forward_fp8", code)
    return out, resid_out


def sptp_prologue_e4m3(x, partials, gamma, eps, h_out=None, y_work=None, q_out=None, scale_out=None, stream=None,
                       write_h=True):
    """Partial sum + residual + RMSNorm with y quantised to E4M3 in the same
    launch.  Returns (h or None, q uint8 [M,d], scale float32 [M])."""
    M, d = x.shape
    P = partials.shape[0]
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
    if s_out is None:
        s_out = torch.empty((P, M, F // P), dtype=torch.bfloat16, device=qy.device)
    if workspace is None:
        workspace = _workspace(SPTP_WS_HEADER_BYTES, qy.device)
    code = lib().sptp_gateup_swiglu_e4m3(_ptr(qy), _ptr(sy), _ptr(qW1g), _ptr(sW1g), _ptr(qW1u), _ptr(sW1u), M, d,
                                         F, P, _ptr(s_out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("sptp_gateup_swiglu_e4m3", code)
    return s_out


def sptp_down_proj_e4m3(qs, ss, qW2, sW2, P, out=None, workspace=None, stream=None):
    _, M, f = qs.shape
    d, F = qW2.shape
    if out is None:
        out = torch.empty((P, M, d), dtype=torch.bfloat16, device=qs.device)
    if workspace is None:
        workspace = _workspace(SPTP_WS_HEADER_BYTES, qs.device)
    code = lib().sptp_down_proj_e4m3(_ptr(qs), _ptr(ss), _ptr(qW2), _ptr(sW2), M, d, F, P, _ptr(out),
                                     _ptr(workspace), workspace.numel(), _stream(stream))
    _check("sptp_down_proj_e4m3", code)
    return out
