"""GPU parity of the attention-side boundary: the column-parallel QKV
projection after the partial sum + residual + RMSNorm prologue, and the
row-parallel output projection, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import sequence_tensor_transformer_gb300 as st
from sequence_tensor_transformer_gb300 import synth

from helpers import (TOL, assert_no_nan, check_errors, dev_tensor, host_f64, nan_tensor, nan_workspace, rel_err,
                     to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    st.load_library()
    torch.cuda.set_device(0)


def qkv_call(T, cfg, variant="auto"):
    dt = st.SPTP_BF16 if cfg.dtype == "bf16" else st.SPTP_FP32
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    ws = nan_workspace(st.sptp_attn_qkv_workspace_size(cfg.M, cfg.d, cfg.N, cfg.P, cfg.chunks, dt))
    qkv, h = nan_tensor((cfg.P, cfg.M, cfg.N // cfg.P), tdt), nan_tensor((cfg.M, cfg.d), tdt)
    st.sptp_attn_qkv_forward(T["x"], T["partials"], T["gamma"], T["Wqkv"], cfg.P, cfg.chunks, cfg.eps, qkv_out=qkv,
                             resid_out=h, workspace=ws, variant=variant)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(qkv, h)
    return qkv, h


def run_qkv(cfg, rows=None, variant="auto"):
    inp = synth.attn_inputs(cfg)
    T = {k: dev_tensor(inp[k], cfg.dtype) for k in ("x", "partials", "gamma", "Wqkv")}
    qkv, h = qkv_call(T, cfg, variant)
    x, parts = inp["x"], inp["partials"]
    if rows is not None:
        x, parts = x[rows], parts[:, rows]
    ref, href = oracle.attn_qkv_boundary(to_f64(x, cfg.dtype), to_f64(parts, cfg.dtype),
                                         to_f64(inp["gamma"], cfg.dtype), to_f64(inp["Wqkv"], cfg.dtype), cfg.P,
                                         cfg.chunks if rows is None else 1, cfg.eps)
    got = host_f64(qkv if rows is None else qkv[:, rows])
    goth = host_f64(h if rows is None else h[rows])
    errs = {p: rel_err(got[p], ref[p]) for p in range(cfg.P)}
    errs["h"] = rel_err(goth, href)
    check_errors(errs, cfg.dtype, cfg.dtype)


@pytest.mark.parametrize("variant", ["pair", "fused"])
@pytest.mark.parametrize("M,d,N,P,C", [(300, 136, 3 * 200, 3, 3), (512, 512, 2 * 640, 2, 4), (64, 128, 512, 2, 2),
                                       (2048, 1024, 4 * 1152, 4, 8), (264, 64, 8 * 40, 8, 8)])
def test_attn_qkv_boundary_bf16(M, d, N, P, C, variant):
    run_qkv(synth.AttnConfig("t", M, d, N, N // 2, P, C, "bf16"), variant=variant)


def test_attn_qkv_boundary_fp32():
    cfg = synth.AttnConfig("t32", 96, 128, 2 * 96, 96, 2, 2, "fp32")
    run_qkv(cfg)
    T = {k: dev_tensor(v, "fp32") for k, v in synth.attn_inputs(cfg).items()}
    for variant in ("fused", "chain", "layers"):
        with pytest.raises(st.SptpError) as e:
            qkv_call(T, cfg, variant)
        assert e.value.code == st.STATUS["unimplemented"]


@pytest.mark.parametrize("variant", ["pair", "fused"])
def test_attn_qkv_boundary_qwen2_7b_shape_sampled_rows(variant):
    cfg = synth.ATTN_QWEN2_7B_SHAPE
    rng = np.random.default_rng(3)
    rows = sorted(set([0, 1, 255, 256, 8191, cfg.M - 1] + list(rng.choice(cfg.M, 12, replace=False))))
    run_qkv(cfg, rows=rows, variant=variant)


def test_attn_out_projection_qwen2_7b_shape_sampled_rows():
    cfg = synth.ATTN_QWEN2_7B_SHAPE
    inp = synth.attn_inputs(cfg)
    a = dev_tensor(inp["attn"], "bf16")
    Wo = dev_tensor(inp["Wo"], "bf16")
    out, ws = nan_tensor((cfg.P, cfg.M, cfg.d)), nan_workspace(st.SPTP_WS_HEADER_BYTES)
    st.sptp_down_proj(a, Wo, cfg.P, out=out, workspace=ws)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(out)
    rows = [0, 5, 4097, cfg.M - 1]
    ref = oracle.rowparallel_projection(to_f64(inp["attn"][:, rows], "bf16"), to_f64(inp["Wo"], "bf16"), cfg.P)
    got = host_f64(out[:, rows])
    check_errors({p: rel_err(got[p], ref[p]) for p in range(cfg.P)}, "bf16")


def test_fused_qkv_boundary_equals_two_launch_path_bitwise():
    """The fused attention-side boundary and prologue + QKV GEMM compute the
    same y and the same tiles: identical outputs."""
    cfg = synth.AttnConfig("bitwise", 1024, 3584, 4 * 1152, 4 * 896, 4, 8, "bf16")
    inp = synth.attn_inputs(cfg)
    T = {k: dev_tensor(inp[k], "bf16") for k in ("x", "partials", "gamma", "Wqkv")}
    res = {v: qkv_call(T, cfg, v) for v in ("pair", "fused")}
    assert torch.equal(res["fused"][1], res["pair"][1])
    assert torch.equal(res["fused"][0], res["pair"][0])
