"""GPU parity of the attention-side boundary: the column-parallel QKV
projection after the partial sum + residual + RMSNorm prologue, and the
row-parallel output projection, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import sequence_tensor_transformer_gb300 as st
from sequence_tensor_transformer_gb300 import synth

from helpers import TOL, dev_tensor, host_f64, rel_err, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    st.load_library()
    torch.cuda.set_device(0)


@pytest.fixture(params=["pair", "single", "fused"])
def gemm_variant(request, monkeypatch):
    """Prologue + CTA-pair or single-CTA QKV GEMM, or the whole boundary as one
    fused persistent launch (SPTP_ATTN_VARIANT=fused; strict mode makes a
    fall-back an error)."""
    if request.param == "fused":
        monkeypatch.setenv("SPTP_ATTN_VARIANT", "fused")
    else:
        monkeypatch.setenv("SPTP_GEMM_VARIANT", request.param)
    return request.param


def run_qkv(cfg, rows=None):
    inp = synth.attn_inputs(cfg)
    T = {k: dev_tensor(inp[k], cfg.dtype) for k in ("x", "partials", "gamma", "Wqkv")}
    dt = st.SPTP_BF16 if cfg.dtype == "bf16" else st.SPTP_FP32
    ws = torch.empty(st.sptp_attn_qkv_workspace_size(cfg.M, cfg.d, cfg.N, cfg.P, cfg.chunks, dt),
                     dtype=torch.uint8, device="cuda:0")
    qkv, h = st.sptp_attn_qkv_forward(T["x"], T["partials"], T["gamma"], T["Wqkv"], cfg.P, cfg.chunks, cfg.eps,
                                      workspace=ws)
    assert st.sptp_read_device_status(ws) == 0
    x, parts = inp["x"], inp["partials"]
    if rows is not None:
        x, parts = x[rows], parts[:, rows]
    ref, href = oracle.attn_qkv_boundary(to_f64(x, cfg.dtype), to_f64(parts, cfg.dtype),
                                         to_f64(inp["gamma"], cfg.dtype), to_f64(inp["Wqkv"], cfg.dtype), cfg.P,
                                         cfg.chunks if rows is None else 1, cfg.eps)
    got = host_f64(qkv if rows is None else qkv[:, rows])
    goth = host_f64(h if rows is None else h[rows])
    for p in range(cfg.P):
        assert rel_err(got[p], ref[p]) <= TOL[cfg.dtype], p
    assert rel_err(goth, href) <= TOL[cfg.dtype]


@pytest.mark.parametrize("M,d,N,P,C", [(300, 136, 3 * 200, 3, 3), (512, 512, 2 * 640, 2, 4), (64, 128, 512, 2, 2),
                                       (2048, 1024, 4 * 1152, 4, 8), (264, 64, 8 * 40, 8, 8)])
def test_attn_qkv_boundary_bf16(M, d, N, P, C, gemm_variant):
    run_qkv(synth.AttnConfig("t", M, d, N, N // 2, P, C, "bf16"))


def test_attn_qkv_boundary_fp32():
    run_qkv(synth.AttnConfig("t32", 96, 128, 2 * 96, 96, 2, 2, "fp32"))


@pytest.mark.parametrize("variant", ["two_launch", "fused"])
def test_attn_qkv_boundary_qwen2_7b_shape_sampled_rows(variant, monkeypatch):
    if variant == "fused":
        monkeypatch.setenv("SPTP_ATTN_VARIANT", "fused")
    cfg = synth.ATTN_QWEN2_7B_SHAPE
    rng = np.random.default_rng(3)
    rows = sorted(set([0, 1, 255, 256, 8191, cfg.M - 1] + list(rng.choice(cfg.M, 12, replace=False))))
    run_qkv(cfg, rows=rows)


def test_attn_out_projection_qwen2_7b_shape_sampled_rows():
    cfg = synth.ATTN_QWEN2_7B_SHAPE
    inp = synth.attn_inputs(cfg)
    a = dev_tensor(inp["attn"], "bf16")
    Wo = dev_tensor(inp["Wo"], "bf16")
    out = st.sptp_down_proj(a, Wo, cfg.P)
    torch.cuda.synchronize()
    rows = [0, 5, 4097, cfg.M - 1]
    ref = oracle.rowparallel_projection(to_f64(inp["attn"][:, rows], "bf16"), to_f64(inp["Wo"], "bf16"), cfg.P)
    got = host_f64(out[:, rows])
    for p in range(cfg.P):
        assert rel_err(got[p], ref[p]) <= TOL["bf16"], p


def test_fused_qkv_boundary_equals_two_launch_path_bitwise(monkeypatch):
    """The fused attention-side boundary and prologue + QKV GEMM compute the
    same y and the same tiles: identical outputs."""
    cfg = synth.AttnConfig("bitwise", 1024, 3584, 4 * 1152, 4 * 896, 4, 8, "bf16")
    inp = synth.attn_inputs(cfg)
    T = {k: dev_tensor(inp[k], "bf16") for k in ("x", "partials", "gamma", "Wqkv")}
    res = {}
    for variant in ("two_launch", "fused"):
        if variant == "fused":
            monkeypatch.setenv("SPTP_ATTN_VARIANT", "fused")
        qkv, h = st.sptp_attn_qkv_forward(T["x"], T["partials"], T["gamma"], T["Wqkv"], cfg.P, cfg.chunks, cfg.eps)
        res[variant] = (qkv.clone(), h.clone())
    torch.cuda.synchronize()
    assert torch.equal(res["fused"][1], res["two_launch"][1])
    assert torch.equal(res["fused"][0], res["two_launch"][0])
