"""The bounds-checked build on the GPU.

compute-sanitizer is not available for these kernels, so the library has a
debug build of its own (build(checked=True) -> libsptp_check.so, compiled
with -DSPTP_BOUNDS_CHECK): every kernel checks the indices and addresses it
computes -- decoded tiles, readiness counters, pending-ring slots and
source shards, the cluster shape, TMA box origins, global loads and stores
-- against the buffers they address, records a failure as SPTP_ERR_BOUNDS
in the workspace status words and skips the access.  These tests run small
cases of every entry point and launch variant through that build, with
NaN-poisoned outputs and workspaces, and require status 0, every output
written, and parity with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import sequence_tensor_transformer_gb300 as st
from oracle import fp8_oracle as f8
from sequence_tensor_transformer_gb300 import synth

from helpers import TOL, assert_no_nan, dev_tensor, host_f64, nan_tensor, nan_workspace, rel_err, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def checked_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sequence_tensor_transformer_gb300 import build
    path = build.build(checked=True)
    normal = st.load_library()
    torch.cuda.set_device(0)
    st.load_library(path, replace=True)
    yield
    st.set_library(normal)


def status_ok(ws):
    code = st.sptp_read_device_status(ws)
    words = ws[:20].view(torch.int32).cpu().tolist()
    assert code == 0, f"status {code} ({st.sptp_status_string(code)}), where {words[1]}, block {words[2]}, " \
                      f"value {words[3]}"


def boundary(M, d, F, P, C, variant, dtype="bf16", seed=0):
    cfg = synth.BoundaryConfig("chk", M, d, F, P, C, dtype, dtype == "bf16", seed=seed)
    inp = synth.boundary_inputs(cfg)
    T = {k: dev_tensor(v, dtype) for k, v in inp.items()}
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dt = st.SPTP_BF16 if dtype == "bf16" else st.SPTP_FP32
    ws = nan_workspace(st.sptp_ffn_workspace_size(M, d, F, P, C, dt))
    out, h = nan_tensor((P, M, d), tdt), nan_tensor((M, d), tdt)
    st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], P, C, cfg.eps, out=out,
                        resid_out=h, workspace=ws, variant=variant)
    status_ok(ws)
    assert_no_nan(out, h)
    f64 = {k: to_f64(v, dtype) for k, v in inp.items()}
    ref, href = oracle.sptp_ffn_forward(f64["x"], f64["partials"], f64["gamma"], f64["W1g"], f64["W1u"], f64["W2"],
                                        P, C, cfg.eps)
    got = host_f64(out)
    for p in range(P):
        assert rel_err(got[p], ref[p]) <= TOL[dtype], p
    assert rel_err(host_f64(h), href) <= TOL[dtype]


@pytest.mark.parametrize("variant", ["pair", "chain", "fused"])
@pytest.mark.parametrize("M,d,F,P,C", [(320, 256, 768, 2, 2), (600, 256, 512, 2, 6), (130, 64, 64, 1, 1),
                                       (1000, 512, 4 * 392, 4, 8), (384, 136, 3 * 200, 3, 3),
                                       (40, 16384, 2 * 64, 2, 2)])
def test_boundary_checked(M, d, F, P, C, variant):
    # d = 16384: rows too wide for the prologue's shared-memory ring and for
    # the fused launch's one-pass block rows (warp-per-row prologue)
    boundary(M, d, F, P, C, variant)


def test_boundary_fp32_checked():
    boundary(96, 136, 3 * 40, 3, 3, "pair", dtype="fp32")


def dtp(P, L, delta, flush, variant, M=200, d=136, f=48, indep=False):
    cfg = synth.DTPConfig("chk", M, d, P * f, P, L, delta, "bf16")
    inp = synth.dtp_inputs(cfg, independent_streams=indep)
    T = {k: dev_tensor(v, "bf16") for k, v in inp.items()}
    ws = nan_workspace(st.dtp_ffn_stack_workspace_size(M, d, cfg.F, P, L, delta, st.SPTP_BF16))
    st.dtp_ffn_stack_forward(T["x_shards"], T["gamma"], T["W1g"], T["W1u"], T["W2"], P, L, delta, flush, cfg.eps,
                             workspace=ws, variant=variant)
    status_ok(ws)
    assert_no_nan(T["x_shards"])
    f64 = {k: to_f64(v, "bf16") for k, v in inp.items()}
    ref = oracle.dtp_ffn_stack_forward(f64["x_shards"], f64["gamma"], f64["W1g"], f64["W1u"], f64["W2"], P, L, delta,
                                       bool(flush), cfg.eps)
    got = host_f64(T["x_shards"])
    for p in range(P):
        assert rel_err(got[p], ref[p]) <= TOL["bf16"], p


@pytest.mark.parametrize("variant", ["fused", "layers"])
@pytest.mark.parametrize("P,L,delta,flush", [(2, 3, 1, 1), (3, 4, 2, 0), (4, 2, 5, 1), (1, 3, 0, 1)])
def test_dtp_stack_checked(P, L, delta, flush, variant):
    dtp(P, L, delta, flush, variant)


@pytest.mark.parametrize("variant", ["fused", "layers"])
def test_dtp_stack_most_sources_checked(variant):
    # P = 8, S = 9: the final flushing update sums 1 + 7 * 9 = 64 sources
    dtp(8, 9, 8, 1, variant, M=40, d=64, f=16, indep=True)


@pytest.mark.parametrize("variant", ["pair", "fused"])
@pytest.mark.parametrize("M,d,N,P,C", [(300, 136, 3 * 200, 3, 3), (264, 64, 8 * 40, 8, 8), (512, 512, 2 * 640, 2, 4)])
def test_attention_boundary_checked(M, d, N, P, C, variant):
    cfg = synth.AttnConfig("chk", M, d, N, N, P, C, "bf16")
    inp = synth.attn_inputs(cfg)
    T = {k: dev_tensor(inp[k], "bf16") for k in ("x", "partials", "gamma", "Wqkv")}
    ws = nan_workspace(st.sptp_attn_qkv_workspace_size(M, d, N, P, C, st.SPTP_BF16))
    qkv, h = nan_tensor((P, M, N // P)), nan_tensor((M, d))
    st.sptp_attn_qkv_forward(T["x"], T["partials"], T["gamma"], T["Wqkv"], P, C, cfg.eps, qkv_out=qkv, resid_out=h,
                             workspace=ws, variant=variant)
    status_ok(ws)
    assert_no_nan(qkv, h)
    ref, href = oracle.attn_qkv_boundary(to_f64(inp["x"], "bf16"), to_f64(inp["partials"], "bf16"),
                                         to_f64(inp["gamma"], "bf16"), to_f64(inp["Wqkv"], "bf16"), P, C, cfg.eps)
    got = host_f64(qkv)
    for p in range(P):
        assert rel_err(got[p], ref[p]) <= TOL["bf16"], p
    # the row-parallel out-projection after attention (a plain store GEMM)
    a = dev_tensor(inp["attn"], "bf16")
    Wo = dev_tensor(inp["Wo"], "bf16")
    out, hdr = nan_tensor((P, M, d)), nan_workspace(st.SPTP_WS_HEADER_BYTES)
    st.sptp_down_proj(a, Wo, P, out=out, workspace=hdr)
    status_ok(hdr)
    assert_no_nan(out)
    ref = oracle.rowparallel_projection(to_f64(inp["attn"], "bf16"), to_f64(inp["Wo"], "bf16"), P)
    got = host_f64(out)
    for p in range(P):
        assert rel_err(got[p], ref[p]) <= TOL["bf16"], p


@pytest.mark.parametrize("M,d,F,P,C", [(320, 256, 768, 2, 2), (384, 144, 3 * 208, 3, 3), (64, 8192, 8 * 128, 8, 8)])
def test_fp8_boundary_checked(M, d, F, P, C):
    # d = 8192 with 8 partials: y is stored and quantised by a second launch
    cfg = synth.BoundaryConfig("chk8", M, d, F, P, C, "bf16", True)
    inp = synth.boundary_inputs(cfg)
    T = {k: dev_tensor(v, "bf16") for k, v in inp.items()}
    qw = st.quantize_ffn_weights_e4m3(T["W1g"], T["W1u"], T["W2"], P)
    ws = nan_workspace(st.sptp_ffn_fp8_workspace_size(M, d, F, P, C))
    out, h = nan_tensor((P, M, d)), nan_tensor((M, d))
    st.sptp_ffn_forward_fp8(T["x"], T["partials"], T["gamma"], qw, P, C, cfg.eps, out=out, resid_out=h, workspace=ws)
    status_ok(ws)
    assert_no_nan(out, h)
    f64 = {k: to_f64(v, "bf16") for k, v in inp.items()}
    ref, href = f8.sptp_ffn_forward_fp8(f64["x"], f64["partials"], f64["gamma"], f64["W1g"], f64["W1u"], f64["W2"], P,
                                        C, cfg.eps)
    got = host_f64(out)
    for p in range(P):
        assert rel_err(got[p], ref[p]) <= TOL["bf16"], p


@pytest.mark.parametrize("L,d,F", [(2, 136, 200), (3, 1024, 3072), (1, 8, 24576)])
def test_permutation_checked(L, d, F):
    """The pipelined launch (the first two) and the two-launch fallback."""
    rng = np.random.default_rng(3)
    W1g, W1u = synth._cast(rng.standard_normal((L, F, d)), "bf16"), synth._cast(rng.standard_normal((L, F, d)), "bf16")
    W2 = synth._cast(rng.standard_normal((L, d, F)), "bf16")
    perm = np.stack([rng.permutation(F) for _ in range(L)]).astype(np.int32)
    hdr = nan_workspace(st.SPTP_WS_HEADER_BYTES)
    outs = st.sptp_permute_ffn_neurons(dev_tensor(W1g, "bf16"), dev_tensor(W1u, "bf16"), dev_tensor(W2, "bf16"),
                                       torch.from_numpy(perm).cuda(), workspace=hdr)
    status_ok(hdr)
    view = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    for l in range(L):
        assert np.array_equal(view(outs[0])[l], W1g[l][perm[l]])
        assert np.array_equal(view(outs[2])[l], W2[l][:, perm[l]])
