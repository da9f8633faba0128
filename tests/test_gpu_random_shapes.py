"""GPU parity on seeded random shapes: every entry point against the oracle on
irregular sizes (M not a tile multiple, d and F/P off the 64/128/256 tile
grid, P from 1 to 8, several chunk counts), to exercise the tile edges, the
zero-filled TMA boxes and the ragged tails of every kernel."""
import numpy as np
import pytest
import torch

import oracle
import sequence_tensor_transformer_gb300 as st
from oracle import fp8_oracle as f8
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


def shapes(seed, n, mult=8):
    """n boundary shapes (M, d, F, P, C) with d % mult == 0 and (F/P) % mult == 0."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        P = int(rng.integers(1, 9))
        C = P * int(rng.integers(1, 4))
        M = C * int(rng.integers(1, 700 // C + 1))
        d = mult * int(rng.integers(2, 1536 // mult + 1))
        F = P * mult * int(rng.integers(1, 640 // mult + 1))
        out.append((M, d, F, P, C))
    return out


def check_boundary(cfg, out, h, ref, href, family):
    got = host_f64(out)
    errs = {p: rel_err(got[p], ref[p]) for p in range(cfg.P)}
    errs["h"] = rel_err(host_f64(h), href)
    check_errors(errs, family)


@pytest.mark.parametrize("variant", ["pair", "chain", "fused"])
@pytest.mark.parametrize("shape", shapes(101, 8))
def test_random_boundary_bf16(shape, variant):
    M, d, F, P, C = shape
    cfg = synth.BoundaryConfig(f"r_{M}_{d}_{F}_{P}_{C}", M, d, F, P, C, "bf16", True, seed=M + d)
    inp = synth.boundary_inputs(cfg)
    T = {k: dev_tensor(v, "bf16") for k, v in inp.items()}
    ws = nan_workspace(st.sptp_ffn_workspace_size(M, d, F, P, C, st.SPTP_BF16))
    out, h = nan_tensor((P, M, d)), nan_tensor((M, d))
    st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], P, C, cfg.eps, out=out,
                        resid_out=h, workspace=ws, variant=variant)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(out, h)
    f64 = {k: to_f64(v, "bf16") for k, v in inp.items()}
    ref, href = oracle.sptp_ffn_forward(f64["x"], f64["partials"], f64["gamma"], f64["W1g"], f64["W1u"], f64["W2"],
                                        P, C, cfg.eps)
    check_boundary(cfg, out, h, ref, href, "bf16")


def fp32_shapes(seed, n):
    """Smaller boundary shapes for the fp32 CUDA-core path, with K (d and
    F/P) off its 32-deep slice and M off its 64-row tile."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        P = int(rng.integers(1, 5))
        C = P * int(rng.integers(1, 3))
        M = C * int(rng.integers(1, 300 // C + 1))
        d = 8 * int(rng.integers(1, 65))
        F = P * 8 * int(rng.integers(1, 49))
        out.append((M, d, F, P, C))
    return out


@pytest.mark.parametrize("shape", fp32_shapes(303, 6))
def test_random_boundary_fp32(shape):
    M, d, F, P, C = shape
    cfg = synth.BoundaryConfig(f"r32_{M}_{d}_{F}_{P}_{C}", M, d, F, P, C, "fp32", False, seed=M + d)
    inp = synth.boundary_inputs(cfg)
    T = {k: dev_tensor(v, "fp32") for k, v in inp.items()}
    ws = nan_workspace(st.sptp_ffn_workspace_size(M, d, F, P, C, st.SPTP_FP32))
    out, h = nan_tensor((P, M, d), torch.float32), nan_tensor((M, d), torch.float32)
    st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], P, C, cfg.eps, out=out,
                        resid_out=h, workspace=ws)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(out, h)
    f64 = {k: to_f64(v, "fp32") for k, v in inp.items()}
    ref, href = oracle.sptp_ffn_forward(f64["x"], f64["partials"], f64["gamma"], f64["W1g"], f64["W1u"], f64["W2"],
                                        P, C, cfg.eps)
    got = host_f64(out)
    errs = {p: rel_err(got[p], ref[p]) for p in range(P)}
    errs["h"] = rel_err(host_f64(h), href)
    check_errors(errs, "fp32", "fp32")


@pytest.mark.parametrize("shape", shapes(202, 8, mult=16))
def test_random_boundary_fp8(shape):
    M, d, F, P, C = shape
    cfg = synth.BoundaryConfig(f"r8_{M}_{d}_{F}_{P}_{C}", M, d, F, P, C, "bf16", True, seed=M + 3 * d)
    inp = synth.boundary_inputs(cfg)
    T = {k: dev_tensor(v, "bf16") for k, v in inp.items()}
    qw = st.quantize_ffn_weights_e4m3(T["W1g"], T["W1u"], T["W2"], P)
    ws = nan_workspace(st.sptp_ffn_fp8_workspace_size(M, d, F, P, C))
    out, h = nan_tensor((P, M, d)), nan_tensor((M, d))
    st.sptp_ffn_forward_fp8(T["x"], T["partials"], T["gamma"], qw, P, C, cfg.eps, out=out, resid_out=h, workspace=ws)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(out, h)
    f64 = {k: to_f64(v, "bf16") for k, v in inp.items()}
    ref, href = f8.sptp_ffn_forward_fp8(f64["x"], f64["partials"], f64["gamma"], f64["W1g"], f64["W1u"],
                                        f64["W2"], P, C, cfg.eps)
    check_boundary(cfg, out, h, ref, href, "e4m3")


@pytest.mark.parametrize("variant", ["fused", "layers"])
@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_random_dtp_stack(seed, variant):
    rng = np.random.default_rng(300 + seed)
    P = int(rng.integers(1, 5))
    L = int(rng.integers(1, 5))
    delta = int(rng.integers(0, 4))
    M = int(rng.integers(1, 600))
    d = 8 * int(rng.integers(2, 129))
    F = P * 8 * int(rng.integers(1, 49))
    flush = int(rng.integers(0, 2))
    cfg = synth.DTPConfig(f"rd_{seed}", M, d, F, P, L, delta, "bf16")
    inp = synth.dtp_inputs(cfg, independent_streams=bool(seed % 2))
    T = {k: dev_tensor(v, "bf16") for k, v in inp.items()}
    ws = nan_workspace(st.dtp_ffn_stack_workspace_size(M, d, F, P, L, delta, st.SPTP_BF16))
    st.dtp_ffn_stack_forward(T["x_shards"], T["gamma"], T["W1g"], T["W1u"], T["W2"], P, L, delta, flush, cfg.eps,
                             workspace=ws, variant=variant)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(T["x_shards"])
    f64 = {k: to_f64(v, "bf16") for k, v in inp.items()}
    ref = oracle.dtp_ffn_stack_forward(f64["x_shards"], f64["gamma"], f64["W1g"], f64["W1u"], f64["W2"], P, L, delta,
                                       bool(flush), cfg.eps)
    got = host_f64(T["x_shards"])
    check_errors({p: rel_err(got[p], ref[p]) for p in range(P)}, "bf16")


@pytest.mark.parametrize("variant", ["pair", "fused"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_attention_boundary(seed, variant):
    rng = np.random.default_rng(400 + seed)
    P = int(rng.integers(1, 9))
    C = P * int(rng.integers(1, 3))
    M = C * int(rng.integers(1, 600 // C + 1))
    d = 8 * int(rng.integers(2, 193))
    N = P * 8 * int(rng.integers(1, 97))
    cfg = synth.AttnConfig(f"ra_{seed}", M, d, N, N, P, C, "bf16")
    inp = synth.attn_inputs(cfg)
    T = {k: dev_tensor(inp[k], "bf16") for k in ("x", "partials", "gamma", "Wqkv")}
    ws = nan_workspace(st.sptp_attn_qkv_workspace_size(M, d, N, P, C, st.SPTP_BF16))
    qkv, h = nan_tensor((P, M, N // P)), nan_tensor((M, d))
    st.sptp_attn_qkv_forward(T["x"], T["partials"], T["gamma"], T["Wqkv"], P, C, cfg.eps, qkv_out=qkv, resid_out=h,
                             workspace=ws, variant=variant)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(qkv, h)
    ref, href = oracle.attn_qkv_boundary(to_f64(inp["x"], "bf16"), to_f64(inp["partials"], "bf16"),
                                         to_f64(inp["gamma"], "bf16"), to_f64(inp["Wqkv"], "bf16"), P, C, cfg.eps)
    got = host_f64(qkv)
    errs = {p: rel_err(got[p], ref[p]) for p in range(P)}
    errs["h"] = rel_err(host_f64(h), href)
    check_errors(errs, "bf16")


def perm_shapes(seed, n):
    """n (L, d, F) shapes with d and F multiples of 8: rows that fit the
    pipelined launch's stage and wider ones that take the two-launch path."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        L = int(rng.integers(1, 4))
        d = 8 * int(rng.integers(1, 257))
        F = 8 * int(rng.integers(1, 1537))
        if L * d * F <= (1 << 24):  # at most 16 M elements per matrix
            out.append((L, d, F))
    return out


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("shape", perm_shapes(211, 8))
def test_random_permutation(shape, dtype):
    """sptp_permute_ffn_neurons moves bytes only: its outputs equal plain
    indexing exactly, whichever launch structure the shape takes."""
    L, d, F = shape
    rng = np.random.default_rng(L * 100003 + d * 31 + F)
    W1g = synth._cast(rng.standard_normal((L, F, d)), dtype)
    W1u = synth._cast(rng.standard_normal((L, F, d)), dtype)
    W2 = synth._cast(rng.standard_normal((L, d, F)), dtype)
    perm = np.stack([rng.permutation(F) for _ in range(L)]).astype(np.int32)
    hdr = nan_workspace(st.SPTP_WS_HEADER_BYTES)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    outs = [torch.full((L, F, d), float("nan"), dtype=tdt, device="cuda:0") for _ in range(2)]
    outs.append(torch.full((L, d, F), float("nan"), dtype=tdt, device="cuda:0"))
    st.lib().sptp_permute_ffn_neurons(
        *[t.data_ptr() for t in (dev_tensor(W1g, dtype), dev_tensor(W1u, dtype), dev_tensor(W2, dtype))],
        torch.from_numpy(perm).cuda().data_ptr(), L, d, F, st.SPTP_BF16 if dtype == "bf16" else st.SPTP_FP32,
        *[t.data_ptr() for t in outs], hdr.data_ptr(), hdr.numel(), torch.cuda.current_stream().cuda_stream)
    assert st.sptp_read_device_status(hdr) == 0
    view = (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)) if dtype == "bf16" else \
        (lambda t: t.cpu().numpy())
    for l in range(L):
        assert np.array_equal(view(outs[0])[l], W1g[l][perm[l]])
        assert np.array_equal(view(outs[1])[l], W1u[l][perm[l]])
        assert np.array_equal(view(outs[2])[l], W2[l][:, perm[l]])
