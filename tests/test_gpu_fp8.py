"""GPU parity of the fp8 (E4M3) boundary variant against the float64 fp8
oracle on the same seeded bf16 inputs.

Bars.  The quantiser is byte work: codes and scales must be bit-exact.  The
GEMMs then see identical codes on both sides, so what remains is the fp32
accumulation order and one bf16 rounding of each output (2^-8 relative at
most, per element), plus rare one-step code flips in the quantisation of s
where the GPU's fp32 SwiGLU and the oracle's float64 one round to different
bf16 neighbours: each moves one term of a K-long sum by one E4M3 step.  The
rel. max error bar of the bf16 path, 2e-2, covers that with a wide margin.
"""
import numpy as np
import pytest
import torch

import oracle
import sequence_tensor_transformer_gb300 as st
from oracle import fp8_oracle as f8
from sequence_tensor_transformer_gb300 import synth

from helpers import TOL, assert_no_nan, check_errors, dev_tensor, host_f64, nan_tensor, nan_workspace, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    st.load_library()
    torch.cuda.set_device(0)


def bf16_array(rng, shape, scale=1.0):
    return synth._cast(rng.standard_normal(shape) * scale, "bf16")


def oracle_codes(a64):
    q, e = f8.quantize_rows_e4m3(a64)
    return f8.e4m3_encode(q), np.ldexp(1.0, e)


# ---------------------------------------------------------------- quantiser

@pytest.mark.parametrize("R,K", [(1, 16), (7, 48), (300, 4096), (64, 7168), (33, 8192), (5, 9000 - 9000 % 16),
                                 (2, 20000)])
def test_quantize_rows_bit_exact(R, K):
    rng = np.random.default_rng(R * 31 + K)
    # rows spanning many binades, an all-zero row, a subnormal-heavy row
    a = bf16_array(rng, (R, K)) if R else np.zeros((0, K), np.uint16)
    mags = 10.0 ** rng.uniform(-20, 20, R)
    a64 = synth.to_f64(a, "bf16") * mags[:, None]
    a = synth._cast(a64, "bf16")
    if R > 2:
        a[1] = 0
        row = synth.to_f64(a[2], "bf16")
        row[: K // 2] *= 2.0 ** -30  # far below the row maximum: subnormal codes
        a[2] = synth._cast(row, "bf16")
    a64 = synth.to_f64(a, "bf16")
    q, sc = st.sptp_quantize_rows_e4m3(dev_tensor(a, "bf16"))
    torch.cuda.synchronize()
    codes, scale = oracle_codes(a64)
    got = q.cpu().numpy()
    assert np.array_equal(got, codes), np.argwhere(got != codes)[:5]
    assert np.array_equal(sc.cpu().double().numpy(), scale)


def test_quantize_rows_edge_values():
    # ties between E4M3 neighbours after scaling, signed zeros, the row max
    vals = np.array([448.0, 84.0, -84.0, 42.0, 2.0 ** -10, -(2.0 ** -10), 3 * 2.0 ** -10, 0.0, -0.0,
                     13 * 2.0 ** -4, 1.0 + 2.0 ** -4, 464.0 / 2, 224.0, 225.0, 1.0, -1.0])
    a = synth._cast(np.tile(vals, (3, 1)) * np.array([[1.0], [2.0 ** -40], [2.0 ** 30]]), "bf16")
    q, sc = st.sptp_quantize_rows_e4m3(dev_tensor(a, "bf16"))
    torch.cuda.synchronize()
    codes, scale = oracle_codes(synth.to_f64(a, "bf16"))
    assert np.array_equal(q.cpu().numpy(), codes)
    assert np.array_equal(sc.cpu().double().numpy(), scale)


def test_quantize_rows_empty_is_a_noop():
    a = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda:0")
    q, sc = st.sptp_quantize_rows_e4m3(a)
    assert q.shape == (0, 64) and sc.shape == (0,)


def test_weight_quantisation_layout_bit_exact():
    rng = np.random.default_rng(5)
    d, F, P = 256, 3 * 160, 3
    W1g, W1u, W2 = bf16_array(rng, (F, d), 0.05), bf16_array(rng, (F, d), 0.05), bf16_array(rng, (d, F), 0.05)
    qw = st.quantize_ffn_weights_e4m3(dev_tensor(W1g, "bf16"), dev_tensor(W1u, "bf16"), dev_tensor(W2, "bf16"), P)
    torch.cuda.synchronize()
    qg, eg, qu, eu, q2, e2 = f8.quantize_ffn_weights(synth.to_f64(W1g, "bf16"), synth.to_f64(W1u, "bf16"),
                                                     synth.to_f64(W2, "bf16"), P)
    got = [t.cpu().numpy() for t in qw]
    assert np.array_equal(got[0], f8.e4m3_encode(qg)) and np.array_equal(got[1], np.ldexp(1.0, eg))
    assert np.array_equal(got[2], f8.e4m3_encode(qu)) and np.array_equal(got[3], np.ldexp(1.0, eu))
    assert np.array_equal(got[4], f8.e4m3_encode(q2)) and np.array_equal(got[5], np.ldexp(1.0, e2))
    assert got[5].shape == (d, P)


@pytest.mark.parametrize("M,d,P", [(1, 16, 1), (37, 144, 2), (300, 1024, 3), (129, 4096, 2), (64, 5120, 4),
                                   (16, 8192, 8)])
def test_prologue_e4m3_equals_prologue_then_quantiser(M, d, P):
    """The fused launch gives the codes of quantising the prologue's own y
    (bit for bit), and they dequantise to within one E4M3 rounding of the
    oracle's bf16 y.  d=8192 with 8 sources takes the two-launch fallback."""
    rng = np.random.default_rng(M * 7 + d)
    x, parts = bf16_array(rng, (M, d)), bf16_array(rng, (P, M, d))
    gamma = synth._cast(1 + 0.1 * rng.standard_normal(d), "bf16")
    X, Pt, G = dev_tensor(x, "bf16"), dev_tensor(parts, "bf16"), dev_tensor(gamma, "bf16")
    h1, q1, s1 = st.sptp_prologue_e4m3(X, Pt, G, 1e-6)
    h0, y0 = st.sptp_prologue(X, Pt, G, 1e-6)
    q0, s0 = st.sptp_quantize_rows_e4m3(y0)
    torch.cuda.synchronize()
    assert torch.equal(h1, h0) and torch.equal(q1, q0) and torch.equal(s1, s0)
    href = synth.to_f64(x, "bf16") + synth.to_f64(parts, "bf16").sum(0)
    yref = f8.round_bf16(oracle.rms_norm(href, synth.to_f64(gamma, "bf16"), 1e-6))
    sc = s1.cpu().double().numpy()
    deq = q1.view(torch.float8_e4m3fn).cpu().double().numpy() * sc[:, None]
    assert np.all(np.abs(deq - yref) <= 0.07 * np.abs(yref) + 2.0 ** -10 * sc[:, None])
    _, e = f8.quantize_rows_e4m3(yref)
    assert np.all(np.abs(np.log2(sc) - e) <= 1)


# ---------------------------------------------------------------- GEMMs

@pytest.mark.parametrize("M,d,F,P", [(64, 128, 512, 2), (300, 144, 2 * 400, 2), (257, 1024, 3 * 384, 3),
                                     (1024, 512, 2048, 4)])
def test_gateup_and_down_e4m3_match_oracle(M, d, F, P):
    rng = np.random.default_rng(M + F)
    y = bf16_array(rng, (M, d))
    W1g, W1u = bf16_array(rng, (F, d), d ** -0.5), bf16_array(rng, (F, d), d ** -0.5)
    W2 = bf16_array(rng, (d, F), F ** -0.5)
    qw = st.quantize_ffn_weights_e4m3(dev_tensor(W1g, "bf16"), dev_tensor(W1u, "bf16"), dev_tensor(W2, "bf16"), P)
    qy, sy = st.sptp_quantize_rows_e4m3(dev_tensor(y, "bf16"))
    hdr = nan_workspace(st.SPTP_WS_HEADER_BYTES)
    s = st.sptp_gateup_swiglu_e4m3(qy, sy, qw[0], qw[1], qw[2], qw[3], P, s_out=nan_tensor((P, M, F // P)),
                                   workspace=hdr)
    assert st.sptp_read_device_status(hdr) == 0
    qs, ss = st.sptp_quantize_rows_e4m3(s)
    out = st.sptp_down_proj_e4m3(qs, ss, qw[4], qw[5], P, out=nan_tensor((P, M, d)), workspace=hdr)
    assert st.sptp_read_device_status(hdr) == 0
    assert_no_nan(s, out)
    ow = f8.quantize_ffn_weights(synth.to_f64(W1g, "bf16"), synth.to_f64(W1u, "bf16"), synth.to_f64(W2, "bf16"), P)
    y64 = synth.to_f64(y, "bf16")
    errs = {}
    for p in range(P):
        ref, it = f8.shard_ffn_fp8(y64, ow, P, p, return_intermediates=True)
        errs[f"s[{p}]"] = rel_err(host_f64(s[p]), it["s"])
        errs[f"out[{p}]"] = rel_err(host_f64(out[p]), ref)
    check_errors(errs, "e4m3")


# ---------------------------------------------------------------- full boundary

def run_fp8(cfg, rows=None):
    inp = synth.boundary_inputs(cfg)
    T = {k: dev_tensor(v, "bf16") for k, v in inp.items()}
    qw = st.quantize_ffn_weights_e4m3(T["W1g"], T["W1u"], T["W2"], cfg.P)
    ws = nan_workspace(st.sptp_ffn_fp8_workspace_size(cfg.M, cfg.d, cfg.F, cfg.P, cfg.chunks))
    out, h = nan_tensor((cfg.P, cfg.M, cfg.d)), nan_tensor((cfg.M, cfg.d))
    st.sptp_ffn_forward_fp8(T["x"], T["partials"], T["gamma"], qw, cfg.P, cfg.chunks, cfg.eps, out=out,
                            resid_out=h, workspace=ws)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(out, h)
    out2, _ = st.sptp_ffn_forward_fp8(T["x"], T["partials"], T["gamma"], qw, cfg.P, cfg.chunks, cfg.eps,
                                      workspace=ws)
    assert st.sptp_read_device_status(ws) == 0
    assert torch.equal(out, out2)  # deterministic
    f64 = {k: synth.to_f64(v, "bf16") for k, v in inp.items()}
    if rows is not None:
        f64["x"], f64["partials"] = f64["x"][rows], f64["partials"][:, rows]
    ref, href = f8.sptp_ffn_forward_fp8(f64["x"], f64["partials"], f64["gamma"], f64["W1g"], f64["W1u"],
                                        f64["W2"], cfg.P, cfg.chunks if rows is None else 1, cfg.eps)
    got = host_f64(out if rows is None else out[:, rows])
    goth = host_f64(h if rows is None else h[rows])
    errs = {f"out[{p}]": rel_err(got[p], ref[p]) for p in range(cfg.P)}
    errs["sum_p out"] = rel_err(got.sum(0), ref.sum(0))
    errs["h"] = rel_err(goth, href)
    return check_errors(errs, "e4m3")


def case(M, d, F, P, C, seed=0):
    return synth.BoundaryConfig(f"f8_{M}_{d}_{F}_{P}_{C}", M, d, F, P, C, "bf16", True, seed=seed)


@pytest.mark.parametrize("M,d,F,P,C", [(320, 256, 768, 2, 2), (384, 144, 3 * 208, 3, 3),
                                       (1000, 512, 4 * 400, 4, 8), (2048, 1024, 8 * 256, 8, 8), (130, 64, 64, 1, 1),
                                       (2, 16, 32, 2, 2), (64, 8192, 8 * 128, 8, 8)])
def test_boundary_fp8_multi_tile_and_ragged(M, d, F, P, C):
    # d=8192 with 8 sources: rows too wide for the prologue's shared-memory
    # ring, so y is stored and quantised by a second launch
    run_fp8(case(M, d, F, P, C))


def test_boundary_fp8_d4096_full_size_sampled_rows():
    cfg = synth.BOUNDARY_D4096
    rng = np.random.default_rng(1)
    rows = sorted(set([0, 1, 255, 256, 4095, 4096, 8191] + list(rng.choice(cfg.M, 25, replace=False))))
    run_fp8(cfg, rows=rows)
    torch.cuda.empty_cache()


def test_boundary_fp8_empty_sequence_is_a_noop():
    z = lambda *s, dt=torch.bfloat16: torch.zeros(s, dtype=dt, device="cuda:0")
    qw = (z(64, 64, dt=torch.uint8), z(64, dt=torch.float32), z(64, 64, dt=torch.uint8), z(64, dt=torch.float32),
          z(64, 64, dt=torch.uint8), z(64, 2, dt=torch.float32))
    out, _ = st.sptp_ffn_forward_fp8(z(0, 64), z(2, 0, 64), z(64), qw, 2, 2, 1e-6)
    assert out.shape == (2, 0, 64)
