"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs.  Bar: rel. max error (max |got - ref| / max |ref|,
per output tensor) <= 2e-2 for bf16 storage with fp32 accumulation and
<= 1e-5 for fp32, plus each family's regression bound (helpers.REGRESSION).
Outputs and workspaces start as NaN and every call's device status is read."""
import numpy as np
import pytest
import torch

import oracle
import sequence_tensor_transformer_gb300 as st
from sequence_tensor_transformer_gb300 import synth

from helpers import (TOL, assert_no_nan, check_errors, dev_tensor, host_f64, nan_tensor, nan_workspace, rel_err,
                     to_f64)

pytestmark = pytest.mark.gpu

# The launch variants of each entry point (sptp_variant): every one of them is
# run by name; a variant that cannot launch is an error, not a fall-back.
BOUNDARY_VARIANTS = ["pair", "chain", "fused"]
DTP_VARIANTS = ["fused", "layers"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    st.load_library()
    torch.cuda.set_device(0)


def case(M, d, F, P, C, dtype, down_from_F=True, seed=0):
    return synth.BoundaryConfig(f"t_{M}_{d}_{F}_{P}_{C}_{dtype}", M, d, F, P, C, dtype, down_from_F, seed=seed)


def boundary_call(T, cfg, chunks=None, variant="auto"):
    """One sptp_ffn_forward into NaN-poisoned outputs and workspace; checks
    the device status and that every output element was written."""
    C = chunks or cfg.chunks
    dt = st.SPTP_BF16 if cfg.dtype == "bf16" else st.SPTP_FP32
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    ws = nan_workspace(st.sptp_ffn_workspace_size(cfg.M, cfg.d, cfg.F, cfg.P, C, dt))
    out = nan_tensor((cfg.P, cfg.M, cfg.d), tdt)
    h = nan_tensor((cfg.M, cfg.d), tdt)
    st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], cfg.P, C, cfg.eps,
                        out=out, resid_out=h, workspace=ws, variant=variant)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(out, h)
    return out, h


def run_boundary(cfg, rows=None, chunks=None, variant="auto"):
    inp = synth.boundary_inputs(cfg)
    T = {k: dev_tensor(v, cfg.dtype) for k, v in inp.items()}
    out, h = boundary_call(T, cfg, chunks, variant)
    if rows is not None:
        # rows are independent (the norm reduces over the hidden dim only), so
        # the oracle evaluates just the sampled rows, as one chunk
        inp["x"], inp["partials"] = inp["x"][rows], inp["partials"][:, rows]
    f64 = {k: to_f64(v, cfg.dtype) for k, v in inp.items()}
    ref, href = oracle.sptp_ffn_forward(f64["x"], f64["partials"], f64["gamma"], f64["W1g"], f64["W1u"],
                                        f64["W2"], cfg.P, cfg.chunks if rows is None else 1, cfg.eps)
    got = host_f64(out if rows is None else out[:, rows])
    goth = host_f64(h if rows is None else h[rows])
    return got, goth, ref, href


def check(got, goth, ref, href, dtype):
    errs = {f"out[{p}]": rel_err(got[p], ref[p]) for p in range(ref.shape[0])}
    errs["sum_p out"] = rel_err(got.sum(0), ref.sum(0))
    errs["h"] = rel_err(goth, href)
    return check_errors(errs, dtype, dtype)


# ---------------------------------------------------------------- step level

@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("M,d,P", [(1, 8, 1), (37, 136, 2), (300, 1000, 3), (129, 4096, 2), (64, 5120, 4)])
def test_prologue_matches_oracle(dtype, M, d, P):
    rng = np.random.default_rng(M * 7 + d)
    x = synth._cast(rng.standard_normal((M, d)), dtype)
    parts = synth._cast(rng.standard_normal((P, M, d)), dtype)
    gamma = synth._cast(1 + 0.1 * rng.standard_normal(d), dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    h, y = nan_tensor((M, d), tdt), nan_tensor((M, d), tdt)
    st.sptp_prologue(dev_tensor(x, dtype), dev_tensor(parts, dtype), dev_tensor(gamma, dtype), 1e-6, h_out=h,
                     y_out=y)
    torch.cuda.synchronize()
    assert_no_nan(h, y)
    href = to_f64(x, dtype) + oracle.reduce_partials(to_f64(parts, dtype))
    yref = oracle.rms_norm(href, to_f64(gamma, dtype), 1e-6)
    # bf16 outputs carry one rounding (2^-9 relative); fp32 a few ulps
    tol = 2 ** -8 if dtype == "bf16" else 2e-6
    assert rel_err(host_f64(h), href) <= tol
    assert rel_err(host_f64(y), yref) <= tol


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("M,d,F,P", [(64, 128, 512, 2), (300, 136, 400, 2), (257, 1024, 3 * 392, 3),
                                     (1024, 512, 2048, 4)])
def test_gateup_swiglu_matches_oracle(dtype, M, d, F, P):
    rng = np.random.default_rng(F + M)
    y = synth._cast(rng.standard_normal((M, d)), dtype)
    W1g = synth._cast(rng.standard_normal((F, d)) / np.sqrt(d), dtype)
    W1u = synth._cast(rng.standard_normal((F, d)) / np.sqrt(d), dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    s, ws = nan_tensor((P, M, F // P), tdt), nan_workspace(st.SPTP_WS_HEADER_BYTES)
    st.sptp_gateup_swiglu(dev_tensor(y, dtype), dev_tensor(W1g, dtype), dev_tensor(W1u, dtype), P, s_out=s,
                          workspace=ws)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(s)
    y64, g64, u64 = to_f64(y, dtype), to_f64(W1g, dtype), to_f64(W1u, dtype)
    f = F // P
    errs = {}
    for p in range(P):
        n = slice(p * f, (p + 1) * f)
        errs[p] = rel_err(host_f64(s[p]), oracle.silu(y64 @ g64[n].T) * (y64 @ u64[n].T))
    check_errors(errs, "bf16_step" if dtype == "bf16" else "fp32", dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("M,d,F,P", [(64, 128, 512, 2), (300, 136, 400, 2), (257, 1000, 3 * 392, 3),
                                     (1024, 512, 2048, 4)])
def test_down_proj_matches_oracle(dtype, M, d, F, P):
    rng = np.random.default_rng(F + 3 * M)
    f = F // P
    s = synth._cast(rng.standard_normal((P, M, f)), dtype)
    W2 = synth._cast(rng.standard_normal((d, F)) / np.sqrt(F), dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out, ws = nan_tensor((P, M, d), tdt), nan_workspace(st.SPTP_WS_HEADER_BYTES)
    st.sptp_down_proj(dev_tensor(s, dtype), dev_tensor(W2, dtype), P, out=out, workspace=ws)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(out)
    s64, w64 = to_f64(s, dtype), to_f64(W2, dtype)
    errs = {p: rel_err(host_f64(out[p]), s64[p] @ w64[:, p * f:(p + 1) * f].T) for p in range(P)}
    check_errors(errs, "bf16_step" if dtype == "bf16" else "fp32", dtype)


# ---------------------------------------------------------------- full boundary

def test_tiny_fp32_config():
    check(*run_boundary(synth.TINY_FP32), "fp32")


@pytest.mark.parametrize("variant", BOUNDARY_VARIANTS)
@pytest.mark.parametrize("M,d,F,P,C", [(320, 256, 768, 2, 2), (384, 136, 3 * 200, 3, 3), (1000, 512, 4 * 392, 4, 8),
                                       (2048, 1024, 8 * 256, 8, 8), (130, 64, 64, 1, 1), (600, 256, 512, 2, 6)])
def test_boundary_bf16_multi_tile_and_ragged(M, d, F, P, C, variant):
    check(*run_boundary(case(M, d, F, P, C, "bf16"), variant=variant), "bf16")


@pytest.mark.parametrize("M,d,F,P,C", [(96, 136, 3 * 40, 3, 3), (200, 256, 2 * 96, 2, 4)])
def test_boundary_fp32_ragged(M, d, F, P, C):
    check(*run_boundary(case(M, d, F, P, C, "fp32", down_from_F=False)), "fp32")


def test_fp32_rejects_the_persistent_variants():
    cfg = case(64, 128, 256, 2, 2, "fp32", down_from_F=False)
    T = {k: dev_tensor(v, "fp32") for k, v in synth.boundary_inputs(cfg).items()}
    for variant in ("chain", "fused", "layers"):
        with pytest.raises(st.SptpError) as e:
            st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], 2, 2, 1e-6,
                                variant=variant)
        assert e.value.code == st.STATUS["unimplemented"]


SAMPLE = [0, 1, 127, 128, 1000, 4095, 4096, 5555, 8191]


def sample_rows(M, n=24, seed=1):
    rng = np.random.default_rng(seed)
    base = [r for r in SAMPLE if r < M] + [M - 1]
    return sorted(set(base + list(rng.choice(M, n, replace=False))))


@pytest.mark.parametrize("variant", BOUNDARY_VARIANTS)
def test_boundary_d4096_full_size_sampled_rows(variant):
    cfg = synth.BOUNDARY_D4096
    check(*run_boundary(cfg, rows=sample_rows(cfg.M), variant=variant), "bf16")


@pytest.mark.parametrize("variant", BOUNDARY_VARIANTS)
def test_boundary_qwen2_7b_shape_full_size_sampled_rows(variant):
    cfg = synth.QWEN2_7B_SHAPE
    check(*run_boundary(cfg, rows=sample_rows(cfg.M, 16), variant=variant), "bf16")


@pytest.mark.parametrize("variant", BOUNDARY_VARIANTS)
@pytest.mark.parametrize("M", [4096, 16384, 65536])
def test_m_sweep_full_size_sampled_rows(M, variant):
    cfg = synth.m_sweep(M)
    check(*run_boundary(cfg, rows=sample_rows(cfg.M, 8), variant=variant), "bf16")
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", BOUNDARY_VARIANTS)
def test_chunked_equals_monolithic_bitwise(variant):
    """The chunk count changes when rows reach the GEMMs (FUSED: a gate/up
    tile waits for every chunk its rows overlap), never what a row computes:
    outputs are identical for every chunking, including chunks that are not
    a multiple of the 256-row tile."""
    cfg = case(1536, 512, 4 * 256, 4, 4, "bf16")
    T = {k: dev_tensor(v, "bf16") for k, v in synth.boundary_inputs(cfg).items()}
    res = [boundary_call(T, cfg, C, variant) for C in (4, 8, 12, 16, 24)]
    for out, h in res[1:]:
        assert torch.equal(out, res[0][0]) and torch.equal(h, res[0][1])


def test_sharded_sum_matches_unsharded_on_gpu():
    """Sum of the P partials vs the P=1 boundary on the same weights."""
    cfg = case(512, 512, 2048, 4, 4, "bf16")
    inp = synth.boundary_inputs(cfg)
    T = {k: dev_tensor(v, "bf16") for k, v in inp.items()}
    out4, h4 = st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], 4, 4, 1e-6)
    one = T["partials"].float().sum(0, keepdim=True).to(torch.bfloat16)
    out1, _ = st.sptp_ffn_forward(T["x"], one.contiguous(), T["gamma"], T["W1g"], T["W1u"], T["W2"], 1, 1, 1e-6)
    torch.cuda.synchronize()
    assert rel_err(host_f64(out4).sum(0), host_f64(out1[0])) <= 2e-2


@pytest.mark.parametrize("variant", BOUNDARY_VARIANTS)
def test_resid_in_place_and_optional(variant):
    cfg = case(256, 256, 512, 2, 2, "bf16")
    T = {k: dev_tensor(v, "bf16") for k, v in synth.boundary_inputs(cfg).items()}
    kw = dict(variant=variant)
    out_a, h_a = st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], 2, 2, 1e-6,
                                     **kw)
    out_b, _ = st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], 2, 2, 1e-6,
                                   write_resid=False, **kw)
    x = T["x"].clone()
    out_c, h_c = st.sptp_ffn_forward(x, T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], 2, 2, 1e-6,
                                     resid_out=x, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(out_a, out_c) and torch.equal(h_a, x)


def test_empty_sequence_is_a_noop():
    T = {k: torch.zeros(s, dtype=torch.bfloat16, device="cuda:0") for k, s in
         (("x", (0, 64)), ("p", (2, 0, 64)), ("g", (64,)), ("w1", (128, 64)), ("w2", (64, 128)))}
    for variant in BOUNDARY_VARIANTS:
        out, h = st.sptp_ffn_forward(T["x"], T["p"], T["g"], T["w1"], T["w1"], T["w2"], 2, 2, 1e-6, variant=variant)
        assert out.shape == (2, 0, 64)


def test_error_codes_on_gpu():
    x = torch.zeros((64, 100), dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(st.SptpError) as e:
        st.sptp_ffn_forward(x, torch.zeros((2, 64, 100), dtype=torch.bfloat16, device="cuda:0"), x[0], x, x,
                            x.t().contiguous(), 2, 2, 1e-6)
    assert e.value.code == st.STATUS["shape"]


# ---------------------------------------------------------------- Delayed TP

def run_dtp(cfg, flush=1, independent=False, rows=None, variant="auto"):
    inp = synth.dtp_inputs(cfg, independent_streams=independent)
    T = {k: dev_tensor(v, cfg.dtype) for k, v in inp.items()}
    dt = st.SPTP_BF16 if cfg.dtype == "bf16" else st.SPTP_FP32
    ws = nan_workspace(st.dtp_ffn_stack_workspace_size(cfg.M, cfg.d, cfg.F, cfg.P, cfg.L, cfg.delta, dt))
    st.dtp_ffn_stack_forward(T["x_shards"], T["gamma"], T["W1g"], T["W1u"], T["W2"], cfg.P, cfg.L, cfg.delta,
                             flush, cfg.eps, workspace=ws, variant=variant)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(T["x_shards"])
    f64 = {k: to_f64(v, cfg.dtype) for k, v in inp.items()}
    ref = oracle.dtp_ffn_stack_forward(f64["x_shards"], f64["gamma"], f64["W1g"], f64["W1u"], f64["W2"], cfg.P,
                                       cfg.L, cfg.delta, bool(flush), cfg.eps, rows=rows)
    got = host_f64(T["x_shards"] if rows is None else T["x_shards"][:, rows])
    return got, ref


@pytest.mark.parametrize("variant", DTP_VARIANTS)
def test_dtp_stack_config_full_size_sampled_rows(variant):
    cfg = synth.DTP_STACK
    for flush in (0, 1):
        got, ref = run_dtp(cfg, flush=flush, rows=sample_rows(cfg.M, 32), variant=variant)
        check_errors({(flush, p): rel_err(got[p], ref[p]) for p in range(cfg.P)}, "bf16")


@pytest.mark.parametrize("variant", DTP_VARIANTS)
@pytest.mark.parametrize("P,L,delta,flush,indep", [(2, 3, 0, 1, False), (3, 4, 2, 0, True), (4, 2, 5, 1, False),
                                                   (1, 3, 1, 1, False), (2, 5, 1, 0, False)])
def test_dtp_small_cases(P, L, delta, flush, indep, variant):
    cfg = synth.DTPConfig("t", 200, 136, P * 48, P, L, delta, "bf16")
    got, ref = run_dtp(cfg, flush=flush, independent=indep, variant=variant)
    check_errors({p: rel_err(got[p], ref[p]) for p in range(P)}, "bf16")


def test_dtp_fp32():
    cfg = synth.DTPConfig("t32", 96, 128, 2 * 64, 2, 3, 1, "fp32")
    got, ref = run_dtp(cfg, flush=1)
    check_errors({p: rel_err(got[p], ref[p]) for p in range(cfg.P)}, "fp32", "fp32")
    with pytest.raises(st.SptpError) as e:
        run_dtp(cfg, flush=1, variant="fused")
    assert e.value.code == st.STATUS["unimplemented"]


@pytest.mark.parametrize("variant", DTP_VARIANTS)
def test_dtp_delta0_equals_chained_boundaries_on_gpu(variant):
    cfg = synth.DTPConfig("t0", 256, 256, 2 * 256, 2, 3, 0, "bf16")
    T = {k: dev_tensor(v, "bf16") for k, v in synth.dtp_inputs(cfg).items()}
    xs = T["x_shards"].clone()
    st.dtp_ffn_stack_forward(xs, T["gamma"], T["W1g"], T["W1u"], T["W2"], 2, 3, 0, 1, 1e-6, variant=variant)
    x = T["x_shards"][0].clone()
    parts = torch.zeros((2,) + x.shape, dtype=torch.bfloat16, device="cuda:0")
    for l in range(3):
        parts, x = st.sptp_ffn_forward(x, parts, T["gamma"][l].contiguous(), T["W1g"][l].contiguous(),
                                       T["W1u"][l].contiguous(), T["W2"][l].contiguous(), 2, 2, 1e-6)
    final = x.float() + parts.float().sum(0)
    torch.cuda.synchronize()
    for p in range(2):
        assert rel_err(host_f64(xs[p]), host_f64(final)) <= 2e-2


# ---------------------------------------------------------------- failure detection

def test_bounded_wait_reports_timeout_without_hanging():
    ws = torch.zeros(st.SPTP_WS_HEADER_BYTES, dtype=torch.uint8, device="cuda:0")
    assert st.sptp_wait_selftest(ws, 2_000_000, False) == 0
    assert st.sptp_read_device_status(ws) == st.STATUS["timeout"]
    words = ws[:20].view(torch.int32).cpu().tolist()
    assert words[1] == 6  # the flag wait gave up first
    assert st.sptp_wait_selftest(ws, 2_000_000, True) == 0
    assert st.sptp_read_device_status(ws) == st.STATUS["timeout"]
    words = ws[:20].view(torch.int32).cpu().tolist()
    assert words[1] == 7 and words[3] == 1  # flag seen, then the barrier wait gave up
    # the context is still usable afterwards
    check(*run_boundary(synth.TINY_FP32), "fp32")


@pytest.mark.parametrize("M,d,F,P,C", [(1024, 4096, 2 * 1024, 2, 2), (512, 3584, 4 * 512, 4, 4),
                                       (300, 1000, 3 * 128, 3, 3)])
def test_every_variant_gives_the_same_bits(M, d, F, P, C):
    """With up to 5 sources and d <= 4096 the fused launch's prologue (one
    row per CTA) reduces in the standalone prologue's order, and every GEMM
    tile runs the same UMMAs in every variant: the outputs match bit for
    bit."""
    cfg = case(M, d, F, P, C, "bf16")
    T = {k: dev_tensor(v, "bf16") for k, v in synth.boundary_inputs(cfg).items()}
    res = {v: boundary_call(T, cfg, variant=v) for v in BOUNDARY_VARIANTS}
    for v in ("chain", "fused"):
        assert torch.equal(res[v][1], res["pair"][1]), v
        assert torch.equal(res[v][0], res["pair"][0]), v
