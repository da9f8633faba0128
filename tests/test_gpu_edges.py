"""GPU parity at the limits the entry points accept: the widest rows
(d = 16384, whose sources do not fit the prologue's shared-memory ring), the
most shards (P = 8), and a Delayed-TP stack whose last stream update adds the
most partials a group may sum (1 + (P - 1) * S = 64)."""
import numpy as np
import pytest
import torch

import oracle
import sequence_tensor_transformer_gb300 as st
from sequence_tensor_transformer_gb300 import synth

from helpers import (TOL, assert_no_nan, check_errors, dev_tensor, host_f64, nan_tensor, nan_workspace, rel_err,
                     to_f64)

pytestmark = pytest.mark.gpu

D_MAX = 16384  # the widest row the entry points accept


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    st.load_library()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_prologue_widest_rows_most_shards(dtype):
    M, d, P = 5, D_MAX, 8
    rng = np.random.default_rng(16384)
    x = synth._cast(rng.standard_normal((M, d)), dtype)
    parts = synth._cast(rng.standard_normal((P, M, d)), dtype)
    gamma = synth._cast(1 + 0.1 * rng.standard_normal(d), dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    h, y = nan_tensor((M, d), tdt), nan_tensor((M, d), tdt)
    st.sptp_prologue(dev_tensor(x, dtype), dev_tensor(parts, dtype), dev_tensor(gamma, dtype), 1e-6, h_out=h, y_out=y)
    torch.cuda.synchronize()
    assert_no_nan(h, y)
    href = to_f64(x, dtype) + oracle.reduce_partials(to_f64(parts, dtype))
    yref = oracle.rms_norm(href, to_f64(gamma, dtype), 1e-6)
    # bf16 outputs carry one rounding (2^-9 relative); fp32 a few ulps of a sum of 9 terms
    tol = 2 ** -8 if dtype == "bf16" else 4e-6
    assert rel_err(host_f64(h), href) <= tol
    assert rel_err(host_f64(y), yref) <= tol


@pytest.mark.parametrize("variant", ["pair", "chain", "fused"])
def test_boundary_widest_rows(variant):
    cfg = synth.BoundaryConfig("edge_d16384", 264, D_MAX, 2 * 64, 2, 2, "bf16", True, seed=7)
    inp = synth.boundary_inputs(cfg)
    T = {k: dev_tensor(v, "bf16") for k, v in inp.items()}
    ws = nan_workspace(st.sptp_ffn_workspace_size(cfg.M, cfg.d, cfg.F, cfg.P, cfg.chunks, st.SPTP_BF16))
    out, h = nan_tensor((cfg.P, cfg.M, cfg.d)), nan_tensor((cfg.M, cfg.d))
    st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], cfg.P, cfg.chunks, cfg.eps,
                        out=out, resid_out=h, workspace=ws, variant=variant)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(out, h)
    f64 = {k: to_f64(v, "bf16") for k, v in inp.items()}
    ref, href = oracle.sptp_ffn_forward(f64["x"], f64["partials"], f64["gamma"], f64["W1g"], f64["W1u"],
                                        f64["W2"], cfg.P, cfg.chunks, cfg.eps)
    got = host_f64(out)
    errs = {p: rel_err(got[p], ref[p]) for p in range(cfg.P)}
    errs["h"] = rel_err(host_f64(h), href)
    check_errors(errs, "bf16")


@pytest.mark.parametrize("variant", ["fused", "layers"])
def test_dtp_stack_most_pending_sources(variant):
    # P = 8, S = min(delta + 1, L) = 9: 1 + 7 * 9 = 64 sources at the final
    # flushing step, the most one stream update may sum
    P, L, delta = 8, 9, 8
    cfg = synth.DTPConfig("edge_sources", 40, 64, P * 16, P, L, delta, "bf16")
    inp = synth.dtp_inputs(cfg, independent_streams=True)
    T = {k: dev_tensor(v, "bf16") for k, v in inp.items()}
    ws = nan_workspace(st.dtp_ffn_stack_workspace_size(cfg.M, cfg.d, cfg.F, P, L, delta, st.SPTP_BF16))
    st.dtp_ffn_stack_forward(T["x_shards"], T["gamma"], T["W1g"], T["W1u"], T["W2"], P, L, delta, 1, cfg.eps,
                             workspace=ws, variant=variant)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(T["x_shards"])
    f64 = {k: to_f64(v, "bf16") for k, v in inp.items()}
    ref = oracle.dtp_ffn_stack_forward(f64["x_shards"], f64["gamma"], f64["W1g"], f64["W1u"], f64["W2"], P, L,
                                       delta, True, cfg.eps)
    got = host_f64(T["x_shards"])
    check_errors({p: rel_err(got[p], ref[p]) for p in range(P)}, "bf16")
