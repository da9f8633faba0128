"""The no-allocation entry point, sptp_ffn_forward_noalloc.

Some callers cannot allocate device memory: a plugin inside a host framework
that owns every device allocation, or a serving loop that must not call
cudaMalloc because it can synchronise the device.  This entry point runs the
same boundary on a scratch array the library declares itself.  The test
calls it through the C ABI twice in a row, on different inputs, and checks
each result against the workspace entry point on the same inputs.  This file
is collected last, so a failure here does not stop the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import sequence_tensor_transformer_gb300 as st
from sequence_tensor_transformer_gb300 import synth

from helpers import TOL, dev_tensor, host_f64, rel_err

pytestmark = pytest.mark.gpu


def _inputs(seed, M=512, d=1024, F=4096, P=2):
    cfg = synth.BoundaryConfig(f"noalloc_{seed}", M, d, F, P, P, "bf16", True, seed=seed)
    return cfg, {k: dev_tensor(v, "bf16") for k, v in synth.boundary_inputs(cfg).items()}


def test_noalloc_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    lib = st.load_library()
    stream = torch.cuda.current_stream()
    for seed in (3, 4):  # two calls in a row share the static scratch
        cfg, T = _inputs(seed)
        M, d, F, P = cfg.M, cfg.d, cfg.F, cfg.P
        out = torch.empty((P, M, d), dtype=torch.bfloat16, device="cuda:0")
        resid = torch.empty((M, d), dtype=torch.bfloat16, device="cuda:0")
        code = lib.sptp_ffn_forward_noalloc(
            T["x"].data_ptr(), T["partials"].data_ptr(), T["gamma"].data_ptr(), T["W1g"].data_ptr(),
            T["W1u"].data_ptr(), T["W2"].data_ptr(), M, d, F, P, P, ctypes.c_float(cfg.eps), st.SPTP_BF16,
            out.data_ptr(), resid.data_ptr(), stream.cuda_stream)
        assert code == 0, st.sptp_status_string(code)
        ref_out, ref_h = st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], P,
                                             P, cfg.eps)
        torch.cuda.synchronize()
        for p in range(P):
            assert rel_err(host_f64(out[p]), host_f64(ref_out[p])) <= TOL["bf16"]
        assert rel_err(host_f64(resid), host_f64(ref_h)) <= TOL["bf16"]


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    lib = st.load_library()
    # bf16, d=4096, F=14336: 8192 tokens need ~300 MB of scratch (> 64 MiB)
    code = lib.sptp_ffn_forward_noalloc(16, 32, 48, 64, 80, 96, 8192, 4096, 14336, 2, 8, ctypes.c_float(1e-6),
                                        st.SPTP_BF16, 1 << 20, None, None)
    assert code == -9
    assert "scratch" in st.sptp_status_string(code)
    # invalid sizes report the same code as the workspace entry point
    assert lib.sptp_ffn_forward_noalloc(16, 32, 48, 64, 80, 96, 64, 100, 512, 2, 2, ctypes.c_float(1e-6),
                                        st.SPTP_BF16, 1 << 20, None, None) == -2
