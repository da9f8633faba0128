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

from helpers import TOL, assert_no_nan, dev_tensor, host_f64, nan_tensor, rel_err

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
        out = nan_tensor((P, M, d))
        resid = nan_tensor((M, d))
        code = lib.sptp_ffn_forward_noalloc(
            T["x"].data_ptr(), T["partials"].data_ptr(), T["gamma"].data_ptr(), T["W1g"].data_ptr(),
            T["W1u"].data_ptr(), T["W2"].data_ptr(), M, d, F, P, P, ctypes.c_float(cfg.eps), st.SPTP_BF16,
            out.data_ptr(), resid.data_ptr(), stream.cuda_stream)
        assert code == 0, st.sptp_status_string(code)
        # the static array's status words: no bounded wait gave up
        assert lib.sptp_noalloc_read_device_status(stream.cuda_stream) == 0
        assert_no_nan(out, resid)
        ref_out, ref_h = st.sptp_ffn_forward(T["x"], T["partials"], T["gamma"], T["W1g"], T["W1u"], T["W2"], P,
                                             P, cfg.eps)
        torch.cuda.synchronize()
        for p in range(P):
            assert rel_err(host_f64(out[p]), host_f64(ref_out[p])) <= TOL["bf16"]
        assert rel_err(host_f64(resid), host_f64(ref_h)) <= TOL["bf16"]


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    lib = st.load_library()
    # distinct 16-byte aligned addresses 4 GiB apart: the argument checks
    # dereference nothing and find no overlap
    a = [(1 << 40) + (i << 32) for i in range(7)]
    # bf16, d=4096, F=14336: 8192 tokens need ~300 MB of scratch (> 64 MiB)
    code = lib.sptp_ffn_forward_noalloc(*a[:6], 8192, 4096, 14336, 2, 8, ctypes.c_float(1e-6),
                                        st.SPTP_BF16, a[6], None, None)
    assert code == st.STATUS["too_large"]
    assert "scratch" in st.sptp_status_string(code)
    # invalid sizes report the same code as the workspace entry point
    assert lib.sptp_ffn_forward_noalloc(*a[:6], 64, 100, 512, 2, 2, ctypes.c_float(1e-6),
                                        st.SPTP_BF16, a[6], None, None) == st.STATUS["shape"]
    # argument errors come before the size limit: a bad chunk count at an
    # oversized M is a shape error, a missing input a null error, an output
    # on top of an input an alias error
    assert lib.sptp_ffn_forward_noalloc(*a[:6], 8192, 4096, 14336, 2, 3, ctypes.c_float(1e-6),
                                        st.SPTP_BF16, a[6], None, None) == st.STATUS["shape"]
    assert lib.sptp_ffn_forward_noalloc(None, *a[1:6], 8192, 4096, 14336, 2, 8, ctypes.c_float(1e-6),
                                        st.SPTP_BF16, a[6], None, None) == st.STATUS["null"]
    assert lib.sptp_ffn_forward_noalloc(*a[:6], 8192, 4096, 14336, 2, 8, ctypes.c_float(1e-6),
                                        st.SPTP_BF16, a[0], None, None) == st.STATUS["alias"]


def test_noalloc_status_words_report_a_timeout():
    """The static array's status words carry the no-allocation path's failure
    detection: a bounded wait that gives up there is reported, and the next
    forward clears it."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    lib = st.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.sptp_noalloc_wait_selftest(2_000_000, 0, stream) == 0
    assert lib.sptp_noalloc_read_device_status(stream) == st.STATUS["timeout"]
    cfg, T = _inputs(5, M=256, d=512, F=1024)
    out = torch.empty((cfg.P, cfg.M, cfg.d), dtype=torch.bfloat16, device="cuda:0")
    code = lib.sptp_ffn_forward_noalloc(
        T["x"].data_ptr(), T["partials"].data_ptr(), T["gamma"].data_ptr(), T["W1g"].data_ptr(),
        T["W1u"].data_ptr(), T["W2"].data_ptr(), cfg.M, cfg.d, cfg.F, cfg.P, cfg.P, ctypes.c_float(cfg.eps),
        st.SPTP_BF16, out.data_ptr(), None, stream)
    assert code == 0
    assert lib.sptp_noalloc_read_device_status(stream) == 0
