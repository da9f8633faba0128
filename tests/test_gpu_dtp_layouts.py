"""GPU parity of neuron-permutation shard maps for Delayed TP: the permutation
kernel against plain indexing (bit-exact: it only moves bytes) and the
permuted Delayed-TP stack against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import sequence_tensor_transformer_gb300 as st
from sequence_tensor_transformer_gb300 import synth

from helpers import TOL, assert_no_nan, check_errors, dev_tensor, host_f64, nan_tensor, nan_workspace, rel_err, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["fused", "layers"])
def dtp_variant(request):
    """Delayed-TP stack as one fused persistent launch (default) or as a
    prologue and two GEMM launches per module."""
    return request.param


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    st.load_library()
    torch.cuda.set_device(0)


def _perms(L, F, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(F) for _ in range(L)]).astype(np.int32)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("L,d,F", [(1, 8, 8), (3, 8, 24), (2, 136, 200), (4, 1024, 3072), (2, 64, 6144),
                                   (1, 6144, 8), (1, 4096, 14336), (1, 16, 24576)])
def test_permutation_kernel_is_exact_indexing(dtype, L, d, F):
    """Both launch structures: the one-launch bulk-copy pipeline (a W1 row of
    each matrix and a W2 row fit its 32 KiB stage: one or many rows per unit)
    and the two-launch fallback for wider rows (F = 24576; in fp32 also
    d = 6144 and F = 14336)."""
    rng = np.random.default_rng(L * d + F)
    W1g = synth._cast(rng.standard_normal((L, F, d)), dtype)
    W1u = synth._cast(rng.standard_normal((L, F, d)), dtype)
    W2 = synth._cast(rng.standard_normal((L, d, F)), dtype)
    perm = _perms(L, F, 5)
    hdr = nan_workspace(st.SPTP_WS_HEADER_BYTES)
    outs = st.sptp_permute_ffn_neurons(dev_tensor(W1g, dtype), dev_tensor(W1u, dtype), dev_tensor(W2, dtype),
                                       torch.from_numpy(perm).cuda(), workspace=hdr)
    assert st.sptp_read_device_status(hdr) == 0
    view = (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)) if dtype == "bf16" else \
        (lambda t: t.cpu().numpy())
    for l in range(L):
        assert np.array_equal(view(outs[0])[l], W1g[l][perm[l]])
        assert np.array_equal(view(outs[1])[l], W1u[l][perm[l]])
        assert np.array_equal(view(outs[2])[l], W2[l][:, perm[l]])


@pytest.mark.parametrize("d,F", [(64, 32), (8, 24576)])
def test_out_of_range_index_is_reported_and_zero_filled(d, F):
    """(64, 32) runs the pipelined launch, (8, 24576) the two-launch fallback."""
    L = 1
    W = [torch.randn((L, F, d), device="cuda:0").to(torch.bfloat16) for _ in range(2)]
    W2 = torch.randn((L, d, F), device="cuda:0").to(torch.bfloat16)
    perm = np.arange(F, dtype=np.int32)[None].copy()
    perm[0, 3] = F + 5
    perm[0, 7] = -1
    ws = torch.zeros(st.SPTP_WS_HEADER_BYTES, dtype=torch.uint8, device="cuda:0")
    g, u, w2 = st.sptp_permute_ffn_neurons(W[0], W[1], W2, torch.from_numpy(perm).cuda(), workspace=ws)
    assert st.sptp_read_device_status(ws) == -2
    for t in (g, u):
        assert torch.count_nonzero(t[0, 3]) == 0 and torch.count_nonzero(t[0, 7]) == 0
    assert torch.count_nonzero(w2[0][:, 3]) == 0 and torch.count_nonzero(w2[0][:, 7]) == 0
    keep = [i for i in range(F) if i not in (3, 7)]
    assert torch.equal(g[0, keep], W[0][0, keep]) and torch.equal(u[0, keep], W[1][0, keep])
    assert torch.equal(w2[0][:, keep], W2[0][:, keep])


def run_permuted_dtp(cfg, perms, flush, rows=None, variant="auto"):
    inp = synth.dtp_inputs(cfg)
    T = {k: dev_tensor(v, cfg.dtype) for k, v in inp.items()}
    hdr = nan_workspace(st.SPTP_WS_HEADER_BYTES)
    g, u, w2 = st.sptp_permute_ffn_neurons(T["W1g"], T["W1u"], T["W2"], torch.from_numpy(perms).cuda(), workspace=hdr)
    assert st.sptp_read_device_status(hdr) == 0
    ws = nan_workspace(st.dtp_ffn_stack_workspace_size(cfg.M, cfg.d, cfg.F, cfg.P, cfg.L, cfg.delta, st.SPTP_BF16))
    st.dtp_ffn_stack_forward(T["x_shards"], T["gamma"], g, u, w2, cfg.P, cfg.L, cfg.delta, flush, cfg.eps,
                             workspace=ws, variant=variant)
    assert st.sptp_read_device_status(ws) == 0
    assert_no_nan(T["x_shards"])
    f64 = {k: to_f64(v, cfg.dtype) for k, v in inp.items()}
    xs = f64["x_shards"] if rows is None else f64["x_shards"][:, rows]
    ref = oracle.dtp_ffn_stack_forward_permuted(xs, f64["gamma"], f64["W1g"], f64["W1u"], f64["W2"], perms,
                                                cfg.P, cfg.L, cfg.delta, bool(flush), cfg.eps)
    got = host_f64(T["x_shards"] if rows is None else T["x_shards"][:, rows])
    return got, ref


def test_permuted_dtp_stack_workload_sampled_rows(dtp_variant):
    cfg = synth.DTP_STACK
    rows = [0, 1, 77, 1024, 2047, 3333, 4095]
    got, ref = run_permuted_dtp(cfg, _perms(cfg.L, cfg.F, 11), 1, rows=rows, variant=dtp_variant)
    check_errors({p: rel_err(got[p], ref[p]) for p in range(cfg.P)}, "bf16")


@pytest.mark.parametrize("P,L,delta,flush", [(2, 3, 1, 0), (3, 2, 0, 1), (4, 3, 2, 1)])
def test_permuted_dtp_small_cases(P, L, delta, flush, dtp_variant):
    cfg = synth.DTPConfig("perm", 160, 136, P * 48, P, L, delta, "bf16")
    got, ref = run_permuted_dtp(cfg, _perms(L, cfg.F, P + L), flush, variant=dtp_variant)
    check_errors({p: rel_err(got[p], ref[p]) for p in range(P)}, "bf16")
