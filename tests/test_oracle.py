"""CPU pins of the float64 oracle.

Each test ties the oracle to something other than itself: library routines
(torch.nn.functional in float64), closed forms, invariants the pages state,
brute force on tiny inputs, and a hand-derived worked example.  A plausible
slip in the oracle (a dropped term, a transposed weight, a wrong shard slice,
an off-by-one in the Delayed-TP delay) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle
from oracle import dtp_ffn_stack_forward, rel_max_error, rms_norm, silu, sptp_ffn_forward
from sequence_tensor_transformer_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_case(M, d, F, P, seed=1, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, d)) * scale
    partials = rng.standard_normal((P, M, d))
    gamma = 1 + 0.1 * rng.standard_normal(d)
    W1g = rng.standard_normal((F, d)) / math.sqrt(d)
    W1u = rng.standard_normal((F, d)) / math.sqrt(d)
    W2 = rng.standard_normal((d, F)) / math.sqrt(F)
    return x, partials, gamma, W1g, W1u, W2


# ------------------------------------------------------------ library pins

def test_rms_norm_matches_torch_library():
    rng = np.random.default_rng(0)
    h = rng.standard_normal((37, 96)) * 3
    g = 1 + 0.1 * rng.standard_normal(96)
    for eps in (1e-6, 0.5):
        ref = Fn.rms_norm(torch.from_numpy(h), (96,), torch.from_numpy(g), eps).numpy()
        assert np.max(np.abs(rms_norm(h, g, eps) - ref)) < 1e-13


def test_silu_matches_torch_and_closed_forms():
    z = np.linspace(-30, 30, 1001)
    ref = Fn.silu(torch.from_numpy(z)).numpy()
    assert np.max(np.abs(silu(z) - ref)) < 1e-14
    assert silu(np.array([0.0]))[0] == 0.0
    assert abs(silu(np.array([1.0]))[0] - 1 / (1 + 1 / math.e)) < 1e-15
    assert abs(silu(np.array([-1.0]))[0] + 1 / (1 + math.e)) < 1e-15
    # far tails: silu(z) -> z for z >> 0 and -> 0 for z << 0, no NaN
    big = silu(np.array([800.0, -800.0]))
    assert big[0] == 800.0 and big[1] == 0.0


def test_unsharded_boundary_matches_torch_functional():
    """P=1, one chunk: the boundary is exactly the library composition
    rms_norm(x + partial) -> linear/silu/linear (SwiGLU FFN)."""
    M, d, F = 21, 40, 56
    x, partials, gamma, W1g, W1u, W2 = rand_case(M, d, F, 1)
    out, h = sptp_ffn_forward(x, partials, gamma, W1g, W1u, W2, 1, 1, 1e-6)
    T = torch.from_numpy
    h_ref = T(x) + T(partials).sum(0)
    y = Fn.rms_norm(h_ref, (d,), T(gamma), 1e-6)
    ref = Fn.linear(Fn.silu(Fn.linear(y, T(W1g))) * Fn.linear(y, T(W1u)), T(W2)).numpy()
    assert rel_max_error(h, h_ref.numpy()) < 1e-15
    assert rel_max_error(out[0], ref) < 1e-12


# ------------------------------------------------------------ invariants

@pytest.mark.parametrize("P", [2, 4, 8])
def test_sharded_sum_equals_unsharded(P):
    """Sum over the P row-parallel partials == the unsharded FFN (P=1)."""
    M, d, F = 16, 32, 64
    x, partials, gamma, W1g, W1u, W2 = rand_case(M, d, F, P)
    outP, hP = sptp_ffn_forward(x, partials, gamma, W1g, W1u, W2, P, P, 1e-6)
    # same h, fed as a single partial of an unsharded boundary
    one = partials.sum(0, keepdims=True)
    out1, h1 = sptp_ffn_forward(x, one, gamma, W1g, W1u, W2, 1, 1, 1e-6)
    assert rel_max_error(hP, h1) < 1e-14
    assert rel_max_error(outP.sum(0), out1[0]) < 1e-12
    # each partial only uses its own neuron block: zeroing block p's weights
    # zeroes partial p and nothing else
    f = F // P
    W1g_z = W1g.copy()
    W1g_z[f:2 * f] = 0
    outz, _ = sptp_ffn_forward(x, partials, gamma, W1g_z, W1u, W2, P, P, 1e-6)
    assert np.all(outz[1] == 0)
    assert rel_max_error(outz[0], outP[0]) < 1e-15


@pytest.mark.parametrize("chunks", [1, 2, 4, 8])
def test_chunked_equals_monolithic(chunks):
    M, d, F, P = 32, 24, 48, 2
    args = rand_case(M, d, F, P)
    ref, href = sptp_ffn_forward(*args, P, 1, 1e-6)
    out, h = sptp_ffn_forward(*args, P, chunks, 1e-6)
    assert rel_max_error(h, href) == 0.0
    assert rel_max_error(out, ref) < 1e-13


def test_row_subset_equals_full():
    M, d, F, P = 40, 24, 48, 4
    args = rand_case(M, d, F, P)
    ref, href = sptp_ffn_forward(*args, P, 4, 1e-6)
    rows = [0, 7, 13, 39]
    out, h = sptp_ffn_forward(*args, P, 4, 1e-6, rows=rows)
    assert rel_max_error(h, href[rows]) == 0.0
    assert rel_max_error(out, ref[:, rows]) < 1e-13


def test_norm_commutes_with_sequence_gather():
    """norm(all_gather(x)) == all_gather(norm(x)): normalising each shard's
    sequence slice and concatenating equals normalising the gathered rows."""
    rng = np.random.default_rng(3)
    h = rng.standard_normal((64, 48))
    g = 1 + 0.1 * rng.standard_normal(48)
    whole = rms_norm(h, g, 1e-6)
    for P in (2, 4, 8):
        parts = np.concatenate([rms_norm(s, g, 1e-6) for s in np.split(h, P)])
        assert np.array_equal(parts, whole)


def test_shard_permutation_only_reorders_partials():
    """Renumbering the shards (permuting neuron blocks consistently in W1g,
    W1u and W2) permutes the partials and leaves their sum unchanged."""
    M, d, F, P = 12, 16, 32, 4
    x, partials, gamma, W1g, W1u, W2 = rand_case(M, d, F, P)
    out, _ = sptp_ffn_forward(x, partials, gamma, W1g, W1u, W2, P, P, 1e-6)
    perm = [2, 0, 3, 1]
    f = F // P
    idx = np.concatenate([np.arange(q * f, (q + 1) * f) for q in perm])
    outp, _ = sptp_ffn_forward(x, partials, gamma, W1g[idx], W1u[idx], W2[:, idx], P, P, 1e-6)
    for new, old in enumerate(perm):
        assert rel_max_error(outp[new], out[old]) < 1e-15
    assert rel_max_error(outp.sum(0), out.sum(0)) < 1e-13


# ------------------------------------------------------------ closed forms

def test_zero_gate_gives_zero_output():
    M, d, F, P = 8, 16, 32, 2
    x, partials, gamma, W1g, W1u, W2 = rand_case(M, d, F, P)
    out, h = sptp_ffn_forward(x, partials, gamma, np.zeros_like(W1g), W1u, W2, P, P, 1e-6)
    assert np.all(out == 0)
    assert rel_max_error(h, x + partials[0] + partials[1]) < 1e-15
    out, _ = sptp_ffn_forward(x, partials, np.zeros_like(gamma), W1g, W1u, W2, P, P, 1e-6)
    assert np.all(out == 0)


def test_rms_norm_closed_forms():
    rng = np.random.default_rng(5)
    h = rng.standard_normal((10, 33)) * 2
    eps = 0.3
    y = rms_norm(h, np.ones(33), eps)
    ms = np.mean(h * h, axis=1)
    assert np.max(np.abs(np.mean(y * y, axis=1) - ms / (ms + eps))) < 1e-14
    c = -1.7
    g = 1 + 0.1 * rng.standard_normal(33)
    yc = rms_norm(np.full((1, 33), c), g, eps)
    assert np.max(np.abs(yc[0] - c * g / math.sqrt(c * c + eps))) < 1e-14


def test_hand_derived_worked_example():
    fx = json.load(open(os.path.join(HERE, "golden", "worked_example_d2.json")))
    A = {k: np.array(fx[k], dtype=np.float64) for k in ("x", "partials", "gamma", "W1g", "W1u", "W2")}
    out, h = sptp_ffn_forward(A["x"], A["partials"], A["gamma"], A["W1g"], A["W1u"], A["W2"],
                              fx["P"], fx["chunks"], fx["eps"])
    assert np.max(np.abs(h - np.array(fx["expected_h"]))) < 1e-12
    assert np.max(np.abs(out - np.array(fx["expected_out"]))) < 1e-12


def test_brute_force_scalar_loops():
    """Tiny case with plain scalar loops over every index."""
    M, d, F, P, eps = 3, 4, 4, 2, 1e-6
    x, partials, gamma, W1g, W1u, W2 = rand_case(M, d, F, P, seed=9)
    out, h = sptp_ffn_forward(x, partials, gamma, W1g, W1u, W2, P, 1, eps)
    f = F // P
    for t in range(M):
        hh = [x[t][j] + sum(partials[p][t][j] for p in range(P)) for j in range(d)]
        ms = sum(v * v for v in hh) / d
        y = [hh[j] * gamma[j] / math.sqrt(ms + eps) for j in range(d)]
        for p in range(P):
            s = []
            for n in range(p * f, (p + 1) * f):
                a = sum(y[j] * W1g[n][j] for j in range(d))
                b = sum(y[j] * W1u[n][j] for j in range(d))
                s.append(a / (1 + math.exp(-a)) * b)
            for i in range(d):
                ref = sum(s[k] * W2[i][p * f + k] for k in range(f))
                assert abs(out[p][t][i] - ref) < 1e-12
        for j in range(d):
            assert abs(h[t][j] - hh[j]) < 1e-15


# ------------------------------------------------------------ Delayed TP

def tp_chain(x0, gamma, W1g, W1u, W2, P, L, eps):
    """L standard-TP boundaries chained through the oracle: the first starts
    from zero partials, each next one consumes the previous partials."""
    parts = np.zeros((P,) + x0.shape)
    x = x0
    for l in range(L):
        out, x = sptp_ffn_forward(x, parts, gamma[l], W1g[l], W1u[l], W2[l], P, P, eps)
        parts = out
    return x + parts.sum(0)


def dtp_case(M, d, F, P, L, seed=2):
    rng = np.random.default_rng(seed)
    x0 = rng.standard_normal((M, d))
    gamma = 1 + 0.1 * rng.standard_normal((L, d))
    W1g = rng.standard_normal((L, F, d)) / math.sqrt(d)
    W1u = rng.standard_normal((L, F, d)) / math.sqrt(d)
    W2 = rng.standard_normal((L, d, F)) / math.sqrt(d)
    return x0, gamma, W1g, W1u, W2


@pytest.mark.parametrize("flush", [0, 1])
@pytest.mark.parametrize("P", [2, 4])
def test_dtp_delta0_equals_standard_tp(P, flush):
    M, d, F, L = 8, 16, 32, 3
    x0, gamma, W1g, W1u, W2 = dtp_case(M, d, F, P, L)
    xs = np.stack([x0] * P)
    got = dtp_ffn_stack_forward(xs, gamma, W1g, W1u, W2, P, L, 0, flush, 1e-6)
    ref = tp_chain(x0, gamma, W1g, W1u, W2, P, L, 1e-6)
    for p in range(P):
        assert rel_max_error(got[p], ref) < 1e-12


@pytest.mark.parametrize("delta", [0, 1, 3])
def test_dtp_single_shard_is_tp_for_any_delay(delta):
    M, d, F, L = 8, 16, 32, 3
    x0, gamma, W1g, W1u, W2 = dtp_case(M, d, F, 1, L)
    got = dtp_ffn_stack_forward(x0[None], gamma, W1g, W1u, W2, 1, L, delta, 1, 1e-6)
    assert rel_max_error(got[0], tp_chain(x0, gamma, W1g, W1u, W2, 1, L, 1e-6)) < 1e-12


def _one_boundary(x, g, W1g, W1u, W2, P):
    """Per-shard partials of one module on input x (zero incoming partials)."""
    out, _ = sptp_ffn_forward(x, np.zeros((P,) + x.shape), g, W1g, W1u, W2, P, P, 1e-6)
    return out


@pytest.mark.parametrize("flush", [0, 1])
def test_dtp_delay_arrival_schedule(flush):
    """Modules with gamma = 0 produce zero partials, which isolates when a
    partial reaches a stream.  L=3, delta=1, modules 0 and 2 active: the
    other shard's module-0 partial must be in x_p before module 2 runs
    (0 + 1 + delta = 2), and the other shard's module-2 partial arrives only
    with the flush."""
    M, d, F, P, L = 6, 16, 32, 2, 3
    x0, gamma, W1g, W1u, W2 = dtp_case(M, d, F, P, L)
    gamma[1] = 0.0
    got = dtp_ffn_stack_forward(np.stack([x0] * P), gamma, W1g, W1u, W2, P, L, 1, flush, 1e-6)
    o0 = _one_boundary(x0, gamma[0], W1g[0], W1u[0], W2[0], P)
    x2 = x0 + o0[0] + o0[1]  # both shards hold the same stream before module 2
    o2 = _one_boundary(x2, gamma[2], W1g[2], W1u[2], W2[2], P)
    for p in range(P):
        q = 1 - p
        ref = x2 + o2[p] + (o2[q] if flush else 0.0)
        assert rel_max_error(got[p], ref) < 1e-12


@pytest.mark.parametrize("flush", [0, 1])
def test_dtp_delay_beyond_stack(flush):
    """delta >= L: no other-shard partial arrives inside the stack; only the
    flush adds them."""
    M, d, F, P, L = 6, 16, 32, 2, 2
    x0, gamma, W1g, W1u, W2 = dtp_case(M, d, F, P, L)
    gamma[1] = 0.0
    got = dtp_ffn_stack_forward(np.stack([x0] * P), gamma, W1g, W1u, W2, P, L, 2, flush, 1e-6)
    o0 = _one_boundary(x0, gamma[0], W1g[0], W1u[0], W2[0], P)
    for p in range(P):
        ref = x0 + o0[p] + (o0[1 - p] if flush else 0.0)
        assert rel_max_error(got[p], ref) < 1e-12


def test_dtp_row_subset_and_independent_streams():
    M, d, F, P, L = 10, 16, 32, 2, 3
    x0, gamma, W1g, W1u, W2 = dtp_case(M, d, F, P, L)
    xs = np.stack([x0, -0.5 * x0])
    full = dtp_ffn_stack_forward(xs, gamma, W1g, W1u, W2, P, L, 1, 1, 1e-6)
    rows = [1, 4, 9]
    sub = dtp_ffn_stack_forward(xs, gamma, W1g, W1u, W2, P, L, 1, 1, 1e-6, rows=rows)
    assert rel_max_error(sub, full[:, rows]) < 1e-13
    assert not np.allclose(full[0], full[1])


# ------------------------------------------------------------ synthetic inputs

def test_bf16_cast_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(4096) * 10 ** rng.uniform(-3, 3, 4096),
                        np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -1 - 2 ** -8])]).astype(np.float32)
    ours = synth._fp32_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_bits_to_f64(ours),
                          torch.from_numpy(v).to(torch.bfloat16).double().numpy())


def test_synthetic_inputs_are_seeded_and_shaped():
    cfg = synth.TINY_FP32
    a = synth.boundary_inputs(cfg)
    b = synth.boundary_inputs(cfg)
    for k in a:
        assert np.array_equal(a[k], b[k])
    assert a["partials"].shape == (2, 64, 128) and a["W2"].shape == (128, 512)
    assert a["x"].dtype == np.float32
    # distribution checks: weight std 1/sqrt(d), gamma around 1
    assert abs(a["W1g"].std() - 128 ** -0.5) < 0.01
    assert abs(a["gamma"].mean() - 1.0) < 0.05
    # block-parallel drawing does not depend on the block split
    big = synth.draw((3, synth.BLOCK // 2 + 5), 1.0, 0.0, "bf16", 0, 7)
    again = synth.draw((3, synth.BLOCK // 2 + 5), 1.0, 0.0, "bf16", 0, 7)
    assert np.array_equal(big, again)


# ------------------------------------------------------------ neuron-permutation shard maps

def _perms(L, F, rng, kind):
    out = []
    for _ in range(L):
        if kind == "identity":
            out.append(np.arange(F))
        elif kind == "within":
            # reorder neurons inside each of the 2 contiguous shards only
            f = F // 2
            out.append(np.concatenate([rng.permutation(f), f + rng.permutation(f)]))
        else:
            out.append(rng.permutation(F))
    return out


def test_permutation_of_a_single_ffn_moves_rows_and_columns_together():
    rng = np.random.default_rng(4)
    W1g, W1u, W2 = rng.standard_normal((8, 3)), rng.standard_normal((8, 3)), rng.standard_normal((3, 8))
    perm = rng.permutation(8)
    a, b, c = oracle.permute_ffn_neurons(W1g, W1u, W2, perm)
    for i in range(8):
        assert np.array_equal(a[i], W1g[perm[i]]) and np.array_equal(b[i], W1u[perm[i]])
        assert np.array_equal(c[:, i], W2[:, perm[i]])
    with pytest.raises(ValueError):
        oracle.permute_ffn_neurons(W1g, W1u, W2, [0] * 8)


@pytest.mark.parametrize("kind", ["identity", "random"])
def test_tp_is_invariant_to_any_neuron_permutation(kind):
    """delta = 0 sums every neuron's contribution, so renumbering neurons
    before sharding cannot change the result (the symmetry DTP breaks)."""
    M, d, F, P, L = 6, 16, 32, 2, 3
    x0, gamma, W1g, W1u, W2 = dtp_case(M, d, F, P, L)
    xs = np.stack([x0] * P)
    ref = dtp_ffn_stack_forward(xs, gamma, W1g, W1u, W2, P, L, 0, 1, 1e-6)
    got = oracle.dtp_ffn_stack_forward_permuted(xs, gamma, W1g, W1u, W2, _perms(L, F, np.random.default_rng(1),
                                                kind), P, L, 0, 1, 1e-6)
    assert rel_max_error(got, ref) < 1e-12


@pytest.mark.parametrize("delta", [1, 2])
def test_dtp_is_invariant_to_reordering_within_shards(delta):
    M, d, F, P, L = 6, 16, 32, 2, 3
    x0, gamma, W1g, W1u, W2 = dtp_case(M, d, F, P, L)
    xs = np.stack([x0] * P)
    ref = dtp_ffn_stack_forward(xs, gamma, W1g, W1u, W2, P, L, delta, 0, 1e-6)
    got = oracle.dtp_ffn_stack_forward_permuted(xs, gamma, W1g, W1u, W2, _perms(L, F, np.random.default_rng(2),
                                                "within"), P, L, delta, 0, 1e-6)
    assert rel_max_error(got, ref) < 1e-12


def test_dtp_depends_on_which_neurons_share_a_shard():
    """With delayed partials a cross-shard renumbering changes the streams:
    the sharding is a modelling decision."""
    M, d, F, P, L = 6, 16, 32, 2, 3
    x0, gamma, W1g, W1u, W2 = dtp_case(M, d, F, P, L)
    xs = np.stack([x0] * P)
    ref = dtp_ffn_stack_forward(xs, gamma, W1g, W1u, W2, P, L, 1, 0, 1e-6)
    got = oracle.dtp_ffn_stack_forward_permuted(xs, gamma, W1g, W1u, W2, _perms(L, F, np.random.default_rng(3),
                                                "random"), P, L, 1, 0, 1e-6)
    assert rel_max_error(got, ref) > 1e-3


# ------------------------------------------------------------ attention-side boundary

def test_attn_qkv_boundary_unsharded_matches_torch_functional():
    M, d, N = 12, 32, 48
    rng = np.random.default_rng(21)
    x, parts = rng.standard_normal((M, d)), rng.standard_normal((2, M, d))
    gamma = 1 + 0.1 * rng.standard_normal(d)
    W = rng.standard_normal((N, d)) / math.sqrt(d)
    qkv2, h2 = oracle.attn_qkv_boundary(x, parts, gamma, W, 2, 2, 1e-6)
    T = torch.from_numpy
    y = Fn.rms_norm(T(x) + T(parts).sum(0), (d,), T(gamma), 1e-6)
    ref = Fn.linear(y, T(W)).numpy()
    assert rel_max_error(np.concatenate([qkv2[0], qkv2[1]], axis=1), ref) < 1e-13
    assert rel_max_error(h2, (T(x) + T(parts).sum(0)).numpy()) < 1e-15


def test_rowparallel_projection_partials_sum_to_the_full_linear():
    rng = np.random.default_rng(22)
    P, M, K, d = 4, 10, 64, 24
    a = rng.standard_normal((P, M, K // P))
    W = rng.standard_normal((d, K))
    out = oracle.rowparallel_projection(a, W, P)
    full = Fn.linear(torch.from_numpy(np.concatenate(list(a), axis=1)), torch.from_numpy(W)).numpy()
    assert rel_max_error(out.sum(0), full) < 1e-13
    W0 = W.copy()
    W0[:, K // P:2 * K // P] = 0
    assert np.all(oracle.rowparallel_projection(a, W0, P)[1] == 0)


def test_attn_qkv_boundary_chunking_and_zero_weights():
    rng = np.random.default_rng(23)
    M, d, N, P = 16, 24, 32, 2
    x, parts = rng.standard_normal((M, d)), rng.standard_normal((P, M, d))
    gamma = 1 + 0.1 * rng.standard_normal(d)
    W = rng.standard_normal((N, d))
    a, ha = oracle.attn_qkv_boundary(x, parts, gamma, W, P, P, 1e-6)
    b, hb = oracle.attn_qkv_boundary(x, parts, gamma, W, P, 8, 1e-6)
    assert rel_max_error(a, b) < 1e-14 and rel_max_error(ha, hb) == 0.0
    z, _ = oracle.attn_qkv_boundary(x, parts, gamma, np.zeros_like(W), P, P, 1e-6)
    assert np.all(z == 0)


# ---------------------------------------------------------------- the parity metric
# rel_max_error is the comparison behind every parity assertion, so it is
# pinned to hand-computed values: max_i |got_i - ref_i| / max_i |ref_i|.

def test_rel_max_error_closed_form():
    assert rel_max_error(np.array([1.0, 2.0]), np.array([1.0, 4.0])) == 0.5
    # a 2-D tensor: the max runs over every element
    assert rel_max_error(np.array([[1.0, 2.0], [3.0, 4.5]]), np.array([[1.0, 2.0], [3.0, 5.0]])) == 0.1


def test_rel_max_error_takes_the_absolute_difference():
    # the largest error is negative (got below ref); a signed max would say 0
    assert rel_max_error(np.array([0.0, 10.0]), np.array([3.0, 10.0])) == 0.3
    # and positive (got above ref); a max of (ref - got) would say 0
    assert rel_max_error(np.array([5.0, 10.0]), np.array([3.0, 10.0])) == 0.2
    # a negative error larger in magnitude than a positive one
    assert rel_max_error(np.array([1.5, 6.0]), np.array([1.0, 10.0])) == 0.4


def test_rel_max_error_normalises_by_the_reference():
    # by max|ref| = 2, not by max|got| = 1
    assert rel_max_error(np.array([0.0, 1.0]), np.array([0.0, 2.0])) == 0.5
    # by max|ref| = 4, not by max(ref) = 1 (the largest reference is negative)
    assert rel_max_error(np.array([-4.0, 2.0]), np.array([-4.0, 1.0])) == 0.25
    # symmetric in sign: negating both changes nothing
    assert rel_max_error(-np.array([-4.0, 2.0]), -np.array([-4.0, 1.0])) == 0.25


def test_rel_max_error_is_a_max_not_a_mean():
    ref = np.ones(1001)
    got = ref.copy()
    got[517] += 0.5
    assert rel_max_error(got, ref) == 0.5


def test_rel_max_error_pairs_elements_by_index():
    # the same multiset of values in another order is an error of 2 / 3
    assert rel_max_error(np.array([1.0, 2.0, 3.0]), np.array([3.0, 2.0, 1.0])) == pytest.approx(2.0 / 3.0, abs=0)


def test_rel_max_error_zero_cases():
    assert rel_max_error(np.zeros(5), np.zeros(5)) == 0.0
    # an all-zero reference: the absolute error
    assert rel_max_error(np.array([0.0, -0.25, 0.0]), np.zeros(3)) == 0.25
    assert rel_max_error(np.zeros((0, 4)), np.zeros((0, 4))) == 0.0
    assert rel_max_error(np.array([2.0, 3.0]), np.array([2.0, 3.0])) == 0.0


def test_rel_max_error_fails_non_finite_outputs():
    ref = np.array([1.0, 2.0, 3.0])
    for bad in (np.nan, np.inf, -np.inf):
        got = ref.copy()
        got[1] = bad
        err = rel_max_error(got, ref)
        assert err == math.inf and not err <= 2e-2
    # inf sorts above every finite error, wherever it sits in a list
    assert max([rel_max_error(np.array([np.nan]), np.array([1.0])), 0.5]) == math.inf
    with pytest.raises(ValueError):
        rel_max_error(ref, np.array([1.0, np.nan, 3.0]))


def test_rel_max_error_rejects_shape_mismatch():
    ref = np.arange(12.0).reshape(4, 3)
    with pytest.raises(ValueError):
        rel_max_error(ref[:1], ref)          # one row against a whole tensor
    with pytest.raises(ValueError):
        rel_max_error(ref, ref.T)
    with pytest.raises(ValueError):
        rel_max_error(ref.reshape(-1), ref)
