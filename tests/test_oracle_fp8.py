"""CPU pins of the fp8 oracle: the roundings against PyTorch's casts, the
scale rule by closed forms, the composition by a hand-derived example,
rigorous per-element quantisation bounds and exact power-of-two
equivariances (each would fail under a dropped rounding, a wrong scale axis
or index, or a scale applied the wrong way round)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_oracle as f8
from sequence_tensor_transformer_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _f32_exact(v):
    # PyTorch casts float64 -> float8 through float32; feed values float32
    # holds exactly so that both sides round once
    return np.asarray(v, dtype=np.float32).astype(np.float64)


def _torch_e4m3(v):
    return torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn)


def test_round_e4m3_matches_torch_cast():
    rng = np.random.default_rng(0)
    v = np.concatenate([np.linspace(-448, 448, 100001), np.geomspace(2.0 ** -14, 448, 40001),
                        -np.geomspace(2.0 ** -14, 448, 40001), rng.uniform(-1, 1, 20000) * 2.0 ** -7])
    # ties between grid values (to even) in a normal binade and among the
    # subnormals, the overflow tie at 464 and signed zeros
    v = np.concatenate([v, [0.0, -0.0, 84.0, -84.0, 42.0, 464.0 - 2 ** -6, 2.0 ** -10, 3 * 2.0 ** -10]])
    v = _f32_exact(v)
    r = f8.round_e4m3(v)
    t = _torch_e4m3(v).to(torch.float64).numpy()
    assert np.array_equal(r, t)
    assert np.array_equal(np.signbit(r), np.signbit(t))


def test_e4m3_grid_fixed_points_and_encoding():
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = ~np.isnan(vals)
    assert finite.sum() == 254  # S.1111.111 is NaN, nothing is infinite
    v = vals[finite]
    assert np.array_equal(f8.round_e4m3(v), v)
    assert np.array_equal(f8.e4m3_encode(v), codes[finite])
    pos = np.unique(np.abs(v))
    assert pos.max() == 448.0 and pos[1] == 2.0 ** -9 and len(pos) == 127
    # exponent fields 1..15 give 15 normal binades of 8 values from 2^-6
    # upward, less the NaN code at the top; 7 subnormals below; and zero
    assert np.sum(pos >= 2.0 ** -6) == 15 * 8 - 1 and np.sum((pos > 0) & (pos < 2.0 ** -6)) == 7
    with pytest.raises(ValueError):
        f8.round_e4m3(np.array([480.0]))
    with pytest.raises(ValueError):
        f8.e4m3_encode(np.array([0.3]))


def test_round_bf16_matches_torch_cast():
    rng = np.random.default_rng(1)
    w = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.uniform(-40, 37, 100000),
                        np.geomspace(1e-45, 3e38, 10000), [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]])
    w = _f32_exact(w)
    r = f8.round_bf16(w)
    t = torch.tensor(w, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(r, t)
    # the synthetic-input cast agrees too
    assert np.array_equal(f8.round_bf16(w[:1000]), synth.to_f64(synth._cast(w[:1000], "bf16"), "bf16"))


def test_row_exponent_closed_forms_and_minimality():
    e = f8.e4m3_row_exponent
    assert e(448.0) == 0 and e(448.0 * (1 + 2 ** -20)) == 1 and e(224.0) == -1 and e(224.5) == 0
    assert e(1.0) == -8 and e(1.75) == -8 and e(1.7500001) == -7
    assert e(0.0) == -126 and e(2.0 ** -200) == -126
    rng = np.random.default_rng(2)
    amax = 10.0 ** rng.uniform(-30, 30, 5000)
    ex = e(amax)
    assert np.all(amax <= 448.0 * np.ldexp(1.0, ex))
    assert np.all(amax > 448.0 * np.ldexp(1.0, ex - 1))


def test_quantize_rows_matches_torch_cast_with_row_scales():
    rng = np.random.default_rng(3)
    a = synth.to_f64(synth._cast(rng.standard_normal((40, 96)) * 10.0 ** rng.uniform(-6, 6, (40, 1)), "bf16"),
                     "bf16")
    a[3] = 0.0
    a[5, :] = a[5, :] * 0 + 2.0 ** -130  # tiny row: clamped exponent
    q, e = f8.quantize_rows_e4m3(a)
    assert e.shape == (40,) and e[3] == -126 and e[5] == -126
    t = _torch_e4m3(a * np.ldexp(1.0, -e)[:, None]).to(torch.float64).numpy()
    assert np.array_equal(q, t)
    m = np.max(np.abs(q), axis=1)
    live = (e > -126)
    # the row maximum lands in (224, 448] before rounding: at least 224 after
    assert np.all(m[live] >= 224.0) and np.all(m <= 448.0)
    # per-row: scaling one row by 2^k shifts only that row's exponent
    a2 = a.copy()
    a2[7] *= 2.0 ** 5
    q2, e2 = f8.quantize_rows_e4m3(a2)
    assert np.array_equal(q2, q) and e2[7] == e[7] + 5 and np.array_equal(np.delete(e2, 7), np.delete(e, 7))


def test_fp8_hand_derived_worked_example():
    fx = json.load(open(os.path.join(HERE, "golden", "fp8_worked_example_d2.json")))
    A = {k: np.array(fx[k], dtype=np.float64) for k in ("x", "partials", "gamma", "W1g", "W1u", "W2")}
    out, h = f8.sptp_ffn_forward_fp8(A["x"], A["partials"], A["gamma"], A["W1g"], A["W1u"], A["W2"], fx["P"],
                                     fx["chunks"], fx["eps"])
    assert np.array_equal(h, np.array(fx["expected_h"]))
    assert np.array_equal(out, np.array(fx["expected_out"]))
    _, eg, _, eu, _, e2 = f8.quantize_ffn_weights(A["W1g"], A["W1u"], A["W2"], fx["P"])
    ex = fx["expected_weight_exponents"]
    assert eg.tolist() == ex["W1g"] and eu.tolist() == ex["W1u"] and e2.tolist() == ex["W2"]


def _rand_ffn(seed, R=24, d=64, F=96, P=2):
    rng = np.random.default_rng(seed)
    y = f8.round_bf16(rng.standard_normal((R, d)))
    W1g = f8.round_bf16(rng.standard_normal((F, d)) / np.sqrt(d) * 2.0 ** rng.integers(-3, 4, (F, 1)))
    W1u = f8.round_bf16(rng.standard_normal((F, d)) / np.sqrt(d))
    W2 = f8.round_bf16(rng.standard_normal((d, F)) / np.sqrt(F) * 2.0 ** rng.integers(-3, 4, (d, 1)))
    return y, W1g, W1u, W2, P


def _dequant_bound(a, qa, ea, b, qb, eb):
    """Rigorous bound on |(qa 2^ea)(qb 2^eb)^T - a b^T| per element: each
    E4M3 rounding errs by at most 2^-4 relative (normal) or half the
    subnormal spacing, 2^-10 * 2^e (absolute)."""
    ta = np.ldexp(1.0, ea)[:, None] * 2.0 ** -10
    tb = np.ldexp(1.0, eb)[:, None] * 2.0 ** -10
    da = 2.0 ** -4 * np.abs(a) + ta
    db = 2.0 ** -4 * np.abs(b) + tb
    return da @ np.abs(b).T + np.abs(a) @ db.T + da @ db.T


@pytest.mark.parametrize("seed", [0, 1])
def test_fp8_shard_gemms_within_quantisation_bounds(seed):
    y, W1g, W1u, W2, P = _rand_ffn(seed)
    qw = f8.quantize_ffn_weights(W1g, W1u, W2, P)
    qg, eg, qu, eu, q2, e2 = qw
    f = W1g.shape[0] // P
    for p in range(P):
        n = slice(p * f, (p + 1) * f)
        out, it = f8.shard_ffn_fp8(y, qw, P, p, return_intermediates=True)
        exact_a = y @ W1g[n].T
        assert np.all(np.abs(it["a"] - exact_a) <= _dequant_bound(y, it["qy"], it["ey"], W1g[n], qg[n], eg[n]))
        assert np.all(np.abs(it["b"] - y @ W1u[n].T) <= _dequant_bound(y, it["qy"], it["ey"], W1u[n], qu[n],
                                                                        eu[n]))
        # the fp8 result is not the exact one (the bound is not vacuous)
        assert np.max(np.abs(it["a"] - exact_a)) > 0
        # s is the bf16 activation of SwiGLU(a, b)
        s_exact = oracle.silu(it["a"]) * it["b"]
        assert np.array_equal(f8.round_bf16(it["s"]), it["s"])
        # one bf16 rounding: at most 2^-8 relative (8 significant bits)
        assert np.all(np.abs(it["s"] - s_exact) <= 2.0 ** -8 * np.abs(s_exact) + 1e-300)
        # s is scaled per token row over the shard's neurons
        assert np.array_equal(it["es"], f8.e4m3_row_exponent(np.max(np.abs(it["s"]), axis=1)))
        W2p = W2[:, n]
        assert np.all(np.abs(out - it["s"] @ W2p.T) <= _dequant_bound(it["s"], it["qs"], it["es"], W2p, q2[:, n],
                                                                       e2[:, p]))


def test_fp8_power_of_two_equivariances():
    y, W1g, W1u, W2, P = _rand_ffn(5)
    f = W1g.shape[0] // P
    base = [f8.shard_ffn_fp8(y, f8.quantize_ffn_weights(W1g, W1u, W2, P), P, p, True) for p in range(P)]
    # a gate row times 2^3: that neuron's gate value times 2^3, nothing else
    g2 = W1g.copy()
    g2[5] *= 8.0
    r = f8.shard_ffn_fp8(y, f8.quantize_ffn_weights(g2, W1u, W2, P), P, 0, True)[1]
    assert np.array_equal(r["a"][:, 5], 8.0 * base[0][1]["a"][:, 5])
    assert np.array_equal(np.delete(r["a"], 5, axis=1), np.delete(base[0][1]["a"], 5, axis=1))
    # a token row times 2^-2: that row's gate/up values times 2^-2
    y2 = y.copy()
    y2[3] *= 0.25
    r = f8.shard_ffn_fp8(y2, f8.quantize_ffn_weights(W1g, W1u, W2, P), P, 1, True)[1]
    assert np.array_equal(r["b"][3], 0.25 * base[1][1]["b"][3])
    assert np.array_equal(np.delete(r["b"], 3, axis=0), np.delete(base[1][1]["b"], 3, axis=0))
    # W2[n][F_1] times 2^4: shard 1's feature n times 2^4; shard 0 unchanged
    # (each shard's W2 segment has its own scale)
    w2 = W2.copy()
    w2[7, f:] *= 16.0
    qw = f8.quantize_ffn_weights(W1g, W1u, w2, P)
    o0, o1 = f8.shard_ffn_fp8(y, qw, P, 0), f8.shard_ffn_fp8(y, qw, P, 1)
    assert np.array_equal(o0, base[0][0])
    assert np.array_equal(o1[:, 7], 16.0 * base[1][0][:, 7])
    assert np.array_equal(np.delete(o1, 7, axis=1), np.delete(base[1][0], 7, axis=1))


def test_fp8_boundary_tracks_the_float64_boundary():
    cfg = synth.BoundaryConfig("fp8_pin", 64, 256, 512, 2, 2, "bf16", True, seed=11)
    inp = {k: synth.to_f64(v, "bf16") for k, v in synth.boundary_inputs(cfg).items()}
    args = (inp["x"], inp["partials"], inp["gamma"], inp["W1g"], inp["W1u"], inp["W2"], cfg.P, cfg.chunks, cfg.eps)
    out8, h8 = f8.sptp_ffn_forward_fp8(*args)
    out, h = oracle.sptp_ffn_forward(*args)
    # h: the fp32 sum of bf16 values, within fp32 rounding of the exact sum
    assert oracle.rel_max_error(h8, h) < 2.0 ** -22
    # two chained E4M3 GEMMs: a few per cent of the output's range, far
    # below what a misplaced scale (a factor of 2 or more) gives
    for p in range(cfg.P):
        err = oracle.rel_max_error(out8[p], out[p])
        assert 1e-4 < err < 0.08, (p, err)
    # chunking and row subsets do not change the fp8 result
    out1, _ = f8.sptp_ffn_forward_fp8(*args[:-2], 1, cfg.eps)
    assert np.array_equal(out1, out8)
    rows = np.array([0, 5, 63, 17])
    outr, hr = f8.sptp_ffn_forward_fp8(*args, rows=rows)
    assert np.array_equal(outr, out8[:, rows]) and np.array_equal(hr, h8[rows])


def test_fp8_decisions_are_taken_in_fp32():
    """The values that decide a code -- y, and s from the fp32 gate/up
    accumulations -- are the kernels' fp32 ones: y equals the bf16 rounding
    of (h * gamma) * (1 / sqrt(mean h^2 + eps)) evaluated with every operation
    rounded to fp32, and a, b hold fp32 values."""
    cfg = synth.BoundaryConfig("fp8_f32", 16, 64, 128, 2, 2, "bf16", True, seed=3)
    inp = {k: synth.to_f64(v, "bf16") for k, v in synth.boundary_inputs(cfg).items()}
    h, y = f8.boundary_rows_fp32(inp["x"], inp["partials"], inp["gamma"], cfg.eps)
    # every fp32 step, written out element by element for one row
    f32 = np.float32
    row = 5
    hr = [f32(inp["x"][row, j]) + (f32(0) + f32(inp["partials"][0, row, j]) + f32(inp["partials"][1, row, j]))
          for j in range(cfg.d)]
    ss = f32(0)
    for v in hr:
        ss = f32(ss + f32(v * v))
    inv = f32(1) / np.sqrt(f32(ss / f32(cfg.d)) + f32(cfg.eps))
    yr = f8.round_bf16(np.array([float(f32(f32(v * f32(inp["gamma"][j])) * inv)) for j, v in enumerate(hr)]))
    assert np.array_equal(h[row], np.array([float(v) for v in hr]))
    # the mean square is an fp32 sum in another order: y agrees within one bf16 step where it differs at all
    assert np.max(np.abs(y[row] - yr)) <= 2.0 ** -7 * np.max(np.abs(yr))
    assert np.mean(y[row] == yr) > 0.9
    qw = f8.quantize_ffn_weights(inp["W1g"], inp["W1u"], inp["W2"], cfg.P)
    _, it = f8.shard_ffn_fp8(y, qw, cfg.P, 1, return_intermediates=True)
    for k in ("a", "b"):
        assert np.array_equal(it[k].astype(np.float32).astype(np.float64), it[k])
