"""Oracle for the fp8 (E4M3) variant of the SP-TP FFN boundary.

TEST INFRASTRUCTURE ONLY: a plain CPU statement of what the fp8 path of the
CUDA library computes (float64, with fp32 where a value decides a code).  Only the tests, the package smoke check and the
benchmark's CPU legs may import it; the product path never calls it.

Source (web page; title and section): "[Feature] Async Tensor Parallelism for
Archon Engine", section "Additional Information" names fp8 (MXFP8) linear
layers inside tensor-parallel blocks as a known limitation; it fixes no
scaling recipe.  Readings taken here, each also listed in the repository's
design notes:

* Every linear layer's input is the bf16 activation (y after RMSNorm, s after
  SwiGLU), as in a bf16 model whose linears run in fp8; the layer quantises
  that bf16 tensor itself.
* Quantisation is row-wise with power-of-two scales: a row r of a [R][K]
  operand (K the reduction axis) gets e_r = the smallest integer >= -126 with
  max_k |a[r][k]| <= 448 * 2^e_r; its codes are q[r][k] = RNE_E4M3(a[r][k] *
  2^-e_r).  A power of two makes a * 2^-e exact, so any implementation that
  quantises the same bf16 value takes the same decision.  (MX formats share
  one power-of-two scale per 32 elements; one scale per row is the plainest
  scaling that a GEMM epilogue can undo exactly.)
* Scale axes: y per token row over d; W1g and W1u per output neuron (row of
  [F][d]) over d; s per token row over the shard's F/P neurons; W2 per output
  feature n and shard p over W2[n][F_p].  Shard p's scales are its own: a
  real TP rank quantises its local shard.
* A GEMM of quantised operands is sum_k qa qb times 2^(e_a + e_b); gate and
  up values are dequantised before SwiGLU.
* Where a value decides a code -- y and s, whose bf16 roundings are then
  quantised to E4M3 -- this oracle computes it in the precision the kernels
  use, fp32 (the sums of partials, the mean square and the norm of y; the
  gate/up accumulations, SwiGLU and the down accumulation), so that both
  sides take each quantisation decision in the same precision.  A float64
  value next to a rounding boundary could otherwise fall on the other side
  of it, and one E4M3 code of s moves a term of a K-long down-projection sum
  by up to an eighth.  The fp32 sums run in numpy's order, not the kernels';
  the products of E4M3 values are exact in fp32.

Parity status: round_bf16 and round_e4m3 are pinned against PyTorch's casts;
e4m3_row_exponent by closed forms and minimality; the composition by a
hand-derived worked example, exact power-of-two equivariances and an error
bound against the float64 boundary.
"""
from __future__ import annotations

import numpy as np


E4M3_MAX = 448.0
MIN_EXPONENT = -126


def _round_to_grid(v: np.ndarray, significant_bits: int, min_normal_exp: int) -> np.ndarray:
    """Round-to-nearest-even onto a binary floating-point grid with
    `significant_bits` bits of significand (implicit bit included) and
    smallest normal binade [2^min_normal_exp, 2^(min_normal_exp+1)); below it
    the spacing stays that of the smallest binade (subnormals)."""
    v = np.asarray(v, dtype=np.float64)
    _, ex = np.frexp(v)  # v = m * 2^ex, 0.5 <= |m| < 1, so the leading bit is 2^(ex-1)
    lead = np.maximum(ex - 1, min_normal_exp)
    ulp = np.ldexp(1.0, lead - (significant_bits - 1))
    return np.rint(v / ulp) * ulp


def round_bf16(v) -> np.ndarray:
    """Round to bfloat16 (8 significant bits, float32's exponent range),
    nearest-even; values past the largest finite bf16 become +-inf."""
    r = _round_to_grid(v, 8, -126)
    big = np.abs(r) >= 2.0 ** 128
    return np.where(big, np.copysign(np.inf, r), r)


def round_e4m3(v) -> np.ndarray:
    """Round to OCP E4M3 (4 significant bits, exponent bias 7, smallest normal
    2^-6, subnormal spacing 2^-9, largest finite 448), nearest-even.  Inputs
    whose rounding leaves [-448, 448] are outside the domain used here."""
    r = _round_to_grid(v, 4, -6)
    if np.any(np.abs(r) > E4M3_MAX):
        raise ValueError("value outside the E4M3 range")
    return r


def e4m3_encode(v) -> np.ndarray:
    """Byte encoding of values on the E4M3 grid: sign << 7 | exponent field
    << 3 | mantissa, exponent field 0 for zero and subnormals."""
    v = np.asarray(v, dtype=np.float64)
    if not np.array_equal(round_e4m3(v), v):
        raise ValueError("value not on the E4M3 grid")
    a = np.abs(v)
    sign = np.signbit(v).astype(np.int64)
    _, ex = np.frexp(a)
    lead = ex - 1
    normal = a >= 2.0 ** -6
    field = np.where(normal, lead + 7, 0)
    mant = np.where(normal, np.ldexp(a, -lead) * 8 - 8, a * 2.0 ** 9)
    code = (sign << 7) | (field.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    return code.astype(np.uint8)


def e4m3_row_exponent(amax) -> np.ndarray:
    """Smallest integer e >= -126 with amax <= 448 * 2^e (elementwise)."""
    amax = np.asarray(amax, dtype=np.float64)
    e = np.full(amax.shape, MIN_EXPONENT, dtype=np.int64)
    # count upwards from -126 until 448 * 2^e covers amax (every row at once)
    while True:
        short = amax > E4M3_MAX * np.ldexp(1.0, e)
        if not np.any(short):
            return e
        e = e + short


def quantize_rows_e4m3(a):
    """Row-wise power-of-two-scaled E4M3 quantisation over the last axis.
    Returns (q, e): q the E4M3 values (float64, on the grid), e the int
    exponents, a ~= q * 2^e[..., None]."""
    a = np.asarray(a, dtype=np.float64)
    e = e4m3_row_exponent(np.max(np.abs(a), axis=-1) if a.shape[-1] else np.zeros(a.shape[:-1]))
    q = round_e4m3(a * np.ldexp(1.0, -e)[..., None])
    return q, e


def quantize_ffn_weights(W1g, W1u, W2, P: int):
    """The fp8 weights of one FFN: W1g/W1u per neuron row over d, W2 per
    (output feature n, shard p) over W2[n][F_p].  Returns
    (qg, eg, qu, eu, q2, e2) with e2 of shape [d, P]."""
    W1g = np.asarray(W1g, dtype=np.float64)
    W1u = np.asarray(W1u, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    d, F = W2.shape
    f = F // P
    qg, eg = quantize_rows_e4m3(W1g)
    qu, eu = quantize_rows_e4m3(W1u)
    q2, e2 = quantize_rows_e4m3(W2.reshape(d, P, f))
    return qg, eg, qu, eu, q2.reshape(d, F), e2


def _f32(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float32)


def _gemm_f32(qa, ea, qb, eb) -> np.ndarray:
    """(sum_k qa[r][k] qb[c][k]) * 2^ea[r] * 2^eb[c] in fp32: the products of
    E4M3 values are exact, the sum is an fp32 sum, and each scale is a power
    of two applied as an fp32 multiplication (row scale first).  Each row is
    its own matrix-vector product, so a row's result does not depend on which
    other rows are evaluated with it (row samples equal the full result)."""
    qa32, qb32 = _f32(qa), _f32(qb)
    acc = np.zeros((qa32.shape[0], qb32.shape[0]), dtype=np.float32)
    for r in range(qa32.shape[0]):
        acc[r] = qb32 @ qa32[r]
    return (acc * _f32(np.ldexp(1.0, ea))[:, None]) * _f32(np.ldexp(1.0, eb))[None, :]


def _silu_f32(a: np.ndarray) -> np.ndarray:
    """silu(a) = a / (1 + e^-a) in fp32 (e^-a overflowing to inf gives -0)."""
    with np.errstate(over="ignore"):
        return a / (np.float32(1.0) + np.exp(-a))


def shard_ffn_fp8(y, qw, P: int, p: int, return_intermediates: bool = False):
    """Shard p's fp8 gate/up GEMM, SwiGLU and fp8 down GEMM on bf16 rows y
    [R][d]; qw = quantize_ffn_weights(...).  The GEMMs accumulate in fp32 and
    SwiGLU runs in fp32, so that s -- whose bf16 rounding decides the E4M3
    codes of the down projection's input -- is computed in the kernels'
    precision.  Returns the partial [R][d] (float64 holding the fp32 values,
    before the output's bf16 rounding)."""
    qg, eg, qu, eu, q2, e2 = qw
    F = qg.shape[0]
    f = F // P
    n = slice(p * f, (p + 1) * f)
    qy, ey = quantize_rows_e4m3(y)
    a = _gemm_f32(qy, ey, qg[n], eg[n])
    b = _gemm_f32(qy, ey, qu[n], eu[n])
    s = round_bf16((_silu_f32(a) * b).astype(np.float64))
    qs, es = quantize_rows_e4m3(s)
    out = _gemm_f32(qs, es, q2[:, n], e2[:, p]).astype(np.float64)
    if return_intermediates:
        return out, dict(qy=qy, ey=ey, a=a.astype(np.float64), b=b.astype(np.float64), s=s, qs=qs, es=es)
    return out


def boundary_rows_fp32(x, partials, gamma, eps):
    """h = x + (partials[0] + partials[1] + ...) and the bf16 activation
    y = bf16((h * gamma) * 1 / sqrt(mean(h^2) + eps)), in fp32 (the partial sum
    and the residual add, the mean square, the norm), as the kernels compute
    the y that the gate/up linear quantises.  Returns (h, y) as float64."""
    r = np.zeros(np.shape(x), dtype=np.float32)
    for q in range(partials.shape[0]):
        r = r + _f32(partials[q])
    h = _f32(x) + r
    ms = np.sum(h * h, axis=-1, dtype=np.float32) / np.float32(h.shape[-1])
    inv = np.float32(1.0) / np.sqrt(ms + np.float32(eps))
    y = round_bf16(((h * _f32(gamma)) * inv[:, None]).astype(np.float64))
    return h.astype(np.float64), y


def sptp_ffn_forward_fp8(x, partials, gamma, W1g, W1u, W2, P: int, chunks: int, eps: float, rows=None):
    """The SP-TP FFN boundary with fp8 linear layers: per chunk the P partials
    are summed, the residual added and the sum RMS-normalised (in fp32,
    boundary_rows_fp32); y is the bf16 activation; every shard runs
    shard_ffn_fp8 on it.  Arguments and return
    value as in the float64 boundary: (out [P, R, d], h [R, d])."""
    M, d = x.shape
    F = W1g.shape[0]
    if partials.shape[0] != P or F % P != 0 or chunks < 1 or M % chunks != 0:
        raise ValueError("bad shape")
    qw = quantize_ffn_weights(W1g, W1u, W2, P)
    sel = np.arange(M) if rows is None else np.asarray(rows)
    out = np.zeros((P, len(sel), d))
    h_out = np.zeros((len(sel), d))
    m = M // chunks
    for c in range(chunks):
        pos = np.nonzero((sel >= c * m) & (sel < (c + 1) * m))[0]
        if len(pos) == 0:
            continue
        r_idx = sel[pos]
        h, y = boundary_rows_fp32(x[r_idx], partials[:, r_idx, :], gamma, eps)
        h_out[pos] = h
        for p in range(P):
            out[p, pos] = shard_ffn_fp8(y, qw, P, p)
    return out, h_out
