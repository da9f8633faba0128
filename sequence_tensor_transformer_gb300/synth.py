"""Seeded synthetic inputs for the SP-TP FFN boundary and the Delayed-TP stack.

This module holds the input recipe only -- shapes, distributions, seeds and
the cast to the storage format.  It contains none of the method's arithmetic
and is the single piece shared by the CUDA path's callers and the oracle.

Recipe (the workloads of the SP-TP FFN boundary; init distributions as the
workload descriptions give them):

* every tensor is drawn from N(0, 1) in float64 and scaled by its standard
  deviation: activations x and row-parallel partials N(0, 1); gate/up weights
  N(0, 1/d); down weights N(0, 1/F) for the bf16 boundary workloads and
  N(0, 1/d) for the fp32 one and the Delayed-TP stack; gamma = 1 + 0.1 N(0, 1);
* a tensor is cut into blocks of ``BLOCK`` elements and block ``b`` of tensor
  ``t`` comes from ``numpy.random.default_rng([seed, t, b])``, so the values do
  not depend on how many threads draw them;
* the float64 draw is then cast to the storage format: fp32 by round to
  nearest even, bf16 by rounding that fp32 value once more to nearest even
  (kept as raw uint16 bit patterns, since numpy has no bf16).  Both sides of a
  comparison read the cast values.

Tensor ids fix the draw identity: x=0, partials=1, gamma=2, W1g=3, W1u=4,
W2=5; for the Delayed-TP stack x=0 and layer l uses ids 10+4l .. 13+4l
(gamma, W1g, W1u, W2).
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

BLOCK = 1 << 22


@dataclasses.dataclass(frozen=True)
class BoundaryConfig:
    """One SP-TP FFN boundary workload: M tokens, hidden d, FFN width F,
    P tensor-parallel shards, ``chunks`` sequence chunks."""

    name: str
    M: int
    d: int
    F: int
    P: int
    chunks: int
    dtype: str  # "bf16" or "fp32"
    down_std_from_F: bool  # down weights N(0, 1/F) instead of N(0, 1/d)
    eps: float = 1e-6
    seed: int = 0


@dataclasses.dataclass(frozen=True)
class DTPConfig:
    """One Delayed-TP stack workload: L FFN sub-layers, delay ``delta``."""

    name: str
    M: int
    d: int
    F: int
    P: int
    L: int
    delta: int
    dtype: str
    eps: float = 1e-6
    seed: int = 0


TINY_FP32 = BoundaryConfig("tiny_fp32_M64_d128_F512_P2_C4", 64, 128, 512, 2, 4, "fp32", False)
BOUNDARY_D4096 = BoundaryConfig("sptp_bf16_M8192_d4096_F14336_P2_C8", 8192, 4096, 14336, 2, 8, "bf16", True)
QWEN2_7B_SHAPE = BoundaryConfig("sptp_bf16_M16384_d3584_F18944_P4_C16", 16384, 3584, 18944, 4, 16, "bf16", True)


def m_sweep(M: int) -> BoundaryConfig:
    """M sweep at d=4096, F=16384, P=8, chunks=P."""
    return BoundaryConfig(f"sptp_bf16_M{M}_d4096_F16384_P8_C8", M, 4096, 16384, 8, 8, "bf16", True)


M_SWEEP = tuple(m_sweep(M) for M in (4096, 8192, 16384, 32768, 65536))
DTP_STACK = DTPConfig("dtp_bf16_L4_M4096_d1024_F3072_P2_delta1", 4096, 1024, 3072, 2, 4, 1, "bf16")


@dataclasses.dataclass(frozen=True)
class AttnConfig:
    """The boundary in front of an attention sub-layer and the row-parallel
    projection after it: N = q + k + v projection rows, Ho = attention width."""

    name: str
    M: int
    d: int
    N: int
    Ho: int
    P: int
    chunks: int
    dtype: str
    eps: float = 1e-6
    seed: int = 0


# Qwen2-7B-shaped attention: 28 query heads and 4 key/value heads of 128
ATTN_QWEN2_7B_SHAPE = AttnConfig("attn_bf16_M16384_d3584_N4608_Ho3584_P4_C16", 16384, 3584,
                                 28 * 128 + 2 * 4 * 128, 28 * 128, 4, 16, "bf16")


# ---------------------------------------------------------------- drawing

def _block(seed: int, tid: int, b: int, n: int) -> np.ndarray:
    return np.random.default_rng([seed, tid, b]).standard_normal(n)


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(16, os.cpu_count() or 1))


def _fp32_to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); return raw bits."""
    u = f32.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def _cast(v64: np.ndarray, dtype: str) -> np.ndarray:
    f32 = v64.astype(np.float32)
    if dtype == "fp32":
        return f32
    if dtype == "bf16":
        return _fp32_to_bf16_bits(f32)
    raise ValueError(dtype)


def draw(shape, std: float, mean: float, dtype: str, seed: int, tid: int) -> np.ndarray:
    """Draw ``mean + std * N(0,1)`` of ``shape`` in float64 and cast it to ``dtype``
    ("bf16" -> uint16 bit patterns, "fp32" -> float32)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    nb = (n + BLOCK - 1) // BLOCK

    def work(b):
        lo = b * BLOCK
        hi = min(n, lo + BLOCK)
        v = _block(seed, tid, b, hi - lo)
        if std != 1.0:
            v *= std
        if mean != 0.0:
            v += mean
        out[lo:hi] = _cast(v, dtype)

    if nb <= 1:
        for b in range(nb):
            work(b)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nb)))
    return out.reshape(shape)


def boundary_inputs(cfg: BoundaryConfig) -> dict:
    """Inputs of one SP-TP FFN boundary call, in storage format:
    x[M][d], partials[P][M][d], gamma[d], W1g[F][d], W1u[F][d], W2[d][F]."""
    M, d, F, P, s, dt = cfg.M, cfg.d, cfg.F, cfg.P, cfg.seed, cfg.dtype
    wd = d ** -0.5
    wdown = F ** -0.5 if cfg.down_std_from_F else wd
    return {
        "x": draw((M, d), 1.0, 0.0, dt, s, 0),
        "partials": draw((P, M, d), 1.0, 0.0, dt, s, 1),
        "gamma": draw((d,), 0.1, 1.0, dt, s, 2),
        "W1g": draw((F, d), wd, 0.0, dt, s, 3),
        "W1u": draw((F, d), wd, 0.0, dt, s, 4),
        "W2": draw((d, F), wdown, 0.0, dt, s, 5),
    }


def dtp_inputs(cfg: DTPConfig, independent_streams: bool = False) -> dict:
    """Inputs of one Delayed-TP stack call, in storage format:
    x_shards[P][M][d] (one N(0,1) tensor replicated to every shard, or one
    independent draw per shard), gamma[L][d], W1g[L][F][d], W1u[L][F][d],
    W2[L][d][F] (all weights N(0, 1/d))."""
    M, d, F, P, L, s, dt = cfg.M, cfg.d, cfg.F, cfg.P, cfg.L, cfg.seed, cfg.dtype
    if independent_streams:
        xs = np.stack([draw((M, d), 1.0, 0.0, dt, s, 1000 + p) for p in range(P)])
    else:
        x0 = draw((M, d), 1.0, 0.0, dt, s, 0)
        xs = np.stack([x0] * P)
    wd = d ** -0.5
    g = np.stack([draw((d,), 0.1, 1.0, dt, s, 10 + 4 * l) for l in range(L)])
    w1g = np.stack([draw((F, d), wd, 0.0, dt, s, 11 + 4 * l) for l in range(L)])
    w1u = np.stack([draw((F, d), wd, 0.0, dt, s, 12 + 4 * l) for l in range(L)])
    w2 = np.stack([draw((d, F), wd, 0.0, dt, s, 13 + 4 * l) for l in range(L)])
    return {"x_shards": xs, "gamma": g, "W1g": w1g, "W1u": w1u, "W2": w2}


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns to float64 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Widen a storage-format array to float64 (exact)."""
    return bf16_bits_to_f64(arr) if dtype == "bf16" else arr.astype(np.float64)


def attn_inputs(cfg: AttnConfig) -> dict:
    """Inputs of the attention-side boundary, in storage format: x[M][d],
    partials[P][M][d], gamma[d], Wqkv[N][d] ~ N(0, 1/d); and of the
    row-parallel output projection: attn[P][M][Ho/P] ~ N(0, 1), Wo[d][Ho] ~
    N(0, 1/Ho).  Tensor ids 20.. keep the draws apart from the FFN's."""
    M, d, N, Ho, P, s, dt = cfg.M, cfg.d, cfg.N, cfg.Ho, cfg.P, cfg.seed, cfg.dtype
    return {
        "x": draw((M, d), 1.0, 0.0, dt, s, 20),
        "partials": draw((P, M, d), 1.0, 0.0, dt, s, 21),
        "gamma": draw((d,), 0.1, 1.0, dt, s, 22),
        "Wqkv": draw((N, d), d ** -0.5, 0.0, dt, s, 23),
        "attn": draw((P, M, Ho // P), 1.0, 0.0, dt, s, 24),
        "Wo": draw((d, Ho), Ho ** -0.5, 0.0, dt, s, 25),
    }
