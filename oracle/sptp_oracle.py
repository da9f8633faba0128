"""Oracle for the SP-TP FFN boundary and the Delayed-TP FFN stack.

TEST INFRASTRUCTURE ONLY.  This is the plain, slow, float64 CPU statement of
what the CUDA library computes.  Only the tests, the package smoke check and
the benchmark's CPU-baseline leg may import it; the product path never calls
it and shares no code with it (the only common module is the seeded input
generator, which holds no arithmetic of the method).

Sources (web pages; title and section):

* "[Feature] Async Tensor Parallelism for Archon Engine", sections
  "TP Communication Is on Activations, Not Weights" and "Potential Solution"
  (intra-layer chunked all-gather + matmul; the sub-layer boundary
  reduce-scatter -> residual add + RMSNorm -> all-gather, and the invariant
  norm(all_gather(x)) == all_gather(norm(x))).
* "Affinity-Aware Sharding for Delayed Tensor Parallelism", Abstract
  (Delayed TP: own partial added at once, other devices' partials delta
  modules later; contiguous neuron sharding is the "naive contiguous" layout).

Readings where the pages leave a step open (each one is also listed in the
design notes of the repository):

* RMSNorm: y = h * gamma / sqrt(mean_j h_j^2 + eps), gamma is the scale itself.
* The FFN is SwiGLU: s = silu(h W1g^T) * (h W1u^T), silu(z) = z / (1 + e^-z);
  weights are stored [out][in] (W1g, W1u: [F][d]; W2: [d][F]).
* Shard p holds neurons F_p = [p F/P, (p+1) F/P) of W1g/W1u (rows) and of W2
  (columns); its down projection is a full-width partial of the next sum.
* Chunk c of C covers rows [c M/C, (c+1) M/C) and belongs to shard
  floor(c P / C); on one device the gather of a chunk is the identity.
* Delayed TP: before module l shard p holds x0 + all own partials of modules
  < l + the other shards' partials of modules < l - delta.  After the last
  module its own last partial is added too; ``flush`` then adds whatever the
  other shards' partials have not yet arrived.  Negative module indices are
  absent (the stack starts with nothing pending).

Parity status: every function here is pinned by the CPU tests (library
routines, closed forms, invariants, brute force, a hand-derived example);
none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np


def reduce_partials(partials: np.ndarray) -> np.ndarray:
    """Sum of the P row-parallel partial outputs (the reduce-scatter's
    arithmetic; page 1, "Potential Solution", sub-layer boundary).

    partials: [P, rows, d] -> [rows, d], summed in ascending shard order."""
    r = np.array(partials[0], dtype=np.float64, copy=True)
    for p in range(1, partials.shape[0]):
        r += partials[p]
    return r


def rms_norm(h: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the hidden (last) dimension (page 1, "Potential Solution":
    the norm reduces over hidden, the gather runs over sequence)."""
    ms = np.mean(h * h, axis=-1, keepdims=True)
    return h / np.sqrt(ms + eps) * gamma


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def shard_ffn(y: np.ndarray, W1g: np.ndarray, W1u: np.ndarray, W2: np.ndarray,
              P: int, p: int) -> np.ndarray:
    """Shard p's column-parallel gate/up projection, SwiGLU and row-parallel
    down projection: a full-width partial of the next residual update
    (page 1, "Potential Solution"; page 2, Abstract: a device's "partial
    output").  y: [rows, d] -> [rows, d]."""
    F = W1g.shape[0]
    f = F // P
    n = slice(p * f, (p + 1) * f)
    a = y @ W1g[n].T
    b = y @ W1u[n].T
    s = silu(a) * b
    return s @ W2[:, n].T


def sptp_ffn_forward(x, partials, gamma, W1g, W1u, W2, P: int, chunks: int, eps: float,
                     rows=None):
    """One SP-TP FFN sub-layer boundary (page 1, "Potential Solution").

    For every sequence chunk c (rows [c M/C, (c+1) M/C), owned by shard
    floor(c P / C)): reduce the P partials of those rows, add the residual,
    RMSNorm; the normed chunk is then all-gathered (the identity here) and
    every shard p runs its gate/up GEMM, SwiGLU and down GEMM on it, giving
    shard p's partial of the next boundary.

    Inputs are float64 arrays: x [M,d], partials [P,M,d], gamma [d],
    W1g/W1u [F,d], W2 [d,F].  ``rows`` optionally restricts the evaluation to
    a subset of token rows (rows are independent: the norm reduces over the
    hidden dimension only).

    Returns (out [P, R, d], h [R, d]) with R = M or len(rows).
    """
    M, d = x.shape
    F = W1g.shape[0]
    if partials.shape[0] != P or F % P != 0 or chunks < 1 or M % chunks != 0:
        raise ValueError("bad shape")
    sel = np.arange(M) if rows is None else np.asarray(rows)
    out = np.zeros((P, len(sel), d))
    h_out = np.zeros((len(sel), d))
    m = M // chunks
    for c in range(chunks):
        lo, hi = c * m, (c + 1) * m
        _owner = (c * P) // chunks  # reduce-scatter destination of this chunk
        pos = np.nonzero((sel >= lo) & (sel < hi))[0]
        if len(pos) == 0:
            continue
        r_idx = sel[pos]
        # reduce-scatter arithmetic + residual add + RMSNorm on the owner
        h = x[r_idx] + reduce_partials(partials[:, r_idx, :])
        y = rms_norm(h, gamma, eps)
        h_out[pos] = h
        # all-gather of the normed chunk (identity on one device), then every
        # shard's column-parallel / row-parallel FFN consumes the chunk
        for p in range(P):
            out[p, pos] = shard_ffn(y, W1g, W1u, W2, P, p)
    return out, h_out


def dtp_ffn_stack_forward(x_shards, gamma, W1g, W1u, W2, P: int, L: int, delta: int,
                          flush: bool, eps: float, rows=None):
    """Delayed-TP stack of L FFN sub-layers (page 2, Abstract).

    Shard p keeps its own residual stream x_p.  Module l on shard p reads
    RMSNorm_l(x_p) and produces o_p^(l) with shard p's neurons.  Shard p adds
    o_p^(l) to x_p at once; another shard q's o_q^(l) reaches x_p delta
    modules later (before module l + 1 + delta).  delta = 0 is standard TP.
    After module L-1 shard p adds its own last partial and the partials that
    arrive at that point; with ``flush`` it also adds every other-shard
    partial still pending.

    Inputs are float64: x_shards [P,M,d], gamma [L,d], W1g/W1u [L,F,d],
    W2 [L,d,F].  Returns the final x_shards [P, R, d].
    """
    if delta < 0 or L < 1:
        raise ValueError("bad delta/L")
    sel = slice(None) if rows is None else np.asarray(rows)
    x = np.array(x_shards[:, sel, :], dtype=np.float64, copy=True)
    o = {}  # (module, shard) -> partial, the pending queue

    def arrive(p, l):
        # updates that land on shard p just before module position l
        if l - 1 >= 0:
            x[p] += o[(l - 1, p)]
        k = l - 1 - delta
        if k >= 0:
            for q in range(P):
                if q != p:
                    x[p] += o[(k, q)]

    for l in range(L):
        for p in range(P):
            arrive(p, l)
        for p in range(P):
            y = rms_norm(x[p], gamma[l], eps)
            o[(l, p)] = shard_ffn(y, W1g[l], W1u[l], W2[l], P, p)
    for p in range(P):
        arrive(p, L)
    if flush:
        for p in range(P):
            for k in range(max(0, L - delta), L):
                for q in range(P):
                    if q != p:
                        x[p] += o[(k, q)]
    return x


def attn_qkv_boundary(x, partials, gamma, Wqkv, P: int, chunks: int, eps: float):
    """The boundary in front of an attention sub-layer (page 1, "Potential
    Solution": there are 4 boundaries per block, between attention and FFN
    sub-layers both ways).  The same reduce-scatter arithmetic, residual add
    and RMSNorm per chunk, then the (identity) all-gather and each shard's
    column-parallel QKV projection: shard p holds rows
    [p N/P, (p+1) N/P) of Wqkv [N][d] (its heads' q, k and v rows).

    Returns (qkv [P, M, N/P], h [M, d])."""
    M, d = x.shape
    N = Wqkv.shape[0]
    if partials.shape[0] != P or N % P != 0 or chunks < 1 or M % chunks != 0:
        raise ValueError("bad shape")
    n = N // P
    qkv = np.zeros((P, M, n))
    h_out = np.zeros((M, d))
    m = M // chunks
    for c in range(chunks):
        rows = slice(c * m, (c + 1) * m)
        h = x[rows] + reduce_partials(partials[:, rows, :])
        y = rms_norm(h, gamma, eps)
        h_out[rows] = h
        for p in range(P):
            qkv[p, rows] = y @ Wqkv[p * n:(p + 1) * n].T
    return qkv, h_out


def rowparallel_projection(a, W, P: int):
    """Row-parallel projection after a sub-layer (page 1, "Potential
    Solution": the sub-layer ends with a reduce-scatter of these partials):
    shard p multiplies its activations a[p] [M][K/P] by its columns
    [p K/P, (p+1) K/P) of W [d][K] and yields a full-width partial."""
    K = W.shape[1]
    k = K // P
    return np.stack([a[p] @ W[:, p * k:(p + 1) * k].T for p in range(P)])


def permute_ffn_neurons(W1g: np.ndarray, W1u: np.ndarray, W2: np.ndarray, perm) -> tuple:
    """One FFN with its neurons renumbered before sharding (page 2, Abstract:
    the dense model is permuted before it is sharded, so the contiguous
    shard p then holds the old neurons perm[F_p]).  New neuron i is old
    neuron perm[i]: rows of W1g/W1u and columns of W2 move together."""
    perm = np.asarray(perm)
    if sorted(perm.tolist()) != list(range(W1g.shape[0])):
        raise ValueError("not a permutation")
    return W1g[perm], W1u[perm], W2[:, perm]


def dtp_ffn_stack_forward_permuted(x_shards, gamma, W1g, W1u, W2, perms, P: int, L: int, delta: int,
                                   flush: bool, eps: float, rows=None):
    """Delayed-TP stack under a neuron-permutation shard map per module
    (page 2, Abstract: with delayed partials the sharding is a modelling
    decision).  perms[l] renumbers module l's neurons before contiguous
    sharding; see permute_ffn_neurons."""
    g1, u1, w2 = [], [], []
    for l in range(L):
        a, b, c = permute_ffn_neurons(W1g[l], W1u[l], W2[l], perms[l])
        g1.append(a)
        u1.append(b)
        w2.append(c)
    return dtp_ffn_stack_forward(x_shards, gamma, np.stack(g1), np.stack(u1), np.stack(w2), P, L, delta, flush,
                                 eps, rows=rows)


def rel_max_error(got: np.ndarray, ref: np.ndarray) -> float:
    """The parity metric: max_i |got_i - ref_i| / max_i |ref_i| over one output
    tensor, element i of `got` against element i of `ref` (the workloads'
    "rel. max error"; absolute max error when `ref` is all zero, 0 when both
    are).

    The two arrays must have the same shape (no broadcasting: a single row
    compared with a whole tensor is an error, not a pass).  A non-finite
    element of `got` gives +inf, so it fails every bound and sorts above
    every finite error; a non-finite `ref` is a fault of the reference and
    raises."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.shape != ref.shape:
        raise ValueError(f"shapes differ: got {got.shape}, ref {ref.shape}")
    if not np.all(np.isfinite(ref)):
        raise ValueError("the reference holds non-finite values")
    if ref.size == 0:
        return 0.0
    if not np.all(np.isfinite(got)):
        return float("inf")
    num = float(np.max(np.abs(got - ref)))
    den = float(np.max(np.abs(ref)))
    if den == 0.0:
        return num
    return num / den
