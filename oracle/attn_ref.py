"""Plain fp64 CPU oracle for large-head-dim attention (forward and backward).

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
arm of ``bench.py`` may call it.  It shares no code with the CUDA path.

What it computes is the plain definition of scaled-dot-product attention, the
"naive_math" variant of the attention-kernel-profiler design notes
(generate_docs.py, DESIGN section 3 "Attention Variants" / "naive_math"):

    scores = Q @ K^T * scale          (scale defaults to 1/sqrt(d_head))
    scores = scores + bias            (additive mask, FFPA Attention Benchmark
                                       page, "Quick Start": compact [1,1,1,Nkv]
                                       key-position bias, or [1,1,Nq,Nkv])
    scores = causal_mask(scores)      (query i sees keys j <= i, top-left)
    P      = softmax(scores)          (max-subtracted)
    O      = P @ V
    lse_i  = log(sum_j exp(scores_ij))   natural log of the scaled, biased scores

Grouped-query attention follows the same notes' "gqa_4kv" variant: K/V heads
are expanded with repeat_interleave, i.e. query head h reads kv head
h // (Hq // Hkv).

The backward is the analytic gradient of L = sum(O * dO):
    dV = P^T dO,  dP = dO V^T,  Delta_i = sum_d dO_id O_id,
    dS = P * (dP - Delta),  dQ = scale dS K,  dK = scale dS^T Q,
with dK/dV summed over the query heads of a GQA group.  The FFPA Attention
Benchmark page ("More Benchmark") splits the same backward into a
preprocess (Delta) and dV, dK, dQ launches; the oracle computes each gradient
directly from its definition instead.

Dropout (the "dropout" rows of the FFPA Attention Benchmark page's "More
Benchmark" tables) drops entries of P after the softmax and scales the kept
ones by 1 / (1 - p), so O = (P * Z) V with Z = keep / (1 - p) and lse that of
the undropped scores.  The backward is the gradient of the same function for
a fixed keep mask:
    dV = (P * Z)^T dO,  dP = (dO V^T) * Z,  Delta_i = sum_d dO_id O_id,
    dS = P * (dP - Delta),  dQ, dK as above.
The pages name no generator, so the keep mask follows a contract written
here (``dropout_keep``): Philox4x32-10 (``oracle.philox``) with key = the
64-bit seed and counter (j // 8, i, b * Hq + h, offset) for query row i and
key j of query head h in batch b; score (i, j) takes the 16-bit field
(j mod 2) of output word (j mod 8) // 2 and is kept when that value is at
least t = min(65535, floor(p * 65536 + 1/2)).

Readings where the pages are silent (each also listed in the design notes):
  * lse is the natural log of the scaled and biased scores.
  * causal with Nq != Nkv is top-left (query i sees keys j <= i).
  * a row with every score at -inf gives O = 0, lse = -inf and zero gradients.
  * the oracle takes the inputs' exact fp16/bf16 values in fp64 and does not
    emulate any rounding of P or of the outputs.

All arrays are numpy float64; shapes are [B, H, N, D] with D contiguous.
"""
from __future__ import annotations

import math

import numpy as np

from .philox import philox4x32_10

__all__ = [
    "dropout_threshold",
    "dropout_keep",
    "kv_head_of",
    "scores_head",
    "probs_head",
    "attn_fwd",
    "attn_fwd_rows",
    "attn_bwd",
    "attn_bwd_sampled",
    "sample_rows",
]


def kv_head_of(h: int, hq: int, hkv: int) -> int:
    """KV head read by query head ``h`` (repeat_interleave expansion, "gqa_4kv")."""
    if hq % hkv != 0:
        raise ValueError("Hkv must divide Hq")
    return h // (hq // hkv)


def _bias_rows(bias, b: int, h: int, rows: np.ndarray, nkv: int) -> np.ndarray | float:
    """Broadcast an additive bias of shape [B|1, H|1, Nq|1, Nkv] to [len(rows), Nkv]."""
    if bias is None:
        return 0.0
    bias = np.asarray(bias, dtype=np.float64)
    if bias.ndim != 4 or bias.shape[3] != nkv:
        raise ValueError("bias must be 4-D [B|1, H|1, Nq|1, Nkv]")
    bb = bias[b if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0]
    if bb.shape[0] == 1:
        return np.broadcast_to(bb[0], (len(rows), nkv))
    return bb[rows]


def dropout_threshold(p: float) -> int:
    """16-bit threshold of drop probability p: a score is kept when its value >= t."""
    p = float(p)
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return min(65535, int(math.floor(p * 65536.0 + 0.5)))


def dropout_keep(b: int, h: int, hq: int, rows, cols, p: float, seed: int, offset: int) -> np.ndarray:
    """Keep mask [len(rows), len(cols)] of query head h of batch b under the contract above."""
    t = dropout_threshold(p)
    i = np.asarray(rows, dtype=np.uint64)[:, None]
    j = np.asarray(cols, dtype=np.uint64)[None, :]
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    x = philox4x32_10((j >> np.uint64(3), i, b * hq + h, int(offset)), (seed & 0xFFFFFFFF, seed >> 32))
    jm = (j & np.uint64(7)) + np.zeros_like(i)
    word = np.choose((jm >> np.uint64(1)).astype(np.int64), x)
    u = (word >> (np.uint64(16) * (jm & np.uint64(1)))) & np.uint64(0xFFFF)
    return u >= np.uint64(t)


def _dropout_z(dropout, b, h, hq, rows, cols):
    """Z = keep / (1 - p) on [rows, cols], or 1.0 without dropout."""
    if dropout is None:
        return 1.0
    p, seed, offset = dropout
    return dropout_keep(b, h, hq, rows, cols, p, seed, offset) / (1.0 - float(p))


def scores_head(q, k, bias, b, h, hkv_idx, scale, causal, rows=None, cols=None) -> np.ndarray:
    """Scaled, biased, causally masked scores S[rows, cols] of one (batch, query head).

    q: [B, Hq, Nq, D]; k: [B, Hkv, Nkv, D].  Masked entries are -inf.
    """
    nq, nkv = q.shape[2], k.shape[2]
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    cols = np.arange(nkv) if cols is None else np.asarray(cols)
    qh = q[b, h][rows]
    kh = k[b, hkv_idx][cols]
    s = (qh @ kh.T) * scale
    bias_r = _bias_rows(bias, b, h, rows, nkv)
    if not np.isscalar(bias_r):
        s = s + bias_r[:, cols]
    if causal:
        s = np.where(cols[None, :] > rows[:, None], -np.inf, s)
    return s


def probs_head(s: np.ndarray):
    """Max-subtracted softmax of each row of S, with the row logsumexp.

    Returns (P, lse).  A row whose scores are all -inf gives P = 0, lse = -inf.
    """
    m = np.max(s, axis=1)
    dead = ~np.isfinite(m)
    m_safe = np.where(dead, 0.0, m)
    e = np.exp(s - m_safe[:, None])
    l = np.sum(e, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(dead[:, None], 0.0, e / np.where(dead, 1.0, l)[:, None])
        lse = np.where(dead, -np.inf, m_safe + np.log(np.where(dead, 1.0, l)))
    return p, lse


def _check(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.shape != k.shape:
        raise ValueError("q [B,Hq,Nq,D], k/v [B,Hkv,Nkv,D] expected")
    if q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError("batch and head dim must match")
    if q.shape[1] % k.shape[1] != 0:
        raise ValueError("Hkv must divide Hq")


def _scale(scale, d):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def attn_fwd(q, k, v, bias=None, causal=False, scale=None, dropout=None):
    """Full forward: O [B,Hq,Nq,D] and lse [B,Hq,Nq] (fp64).

    dropout: None or (p, seed, offset) under the contract above.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    _check(q, k, v)
    bsz, hq, nq, d = q.shape
    hkv = k.shape[1]
    scale = _scale(scale, d)
    o = np.zeros(q.shape)
    lse = np.zeros((bsz, hq, nq))
    for b in range(bsz):
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            p, lse[b, h] = probs_head(scores_head(q, k, bias, b, h, g, scale, causal))
            z = _dropout_z(dropout, b, h, hq, np.arange(nq), np.arange(k.shape[2]))
            o[b, h] = (p * z) @ v[b, g]
    return o, lse


def attn_fwd_rows(q, k, v, b, h, rows, bias=None, causal=False, scale=None, dropout=None):
    """Forward for selected query rows of one (batch, head): O[rows] and lse[rows]."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    _check(q, k, v)
    scale = _scale(scale, q.shape[3])
    g = kv_head_of(h, q.shape[1], k.shape[1])
    p, lse = probs_head(scores_head(q, k, bias, b, h, g, scale, causal, rows=rows))
    z = _dropout_z(dropout, b, h, q.shape[1], rows, np.arange(k.shape[2]))
    return (p * z) @ v[b, g], lse


def attn_bwd(q, k, v, do, bias=None, causal=False, scale=None, dropout=None):
    """Full analytic backward: (dQ, dK, dV), fp64, dK/dV summed over each GQA group."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    _check(q, k, v)
    bsz, hq, nq, d = q.shape
    hkv = k.shape[1]
    scale = _scale(scale, d)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(bsz):
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            p, _ = probs_head(scores_head(q, k, bias, b, h, g, scale, causal))
            z = _dropout_z(dropout, b, h, hq, np.arange(q.shape[2]), np.arange(k.shape[2]))
            o = (p * z) @ v[b, g]
            dv[b, g] += (p * z).T @ do[b, h]
            dp = (do[b, h] @ v[b, g].T) * z
            delta = np.sum(do[b, h] * o, axis=1)
            ds = p * (dp - delta[:, None])
            dq[b, h] = scale * (ds @ k[b, g])
            dk[b, g] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


def attn_bwd_sampled(q, k, v, do, b, h_kv, q_rows, kv_rows, bias=None, causal=False, scale=None,
                     block=1024, dropout=None):
    """Exact gradients at selected rows, for shapes too large for the full backward.

    For kv head ``h_kv`` of batch ``b``: returns
      dq:  {h: dQ[b, h, rows_h]} for each query head h of the group, where
           rows_h = q_rows[h] if q_rows is a dict, else q_rows,
      dk, dv: dK[b, h_kv, kv_rows], dV[b, h_kv, kv_rows] (summed over the group).
    Every P_ij needed is normalised by the full-row statistics (lse, Delta) that
    the oracle computes itself over all keys, in row blocks of ``block``.
    """
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    _check(q, k, v)
    hq, nq, d = q.shape[1], q.shape[2], q.shape[3]
    hkv = k.shape[1]
    scale = _scale(scale, d)
    group = hq // hkv
    kv_rows = np.asarray(kv_rows)
    dq_out = {}
    dk = np.zeros((len(kv_rows), d))
    dv = np.zeros((len(kv_rows), d))
    for h in range(h_kv * group, (h_kv + 1) * group):
        # full-row statistics over all keys: lse_i and Delta_i = sum_d dO_id O_id
        lse = np.empty(nq)
        delta = np.empty(nq)
        for r0 in range(0, nq, block):
            rows = np.arange(r0, min(nq, r0 + block))
            p, lse[rows] = probs_head(scores_head(q, k, bias, b, h, h_kv, scale, causal, rows=rows))
            z = _dropout_z(dropout, b, h, hq, rows, np.arange(k.shape[2]))
            delta[rows] = np.sum(do[b, h][rows] * ((p * z) @ v[b, h_kv]), axis=1)
        # dQ at the sampled query rows (needs those rows of P and dP over all keys)
        rows_h = np.asarray(q_rows[h] if isinstance(q_rows, dict) else q_rows)
        p, _ = probs_head(scores_head(q, k, bias, b, h, h_kv, scale, causal, rows=rows_h))
        z = _dropout_z(dropout, b, h, hq, rows_h, np.arange(k.shape[2]))
        dp = (do[b, h][rows_h] @ v[b, h_kv].T) * z
        ds = p * (dp - delta[rows_h][:, None])
        dq_out[h] = scale * (ds @ k[b, h_kv])
        # dK/dV at the sampled key rows (needs those columns of P over all queries)
        s_cols = scores_head(q, k, bias, b, h, h_kv, scale, causal, cols=kv_rows)
        with np.errstate(invalid="ignore"):
            p_cols = np.where(np.isfinite(lse)[:, None], np.exp(s_cols - np.where(
                np.isfinite(lse), lse, 0.0)[:, None]), 0.0)
        z = _dropout_z(dropout, b, h, hq, np.arange(nq), kv_rows)
        dv += (p_cols * z).T @ do[b, h]
        dp_cols = (do[b, h] @ v[b, h_kv][kv_rows].T) * z
        ds_cols = p_cols * (dp_cols - delta[:, None])
        dk += scale * (ds_cols.T @ q[b, h])
    return dq_out, dk, dv


def sample_rows(n: int, count: int, seed: int) -> np.ndarray:
    """Seeded sample of ``count`` distinct row indices in [0, n), always with 0 and n-1."""
    if count >= n:
        return np.arange(n)
    rng = np.random.default_rng(seed)
    picked = set(rng.choice(n, count, replace=False).tolist())
    picked.discard(0)
    picked.discard(n - 1)
    rest = sorted(picked)[: count - 2]
    return np.array(sorted([0, n - 1] + rest), dtype=np.int64)
