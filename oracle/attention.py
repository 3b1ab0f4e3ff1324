"""Oracle single-token decode attention (float64) and its split-K partial/combine form.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Definition (rMLX issue #292, "Root cause": single-token flash-decode SDPA over the KV
prefix; the quantized variants attend over the dequantized store values):

  for sequence b and query head h, with G = Hq / Hkv and kv = h // G,
    s_t   = scale * sum_j q[b, h, j] * K^[b, kv, t, j]        for t < L_b
    p     = softmax(s)                                         (computed stably)
    out_h = sum_t p_t * V^[b, kv, t, :]
  L_b == 0 gives out_h = 0.

Split-K form (flash-decode): partition [0, L_b) into ranges r; per range
    m_r = max_{t in r} s_t,  l_r = sum_{t in r} exp(s_t - m_r),
    acc_r = sum_{t in r} exp(s_t - m_r) * V^_t
and combine M = max_r m_r,  out = sum_r exp(m_r - M) acc_r / sum_r exp(m_r - M) l_r.
The two forms are equal in exact arithmetic.

Pinned by tests/test_oracle_attention.py: hand-derived cases (tests/golden/attention_cases.json),
closed forms (identical keys -> mean of V, dominant score -> that V row, L = 1, zero
scale -> mean), brute force with pure-Python loops on tiny inputs, token-permutation
invariance, GQA head mapping, and split invariance of the partial/combine form.
"""

from __future__ import annotations

import math

import numpy as np


def attend_one(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """One query row against one head's prefix. q [D], k [L, D], v [L, D] (float64)."""
    if k.shape[0] == 0:
        return np.zeros(v.shape[1], dtype=np.float64)
    s = scale * (k @ q)
    m = s.max()
    e = np.exp(s - m)
    return (e @ v) / e.sum()


def attention(q: np.ndarray, k_seqs, v_seqs, num_kv_heads: int, scale: float | None = None):
    """Batched decode attention.

    q: float64 [B, Hq, D]; k_seqs / v_seqs: per-sequence float64 arrays [L_b, Hkv, D]
    (the dequantized store values).  scale defaults to 1/sqrt(D).  Returns float64 [B, Hq, D].
    """
    bsz, hq, dim = q.shape
    group = hq // num_kv_heads
    if scale is None:
        scale = 1.0 / math.sqrt(dim)
    out = np.zeros((bsz, hq, dim), dtype=np.float64)
    for b in range(bsz):
        for h in range(hq):
            kv = h // group
            out[b, h] = attend_one(q[b, h], k_seqs[b][:, kv, :], v_seqs[b][:, kv, :], scale)
    return out


def partials(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, bounds):
    """Split-K partials (m_r, l_r, acc_r) of one query row over token ranges ``bounds``."""
    out = []
    for lo, hi in bounds:
        if hi <= lo:
            continue
        s = scale * (k[lo:hi] @ q)
        m = s.max()
        e = np.exp(s - m)
        out.append((m, e.sum(), e @ v[lo:hi]))
    return out


def combine(parts, dim: int) -> np.ndarray:
    """Merge split-K partials into the attention output."""
    if not parts:
        return np.zeros(dim, dtype=np.float64)
    big_m = max(p[0] for p in parts)
    num = sum(math.exp(m - big_m) * acc for m, _, acc in parts)
    den = sum(math.exp(m - big_m) * l for m, l, _ in parts)
    return num / den


def attend_one_split(q, k, v, scale, chunk: int) -> np.ndarray:
    """attend_one computed through fixed-size token chunks and the combine."""
    n = k.shape[0]
    bounds = [(lo, min(lo + chunk, n)) for lo in range(0, n, chunk)]
    return combine(partials(q, k, v, scale, bounds), v.shape[1])


def attend_tokens(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Several query tokens of one head against one sequence whose last T positions are
    those tokens (speculative drafts, verified together): query i (of T) attends to the
    positions [0, L - T + i], i.e. causal among the drafts.

    q: float64 [T, D]; k, v: float64 [L, D] -> [T, D].  Query i is ``attend_one`` on the
    first L - T + 1 + i positions (zeros where that count is <= 0).
    """
    T = q.shape[0]
    L = k.shape[0]
    out = np.zeros((T, v.shape[1]))
    for i in range(T):
        n = L - T + 1 + i
        if n > 0:
            out[i] = attend_one(q[i], k[:n], v[:n], scale)
    return out

