"""Seeded synthetic inputs for the decode-attention workloads.

Shared by the tests (which feed the same arrays to the oracle and to the library) and by
bench.py.  This module holds no codec or attention arithmetic: it draws numbers, rounds
them to bf16 (the input precision of every workload) and lays out page tables.

Workload recipes (all values are drawn with NumPy's PCG64 from an explicit seed, then
rounded to bf16 with round-to-nearest-even):

  tiny     B=1, Hq=4, Hkv=1, D=128, L=256; q, K, V ~ N(0, 1).
  layer8b  B=1, Hq=32, Hkv=8, D=128, L in {4096, 16384, 65536}; q, K, V ~ N(0, 1).
  longctx  B=1, Hq=32, Hkv=2, D=256, L in {32768, 131072, 204800}; q ~ N(0, 1);
           K, V ~ N(0, 1) * s[kv_head, channel], s = exp(U(ln 0.25, ln 4)), drawn
           independently for K and for V.
  ragged   B=64, L_b ~ U{1024, ..., 32768}, Hq=32, Hkv=8, D=128; q, K, V ~ N(0, 1);
           256-token pages placed by a seeded random permutation of all pages.
  resident B=1, Hq=32, Hkv=8, D=128, 65536-token prefix then 128 appended rows;
           K, V ~ Student-t(df=3) * s[kv_head, channel] (same log-uniform range); q ~ N(0, 1).

These stand in for the full models the source pages measure (they need trained weights
that are not used here).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    # finite inputs: u < 0xFF800000, so the rounding increment cannot wrap
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def channel_scales(rng: np.random.Generator, num_kv_heads: int, head_dim: int,
                   lo: float = 0.25, hi: float = 4.0) -> np.ndarray:
    """Per-(kv_head, channel) multipliers, log-uniform in [lo, hi]."""
    return np.exp(rng.uniform(np.log(lo), np.log(hi), size=(num_kv_heads, head_dim)))


@dataclass
class DecodeInputs:
    """One batch of decode inputs (host arrays, bf16 as uint16 bit patterns)."""

    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    seq_lens: np.ndarray            # int32 [B]
    q: np.ndarray                   # uint16 [B, Hq, D]
    k_rows: list = field(default_factory=list)   # per sequence uint16 [L_b, Hkv, D]
    v_rows: list = field(default_factory=list)
    page_table: np.ndarray = None   # int32 [B, max_pages], -1 where unused
    num_pages: int = 0

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])


def make_page_table(rng, capacities, page_size: int, permute: bool = True):
    """Assign ceil(cap_b / page_size) pages to each sequence.

    With ``permute`` the physical pages are a seeded random permutation of all pages
    (pages of one sequence land anywhere in the store); otherwise they are consecutive.
    Returns (page_table int32 [B, max_pages] with -1 past each sequence's end, num_pages).
    """
    need = [max(1, -(-int(c) // page_size)) for c in capacities]
    total = int(sum(need))
    order = rng.permutation(total) if permute else np.arange(total)
    table = np.full((len(need), max(need)), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = order[pos:pos + n]
        pos += n
    return table, total


def _draw(rng, kind, shape, scales=None):
    if kind == "normal":
        x = rng.standard_normal(shape, dtype=np.float32)
    elif kind == "t3":
        x = rng.standard_t(3, size=shape).astype(np.float32)
    else:
        raise ValueError(kind)
    if scales is not None:
        x = (x * scales).astype(np.float32)
    return f32_to_bf16_bits(x)


def make_inputs(seq_lens, num_q_heads: int, num_kv_heads: int, head_dim: int, seed: int,
                page_size: int = 256, dist: str = "normal", channel_scaled: bool = False,
                permute_pages: bool = True, extra_capacity: int = 0) -> DecodeInputs:
    """Draw q and the K/V prefixes of a batch, and place its pages.

    ``extra_capacity`` reserves room for that many appended tokens per sequence.
    """
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    bsz = seq_lens.shape[0]
    ks = vs = None
    if channel_scaled:
        ks = channel_scales(rng, num_kv_heads, head_dim)
        vs = channel_scales(rng, num_kv_heads, head_dim)
    q = _draw(rng, "normal", (bsz, num_q_heads, head_dim))
    k_rows, v_rows = [], []
    for b in range(bsz):
        shape = (int(seq_lens[b]), num_kv_heads, head_dim)
        k_rows.append(_draw(rng, dist, shape, ks))
        v_rows.append(_draw(rng, dist, shape, vs))
    table, num_pages = make_page_table(rng, seq_lens + extra_capacity, page_size,
                                       permute=permute_pages)
    inp = DecodeInputs(num_q_heads, num_kv_heads, head_dim, page_size, seq_lens, q,
                       k_rows, v_rows, table, num_pages)
    inp.k_channel_scales, inp.v_channel_scales = ks, vs
    return inp


def ragged_lengths(seed: int, batch: int = 64, lo: int = 1024, hi: int = 32768) -> np.ndarray:
    """Integer sequence lengths, uniform on [lo, hi] inclusive."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=batch).astype(np.int32)


# Named workloads: (num_q_heads, num_kv_heads, head_dim, dist, channel_scaled, lengths)
WORKLOADS = {
    "tiny": dict(num_q_heads=4, num_kv_heads=1, head_dim=128, dist="normal",
                 channel_scaled=False, kv_lens=(256,)),
    "layer8b": dict(num_q_heads=32, num_kv_heads=8, head_dim=128, dist="normal",
                    channel_scaled=False, kv_lens=(4096, 16384, 65536)),
    "longctx": dict(num_q_heads=32, num_kv_heads=2, head_dim=256, dist="normal",
                    channel_scaled=True, kv_lens=(32768, 131072, 204800)),
    "ragged": dict(num_q_heads=32, num_kv_heads=8, head_dim=128, dist="normal",
                   channel_scaled=False, kv_lens=None),
    "resident": dict(num_q_heads=32, num_kv_heads=8, head_dim=128, dist="t3",
                     channel_scaled=True, kv_lens=(65536,)),
}
