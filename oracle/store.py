"""Oracle model of the paged, structure-of-arrays KV store layout.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The store keeps the quantized prefix resident on the device, the fix direction of rMLX
issue #295 ("Fix direction": keep the prefix resident, read the quant store directly, no
per-step host restage).  Its byte layout is the library's documented format:

  store  = num_pages pages; page p = num_kv_heads slabs; slab (p, h) =
           [page_size rows x row_bytes]  (quantized or 16-bit row data)
           [page_size rows x n_scales x 2 bytes]  (fp16 scale bits; absent for 16-bit codecs)
  token position pos of sequence b lives in page page_table[b, pos // page_size],
  row pos % page_size of every head's slab.

This module only computes where a row lives and writes/reads rows at that place; it
holds no codec arithmetic.  Pinned by tests/test_oracle_store.py (hand-computed offsets,
write/read round trip, slabs never overlap).
"""

from __future__ import annotations

import numpy as np

from .codec import row_bytes, scale_count


def slab_bytes(codec: str, head_dim: int, page_size: int) -> int:
    return page_size * (row_bytes(codec, head_dim) + 2 * scale_count(codec, head_dim))


def store_bytes(codec: str, num_kv_heads: int, head_dim: int, page_size: int,
                num_pages: int) -> int:
    return num_pages * num_kv_heads * slab_bytes(codec, head_dim, page_size)


def row_offsets(codec: str, num_kv_heads: int, head_dim: int, page_size: int,
                page: int, row: int, head: int):
    """(byte offset of the row data, byte offset of its first scale) inside the store."""
    slab = (page * num_kv_heads + head) * slab_bytes(codec, head_dim, page_size)
    rb = row_bytes(codec, head_dim)
    data = slab + row * rb
    scales = slab + page_size * rb + row * 2 * scale_count(codec, head_dim)
    return data, scales


def write_rows(buf: np.ndarray, codec: str, num_kv_heads: int, head_dim: int, page_size: int,
               page_table_row: np.ndarray, positions: np.ndarray, packed: np.ndarray,
               scales: np.ndarray) -> None:
    """Write encoded rows of one sequence into a store buffer (uint8, 1-D).

    positions: int [N]; packed: uint8 [N, Hkv, row_bytes]; scales: uint16 [N, Hkv, nb].
    """
    rb = row_bytes(codec, head_dim)
    nb = scale_count(codec, head_dim)
    for i, pos in enumerate(np.asarray(positions)):
        page = int(page_table_row[pos // page_size])
        for h in range(num_kv_heads):
            d_off, s_off = row_offsets(codec, num_kv_heads, head_dim, page_size, page,
                                       int(pos % page_size), h)
            buf[d_off:d_off + rb] = packed[i, h]
            if nb:
                buf[s_off:s_off + 2 * nb] = np.ascontiguousarray(scales[i, h]).view(np.uint8)


def read_rows(buf: np.ndarray, codec: str, num_kv_heads: int, head_dim: int, page_size: int,
              page_table_row: np.ndarray, positions: np.ndarray):
    """Gather rows of one sequence from a store buffer.

    Returns (packed uint8 [N, Hkv, row_bytes], scales uint16 [N, Hkv, nb]).
    """
    rb = row_bytes(codec, head_dim)
    nb = scale_count(codec, head_dim)
    positions = np.asarray(positions)
    packed = np.empty((len(positions), num_kv_heads, rb), np.uint8)
    scales = np.empty((len(positions), num_kv_heads, nb), np.uint16)
    pt = np.asarray(page_table_row)
    pages = pt[positions // page_size].astype(np.int64)
    rows = (positions % page_size).astype(np.int64)
    sb = slab_bytes(codec, head_dim, page_size)
    for h in range(num_kv_heads):
        slab = (pages * num_kv_heads + h) * sb
        d_off = slab + rows * rb
        idx = d_off[:, None] + np.arange(rb)[None, :]
        packed[:, h, :] = buf[idx]
        if nb:
            s_off = slab + page_size * rb + rows * 2 * nb
            sidx = s_off[:, None] + np.arange(2 * nb)[None, :]
            scales[:, h, :] = np.ascontiguousarray(buf[sidx]).view(np.uint16).reshape(-1, nb)
    return packed, scales
