"""Pins of the oracle's paged store layout (CPU)."""

import numpy as np

from oracle import codec, store


def test_hand_offsets_q8():
    # q8_0, D=128, Hkv=8, page 256: row 128 B, 4 scales (8 B); slab = 256*(128+8) = 34816 B
    assert store.slab_bytes("q8_0", 128, 256) == 34816
    assert store.store_bytes("q8_0", 8, 128, 256, 10) == 10 * 8 * 34816
    d, s = store.row_offsets("q8_0", 8, 128, 256, page=2, row=3, head=5)
    slab = (2 * 8 + 5) * 34816
    assert d == slab + 3 * 128
    assert s == slab + 256 * 128 + 3 * 8


def test_hand_offsets_16bit_and_q4():
    assert store.slab_bytes("bf16", 256, 256) == 256 * 512
    d, s = store.row_offsets("f16", 2, 256, 256, page=1, row=255, head=1)
    assert d == 3 * 256 * 512 + 255 * 512
    assert store.slab_bytes("q4s", 128, 256) == 256 * (64 + 8)


def test_slabs_tile_the_store_without_overlap():
    for name in ("bf16", "q8_0", "q4s"):
        hkv, dim, page, pages = 3, 64, 64, 4
        seen = np.zeros(store.store_bytes(name, hkv, dim, page, pages), dtype=np.int32)
        rb = codec.row_bytes(name, dim)
        nb = codec.scale_count(name, dim)
        for p in range(pages):
            for h in range(hkv):
                for r in range(page):
                    d, s = store.row_offsets(name, hkv, dim, page, p, r, h)
                    seen[d:d + rb] += 1
                    if nb:
                        seen[s:s + 2 * nb] += 1
        assert np.all(seen == 1)


def test_write_read_roundtrip_permuted_pages():
    rng = np.random.default_rng(0)
    name, hkv, dim, page = "q8_0", 2, 64, 64
    table = np.array([3, 0, 2, 1], dtype=np.int32)
    buf = np.zeros(store.store_bytes(name, hkv, dim, page, 4), np.uint8)
    pos = np.arange(200)
    packed = rng.integers(0, 256, size=(200, hkv, dim), dtype=np.uint8)
    scales = rng.integers(0, 1 << 16, size=(200, hkv, dim // 32), dtype=np.uint16)
    store.write_rows(buf, name, hkv, dim, page, table, pos, packed, scales)
    p2, s2 = store.read_rows(buf, name, hkv, dim, page, table, pos)
    assert np.array_equal(p2, packed) and np.array_equal(s2, scales)
    # token 70 is row 6 of logical page 1 -> physical page 0
    d, _ = store.row_offsets(name, hkv, dim, page, 0, 6, 1)
    assert np.array_equal(buf[d:d + dim], packed[70, 1])
