"""Decode parity at the edges of what the library accepts: every page size class, the
largest head_dim and group at the largest page, a split into many chunks (the two-level
merge with many groups), and a batch with more (sequence, KV head) units than resident CTAs
and sequences of a single token."""

import numpy as np
import pytest
import torch

from kvq_testutil import assert_close, build_store, device_inputs, kvq, oracle_out
from workloads import make_inputs

pytestmark = pytest.mark.gpu


def decode(inp, kc, vc, **kw):
    k = kvq()
    ks, vs = build_store(inp, kc, "k"), build_store(inp, vc, "v")
    q, sl, pt = device_inputs(inp)
    out = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=int(inp.seq_lens.max()), **kw)
    torch.cuda.synchronize()
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("page_size", [64, 128, 512, 1024])
@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q4s"), ("bf16", "bf16")])
def test_page_sizes(page_size, kc, vc):
    # lengths with a ragged tail inside a page and one ending exactly on a page boundary
    inp = make_inputs([3001, 2 * page_size], 16, 4, 128, seed=60 + page_size, page_size=page_size)
    assert_close(decode(inp, kc, vc), oracle_out(inp, kc, vc), f"page {page_size} {kc}/{vc}")


@pytest.mark.parametrize("page_size", [64, 128])
@pytest.mark.parametrize("hq,hkv,d", [(32, 2, 256), (32, 2, 128), (64, 8, 128)])
def test_small_pages_for_the_wide_groups(page_size, hq, hkv, d):
    # heads-on-M (GQA 16:1) and three-pipeline 8-head warps (GQA 8:1) where every tile is
    # a whole page or half of one, with a ragged tail
    inp = make_inputs([2000, 3 * page_size + 5], hq, hkv, d, seed=74 + page_size + d, page_size=page_size,
                      channel_scaled=True)
    assert_close(decode(inp, "q8_0", "q8_0"), oracle_out(inp, "q8_0", "q8_0"),
                 f"page {page_size} GQA {hq // hkv}:1 D={d}")


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q8_0"), ("f16", "f16")])
def test_largest_head_dim_and_group_at_the_largest_page(kc, vc):
    # head_dim 256, 16 query heads per KV head, 1024-token pages, channel-scaled values
    inp = make_inputs([5000], 32, 2, 256, seed=70, page_size=1024, channel_scaled=True)
    assert_close(decode(inp, kc, vc), oracle_out(inp, kc, vc), f"D256 G16 P1024 {kc}/{vc}")


@pytest.mark.parametrize("hkv", [8, 4])
def test_many_chunks_two_level_merge(hkv):
    # 64-token chunks over 16384 tokens: 256 partials per (sequence, KV head).  With 4 query
    # heads per KV head they are 4096 per-warp records for the merge kernel; with 8 the
    # kernel merges them in place, in 16 groups and then across the groups
    inp = make_inputs([16384], 32, hkv, 128, seed=71)
    got = decode(inp, "q8_0", "q8_0", chunk_tokens=64)
    want = oracle_out(inp, "q8_0", "q8_0", heads=[0, 5, 13, 31])
    assert_close(got, want, f"256 chunks, {32 // hkv} heads per KV head")
    # the default split and the 64-token split agree to rounding
    ref = decode(inp, "q8_0", "q8_0")
    assert np.max(np.abs(got - ref)) < 1e-4


def test_in_place_merge_beyond_the_record_limit():
    # 64-token chunks over 65536 tokens at 4 query heads per KV head: 16384 per-warp records
    # would exceed the record limit, so the kernel merges in place (1024 partials, 64 groups)
    inp = make_inputs([65536], 8, 2, 128, seed=73)
    got = decode(inp, "q8_0", "q8_0", chunk_tokens=64)
    want = oracle_out(inp, "q8_0", "q8_0", heads=[0, 3, 6])
    assert_close(got, want, "1024 chunks in place")


def test_more_units_than_resident_ctas_and_single_token_sequences():
    # 160 sequences x 8 KV heads = 1280 units, lengths 1..700 (every one shorter than a chunk)
    rng = np.random.default_rng(72)
    lens = rng.integers(1, 701, size=160)
    lens[:4] = [1, 1, 64, 65]
    inp = make_inputs(lens, 32, 8, 64, seed=72, page_size=64)
    got = decode(inp, "q4s", "q4s")
    want = oracle_out(inp, "q4s", "q4s", seqs=[0, 1, 2, 3, 50, 159], heads=[0, 7, 30])
    assert_close(got, want, "1280 units")
