"""Fused flash-decode parity against the oracle run on the same dequantized values."""

import math

import numpy as np
import pytest
import torch

from kvq_testutil import (assert_close, bf16_tensor, build_store, device_inputs, kvq, oracle_out,
                          oracle_values)
from workloads import make_inputs, ragged_lengths

pytestmark = pytest.mark.gpu

PAIRS = [("bf16", "bf16"), ("f16", "f16"), ("q8_0", "bf16"), ("q8_0", "q8_0"),
         ("q4s", "q4s"), ("q8_0", "q4s"), ("q4s", "q8_0"), ("q4s", "bf16")]
VARIANTS = [1, 2]


def run_decode(inp, kc, vc, **kw):
    k = kvq()
    ks = build_store(inp, kc, "k")
    vs = build_store(inp, vc, "v")
    q, sl, pt = device_inputs(inp)
    out = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=int(inp.seq_lens.max()), **kw)
    torch.cuda.synchronize()
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    return out.cpu().numpy(), (ks, vs, q, sl, pt)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("bf16", "bf16")])
def test_tiny_workload(kc, vc, variant):
    # B=1, 4 query heads on 1 KV head, D=128, L=256, N(0,1) bf16
    inp = make_inputs([256], 4, 1, 128, seed=0)
    got, _ = run_decode(inp, kc, vc, variant=variant)
    assert_close(got, oracle_out(inp, kc, vc), f"tiny {kc}/{vc}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("kc,vc", PAIRS)
def test_layer8b_reduced(kc, vc, variant):
    # 32/8 heads, D=128, a length spanning several chunks plus a ragged tail
    inp = make_inputs([3001], 32, 8, 128, seed=11)
    got, _ = run_decode(inp, kc, vc, variant=variant, chunk_tokens=512)
    assert_close(got, oracle_out(inp, kc, vc), f"layer8b {kc}/{vc}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("kc,vc", [("f16", "f16"), ("bf16", "bf16"), ("q8_0", "q8_0"),
                                   ("q4s", "q4s")])
def test_longctx_reduced(kc, vc, variant):
    # 32/2 heads (GQA 16:1), D=256, per-channel scales log-uniform in [0.25, 4]
    inp = make_inputs([2500], 32, 2, 256, seed=12, channel_scaled=True)
    got, _ = run_decode(inp, kc, vc, variant=variant, chunk_tokens=1024)
    assert_close(got, oracle_out(inp, kc, vc), f"longctx {kc}/{vc}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q4s")])
def test_ragged_paged_batch(kc, vc, variant):
    lens = [1, 63, 64, 65, 700, 2049, 256, 0]
    inp = make_inputs(lens, 32, 8, 128, seed=13)
    got, _ = run_decode(inp, kc, vc, variant=variant)
    want = oracle_out(inp, kc, vc)
    assert_close(got, want, f"ragged {kc}/{vc}")
    assert np.all(got[7] == 0.0)  # the empty sequence yields zeros


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("head_dim", [128, 256])
@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q4s")])
def test_ragged_batch_gqa16(kc, vc, head_dim, variant):
    # GQA 16:1 (q8_0: the heads-on-M loop and its chunk merge, where CTAs past a short
    # sequence write empty partials; q4s: the tokens-on-M loop over two 8-head groups)
    lens = [1, 63, 64, 65, 700, 2049, 0, 3000]
    inp = make_inputs(lens, 32, 2, head_dim, seed=131, channel_scaled=True)
    got, _ = run_decode(inp, kc, vc, variant=variant)
    assert_close(got, oracle_out(inp, kc, vc), f"ragged GQA 16:1 D={head_dim} {kc}/{vc}")
    assert np.all(got[6] == 0.0)  # the empty sequence yields zeros


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q4s"), ("bf16", "bf16")])
def test_ragged_batch_gqa8(kc, vc):
    # 8 query heads per KV head: three pipelines of 8-head warps per CTA, a ragged batch
    # (pipelines of one CTA finish at different times; empty and one-token sequences)
    inp = make_inputs([5, 1, 0, 64, 1500, 4100], 64, 8, 128, seed=134)
    got, _ = run_decode(inp, kc, vc)
    assert_close(got, oracle_out(inp, kc, vc), f"ragged GQA 8:1 {kc}/{vc}")
    assert np.all(got[2] == 0.0)


@pytest.mark.parametrize("head_dim", [128, 256])
def test_heavy_tailed_values_gqa16(head_dim):
    # Student-t values and keys with per-channel scales at GQA 16:1: the heads-on-M loop's
    # V-scale bound and lazy max under large magnitudes
    inp = make_inputs([3000, 1200], 32, 2, head_dim, seed=132, dist="t3", channel_scaled=True)
    got, _ = run_decode(inp, "q8_0", "q8_0")
    assert_close(got, oracle_out(inp, "q8_0", "q8_0"), f"t3 GQA 16:1 D={head_dim}")


def test_page_permutation_invariance_gqa16():
    # the heads-on-M loop's result depends on the positions only, not on where the pages are
    a = make_inputs([2600, 700], 32, 2, 256, seed=133, permute_pages=True)
    b = make_inputs([2600, 700], 32, 2, 256, seed=133, permute_pages=False)
    assert not np.array_equal(a.page_table, b.page_table)
    ga, _ = run_decode(a, "q8_0", "q8_0", chunk_tokens=256)
    gb, _ = run_decode(b, "q8_0", "q8_0", chunk_tokens=256)
    assert np.array_equal(ga, gb)


@pytest.mark.parametrize("batch", [3, 16])
def test_mid_size_batches(batch):
    # 24 units (single-pipeline CTAs filling the slots in one wave) and 128 units (four-
    # pipeline CTAs with capped chunks), ragged lengths, both merge paths
    lens = [int(x) for x in np.random.default_rng(135 + batch).integers(1, 6000, size=batch)]
    inp = make_inputs(lens, 32, 8, 128, seed=135 + batch)
    for kc, vc in (("q8_0", "q8_0"), ("q4s", "q4s"), ("bf16", "bf16"), ("q8_0", "bf16")):
        got, _ = run_decode(inp, kc, vc)
        assert_close(got, oracle_out(inp, kc, vc), f"B={batch} {kc}/{vc}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q8_0", "q4s")])
def test_heavy_tailed_values(kc, vc, variant):
    inp = make_inputs([1500], 32, 8, 128, seed=14, dist="t3", channel_scaled=True)
    got, _ = run_decode(inp, kc, vc, variant=variant)
    assert_close(got, oracle_out(inp, kc, vc), f"t3 {kc}/{vc}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("group,head_dim", [(1, 128), (2, 64), (8, 128), (16, 128), (4, 256),
                                            (8, 64), (6, 128), (2, 256), (12, 128)])
def test_group_and_head_dim_sweep(group, head_dim, variant):
    inp = make_inputs([777, 129], 2 * group, 2, head_dim, seed=15)
    got, _ = run_decode(inp, "q8_0", "q8_0", variant=variant)
    assert_close(got, oracle_out(inp, "q8_0", "q8_0"), f"G={group} D={head_dim}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_split_invariance(variant):
    inp = make_inputs([4100], 16, 4, 128, seed=16)
    want = oracle_out(inp, "q8_0", "q8_0")
    outs = []
    for chunk in (64, 128, 512, 2048, 4160):
        got, _ = run_decode(inp, "q8_0", "q8_0", variant=variant, chunk_tokens=chunk)
        assert_close(got, want, f"chunk={chunk}")
        outs.append(got)
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) < 1e-3


@pytest.mark.parametrize("variant", VARIANTS)
def test_page_permutation_invariance(variant):
    a = make_inputs([1800, 900], 8, 2, 128, seed=17, permute_pages=True)
    b = make_inputs([1800, 900], 8, 2, 128, seed=17, permute_pages=False)
    assert not np.array_equal(a.page_table, b.page_table)
    ga, _ = run_decode(a, "q4s", "q4s", variant=variant, chunk_tokens=256)
    gb, _ = run_decode(b, "q4s", "q4s", variant=variant, chunk_tokens=256)
    assert np.array_equal(ga, gb)


@pytest.mark.parametrize("variant", VARIANTS)
def test_closed_forms_on_device(variant):
    # identical keys -> mean of the dequantized V; a single token -> that V row
    inp = make_inputs([500, 1], 4, 1, 128, seed=18)
    inp.k_rows[0][:] = inp.k_rows[0][0:1]
    got, _ = run_decode(inp, "q8_0", "q8_0", variant=variant)
    _, vs = oracle_values(inp, "q8_0", "q8_0")
    for h in range(4):
        assert np.max(np.abs(got[0, h] - vs[0][:, 0].mean(axis=0))) < 2e-3
        assert np.max(np.abs(got[1, h] - vs[1][0, 0])) < 2e-3


@pytest.mark.parametrize("variant", VARIANTS)
def test_explicit_softmax_scale(variant):
    inp = make_inputs([640], 8, 2, 128, seed=19)
    got, _ = run_decode(inp, "q8_0", "bf16", variant=variant, softmax_scale=0.3)
    assert_close(got, oracle_out(inp, "q8_0", "bf16", scale=0.3), "scale=0.3")


@pytest.mark.parametrize("variant", VARIANTS)
def test_stale_rows_past_length_are_ignored(variant):
    # rows past seq_len hold NaN bit patterns: they must not reach the output
    inp = make_inputs([300], 8, 2, 128, seed=20)
    k = kvq()
    ks = build_store(inp, "bf16", "k")
    vs = build_store(inp, "bf16", "v")
    P = inp.page_size
    for st in (ks, vs):
        raw = st.buf.view(torch.int16).view(inp.num_pages, 2, P, 128)
        last = int(inp.page_table[0, 300 // P])
        raw[last, :, 300 % P:, :] = 0x7FC0  # bf16 quiet NaN
    q, sl, pt = device_inputs(inp)
    out = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=300, variant=variant)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert_close(got, oracle_out(inp, "bf16", "bf16"), "stale NaN rows")


def test_workspace_counters_return_to_zero():
    # the split-K merge counts arrivals in the workspace; each call must leave it reusable
    inp = make_inputs([5000, 3000], 16, 4, 128, seed=21)
    k = kvq()
    ks = build_store(inp, "q8_0", "k")
    vs = build_store(inp, "q8_0", "v")
    q, sl, pt = device_inputs(inp)
    need = k.kvq_decode_workspace_bytes(ks, vs, 2, 16, 5000, chunk_tokens=256)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    k.kvq_decode_workspace_init(ws)
    outs = [k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=5000, workspace=ws,
                               chunk_tokens=256).cpu().numpy() for _ in range(3)]
    assert k.kvq_store_get_error(ks) == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    assert_close(outs[0], oracle_out(inp, "q8_0", "q8_0"), "reused workspace")


def test_dirty_workspace_is_reported():
    # 16 query heads on 2 KV heads (8 per KV head): the
    # kernel merges the split in place with arrival counters, so counters that are not zero
    # at the start are reported
    inp = make_inputs([3000], 16, 2, 128, seed=22)
    k = kvq()
    ks = build_store(inp, "q8_0", "k")
    vs = build_store(inp, "q8_0", "v")
    q, sl, pt = device_inputs(inp)
    need = k.kvq_decode_workspace_bytes(ks, vs, 1, 16, 3000, chunk_tokens=256)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=3000, workspace=ws, chunk_tokens=256)
    assert k.kvq_store_get_error(ks) == 5
    k.kvq_decode_workspace_init(ws)
    out = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=3000, workspace=ws, chunk_tokens=256)
    assert k.kvq_store_get_error(ks) == 0
    assert_close(out.cpu().numpy(), oracle_out(inp, "q8_0", "q8_0"), "after re-init")


def test_dirty_workspace_record_mode_keeps_no_state():
    # at most 4 query heads per KV head: every warp rewrites its record on every call and
    # a separate kernel merges them, so a workspace full of garbage gives the same output
    inp = make_inputs([3000], 8, 2, 128, seed=22)
    k = kvq()
    ks = build_store(inp, "q8_0", "k")
    vs = build_store(inp, "q8_0", "v")
    q, sl, pt = device_inputs(inp)
    need = k.kvq_decode_workspace_bytes(ks, vs, 1, 8, 3000, chunk_tokens=256)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    dirty = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=3000, workspace=ws, chunk_tokens=256)
    assert k.kvq_store_get_error(ks) == 0
    ws.zero_()
    clean = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=3000, workspace=ws, chunk_tokens=256)
    assert torch.equal(dirty, clean)
    assert_close(clean.cpu().numpy(), oracle_out(inp, "q8_0", "q8_0"), "record mode")


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q8_0", "q4s")])
def test_resident_append_decode_loop(kc, vc):
    # resident-loop workload at reduced size: a heavy-tailed prefix, then steps of
    # kvq_append_kv (encode one K and V row, seq_lens += 1) + kvq_flash_decode, all on the
    # device; outputs checked against the oracle at several steps
    L0, steps = 1000, 24
    inp = make_inputs([L0 + steps], 32, 8, 128, seed=23, dist="t3", channel_scaled=True)
    k = kvq()
    ks = k.kvq_store_create(kc, 8, 128, inp.page_size, inp.num_pages)
    vs = k.kvq_store_create(vc, 8, 128, inp.page_size, inp.num_pages)
    pt = torch.from_numpy(inp.page_table).cuda()
    seq = torch.zeros(1, dtype=torch.int32, device="cuda")
    krows, vrows = bf16_tensor(inp.k_rows[0]), bf16_tensor(inp.v_rows[0])
    k.kvq_append_kv(ks, vs, krows[None, :L0].contiguous(), vrows[None, :L0].contiguous(), seq, pt)
    q = bf16_tensor(inp.q)
    ws = torch.zeros(k.kvq_decode_workspace_bytes(ks, vs, 1, 32, L0 + steps), dtype=torch.uint8, device="cuda")
    outs = {}
    for step in range(steps):
        k.kvq_append_kv(ks, vs, krows[None, L0 + step:L0 + step + 1].contiguous(),
                        vrows[None, L0 + step:L0 + step + 1].contiguous(), seq, pt)
        out = k.kvq_flash_decode(q, ks, vs, seq, pt, max_len_hint=L0 + steps, workspace=ws)
        if step in (0, 7, steps - 1):
            outs[step] = out.cpu().numpy()
    assert int(seq.item()) == L0 + steps
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    for step, got in outs.items():
        L = L0 + step + 1
        sub = make_inputs([L], 32, 8, 128, seed=23, dist="t3", channel_scaled=True)
        sub.k_rows[0] = inp.k_rows[0][:L]
        sub.v_rows[0] = inp.v_rows[0][:L]
        sub.q = inp.q
        assert_close(got, oracle_out(sub, kc, vc), f"step {step}")


@pytest.mark.parametrize("kc,vc", PAIRS)
def test_heavy_tailed_large_magnitude_keys(kc, vc):
    # Student-t keys and values times per-channel scales up to 4 (blocks with amax ~ 50+):
    # the integer-code offsets must not cost precision (a 1024-based 4-bit K fragment with
    # a seeded accumulator missed the tolerance here)
    inp = make_inputs([3000, 1200], 32, 8, 128, seed=97, dist="t3", channel_scaled=True)
    ks, vs = build_store(inp, kc, "k"), build_store(inp, vc, "v")
    q, seq, pt = device_inputs(inp)
    got = kvq().kvq_flash_decode(q, ks, vs, seq, pt).cpu().numpy()
    assert_close(got, oracle_out(inp, kc, vc), f"{kc}/{vc}")
