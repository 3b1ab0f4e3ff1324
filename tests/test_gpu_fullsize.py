"""Parity at the workloads' full sizes, in the launch configuration bench.py times (default
planner, tensor-core kernel), on sampled outputs the oracle computes one by one."""

import math

import numpy as np
import pytest
import torch

from kvq_testutil import ATOL, RTOL_L2, bf16_tensor, compare, device_inputs, kvq
from oracle import attention as oatt
from oracle import codec as ocodec
from workloads import make_inputs, ragged_lengths

pytestmark = pytest.mark.gpu


def upload(inp, codec, which):
    k = kvq()
    st = k.kvq_store_create(codec, inp.num_kv_heads, inp.head_dim, inp.page_size, inp.num_pages)
    rows_all = inp.k_rows if which == "k" else inp.v_rows
    pt = torch.from_numpy(inp.page_table).cuda()
    for b in range(inp.batch):
        seq0 = torch.zeros(1, dtype=torch.int32, device="cuda")
        k.kvq_append(st, bf16_tensor(rows_all[b][None]), seq0, pt[b:b + 1].contiguous())
    return st


def sampled_oracle(inp, kc, vc, picks):
    """Oracle output for (b, h) pairs: only that KV head's rows are dequantized."""
    q = ocodec.bf16_bits_to_f64(inp.q)
    group = inp.num_q_heads // inp.num_kv_heads
    D = inp.head_dim
    out = {}
    cache = {}
    for b, h in picks:
        kv = h // group
        if (b, kv) not in cache:
            kd = ocodec.dequantized(inp.k_rows[b][:, kv, :], kc)
            vd = ocodec.dequantized(inp.v_rows[b][:, kv, :], vc)
            cache[(b, kv)] = (kd, vd)
        kd, vd = cache[(b, kv)]
        out[(b, h)] = oatt.attend_one(q[b, h], kd, vd, 1 / math.sqrt(D))
    return out


def check(got, want):
    g = np.stack([got[b, h] for (b, h) in want])
    w = np.stack([want[k] for k in want])
    mx, rl2 = compare(g, w)
    assert mx <= ATOL and rl2 <= RTOL_L2, (mx, rl2)


def decode(inp, ks, vs):
    k = kvq()
    q, sl, pt = device_inputs(inp)
    out = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=int(inp.seq_lens.max()))
    torch.cuda.synchronize()
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("kc,vc", [("bf16", "bf16"), ("q8_0", "bf16"), ("q8_0", "q8_0"),
                                   ("q4s", "q4s"), ("q8_0", "q4s")])
def test_layer8b_65536(kc, vc):
    inp = make_inputs([65536], 32, 8, 128, seed=101)
    got = decode(inp, upload(inp, kc, "k"), upload(inp, vc, "v"))
    check(got, sampled_oracle(inp, kc, vc, [(0, h) for h in (0, 5, 13, 31)]))


@pytest.mark.parametrize("kc,vc", [("f16", "f16"), ("q8_0", "q8_0")])
def test_longctx_204800(kc, vc):
    inp = make_inputs([204800], 32, 2, 256, seed=102, channel_scaled=True)
    got = decode(inp, upload(inp, kc, "k"), upload(inp, vc, "v"))
    check(got, sampled_oracle(inp, kc, vc, [(0, 0), (0, 15), (0, 16), (0, 31)]))


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q4s")])
def test_ragged_paged_batch_full(kc, vc):
    lens = ragged_lengths(103, 64)
    inp = make_inputs(lens, 32, 8, 128, seed=104)
    got = decode(inp, upload(inp, kc, "k"), upload(inp, vc, "v"))
    longest, shortest = int(np.argmax(lens)), int(np.argmin(lens))
    check(got, sampled_oracle(inp, kc, vc, [(longest, 3), (shortest, 30), (7, 17), (40, 8)]))


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q8_0", "q4s")])
def test_resident_loop_full(kc, vc):
    # 65536-token heavy-tailed prefix, then 128 steps of kvq_append_kv + kvq_flash_decode
    L0, steps = 65536, 128
    inp = make_inputs([L0 + steps], 32, 8, 128, seed=105, dist="t3", channel_scaled=True)
    k = kvq()
    ks = k.kvq_store_create(kc, 8, 128, inp.page_size, inp.num_pages)
    vs = k.kvq_store_create(vc, 8, 128, inp.page_size, inp.num_pages)
    pt = torch.from_numpy(inp.page_table).cuda()
    seq = torch.zeros(1, dtype=torch.int32, device="cuda")
    krows, vrows = bf16_tensor(inp.k_rows[0]), bf16_tensor(inp.v_rows[0])
    k.kvq_append_kv(ks, vs, krows[None, :L0].contiguous(), vrows[None, :L0].contiguous(), seq, pt)
    q = bf16_tensor(inp.q)
    ws = torch.zeros(k.kvq_decode_workspace_bytes(ks, vs, 1, 32, L0 + steps), dtype=torch.uint8,
                     device="cuda")
    out = None
    for step in range(steps):
        k.kvq_append_kv(ks, vs, krows[None, L0 + step:L0 + step + 1].contiguous(),
                        vrows[None, L0 + step:L0 + step + 1].contiguous(), seq, pt)
        out = k.kvq_flash_decode(q, ks, vs, seq, pt, max_len_hint=L0 + steps, workspace=ws)
    got = out.cpu().numpy()
    assert int(seq.item()) == L0 + steps
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    check(got, sampled_oracle(inp, kc, vc, [(0, 0), (0, 9), (0, 22), (0, 31)]))


def oracle_all_heads(inp, kc, vc, L):
    """Oracle output of every query head of sequence 0 over its first L positions, one KV
    head's rows dequantized at a time."""
    q = ocodec.bf16_bits_to_f64(inp.q)
    group = inp.num_q_heads // inp.num_kv_heads
    D = inp.head_dim
    out = np.zeros((inp.num_q_heads, D))
    for kv in range(inp.num_kv_heads):
        kd = ocodec.dequantized(inp.k_rows[0][:L, kv, :], kc)
        vd = ocodec.dequantized(inp.v_rows[0][:L, kv, :], vc)
        for h in range(kv * group, (kv + 1) * group):
            out[h] = oatt.attend_one(q[0, h], kd, vd, 1 / math.sqrt(D))
    return out


def prefix(inp, kc, vc, L0):
    """Stores holding the first L0 rows of sequence 0 (one bulk append), seq_lens = [L0]."""
    k = kvq()
    ks = k.kvq_store_create(kc, inp.num_kv_heads, inp.head_dim, inp.page_size, inp.num_pages)
    vs = k.kvq_store_create(vc, inp.num_kv_heads, inp.head_dim, inp.page_size, inp.num_pages)
    pt = torch.from_numpy(inp.page_table).cuda()
    seq = torch.zeros(1, dtype=torch.int32, device="cuda")
    krows, vrows = bf16_tensor(inp.k_rows[0]), bf16_tensor(inp.v_rows[0])
    k.kvq_append_kv(ks, vs, krows[None, :L0].contiguous(), vrows[None, :L0].contiguous(), seq, pt, advance=True)
    return ks, vs, seq, pt, krows, vrows


def check_new_rows(ks, vs, inp, kc, vc, positions):
    from kvq_testutil import expected_rows, store_rows
    for which, st, codec in (("k", ks, kc), ("v", vs, vc)):
        gp, gs = store_rows(st, inp, 0, positions)
        ep, es = expected_rows(inp, which, codec, 0, positions)
        assert np.array_equal(gp, ep) and np.array_equal(gs, es), which


def test_fused_step_layer8b_65536_all_heads():
    # the step bench.py times: kvq_flash_decode_append from a 65536-token q8_0 prefix at 32
    # query heads on 8 KV heads, default planner (one wave of CTAs, per-warp records and the
    # merge kernel), hint sized as the bench sizes it; every head against the oracle and the
    # appended row bit-exact
    L0 = 65536
    inp = make_inputs([L0 + 1], 32, 8, 128, seed=106)
    k = kvq()
    ks, vs, seq, pt, krows, vrows = prefix(inp, "q8_0", "q8_0", L0)
    out = k.kvq_flash_decode_append(bf16_tensor(inp.q), krows[L0][None].contiguous(), vrows[L0][None].contiguous(),
                                    ks, vs, seq, pt, max_len_hint=L0 + 203)
    got = out.cpu().numpy()[0]
    assert int(seq.item()) == L0 + 1
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    check_new_rows(ks, vs, inp, "q8_0", "q8_0", [L0])
    mx, rl2 = compare(got, oracle_all_heads(inp, "q8_0", "q8_0", L0 + 1))
    assert mx <= ATOL and rl2 <= RTOL_L2, (mx, rl2)


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q8_0", "q4s")])
def test_fused_resident_loop_full(kc, vc):
    # the resident-loop workload as the bench runs it: 128 one-launch steps (encode the new
    # K/V row, attend, advance the length) from a heavy-tailed 65536-token prefix, nothing
    # restaged through the host; checked at the last step (all heads) and every appended row
    L0, steps = 65536, 128
    inp = make_inputs([L0 + steps], 32, 8, 128, seed=107, dist="t3", channel_scaled=True)
    k = kvq()
    ks, vs, seq, pt, krows, vrows = prefix(inp, kc, vc, L0)
    q = bf16_tensor(inp.q)
    hint = L0 + steps
    ws = torch.zeros(k.kvq_decode_workspace_bytes(ks, vs, 1, 32, hint), dtype=torch.uint8, device="cuda")
    out = None
    for step in range(steps):
        out = k.kvq_flash_decode_append(q, krows[L0 + step][None].contiguous(), vrows[L0 + step][None].contiguous(),
                                        ks, vs, seq, pt, max_len_hint=hint, workspace=ws)
    got = out.cpu().numpy()[0]
    assert int(seq.item()) == L0 + steps
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    check_new_rows(ks, vs, inp, kc, vc, list(range(L0, L0 + steps)))
    mx, rl2 = compare(got, oracle_all_heads(inp, kc, vc, L0 + steps))
    assert mx <= ATOL and rl2 <= RTOL_L2, (mx, rl2)
