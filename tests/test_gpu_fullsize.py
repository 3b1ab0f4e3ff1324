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
