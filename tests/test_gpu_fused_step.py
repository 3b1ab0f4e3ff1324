"""kvq_flash_decode_append: the decode kernel encodes the new token's K/V rows itself
(bit-exact with the oracle encode), attends over the grown sequence (oracle tolerance),
and advances seq_lens on the device."""

import numpy as np
import pytest
import torch

from kvq_testutil import assert_close, bf16_tensor, expected_rows, kvq, oracle_out, store_rows
from workloads import make_inputs

pytestmark = pytest.mark.gpu

PAIRS = [("q8_0", "q8_0"), ("q8_0", "q4s"), ("q4s", "q4s"), ("q8_0", "bf16"), ("bf16", "bf16"),
         ("f16", "f16"), ("q4s", "q8_0"), ("q4s", "bf16")]


def prefix_stores(inp, kc, vc, prefix):
    """Stores holding the first prefix[b] rows of each sequence; seq_lens = prefix."""
    k = kvq()
    ks = k.kvq_store_create(kc, inp.num_kv_heads, inp.head_dim, inp.page_size, inp.num_pages)
    vs = k.kvq_store_create(vc, inp.num_kv_heads, inp.head_dim, inp.page_size, inp.num_pages)
    pt = torch.from_numpy(inp.page_table).cuda()
    for b, n in enumerate(prefix):
        if n:
            seq0 = torch.zeros(1, dtype=torch.int32, device="cuda")
            k.kvq_append_kv(ks, vs, bf16_tensor(inp.k_rows[b][None, :n]), bf16_tensor(inp.v_rows[b][None, :n]),
                            seq0, pt[b:b + 1].contiguous(), advance=False)
    seq = torch.tensor(list(prefix), dtype=torch.int32, device="cuda")
    return ks, vs, seq, pt


def new_rows(inp, prefix):
    k = np.stack([inp.k_rows[b][n] for b, n in enumerate(prefix)])
    v = np.stack([inp.v_rows[b][n] for b, n in enumerate(prefix)])
    return bf16_tensor(k), bf16_tensor(v)


def check_rows(inp, ks, vs, kc, vc, prefix):
    for b, n in enumerate(prefix):
        for which, st, codec in (("k", ks, kc), ("v", vs, vc)):
            gp, gs = store_rows(st, inp, b, [n])
            ep, es = expected_rows(inp, which, codec, b, [n])
            assert np.array_equal(gp, ep) and np.array_equal(gs, es), (which, b, n)


@pytest.mark.parametrize("kc,vc", PAIRS)
@pytest.mark.parametrize("L0,chunk", [(0, 0), (63, 0), (64, 64), (1000, 0), (1000, 128), (4095, 1024)])
def test_fused_step_matches_oracle(kc, vc, L0, chunk):
    # chunk 64: the new token's CTA has one tile (issued up front); chunk 1024 at 4096
    # tokens: its tile comes from the refill path
    inp = make_inputs([L0 + 1], 16, 4, 128, seed=300 + L0, page_size=256)
    ks, vs, seq, pt = prefix_stores(inp, kc, vc, [L0])
    kn, vn = new_rows(inp, [L0])
    k = kvq()
    out = k.kvq_flash_decode_append(bf16_tensor(inp.q), kn, vn, ks, vs, seq, pt, chunk_tokens=chunk)
    got = out.cpu().numpy()
    assert seq.cpu().tolist() == [L0 + 1]
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    check_rows(inp, ks, vs, kc, vc, [L0])
    assert_close(got, oracle_out(inp, kc, vc), f"{kc}/{vc} L0={L0} chunk={chunk}")


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q4s")])
def test_fused_ragged_batch(kc, vc):
    # empty, tile- and page-boundary and long sequences in one batch, permuted pages
    prefix = [0, 63, 64, 255, 256, 3000, 511, 1]
    inp = make_inputs([n + 1 for n in prefix], 32, 8, 128, seed=31)
    ks, vs, seq, pt = prefix_stores(inp, kc, vc, prefix)
    kn, vn = new_rows(inp, prefix)
    k = kvq()
    out = k.kvq_flash_decode_append(bf16_tensor(inp.q), kn, vn, ks, vs, seq, pt)
    got = out.cpu().numpy()
    assert seq.cpu().tolist() == [n + 1 for n in prefix]
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    check_rows(inp, ks, vs, kc, vc, prefix)
    assert_close(got, oracle_out(inp, kc, vc), "ragged fused step")


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q4s")])
def test_fused_step_many_units(kc, vc):
    # 24 sequences x 8 KV heads = 192 units, more than the SMs: single-pipeline CTAs that
    # merge in place and advance the lengths by tickets (no merge kernel)
    prefix = [int(x) for x in np.random.default_rng(39).integers(0, 2500, size=24)]
    prefix[3], prefix[10] = 0, 255
    inp = make_inputs([n + 1 for n in prefix], 32, 8, 128, seed=39)
    ks, vs, seq, pt = prefix_stores(inp, kc, vc, prefix)
    kn, vn = new_rows(inp, prefix)
    k = kvq()
    got = k.kvq_flash_decode_append(bf16_tensor(inp.q), kn, vn, ks, vs, seq, pt).cpu().numpy()
    assert seq.cpu().tolist() == [n + 1 for n in prefix]
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    check_rows(inp, ks, vs, kc, vc, prefix)
    assert_close(got, oracle_out(inp, kc, vc), f"{kc}/{vc} 24-sequence fused step")


def test_fused_equals_append_then_decode():
    prefix = [700, 1500]
    inp = make_inputs([n + 1 for n in prefix], 32, 8, 128, seed=32, dist="t3", channel_scaled=True)
    k = kvq()
    kn, vn = new_rows(inp, prefix)
    q = bf16_tensor(inp.q)
    ks, vs, seq, pt = prefix_stores(inp, "q8_0", "q4s", prefix)
    fused = k.kvq_flash_decode_append(q, kn, vn, ks, vs, seq, pt, max_len_hint=1536)
    ks2, vs2, seq2, pt2 = prefix_stores(inp, "q8_0", "q4s", prefix)
    k.kvq_append_kv(ks2, vs2, kn[:, None].contiguous(), vn[:, None].contiguous(), seq2, pt2, advance=True)
    twostep = k.kvq_flash_decode(q, ks2, vs2, seq2, pt2, max_len_hint=1536)
    assert torch.equal(ks.buf, ks2.buf) and torch.equal(vs.buf, vs2.buf)
    assert torch.equal(seq, seq2)
    # same split, same arithmetic: the outputs agree to the last bit
    assert torch.equal(fused, twostep)


def test_fused_without_advance():
    prefix = [500]
    inp = make_inputs([501], 32, 8, 128, seed=33)
    ks, vs, seq, pt = prefix_stores(inp, "q8_0", "q8_0", prefix)
    kn, vn = new_rows(inp, prefix)
    k = kvq()
    out = k.kvq_flash_decode_append(bf16_tensor(inp.q), kn, vn, ks, vs, seq, pt, advance=False)
    assert seq.cpu().tolist() == [500]
    check_rows(inp, ks, vs, "q8_0", "q8_0", prefix)
    assert_close(out.cpu().numpy(), oracle_out(inp, "q8_0", "q8_0"), "no advance")


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q8_0", "q4s")])
def test_fused_resident_loop(kc, vc):
    # 40 fused steps from a heavy-tailed prefix with one workspace (its counters return to
    # zero after every call); checked against the oracle at three steps
    L0, steps = 900, 40
    inp = make_inputs([L0 + steps], 32, 8, 128, seed=34, dist="t3", channel_scaled=True)
    ks, vs, seq, pt = prefix_stores(inp, kc, vc, [L0])
    k = kvq()
    q = bf16_tensor(inp.q)
    hint = L0 + steps
    ws = torch.zeros(k.kvq_decode_workspace_bytes(ks, vs, 1, 32, hint), dtype=torch.uint8, device="cuda")
    krows, vrows = bf16_tensor(inp.k_rows[0]), bf16_tensor(inp.v_rows[0])
    outs = {}
    for step in range(steps):
        out = k.kvq_flash_decode_append(q, krows[L0 + step][None].contiguous(), vrows[L0 + step][None].contiguous(),
                                        ks, vs, seq, pt, max_len_hint=hint, workspace=ws)
        if step in (0, 17, steps - 1):
            outs[step] = out.cpu().numpy()
    assert int(seq.item()) == L0 + steps
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    for step, got in outs.items():
        L = L0 + step + 1
        sub = make_inputs([L], 32, 8, 128, seed=34, dist="t3", channel_scaled=True)
        sub.k_rows[0], sub.v_rows[0], sub.q = inp.k_rows[0][:L], inp.v_rows[0][:L], inp.q
        assert_close(got, oracle_out(sub, kc, vc), f"step {step}")


def test_fused_full_store_is_a_fault():
    # the sequence already fills its pages: no append, no advance, KVQ_DEVICE_BAD_SEQ_LEN
    inp = make_inputs([256], 8, 2, 128, seed=35, page_size=256)
    ks, vs, seq, pt = prefix_stores(inp, "q8_0", "q8_0", [256])
    before = ks.buf.clone()
    k = kvq()
    kn = bf16_tensor(inp.k_rows[0][:1])
    vn = bf16_tensor(inp.v_rows[0][:1])
    k.kvq_flash_decode_append(bf16_tensor(inp.q), kn, vn, ks, vs, seq, pt)
    assert k.kvq_store_get_error(ks) == 3
    assert k.kvq_store_get_error(vs) == 3
    assert seq.cpu().tolist() == [256]
    assert torch.equal(ks.buf, before)


def test_fused_cuda_core_variant_is_unsupported():
    inp = make_inputs([10], 8, 2, 128, seed=36)
    ks, vs, seq, pt = prefix_stores(inp, "q8_0", "q8_0", [9])
    kn, vn = new_rows(inp, [9])
    k = kvq()
    with pytest.raises(k.KvqError):
        k.kvq_flash_decode_append(bf16_tensor(inp.q), kn, vn, ks, vs, seq, pt, variant=1)
    assert seq.cpu().tolist() == [9]


def test_bound_step_equals_the_plain_call():
    # kvq.DecodeAppendStep (arguments marshalled once, buffers refilled in place) gives the
    # same stores, lengths and outputs as kvq_flash_decode_append
    L0, steps = 600, 5
    inp = make_inputs([L0 + steps], 32, 8, 128, seed=37)
    k = kvq()
    q = bf16_tensor(inp.q)
    krows, vrows = bf16_tensor(inp.k_rows[0]), bf16_tensor(inp.v_rows[0])
    hint = L0 + steps
    ks, vs, seq, pt = prefix_stores(inp, "q8_0", "q8_0", [L0])
    ws = torch.zeros(k.kvq_decode_workspace_bytes(ks, vs, 1, 32, hint), dtype=torch.uint8, device="cuda")
    kn = torch.empty((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    out = torch.empty((1, 32, 128), dtype=torch.float32, device="cuda")
    bound = k.DecodeAppendStep(q, kn, vn, ks, vs, seq, pt, out, ws, hint)
    ks2, vs2, seq2, pt2 = prefix_stores(inp, "q8_0", "q8_0", [L0])
    for st in range(steps):
        kn.copy_(krows[L0 + st][None]); vn.copy_(vrows[L0 + st][None])
        bound()
        ref = k.kvq_flash_decode_append(q, krows[L0 + st][None].contiguous(), vrows[L0 + st][None].contiguous(),
                                        ks2, vs2, seq2, pt2, max_len_hint=hint)
        assert torch.equal(out, ref)
    assert torch.equal(seq, seq2) and torch.equal(ks.buf, ks2.buf) and torch.equal(vs.buf, vs2.buf)


def test_fused_steps_replay_from_a_cuda_graph():
    # 6 fused steps captured once and replayed: the device-side length advance and the
    # encode/decode of each step happen inside the graph, matching eager steps bit for bit
    L0, steps = 500, 6
    inp = make_inputs([L0 + 2 * steps], 32, 8, 128, seed=38)
    k = kvq()
    q = bf16_tensor(inp.q)
    krow = bf16_tensor(inp.k_rows[0][L0:L0 + 1])
    vrow = bf16_tensor(inp.v_rows[0][L0:L0 + 1])
    hint = L0 + 2 * steps
    outs = []
    for mode in ("eager", "graph"):
        ks, vs, seq, pt = prefix_stores(inp, "q8_0", "q8_0", [L0])
        ws = torch.zeros(k.kvq_decode_workspace_bytes(ks, vs, 1, 32, hint), dtype=torch.uint8, device="cuda")
        out = torch.empty((1, 32, 128), dtype=torch.float32, device="cuda")
        step = k.DecodeAppendStep(q, krow, vrow, ks, vs, seq, pt, out, ws, hint)
        if mode == "eager":
            for _ in range(steps):
                step()
        else:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(steps):
                    step()
            graph.replay()
        torch.cuda.synchronize()
        assert int(seq.item()) == L0 + steps
        outs.append((out.clone(), ks.buf.clone(), vs.buf.clone()))
    assert all(torch.equal(a, b) for a, b in zip(outs[0], outs[1]))


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q4s")])
def test_step_reads_and_writes_pinned_host_buffers(kc, vc):
    # q, k_new, v_new and out in pinned host memory (one slot per step): the kernel reads
    # the inputs and writes the output across the host link in place, giving the same
    # stores, lengths and outputs as the step on device buffers
    L0, steps = 700, 4
    inp = make_inputs([L0 + steps], 32, 8, 128, seed=39)
    k = kvq()
    q = bf16_tensor(inp.q)
    krows, vrows = bf16_tensor(inp.k_rows[0]), bf16_tensor(inp.v_rows[0])
    hint = L0 + steps
    ks, vs, seq, pt = prefix_stores(inp, kc, vc, [L0])
    ws = torch.zeros(k.kvq_decode_workspace_bytes(ks, vs, 1, 32, hint), dtype=torch.uint8, device="cuda")
    hq = q.cpu().pin_memory()
    hk = [krows[L0 + st][None].cpu().pin_memory() for st in range(steps)]
    hv = [vrows[L0 + st][None].cpu().pin_memory() for st in range(steps)]
    hout = [torch.empty((1, 32, 128), dtype=torch.float32).pin_memory() for _ in range(steps)]
    bound = [k.DecodeAppendStep(hq, hk[st], hv[st], ks, vs, seq, pt, hout[st], ws, hint) for st in range(steps)]
    for st in range(steps):
        bound[st]()
    torch.cuda.synchronize()
    ks2, vs2, seq2, pt2 = prefix_stores(inp, kc, vc, [L0])
    for st in range(steps):
        ref = k.kvq_flash_decode_append(q, krows[L0 + st][None].contiguous(), vrows[L0 + st][None].contiguous(),
                                        ks2, vs2, seq2, pt2, max_len_hint=hint)
        assert torch.equal(hout[st], ref.cpu()), st
    assert torch.equal(seq, seq2) and torch.equal(ks.buf, ks2.buf) and torch.equal(vs.buf, vs2.buf)
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0


def test_pageable_host_buffers_are_rejected():
    # only pinned CPU tensors are accepted in place of device buffers (host check, nothing
    # is launched)
    inp = make_inputs([300], 32, 8, 128, seed=40)
    k = kvq()
    ks, vs, seq, pt = prefix_stores(inp, "q8_0", "q8_0", [299])
    ws = torch.zeros(k.kvq_decode_workspace_bytes(ks, vs, 1, 32, 300), dtype=torch.uint8, device="cuda")
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16)           # pageable
    kn = torch.zeros((1, 8, 128), dtype=torch.bfloat16).pin_memory()
    out = torch.empty((1, 32, 128), dtype=torch.float32).pin_memory()
    with pytest.raises(TypeError):
        k.DecodeAppendStep(q, kn, kn, ks, vs, seq, pt, out, ws, 300)


def test_pointer_kind_tells_device_mapped_host_and_pageable():
    k = kvq()
    d = torch.empty(64, dtype=torch.uint8, device="cuda")
    h = torch.empty(64, dtype=torch.uint8).pin_memory()
    p = torch.empty(64, dtype=torch.uint8)
    assert k.pointer_kind(d.data_ptr()) == 0
    assert k.pointer_kind(h.data_ptr()) == 1
    assert k.pointer_kind(p.data_ptr()) == -1
