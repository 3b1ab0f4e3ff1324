"""Faults in device data are recorded, never trapped; bad host arguments are refused."""

import numpy as np
import pytest
import torch

from kvq_testutil import bf16_tensor, build_store, device_inputs, kvq
from workloads import make_inputs

pytestmark = pytest.mark.gpu


def test_bad_page_id_in_append_is_recorded():
    k = kvq()
    st = k.kvq_store_create("q8_0", 2, 128, 64, 4)
    rows = torch.zeros((1, 3, 2, 128), dtype=torch.bfloat16, device="cuda")
    pt = torch.tensor([[0, 99]], dtype=torch.int32, device="cuda")
    seq = torch.tensor([63], dtype=torch.int32, device="cuda")   # rows 63, 64, 65
    k.kvq_append(st, rows, seq, pt)
    assert k.kvq_store_get_error(st) == 1
    assert k.kvq_store_get_error(st) == 0   # the read clears it


def test_position_past_page_table_is_recorded():
    k = kvq()
    st = k.kvq_store_create("q4s", 1, 64, 64, 2)
    rows = torch.zeros((1, 2, 1, 64), dtype=torch.bfloat16, device="cuda")
    pt = torch.tensor([[0, 1]], dtype=torch.int32, device="cuda")
    seq = torch.tensor([127], dtype=torch.int32, device="cuda")  # 127 ok, 128 past the end
    k.kvq_append(st, rows, seq, pt)
    assert k.kvq_store_get_error(st) == 2


@pytest.mark.parametrize("variant", [1, 2])
def test_bad_page_in_decode_is_recorded(variant):
    inp = make_inputs([500], 8, 2, 128, seed=1)
    k = kvq()
    ks = build_store(inp, "q8_0", "k")
    vs = build_store(inp, "q8_0", "v")
    q, sl, pt = device_inputs(inp)
    pt[0, 1] = 10_000
    out = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=500, variant=variant)
    torch.cuda.synchronize()
    assert k.kvq_store_get_error(ks) == 1
    assert np.all(np.isfinite(out.cpu().numpy()))


@pytest.mark.parametrize("variant", [1, 2])
def test_seq_len_past_hint_is_recorded(variant):
    inp = make_inputs([500], 8, 2, 128, seed=2)
    k = kvq()
    ks = build_store(inp, "q8_0", "k")
    vs = build_store(inp, "q8_0", "v")
    q, sl, pt = device_inputs(inp)
    out = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=128, chunk_tokens=64,
                             variant=variant)
    torch.cuda.synchronize()
    assert k.kvq_store_get_error(ks) == 3
    assert np.all(np.isfinite(out.cpu().numpy()))


def test_host_argument_checks():
    k = kvq()
    inp = make_inputs([64], 8, 2, 128, seed=3)
    ks = build_store(inp, "q8_0", "k")
    vs = build_store(inp, "bf16", "v")
    q, sl, pt = device_inputs(inp)
    other_page = k.kvq_store_create("bf16", 2, 128, 128, inp.num_pages)
    with pytest.raises(k.KvqError) as e:   # K and V stores must share the page size
        k.kvq_flash_decode(q, ks, other_page, sl, pt, max_len_hint=64)
    assert e.value.status == k.KVQ_ERR_INVALID_ARG
    with pytest.raises(k.KvqError) as e:   # chunk must be a multiple of 64
        k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=64, chunk_tokens=100)
    assert e.value.status == k.KVQ_ERR_INVALID_ARG
    with pytest.raises(k.KvqError) as e:   # workspace too small
        k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=64,
                           workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == k.KVQ_ERR_WORKSPACE
    with pytest.raises(k.KvqError) as e:   # hint beyond the page table's capacity
        k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=10 ** 6)
    assert e.value.status == k.KVQ_ERR_INVALID_ARG
    with pytest.raises(k.KvqError) as e:   # Hq not a multiple of Hkv
        k.kvq_flash_decode(q[:, :7].contiguous(), ks, vs, sl, pt, max_len_hint=64)
    assert e.value.status == k.KVQ_ERR_INVALID_ARG
    with pytest.raises(k.KvqError) as e:   # unsupported pair (no kernel built for it)
        k4 = k.kvq_store_create("bf16", 2, 128, 256, inp.num_pages)   # 16-bit K, quantized V
        vb = k.kvq_store_create("q8_0", 2, 128, 256, inp.num_pages)
        k.kvq_flash_decode(q, k4, vb, sl, pt, max_len_hint=64)
    assert e.value.status == k.KVQ_ERR_UNSUPPORTED
    with pytest.raises(k.KvqError) as e:   # store buffer too small
        k.kvq_store_create("q8_0", 2, 128, 256, 4,
                           buf=torch.zeros(100, dtype=torch.uint8, device="cuda"))
    assert e.value.status == k.KVQ_ERR_INVALID_ARG


def test_zero_rows_append_is_a_no_op():
    k = kvq()
    st = k.kvq_store_create("q8_0", 1, 128, 64, 1)
    before = k.kvq_launch_count()
    k.kvq_append(st, torch.zeros((1, 0, 1, 128), dtype=torch.bfloat16, device="cuda"),
                 torch.zeros(1, dtype=torch.int32, device="cuda"),
                 torch.zeros((1, 1), dtype=torch.int32, device="cuda"))
    assert k.kvq_launch_count() == before
    _ = bf16_tensor(np.zeros(4, np.uint16))


def test_read_probe_reads_and_leaves_sink():
    k = kvq()
    buf = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_read_probe(buf, sink)
    k.kvq_read_probe(buf[:1000].clone(), sink)   # a ragged length (tail below 16 bytes unread)
    torch.cuda.synchronize()
    assert int(sink.item()) == 0
    with pytest.raises(k.KvqError):
        k.kvq_read_probe(buf[1:17], sink)          # not 16-byte aligned


@pytest.mark.parametrize("hq,hkv,d,kc,skip", [
    (32, 8, 128, "q8_0", 1),     # lean tile loop, per-warp records merged by a second kernel
    (32, 8, 128, "q4s", 0),      # the very first tile never issued: nothing to drain in that stage
    (16, 2, 128, "q8_0", 1),     # 8 heads per KV head: generic loop, in-place merge
    (64, 4, 256, "q8_0", 1),     # GQA 16:1, head dim 256
])
def test_device_timeout_is_recorded_and_the_next_call_runs(hq, hkv, d, kc, skip):
    # A tile that the producer never issues (no copy, no arrival) leaves its consumers waiting
    # on a stage with nothing in flight; their bounded waits run out, the kernel records
    # KVQ_DEVICE_TIMEOUT, drains every copy it did issue and exits.  The context stays usable.
    inp = make_inputs([8000, 1700], hq, hkv, d, seed=43)
    k = kvq()
    ks = build_store(inp, kc, "k")
    vs = build_store(inp, kc, "v")
    q, sl, pt = device_inputs(inp)
    want = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=8000, variant=2)
    assert k.kvq_store_get_error(ks) == 0
    try:
        k.kvq_set_fault_injection(4096, skip)
        k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=8000, variant=2)
        assert k.kvq_store_get_error(ks) == 4   # KVQ_DEVICE_TIMEOUT
    finally:
        k.kvq_set_fault_injection(0, -1)
    got = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=8000, variant=2)
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    assert torch.equal(got, want)



@pytest.mark.parametrize("kc,vc,skip", [("q8_0", "q8_0", 2), ("f16", "f16", 0), ("q8_0", "f16", 1),
                                        ("q4s", "q4s", 1)])
def test_prefill_device_timeout_is_recorded_and_the_next_call_runs(kc, vc, skip):
    # The tensor-core prefill (head_dim 128): a tile that the producer never issues (no copy,
    # no arrival) leaves the waits on it to run out; the CTA raises its abort flag, every
    # role leaves its loop (the row-pair exchanges are bounded waits too), the copies it did
    # issue are waited for, KVQ_DEVICE_TIMEOUT is recorded, and the next call is exact.
    inp = make_inputs([1500, 300], 16, 4, 128, seed=47)
    k = kvq()
    ks = build_store(inp, kc, "k")
    vs = build_store(inp, vc, "v")
    _, sl, pt = device_inputs(inp)
    T = 100
    rng = np.random.default_rng(48)
    q = torch.from_numpy(rng.standard_normal((inp.batch, T, 16, 128), dtype=np.float32)).cuda().to(torch.bfloat16)
    want = k.kvq_prefill_attention(q, ks, vs, sl, pt)
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    try:
        k.kvq_set_fault_injection(4096, skip)
        k.kvq_prefill_attention(q, ks, vs, sl, pt)
        assert k.kvq_store_get_error(ks) == 4   # KVQ_DEVICE_TIMEOUT
    finally:
        k.kvq_set_fault_injection(0, -1)
    got = k.kvq_prefill_attention(q, ks, vs, sl, pt)
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    assert torch.equal(got, want)
