"""kvq_dequantize (the separate-pass comparison arm): bit-exact against the oracle's
rounding of d * q, rows past each sequence untouched, and a 16-bit decode over its output
within tolerance of the oracle on the same rounded values."""

import math

import numpy as np
import pytest
import torch

from kvq_testutil import assert_close, bf16_tensor, build_store, device_inputs, kvq
from oracle import attention as oatt
from oracle import codec as ocodec
from oracle import store as ostore
from workloads import make_inputs

pytestmark = pytest.mark.gpu


def expected_16(inp, which, src, target, b):
    rows = (inp.k_rows if which == "k" else inp.v_rows)[b]
    n, H, D = rows.shape
    packed, scales = ocodec.encode_rows(rows.reshape(-1, D), src)
    return ocodec.dequantized_16(packed, scales, src, D, target).reshape(n, H, D)


def dst_rows(dst, inp, b, n):
    buf = dst.buf.cpu().numpy()
    packed, _ = ostore.read_rows(buf, dst.codec, inp.num_kv_heads, inp.head_dim, inp.page_size,
                                 inp.page_table[b], np.arange(n))
    return packed.view(np.uint16).reshape(n, inp.num_kv_heads, inp.head_dim)


@pytest.mark.parametrize("src", ["q8_0", "q4s"])
@pytest.mark.parametrize("target", ["f16", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128, 256])
def test_dequantize_bit_exact(src, target, head_dim):
    inp = make_inputs([300, 1, 77], 4, 2, head_dim, seed=head_dim + 11, dist="t3", channel_scaled=True,
                      page_size=64, extra_capacity=40)
    k = kvq()
    st = build_store(inp, src, "k")
    dst = k.kvq_store_create(target, inp.num_kv_heads, head_dim, inp.page_size, inp.num_pages)
    dst.buf.fill_(0xA5)   # rows past each sequence must keep this pattern
    _, seq, pt = device_inputs(inp)
    k.kvq_dequantize(st, dst, seq, pt)
    torch.cuda.synchronize()
    assert k.kvq_store_get_error(dst) == 0
    for b in range(inp.batch):
        n = int(inp.seq_lens[b])
        assert np.array_equal(dst_rows(dst, inp, b, n), expected_16(inp, "k", src, target, b)), b
        # the slots reserved past the length were not written
        cap = int((inp.page_table[b] >= 0).sum()) * inp.page_size
        if cap > n:
            buf = dst.buf.cpu().numpy()
            tail, _ = ostore.read_rows(buf, target, inp.num_kv_heads, head_dim, inp.page_size,
                                       inp.page_table[b], np.arange(n, cap))
            assert (tail == 0xA5).all()


@pytest.mark.parametrize("src,target", [("q8_0", "f16"), ("q4s", "f16"), ("q8_0", "bf16")])
def test_unfused_decode_matches_oracle(src, target):
    inp = make_inputs([1500, 640], 32, 8, 128, seed=51, channel_scaled=True)
    k = kvq()
    ks, vs = build_store(inp, src, "k"), build_store(inp, src, "v")
    kd = k.kvq_store_create(target, 8, 128, inp.page_size, inp.num_pages)
    vd = k.kvq_store_create(target, 8, 128, inp.page_size, inp.num_pages)
    q, seq, pt = device_inputs(inp)
    k.kvq_dequantize(ks, kd, seq, pt)
    k.kvq_dequantize(vs, vd, seq, pt)
    got = k.kvq_flash_decode(q, kd, vd, seq, pt).cpu().numpy()
    to64 = ocodec.f16_bits_to_f64 if target == "f16" else ocodec.bf16_bits_to_f64
    qf = ocodec.bf16_bits_to_f64(inp.q)
    want = np.full(got.shape, np.nan)
    for b in range(inp.batch):
        kv = to64(expected_16(inp, "k", src, target, b))
        vv = to64(expected_16(inp, "v", src, target, b))
        for h in range(32):
            want[b, h] = oatt.attend_one(qf[b, h], kv[:, h // 4], vv[:, h // 4], 1 / math.sqrt(128))
    assert_close(got, want, f"{src}->{target}")


def test_dequantize_rejects_mismatched_stores():
    k = kvq()
    a = k.kvq_store_create("q8_0", 2, 128, 64, 4)
    b = k.kvq_store_create("f16", 2, 64, 64, 4)
    c = k.kvq_store_create("q8_0", 2, 128, 64, 4)
    seq = torch.zeros(1, dtype=torch.int32, device="cuda")
    pt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(k.KvqError):
        k.kvq_dequantize(a, b, seq, pt)      # head_dim differs
    with pytest.raises(k.KvqError):
        k.kvq_dequantize(a, c, seq, pt)      # target is not a 16-bit store
