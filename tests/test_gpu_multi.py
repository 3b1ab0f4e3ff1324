"""kvq_flash_decode_multi: several query tokens per sequence (speculative drafts, causal
among themselves) against the oracle's attend_tokens on the same dequantized values."""

import math

import numpy as np
import pytest
import torch

from kvq_testutil import assert_close, bf16_tensor, build_store, device_inputs, kvq, oracle_values
from oracle import attention as oatt
from oracle import codec as ocodec
from workloads import f32_to_bf16_bits, make_inputs

pytestmark = pytest.mark.gpu


def run(inp, kc, vc, T, seed, chunk=0):
    rng = np.random.default_rng(seed)
    qbits = f32_to_bf16_bits(rng.standard_normal((inp.batch, inp.num_q_heads, T, inp.head_dim),
                                                 dtype=np.float32))
    k = kvq()
    ks, vs = build_store(inp, kc, "k"), build_store(inp, vc, "v")
    _, seq, pt = device_inputs(inp)
    got = k.kvq_flash_decode_multi(bf16_tensor(qbits), ks, vs, seq, pt, chunk_tokens=chunk).cpu().numpy()
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    kd, vd = oracle_values(inp, kc, vc)
    q = ocodec.bf16_bits_to_f64(qbits)
    group = inp.num_q_heads // inp.num_kv_heads
    want = np.zeros(got.shape)
    for b in range(inp.batch):
        for h in range(inp.num_q_heads):
            kv = h // group
            want[b, h] = oatt.attend_tokens(q[b, h], kd[b][:, kv], vd[b][:, kv], 1 / math.sqrt(inp.head_dim))
    return got, want


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q4s"), ("bf16", "bf16"), ("q8_0", "q4s")])
@pytest.mark.parametrize("hq,hkv,T", [(32, 8, 2), (32, 8, 3), (32, 8, 4), (16, 8, 8), (8, 8, 16)])
def test_multi_token_matches_oracle(kc, vc, hq, hkv, T):
    inp = make_inputs([700, 130, T, T + 1], hq, hkv, 128, seed=60 + T, dist="t3", channel_scaled=True)
    got, want = run(inp, kc, vc, T, seed=70 + T)
    assert_close(got, want, f"{kc}/{vc} G={hq // hkv} T={T}")


@pytest.mark.parametrize("chunk", [64, 128, 1024])
def test_multi_token_split_invariance(chunk):
    # the masked tail lands in different CTAs / tiles depending on the split
    inp = make_inputs([1000, 257], 32, 8, 128, seed=81)
    got, want = run(inp, "q8_0", "q8_0", 4, seed=82, chunk=chunk)
    assert_close(got, want, f"chunk {chunk}")


@pytest.mark.parametrize("head_dim", [64, 256])
def test_multi_token_head_dims(head_dim):
    inp = make_inputs([500, 66], 16, 2, head_dim, seed=83)
    got, want = run(inp, "q8_0", "q4s", 2, seed=84)
    assert_close(got, want, f"D={head_dim}")


def test_sequence_shorter_than_drafts_gives_zeros_for_unseeing_queries():
    inp = make_inputs([1, 40], 8, 2, 128, seed=85)
    got, want = run(inp, "q8_0", "q8_0", 3, seed=86)
    assert np.array_equal(got[0, :, 0], np.zeros_like(got[0, :, 0]))   # sees no position
    assert np.array_equal(got[0, :, 1], np.zeros_like(got[0, :, 1]))
    assert_close(got, want, "short sequence")


def test_one_token_equals_single_decode():
    inp = make_inputs([900], 32, 8, 128, seed=87)
    k = kvq()
    ks, vs = build_store(inp, "q8_0", "k"), build_store(inp, "q8_0", "v")
    q, seq, pt = device_inputs(inp)
    single = k.kvq_flash_decode(q, ks, vs, seq, pt)
    multi = k.kvq_flash_decode_multi(q[:, :, None].contiguous(), ks, vs, seq, pt)
    assert torch.equal(single, multi[:, :, 0])


@pytest.mark.parametrize("hq,hkv,T,d", [(32, 2, 2, 256), (32, 2, 2, 128), (32, 8, 8, 128), (32, 8, 5, 128),
                                        (48, 2, 1, 256), (24, 2, 2, 256)])
def test_more_than_16_query_rows(hq, hkv, T, d):
    # 17..32 query rows per KV head (q8_0 K and V): two 16-row groups of the heads-on-M loop,
    # the second one partly empty for 20 and 24 rows
    inp = make_inputs([1500, 200, T, T + 3], hq, hkv, d, seed=90 + T, dist="t3", channel_scaled=True)
    got, want = run(inp, "q8_0", "q8_0", T, seed=91 + T)
    assert_close(got, want, f"G={hq // hkv} T={T} D={d}")


def test_too_many_query_rows_is_unsupported():
    inp = make_inputs([100], 32, 8, 128, seed=88)
    k = kvq()
    ks, vs = build_store(inp, "q8_0", "k"), build_store(inp, "q8_0", "v")
    _, seq, pt = device_inputs(inp)
    q = torch.zeros((1, 32, 9, 128), dtype=torch.bfloat16, device="cuda")   # G * T = 36 > 32
    with pytest.raises(k.KvqError):
        k.kvq_flash_decode_multi(q, ks, vs, seq, pt)
    k4, v4 = build_store(inp, "q4s", "k"), build_store(inp, "q4s", "v")
    with pytest.raises(k.KvqError):   # beyond 16 rows only q8_0 K and V
        k.kvq_flash_decode_multi(q[:, :, :5].contiguous(), k4, v4, seq, pt)
    with pytest.raises(k.KvqError):   # the CUDA-core kernel has no multi-token form
        k.kvq_flash_decode_multi(q[:, :, :2].contiguous(), ks, vs, seq, pt, variant=1)
