"""kvq_prefill_attention: a chunk of T prompt tokens (the last T positions, already
appended) attending causally over the quantized store, against the oracle's
attend_tokens on the same dequantized values."""

import math

import numpy as np
import pytest
import torch

from kvq_testutil import assert_close, bf16_tensor, build_store, device_inputs, kvq, oracle_values
from oracle import attention as oatt
from oracle import codec as ocodec
from workloads import f32_to_bf16_bits, make_inputs

pytestmark = pytest.mark.gpu

PAIRS = [("q8_0", "q8_0"), ("q4s", "q4s"), ("q8_0", "q4s"), ("f16", "f16"), ("bf16", "bf16"),
         ("q8_0", "bf16"), ("q4s", "q8_0"), ("q4s", "bf16"), ("q8_0", "f16"), ("f16", "q8_0")]


def run(inp, kc, vc, T, seed):
    rng = np.random.default_rng(seed)
    qbits = f32_to_bf16_bits(rng.standard_normal((inp.batch, T, inp.num_q_heads, inp.head_dim),
                                                 dtype=np.float32))
    k = kvq()
    ks, vs = build_store(inp, kc, "k"), build_store(inp, vc, "v")
    _, seq, pt = device_inputs(inp)
    got = k.kvq_prefill_attention(bf16_tensor(qbits), ks, vs, seq, pt).cpu().numpy()
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
    kd, vd = oracle_values(inp, kc, vc)
    q = ocodec.bf16_bits_to_f64(qbits)
    group = inp.num_q_heads // inp.num_kv_heads
    want = np.zeros(got.shape)
    for b in range(inp.batch):
        for h in range(inp.num_q_heads):
            kv = h // group
            want[b, :, h] = oatt.attend_tokens(q[b, :, h], kd[b][:, kv], vd[b][:, kv],
                                               1 / math.sqrt(inp.head_dim))
    return got, want


@pytest.mark.parametrize("kc,vc", PAIRS)
def test_prefill_matches_oracle(kc, vc):
    # two sequences: a 300-token chunk after a 700-token prefix, and a 77-token prompt alone
    inp = make_inputs([1000, 77], 16, 4, 128, seed=201, dist="t3", channel_scaled=True)
    got, want = run(inp, kc, vc, 77, seed=202)   # T = 77: sequence 1 is all chunk
    assert_close(got, want, f"{kc}/{vc}")


@pytest.mark.parametrize("hq,hkv,T,L", [(32, 8, 64, 64), (32, 8, 129, 1500), (8, 8, 40, 300),
                                        (32, 2, 10, 2000), (16, 8, 1, 500)])
def test_prefill_shapes(hq, hkv, T, L):
    # G in {1, 2, 4, 16}; chunks smaller, equal and larger than a 64-row CTA; T = 1 is decode
    inp = make_inputs([L], hq, hkv, 128, seed=203 + T)
    got, want = run(inp, "q8_0", "q8_0", T, seed=204 + T)
    assert_close(got, want, f"G={hq // hkv} T={T} L={L}")


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("f16", "f16")])
def test_prefill_head_dim_64(kc, vc):
    inp = make_inputs([400, 130], 8, 2, 64, seed=205)
    got, want = run(inp, kc, vc, 33, seed=206)
    assert_close(got, want, "D=64")


def test_prefill_chunk_longer_than_sequence_gives_zeros_for_blind_queries():
    # seq_len 5 with T = 8: query i sees positions <= i - 3, none for i < 3
    inp = make_inputs([5], 8, 2, 128, seed=207)
    got, want = run(inp, "q8_0", "q8_0", 8, seed=208)
    assert np.array_equal(got[0, :3], np.zeros_like(got[0, :3]))
    assert_close(got, want, "short")


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q8_0"), ("f16", "f16"), ("bf16", "bf16")])
def test_prefill_head_dim_256(kc, vc):
    # GQA 16:1 at head_dim 256 (the long-context shape), heavy-tailed channel-scaled values
    inp = make_inputs([900, 70], 32, 2, 256, seed=209, dist="t3", channel_scaled=True)
    got, want = run(inp, kc, vc, 70, seed=210)
    assert_close(got, want, f"D=256 {kc}/{vc}")


def _rescaled(rows, factor):
    return f32_to_bf16_bits((ocodec.bf16_bits_to_f64(rows) * factor).astype(np.float32))


def test_prefill_magnitudes_past_the_f16_range():
    # V up to ~2e5 (q8_0 scales near 1500: d q alone would overflow f16) and K down at
    # ~1/64: the tensor-core kernel's per-tile powers of two must keep both exact; compared
    # in units of the V factor
    inp = make_inputs([1500, 90], 16, 4, 128, seed=213, dist="t3")
    fv = 4.0e4
    inp.k_rows = [_rescaled(x, 1.0 / 64.0) for x in inp.k_rows]
    inp.v_rows = [_rescaled(x, fv) for x in inp.v_rows]
    got, want = run(inp, "q8_0", "q8_0", 90, seed=214)
    assert np.isfinite(got).all()
    assert_close(got / fv, want / fv, "q8_0 magnitudes")


@pytest.mark.parametrize("page_size", [64, 1024])
def test_prefill_page_sizes(page_size):
    # tiles from pages of one tile and of sixteen; chunks spanning several 128-row CTAs
    inp = make_inputs([2100, 333], 32, 8, 128, seed=215, page_size=page_size)
    for kc, vc in (("q8_0", "q8_0"), ("f16", "f16")):
        got, want = run(inp, kc, vc, 200, seed=216)
        assert_close(got, want, f"page {page_size} {kc}/{vc}")


def test_prefill_unsupported_pair():
    k = kvq()
    inp = make_inputs([100], 8, 2, 128, seed=211)
    ks, vs = build_store(inp, "bf16", "k"), build_store(inp, "q8_0", "v")   # 16-bit K, quantized V
    _, seq, pt = device_inputs(inp)
    q = torch.zeros((1, 4, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(k.KvqError) as e:
        k.kvq_prefill_attention(q, ks, vs, seq, pt)
    assert e.value.status == k.KVQ_ERR_UNSUPPORTED
