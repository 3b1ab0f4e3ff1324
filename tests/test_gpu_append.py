"""On-device encode (kvq_append) must match the oracle encode bit for bit."""

import json
import os

import numpy as np
import pytest
import torch

from kvq_testutil import bf16_tensor, build_store, expected_rows, kvq, store_rows
from oracle import codec as ocodec
from workloads import f32_to_bf16_bits, make_inputs

pytestmark = pytest.mark.gpu

CODECS = ["bf16", "f16", "q8_0", "q4s"]


@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("dist,scaled", [("normal", False), ("t3", True)])
def test_append_bit_exact(codec, head_dim, dist, scaled):
    inp = make_inputs([300, 77], 4, 2, head_dim, seed=head_dim + 7, dist=dist,
                      channel_scaled=scaled, page_size=64)
    for which in ("k", "v"):
        st = build_store(inp, codec, which, chunk_rows=129)
        for b in range(inp.batch):
            pos = np.arange(inp.seq_lens[b])
            gp, gs = store_rows(st, inp, b, pos)
            ep, es = expected_rows(inp, which, codec, b, pos)
            assert np.array_equal(gp, ep), f"{codec} {which} b={b}: row bytes differ"
            assert np.array_equal(gs, es), f"{codec} {which} b={b}: scales differ"


@pytest.mark.parametrize("codec", ["q8_0", "q4s"])
def test_append_golden_blocks(codec):
    """The hand-derived blocks (ties, subnormal scales, zero blocks) encoded on the GPU."""
    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "codec_blocks.json")))
    rows = []
    for c in cases["cases"]:
        if c["codec"] != codec:
            continue
        x = np.zeros(128, np.float32)
        for k, v in c["x"].items():
            x[int(k)] = float.fromhex(v)
            x[64 + int(k)] = -float.fromhex(v)   # the mirrored block in the same row
        rows.append((c, f32_to_bf16_bits(x)))
    k = kvq()
    st = k.kvq_store_create(codec, 1, 128, 64, 1)
    pt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    data = np.stack([r for _, r in rows])[None, :, None, :]
    k.kvq_append(st, bf16_tensor(data), torch.zeros(1, dtype=torch.int32, device="cuda"), pt)
    buf = st.buf.cpu().numpy()
    rb = 128 if codec == "q8_0" else 64
    for i, (c, _) in enumerate(rows):
        scales = buf[64 * rb + i * 8: 64 * rb + i * 8 + 8].view(np.uint16)
        assert int(scales[0]) == int(c["d_bits"], 16), c["name"]
        assert int(scales[2]) == int(c["d_bits"], 16), c["name"]
        want = np.zeros(32, np.int64)
        for kk, v in c["q"].items():
            want[int(kk)] = v
        row = buf[i * rb:(i + 1) * rb]
        if codec == "q8_0":
            q = row.view(np.int8).astype(np.int64)
        else:
            q = np.empty(128, np.int64)
            q[0::2] = (row & 15).astype(np.int64) - 8
            q[1::2] = (row >> 4).astype(np.int64) - 8
        assert np.array_equal(q[:32], want), c["name"]
        assert np.array_equal(q[64:96], -want), c["name"]


def test_row_by_row_equals_bulk():
    inp = make_inputs([200], 8, 2, 128, seed=3, page_size=64)
    bulk = build_store(inp, "q8_0", "k")
    k = kvq()
    inc = k.kvq_store_create("q8_0", 2, 128, 64, inp.num_pages)
    seq = torch.zeros(1, dtype=torch.int32, device="cuda")
    pt = torch.from_numpy(inp.page_table).cuda()
    rows = bf16_tensor(inp.k_rows[0][None])
    for i in range(200):
        k.kvq_append(inc, rows[:, i:i + 1].contiguous(), seq, pt)
        k.kvq_seq_lens_add(seq, 1)
    assert int(seq.item()) == 200
    assert torch.equal(bulk.buf, inc.buf)


def test_batched_append_two_sequences():
    inp = make_inputs([96, 96], 4, 2, 128, seed=5, page_size=64)
    k = kvq()
    st = k.kvq_store_create("q4s", 2, 128, 64, inp.num_pages)
    rows = bf16_tensor(np.stack(inp.k_rows))
    seq = torch.zeros(2, dtype=torch.int32, device="cuda")
    k.kvq_append(st, rows, seq, torch.from_numpy(inp.page_table).cuda())
    for b in range(2):
        gp, gs = store_rows(st, inp, b, np.arange(96))
        ep, es = expected_rows(inp, "k", "q4s", b, np.arange(96))
        assert np.array_equal(gp, ep) and np.array_equal(gs, es)


@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q8_0", "q4s"), ("bf16", "bf16")])
@pytest.mark.parametrize("n_new", [1, 3, 200])
def test_append_kv_matches_oracle_and_advances(kc, vc, n_new):
    # K and V rows of a step in one launch, seq_lens advanced afterwards; 200 rows per
    # sequence take several CTAs (advance in a second launch)
    inp = make_inputs([n_new, n_new], 8, 2, 128, seed=40 + n_new, page_size=64)
    k = kvq()
    ks = k.kvq_store_create(kc, 2, 128, 64, inp.num_pages)
    vs = k.kvq_store_create(vc, 2, 128, 64, inp.num_pages)
    seq = torch.zeros(2, dtype=torch.int32, device="cuda")
    k.kvq_append_kv(ks, vs, bf16_tensor(np.stack(inp.k_rows)), bf16_tensor(np.stack(inp.v_rows)), seq,
                    torch.from_numpy(inp.page_table).cuda(), advance=True)
    assert seq.cpu().tolist() == [n_new, n_new]
    for b in range(2):
        for which, st, codec in (("k", ks, kc), ("v", vs, vc)):
            gp, gs = store_rows(st, inp, b, np.arange(n_new))
            ep, es = expected_rows(inp, which, codec, b, np.arange(n_new))
            assert np.array_equal(gp, ep) and np.array_equal(gs, es), (which, b)
    assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0


def _tie_rows(codec, n_rows=96):
    """Rows whose blocks put x / d exactly on rounding boundaries k + 1/2 (d a power of two,
    x = (k + 1/2) d is a bf16), next to them (one bf16 step either side), and at subnormal
    scales; every block also holds +-amax so that d = amax / c is the intended scale."""
    c = 127 if codec == "q8_0" else 7
    rng = np.random.default_rng(11)
    rows = np.zeros((n_rows, 128), np.float32)
    for r in range(n_rows):
        e = int(rng.integers(-30, 6))                 # down to subnormal fp16 scales
        d = 2.0 ** e
        for blk in range(4):
            k = rng.integers(0, c, size=32).astype(np.float64)
            x = (k + 0.5) * d * rng.choice([-1.0, 1.0], size=32)
            x[0] = c * d                                 # amax: d = fp16(amax / c) = 2^e
            rows[r, 32 * blk:32 * blk + 32] = x
    bits = f32_to_bf16_bits(rows)
    # nudge a third of the elements one bf16 step up or down (near-ties)
    nudge = rng.integers(-1, 2, size=bits.shape).astype(np.int64)
    nudge[:, ::32] = 0
    bits = (bits.astype(np.int64) + nudge).astype(np.uint16)
    return bits


@pytest.mark.parametrize("codec", ["q8_0", "q4s"])
@pytest.mark.parametrize("n_new", [1, 96])   # one row per launch (decode path) and the bulk path
def test_append_ties_and_subnormal_scales_bit_exact(codec, n_new):
    bits = _tie_rows(codec)
    k = kvq()
    st = k.kvq_store_create(codec, 1, 128, 128, 1)
    pt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    seq = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = bf16_tensor(bits[None, :, None, :])
    for lo in range(0, 96, n_new):
        k.kvq_append(st, rows[:, lo:lo + n_new].contiguous(), seq, pt)
        k.kvq_seq_lens_add(seq, n_new)
    torch.cuda.synchronize()
    buf = st.buf.cpu().numpy()
    rb = 128 if codec == "q8_0" else 64
    ep, es = ocodec.encode_rows(bits, codec)
    assert np.array_equal(buf[:96 * rb].reshape(96, rb), ep)
    assert np.array_equal(buf[128 * rb:128 * rb + 96 * 8].view(np.uint16).reshape(96, 4), es)
