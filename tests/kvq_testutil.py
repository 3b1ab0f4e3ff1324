"""Helpers for the GPU parity tests: feed one set of seeded inputs to the library (through
the C ABI binding) and to the oracle, and compare."""

from __future__ import annotations

import math

import numpy as np
import torch

from oracle import attention as oatt
from oracle import codec as ocodec
from oracle import store as ostore

ATOL = 2e-3      # max-abs tolerance on the attention output
RTOL_L2 = 1e-3   # relative-L2 tolerance on the attention output


def kvq():
    from flash_decode_quantized_gb300 import kvq as _k
    return _k


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def build_store(inp, codec: str, which: str, chunk_rows: int = 1 << 16):
    """Create a store sized for ``inp`` and append every sequence's rows through kvq_append."""
    k = kvq()
    store = k.kvq_store_create(codec, inp.num_kv_heads, inp.head_dim, inp.page_size, inp.num_pages)
    rows_all = inp.k_rows if which == "k" else inp.v_rows
    pt = torch.from_numpy(inp.page_table).cuda()
    for b in range(inp.batch):
        rows = rows_all[b]
        for lo in range(0, rows.shape[0], chunk_rows):
            part = rows[lo:lo + chunk_rows]
            seq0 = torch.tensor([lo], dtype=torch.int32, device="cuda")
            k.kvq_append(store, bf16_tensor(part[None]), seq0, pt[b:b + 1].contiguous())
    return store


def device_inputs(inp):
    return (bf16_tensor(inp.q), torch.from_numpy(inp.seq_lens).cuda(),
            torch.from_numpy(inp.page_table).cuda())


def oracle_values(inp, k_codec: str, v_codec: str, seqs=None):
    """Dequantized K/V per sequence (float64 [L, Hkv, D]) as the oracle encodes them."""
    seqs = range(inp.batch) if seqs is None else seqs
    ks, vs = {}, {}
    for b in seqs:
        kr, vr = inp.k_rows[b], inp.v_rows[b]
        L, H, D = kr.shape
        ks[b] = ocodec.dequantized(kr.reshape(-1, D), k_codec).reshape(L, H, D)
        vs[b] = ocodec.dequantized(vr.reshape(-1, D), v_codec).reshape(L, H, D)
    return ks, vs


def oracle_out(inp, k_codec, v_codec, scale=None, seqs=None, heads=None):
    """Oracle attention for the selected sequences / query heads; float64 [B, Hq, D] with
    NaN where not computed."""
    seqs = list(range(inp.batch)) if seqs is None else list(seqs)
    heads = list(range(inp.num_q_heads)) if heads is None else list(heads)
    ks, vs = oracle_values(inp, k_codec, v_codec, seqs)
    D = inp.head_dim
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    q = ocodec.bf16_bits_to_f64(inp.q)
    group = inp.num_q_heads // inp.num_kv_heads
    out = np.full((inp.batch, inp.num_q_heads, D), np.nan)
    for b in seqs:
        for h in heads:
            kv = h // group
            out[b, h] = oatt.attend_one(q[b, h], ks[b][:, kv], vs[b][:, kv], scale)
    return out


def compare(got: np.ndarray, want: np.ndarray):
    """(max-abs error, relative-L2 error) over the entries the oracle computed."""
    mask = ~np.isnan(want)
    g, w = got[mask].astype(np.float64), want[mask]
    err = np.abs(g - w)
    denom = max(np.linalg.norm(w), 1e-30)
    return float(err.max(initial=0.0)), float(np.linalg.norm(g - w) / denom)


def assert_close(got, want, what=""):
    mx, rl2 = compare(got, want)
    assert mx <= ATOL and rl2 <= RTOL_L2, f"{what}: max-abs {mx:.3g}, rel-L2 {rl2:.3g}"
    return mx, rl2


def store_rows(store, inp, b, positions):
    """Read rows of sequence b back from a device store: (packed, scales) per the layout."""
    buf = store.buf.cpu().numpy()
    return ostore.read_rows(buf, store.codec, inp.num_kv_heads, inp.head_dim, inp.page_size,
                            inp.page_table[b], np.asarray(positions))


def expected_rows(inp, which, codec, b, positions):
    rows = (inp.k_rows if which == "k" else inp.v_rows)[b][np.asarray(positions)]
    n, H, D = rows.shape
    packed, scales = ocodec.encode_rows(rows.reshape(-1, D), codec)
    return packed.reshape(n, H, -1), scales.reshape(n, H, -1)
