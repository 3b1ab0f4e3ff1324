"""Pins of the oracle block codecs against hand-derived blocks and codec invariants (CPU)."""

import json
import os

import numpy as np
import pytest

from oracle import codec
from workloads import f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "codec_blocks.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)


def _block_bits(case, dim=32):
    x = np.zeros(dim, dtype=np.float64)
    for k, v in case["x"].items():
        x[int(k)] = float.fromhex(v)
    bits = f32_to_bf16_bits(x.astype(np.float32))
    # every golden input is exactly a bf16 value
    assert np.array_equal(codec.bf16_bits_to_f64(bits), x)
    return bits[None, :]


@pytest.mark.parametrize("case", _cases()["cases"], ids=lambda c: c["name"])
def test_golden_block(case):
    bits = _block_bits(case)
    q, d_bits = codec.quantize_rows(bits, case["codec"])
    assert int(d_bits[0, 0]) == int(case["d_bits"], 16)
    want = np.zeros(32, dtype=np.int32)
    for k, v in case["q"].items():
        want[int(k)] = v
    assert np.array_equal(q[0], want)
    packed, scales = codec.encode_rows(bits, case["codec"])
    if "bytes" in case:
        assert packed[0].tobytes().hex() == case["bytes"]
    assert np.array_equal(codec.unpack_codes(packed, case["codec"], 32)[0], want)


def test_golden_f16_control():
    for x_hex, want in _cases()["f16_cases"]["values"]:
        bits = f32_to_bf16_bits(np.array([float.fromhex(x_hex)], np.float32))
        packed, _ = codec.encode_rows(bits[None, :], "f16")
        assert int(packed.view(np.uint16)[0, 0]) == int(want, 16), x_hex


def test_q8_bytes_are_twos_complement():
    q = np.array([[127, -127, -1, 0, 1, -64] + [0] * 26], dtype=np.int32)
    assert codec.pack_codes(q, "q8_0")[0, :6].tobytes().hex() == "7f81ff0001c0"


def test_q4_nibble_order_words():
    # element 8w+e sits in bits 4e..4e+3 of little-endian uint32 word w
    q = np.arange(32, dtype=np.int32) % 15 - 7
    packed = codec.pack_codes(q[None, :], "q4s")
    words = packed.view("<u4")[0]
    for j in range(32):
        w, e = divmod(j, 8)
        assert ((int(words[w]) >> (4 * e)) & 0xF) - 8 == q[j]


def _random_rows(seed, n, dim, scale=1.0, dist="normal"):
    rng = np.random.default_rng(seed)
    if dist == "normal":
        x = rng.standard_normal((n, dim)) * scale
    else:
        x = rng.standard_t(3, size=(n, dim)) * scale
    return f32_to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("name", ["q8_0", "q4s"])
@pytest.mark.parametrize("scale,dist", [(1.0, "normal"), (37.0, "t3"), (1e-3, "normal")])
def test_roundtrip_bound_and_range(name, scale, dist):
    c = codec.QMAX[name]
    bits = _random_rows(1, 512, 128, scale, dist)
    x = codec.bf16_bits_to_f64(bits)
    q, d_bits = codec.quantize_rows(bits, name)
    d = codec.f16_bits_to_f64(d_bits)
    assert np.abs(q).max() <= c
    xb = x.reshape(512, 4, 32)
    qb = q.reshape(512, 4, 32)
    err = np.abs(xb - d[:, :, None] * qb)
    # |x - d q| <= d/2, up to the fp32 rounding of the quotient x/d (<= 2^-24 |x/d| * d)
    bound = d[:, :, None] / 2 + np.abs(xb) * 2.0 ** -23
    normal = d >= 2.0 ** -14
    assert np.all((err <= bound)[normal])
    # a normal scale is within 2^-11 of amax/c, so the largest element maps to +-c
    amax_code = np.abs(qb).max(axis=2)
    assert np.all(amax_code[normal] == c)


def test_brute_force_single_element_blocks():
    # every finite bf16 value alone in a block: with a normal fp16 scale the code is +-127
    # and decoding reproduces the value to within d/2.
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        x = codec.bf16_bits_to_f64(bits)
    keep = np.isfinite(x) & (np.abs(x) >= 127 * 2.0 ** -14) & (np.abs(x) < 127 * 65504.0)
    bits = bits[keep]
    rows = np.zeros((bits.shape[0], 32), dtype=np.uint16)
    rows[:, 5] = bits
    q, d_bits = codec.quantize_rows(rows, "q8_0")
    x = codec.bf16_bits_to_f64(bits)
    assert np.array_equal(q[:, 5], np.sign(x).astype(np.int32) * 127)
    assert not np.any(np.delete(q, 5, axis=1))
    d = codec.f16_bits_to_f64(d_bits[:, 0])
    assert np.all(np.abs(x - 127 * np.sign(x) * d) <= d / 2)


@pytest.mark.parametrize("name", ["bf16", "f16", "q8_0", "q4s"])
def test_pack_unpack_roundtrip(name):
    bits = _random_rows(2, 64, 256)
    packed, scales = codec.encode_rows(bits, name)
    assert packed.shape == (64, codec.row_bytes(name, 256))
    assert scales.shape == (64, codec.scale_count(name, 256))
    if name in codec.QMAX:
        q, _ = codec.quantize_rows(bits, name)
        assert np.array_equal(codec.unpack_codes(packed, name, 256), q)
    xhat = codec.decode_rows(packed, scales, name, 256)
    x = codec.bf16_bits_to_f64(bits)
    if name == "bf16":
        assert np.array_equal(xhat, x)
    elif name == "f16":
        assert np.max(np.abs(xhat - x) / np.abs(x)) <= 2.0 ** -11


def test_q4_error_larger_than_q8():
    bits = _random_rows(3, 256, 128)
    x = codec.bf16_bits_to_f64(bits)
    e8 = np.abs(codec.dequantized(bits, "q8_0") - x).mean()
    e4 = np.abs(codec.dequantized(bits, "q4s") - x).mean()
    # uniform rounding error d/4 on average, d = amax/127 vs amax/7
    assert 10 < e4 / e8 < 30


def test_dequantized_16_hand_values():
    """The separate dequantize pass's 16-bit values, derived by hand: exact products d*q
    rounded once to nearest even (ties included)."""
    # one q8_0 row of 32 elements: codes at 0..3, the rest zero; scales per block below
    cases = [
        # (scale bits, code, f16 bits, bf16 bits, why)
        (0x6156, 3, 0x6800, 0x4500, "683*3 = 2049: tie between 2048 and 2050 (f16) / 2048 and 2064 (bf16) -> 2048"),
        (0x3555, 127, 0x514A, 0x4229, "0.333251953125*127 = 42.322998...: f16 step 1/32 -> 42.3125, bf16 step 1/4 -> 42.25"),
        (0x3800, -7, 0xC300, 0xC060, "0.5*-7 = -3.5 exact in both"),
        (0x3555, -7, 0xC0AA, 0xC015, "-2.332763671875: f16 step 1/512 -> -2.33203125, bf16 step 1/64 -> -2.328125"),
    ]
    for sbits, q, f16_bits, bf16_bits, why in cases:
        packed = np.zeros((1, 32), np.uint8)
        packed[0, 5] = np.uint8(q & 0xFF)
        scales = np.array([[sbits]], np.uint16)
        got16 = codec.dequantized_16(packed, scales, "q8_0", 32, "f16")
        gotb = codec.dequantized_16(packed, scales, "q8_0", 32, "bf16")
        assert int(got16[0, 5]) == f16_bits, why
        assert int(gotb[0, 5]) == bf16_bits, why
        assert int(got16[0, 0]) == 0 and int(gotb[0, 0]) == 0
    # q4s: code -7 is nibble 1 (low nibble of byte 0 holds element 0)
    packed = np.zeros((1, 16), np.uint8)
    packed[0, 0] = 0x81            # element 0: u = 1 -> q = -7; element 1: u = 8 -> q = 0
    scales = np.array([[0x3555]], np.uint16)
    got = codec.dequantized_16(packed, scales, "q4s", 32, "f16")
    assert int(got[0, 0]) == 0xC0AA and int(got[0, 1]) == 0
