"""Oracle block codecs: q8_0, 4-bit symmetric (q4s), and the bf16 / f16 control stores.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Codec contract (q8_0 is the quantized KV type of "halobench record clm-0022", METHOD and
depth tables; the 4-bit-V family is named in rMLX issue #292, correction table; neither
page prints the arithmetic, so the rule below is the library's contract):

  for every stored row (one token, one KV head) and every block of 32 consecutive
  elements along head_dim, with the inputs x_j given as bf16:
    amax = max_j |x_j|
    d32  = amax / c                  (IEEE fp32 quotient; c = 127 for q8_0, 7 for q4s)
    d    = fp16(d32)                 (round to nearest even, subnormals kept)
    q_j  = 0                         if d == 0
         = clamp(round_half_away(fp32(x_j / d)), -c, c)   otherwise
  dequantized value: x^_j = d * q_j (exact in float64)

Packing:
  q8_0: one int8 (two's complement) per element, element order.
  q4s : u_j = q_j + 8 in [1, 15]; block element 2k sits in the low nibble of block byte k
        and element 2k+1 in its high nibble, so 32 elements fill 16 bytes (read as four
        little-endian uint32 words, element 8w+e is bits 4e..4e+3 of word w).
  scales: the fp16 bit pattern of d, one per block, block order.
  bf16 control: the input bits unchanged.  f16 control: fp16(x) with round to nearest even.

Floating point decides the integer codes, so the oracle takes those decisions in the
precision the contract names (fp32 quotient, fp16 scale) and does everything else in
float64.

Pinned by tests/test_oracle_codec.py against hand-derived blocks (tests/golden/codec_blocks.json),
the round-trip bound, |q| <= c, "some |q_j| == c" and brute force over all 2^16 bf16
inputs of a 1-element block position.
"""

from __future__ import annotations

import numpy as np

BLOCK = 32
CODEC_IDS = {"bf16": 0, "f16": 1, "q8_0": 2, "q4s": 3}
QMAX = {"q8_0": 127, "q4s": 7}


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns (uint16) -> exact float64 values."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def f64_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values that are exactly representable in fp32 to fp16 (nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float16).view(np.uint16)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values that are exactly representable in fp32 to bf16 (nearest even;
    finite inputs)."""
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def row_bytes(codec: str, head_dim: int) -> int:
    """Bytes of one stored row (one token of one KV head), excluding scales."""
    return {"bf16": 2 * head_dim, "f16": 2 * head_dim, "q8_0": head_dim,
            "q4s": head_dim // 2}[codec]


def scale_count(codec: str, head_dim: int) -> int:
    """fp16 scales per stored row."""
    return head_dim // BLOCK if codec in QMAX else 0


def _round_half_away(r: np.ndarray) -> np.ndarray:
    return np.sign(r) * np.floor(np.abs(r) + 0.5)


def quantize_rows(x_bits: np.ndarray, codec: str):
    """Block-quantize rows of bf16 bits.

    x_bits: uint16 [N, D] (bf16 bit patterns), D a multiple of 32.
    Returns (q int32 [N, D], d_bits uint16 [N, D/32]).
    """
    c = QMAX[codec]
    x = bf16_bits_to_f64(x_bits)
    n, dim = x.shape
    assert dim % BLOCK == 0
    xb = x.reshape(n, dim // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=2)
    # fp32 quotient amax / c: the float64 quotient of two fp32 values rounded once more to
    # fp32 is the correctly rounded fp32 quotient (53 >= 2*24 + 2).
    d32 = (amax / c).astype(np.float32)
    d_bits = d32.astype(np.float16).view(np.uint16)
    d = f16_bits_to_f64(d_bits)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (xb / d[:, :, None]).astype(np.float32).astype(np.float64)
    q = np.clip(_round_half_away(r), -c, c)
    q = np.where((d == 0)[:, :, None], 0.0, q)
    return q.reshape(n, dim).astype(np.int32), d_bits


def pack_codes(q: np.ndarray, codec: str) -> np.ndarray:
    """Integer codes [N, D] -> packed row bytes uint8 [N, row_bytes]."""
    if codec == "q8_0":
        return q.astype(np.int8).view(np.uint8)
    if codec == "q4s":
        u = (q + 8).astype(np.uint8)
        return (u[:, 0::2] | (u[:, 1::2] << np.uint8(4))).astype(np.uint8)
    raise ValueError(codec)


def unpack_codes(packed: np.ndarray, codec: str, head_dim: int) -> np.ndarray:
    """Packed row bytes uint8 [N, row_bytes] -> integer codes int32 [N, D]."""
    packed = np.asarray(packed, dtype=np.uint8)
    if codec == "q8_0":
        return packed.view(np.int8).astype(np.int32)
    if codec == "q4s":
        q = np.empty((packed.shape[0], head_dim), dtype=np.int32)
        q[:, 0::2] = (packed & 0x0F).astype(np.int32) - 8
        q[:, 1::2] = (packed >> 4).astype(np.int32) - 8
        return q
    raise ValueError(codec)


def encode_rows(x_bits: np.ndarray, codec: str):
    """bf16 rows [N, D] -> (row bytes uint8 [N, row_bytes], scale bits uint16 [N, nb]).

    The 16-bit codecs have no scales (an [N, 0] array is returned).
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    n, dim = x_bits.shape
    if codec == "bf16":
        return x_bits.copy().view(np.uint8).reshape(n, 2 * dim), np.zeros((n, 0), np.uint16)
    if codec == "f16":
        h = f64_to_f16_bits(bf16_bits_to_f64(x_bits))
        return h.view(np.uint8).reshape(n, 2 * dim), np.zeros((n, 0), np.uint16)
    q, d_bits = quantize_rows(x_bits, codec)
    return pack_codes(q, codec), d_bits


def decode_rows(packed: np.ndarray, scales: np.ndarray, codec: str, head_dim: int) -> np.ndarray:
    """Stored rows -> dequantized float64 values [N, D]: x^_j = d_block(j) * q_j."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    n = packed.shape[0]
    if codec == "bf16":
        return bf16_bits_to_f64(packed.view(np.uint16).reshape(n, head_dim))
    if codec == "f16":
        return f16_bits_to_f64(packed.view(np.uint16).reshape(n, head_dim))
    q = unpack_codes(packed, codec, head_dim).astype(np.float64)
    d = f16_bits_to_f64(scales)
    return (q.reshape(n, head_dim // BLOCK, BLOCK) * d[:, :, None]).reshape(n, head_dim)


def dequantized(x_bits: np.ndarray, codec: str) -> np.ndarray:
    """encode then decode: the values a decode kernel must attend over."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    packed, scales = encode_rows(x_bits, codec)
    return decode_rows(packed, scales, codec, x_bits.shape[1])


def dequantized_16(packed: np.ndarray, scales: np.ndarray, codec: str, head_dim: int,
                   target: str) -> np.ndarray:
    """The 16-bit rows a separate dequantize pass writes (the "stock" arm of halobench
    record clm-0022, METHOD and depth tables: quantized KV converted in its own pass, then
    read by a 16-bit decode): bits of fp16_rn(d * q) for target "f16", bf16_rn(d * q) for
    "bf16".  d * q (11-bit scale times a code of at most 8 bits) is exact in fp32, so one
    rounding from the exact product."""
    x = decode_rows(packed, scales, codec, head_dim)
    if target == "f16":
        return f64_to_f16_bits(x)
    if target == "bf16":
        return f64_to_bf16_bits(x)
    raise ValueError(target)

