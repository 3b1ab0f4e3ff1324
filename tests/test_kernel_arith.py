"""Bit-level arithmetic the CUDA kernels rely on, checked exhaustively in float64 / float16
on the CPU (numpy only; no oracle, no CUDA).

Decode (the magic-number conversions of integer codes to f16 in registers):

* an 8-bit code q, its byte flipped to q + 128 and placed under the f16 exponent byte 0x64,
  is the f16 value 1152 + q, and one f16 subtraction of 1152 gives q exactly;
* a 4-bit code stored as u = q + 8: in mantissa bits 0-3 under 0x64 it is 1024 + u (less
  1032 gives q); in bits 4-7 under 0x64 it is 1024 + 16 u, and one fma with (1/16, -72) gives
  q; in bits 4-7 under 0x48 (the K form) it is 9 + q / 8.

Tensor-core prefill:

* a quantized tile becomes two f16 operands, hi = d q rounded and nlo = hi - d q (stored
  negated, read with the MMA's negate-B bit), with d the block scale times the tile's power
  of two 2^-sigma: sigma = e - 22 (e the biased exponent of the tile's largest scale) must
  put every prescaled scale below 2^8, and there hi - nlo must equal d q exactly for every
  f16 d and every code q of q8_0 (and so of q4s);
* a q4s byte b becomes the f16 pair of its two codes through the bits
  (b | b << 16) & 0x00F0000F | 0x64006400 and one fma with the per-half constants
  (1, 1/16) and (-1032, -72) (bit patterns 0x3C00, 0x2C00, 0xE408, 0xD480)."""

import numpy as np


def f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def rn16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


ALL_F16 = np.arange(1, 0x7C00, dtype=np.uint16)   # every positive finite f16, subnormals included


def test_hi_lo_split_is_exact_for_every_prescaled_f16_scale_and_code():
    # every f16 value below 2^8 (the prescaled range), subnormals included
    d = f16(ALL_F16[f16(ALL_F16) < 256.0])[:, None]
    q = np.arange(-127, 128, dtype=np.float64)[None, :]
    p = d * q                       # exact in float64 (11 x 7 significant bits)
    hi = rn16(p)
    nlo = rn16(hi - p)              # what the kernel's fma(q, -d, hi) rounds once
    assert np.all(np.isfinite(hi))
    assert np.array_equal(hi - nlo, p)


def test_tile_exponent_keeps_hi_below_2_to_15():
    bits = ALL_F16
    e = (bits >> 10).astype(np.int64)            # biased exponent of the tile's largest scale
    sigma = e - 22
    ds = f16(bits) * np.exp2(-sigma.astype(np.float64))
    assert np.array_equal(rn16(ds), ds)          # the prescaled largest scale is an exact f16
    assert ds.min() >= 0.25 and ds.max() < 256.0
    assert np.all(rn16(127.0 * ds) < 2.0 ** 15)  # |d q| 2^-sigma stays in range for |q| <= 127


def test_smaller_scales_of_a_tile_prescale_exactly_above_the_f16_normal_range():
    # d <= d_max: d 2^-sigma is exact whenever it is a normal f16 (a power-of-two shift);
    # below 2^-14 it is rounded to the subnormal grid (absolute error <= 2^-25, against a
    # prescaled maximum of at least 2^7 in the same tile)
    for e_max in range(1, 31):
        sigma = e_max - 22
        d = f16(ALL_F16[(ALL_F16 >> 10) <= e_max])
        ds = d * 2.0 ** (-sigma)
        got = rn16(ds)
        normal = ds >= 2.0 ** -14
        assert np.array_equal(got[normal], ds[normal])
        assert np.abs(got - ds).max() <= 2.0 ** -25


def test_q4s_byte_to_code_pair():
    mul_lo, mul_hi = f16(0x3C00), f16(0x2C00)     # 1, 1/16
    add_lo, add_hi = f16(0xE408), f16(0xD480)     # -1032, -72
    assert (mul_lo, mul_hi, add_lo, add_hi) == (1.0, 1.0 / 16, -1032.0, -72.0)
    b = np.arange(256, dtype=np.uint32)
    x = ((b | (b << 16)) & 0x00F0000F) | 0x64006400
    lo = f16(x & 0xFFFF)                          # 1024 + low nibble
    hi = f16(x >> 16)                             # 1024 + 16 high nibble
    assert np.array_equal(lo, 1024.0 + (b & 15)) and np.array_equal(hi, 1024.0 + 16.0 * (b >> 4))
    q_lo = rn16(lo * mul_lo + add_lo)             # fma: exact product and sum, one rounding
    q_hi = rn16(hi * mul_hi + add_hi)
    assert np.array_equal(q_lo, (b & 15).astype(np.float64) - 8)
    assert np.array_equal(q_hi, (b >> 4).astype(np.float64) - 8)


def test_8bit_code_under_0x64_less_1152_is_the_code():
    q = np.arange(-128, 128)
    u = (q + 128) & 0xFF                          # the byte after the sign flip (xor 0x80)
    x = f16(0x6400 | u)
    assert np.array_equal(x, 1152.0 + q)
    assert np.array_equal(rn16(x - f16(0x6480)), q.astype(np.float64))   # 0x6480 = 1152


def test_4bit_code_forms():
    q = np.arange(-8, 8)
    u = q + 8
    low = f16(0x6400 | u)                          # mantissa bits 0-3
    assert np.array_equal(low, 1032.0 + q) and np.array_equal(rn16(low - f16(0x6408)), q.astype(np.float64))
    high = f16(0x6400 | (u << 4))                  # mantissa bits 4-7
    assert np.array_equal(rn16(high * f16(0x2C00) + f16(0xD480)), q.astype(np.float64))   # (x / 16) - 72
    k_form = f16(0x4800 | (u << 4))                # the K codes: 8 + u / 8
    assert np.array_equal(k_form, 9.0 + q / 8.0)
