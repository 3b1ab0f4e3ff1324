"""Pins of the oracle attention and its split-K form (CPU)."""

import json
import math
import os

import numpy as np
import pytest

from oracle import attention

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "attention_cases.json")


def _num(v):
    if isinstance(v, str):
        return math.log(float(v[2:]))
    return float(v)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_golden_cases(case):
    q = np.array(case["q"], dtype=np.float64)
    k = np.array([[_num(x) for x in row] for row in case["k"]], dtype=np.float64)
    v = np.array(case["v"], dtype=np.float64)
    out = attention.attend_one(q, k, v, case["scale"])
    assert np.allclose(out, case["out"], rtol=0, atol=1e-12)
    # the split form through every chunk size reaches the same values
    for chunk in (1, 2, 3):
        assert np.allclose(attention.attend_one_split(q, k, v, case["scale"], chunk),
                           case["out"], rtol=0, atol=1e-12)


def _brute(q, k, v, scale):
    L, D = k.shape
    s = [scale * sum(q[j] * k[t][j] for j in range(D)) for t in range(L)]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    z = sum(w)
    return [sum(w[t] * v[t][j] for t in range(L)) / z for j in range(D)]


@pytest.mark.parametrize("seed", range(5))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    L, D = rng.integers(1, 9), rng.integers(1, 6)
    q, k, v = rng.normal(size=D), rng.normal(size=(L, D)) * 3, rng.normal(size=(L, D))
    scale = float(rng.uniform(0.1, 2))
    assert np.allclose(attention.attend_one(q, k, v, scale), _brute(q, k, v, scale),
                       rtol=0, atol=1e-12)


def test_closed_forms():
    rng = np.random.default_rng(7)
    D, L = 16, 50
    q = rng.normal(size=D)
    v = rng.normal(size=(L, D))
    # identical keys: uniform weights -> mean of V
    k = np.tile(rng.normal(size=D), (L, 1))
    assert np.allclose(attention.attend_one(q, k, v, 0.3), v.mean(axis=0), atol=1e-12)
    # zero scale: uniform weights too
    k = rng.normal(size=(L, D))
    assert np.allclose(attention.attend_one(q, k, v, 0.0), v.mean(axis=0), atol=1e-12)
    # one dominant score: that V row
    k2 = k.copy()
    k2[17] = q * 1e4
    assert np.allclose(attention.attend_one(q, k2, v, 1.0), v[17], atol=1e-12)
    # a single token: its V row
    assert np.allclose(attention.attend_one(q, k[:1], v[:1], 1.0), v[0], atol=1e-15)
    # empty prefix: zeros
    assert np.all(attention.attend_one(q, k[:0], v[:0], 1.0) == 0)


def test_token_permutation_invariance():
    rng = np.random.default_rng(8)
    q, k, v = rng.normal(size=32), rng.normal(size=(300, 32)), rng.normal(size=(300, 32))
    perm = rng.permutation(300)
    a = attention.attend_one(q, k, v, 0.2)
    b = attention.attend_one(q, k[perm], v[perm], 0.2)
    assert np.allclose(a, b, atol=1e-13)


def test_gqa_head_mapping_and_default_scale():
    rng = np.random.default_rng(9)
    B, Hq, Hkv, D, L = 2, 6, 2, 16, 10
    q = rng.normal(size=(B, Hq, D))
    ks = [rng.normal(size=(L, Hkv, D)) for _ in range(B)]
    vs = [rng.normal(size=(L, Hkv, D)) + 10 * np.arange(Hkv)[None, :, None] for _ in range(B)]
    out = attention.attention(q, ks, vs, Hkv)
    for b in range(B):
        for h in range(Hq):
            kv = h // 3   # contiguous groups of G = 3 query heads
            want = attention.attend_one(q[b, h], ks[b][:, kv], vs[b][:, kv], 1 / math.sqrt(D))
            assert np.allclose(out[b, h], want, atol=1e-13)
            # the group's KV head shows in the output's offset (10 * kv)
            assert abs(out[b, h].mean() - 10 * kv) < 3
    # G = 1 is plain multi-head attention
    out1 = attention.attention(q[:, :2], [k[:, :2] for k in ks], [v[:, :2] for v in vs], 2)
    for h in range(2):
        assert np.allclose(out1[0, h], attention.attend_one(q[0, h], ks[0][:, h], vs[0][:, h],
                                                            0.25), atol=1e-13)


@pytest.mark.parametrize("chunk", [1, 7, 64, 256, 1000])
def test_split_invariance(chunk):
    rng = np.random.default_rng(10)
    q, k, v = rng.normal(size=64), rng.normal(size=(777, 64)) * 2, rng.normal(size=(777, 64))
    whole = attention.attend_one(q, k, v, 0.125)
    split = attention.attend_one_split(q, k, v, 0.125, chunk)
    assert np.max(np.abs(whole - split)) < 1e-12


def test_zero_length_sequence_in_batch():
    rng = np.random.default_rng(11)
    q = rng.normal(size=(2, 2, 8))
    ks = [np.zeros((0, 1, 8)), rng.normal(size=(5, 1, 8))]
    vs = [np.zeros((0, 1, 8)), rng.normal(size=(5, 1, 8))]
    out = attention.attention(q, ks, vs, 1)
    assert np.all(out[0] == 0) and np.all(np.isfinite(out[1]))


def test_attend_tokens_hand_case():
    # all scores equal: each draft query averages the positions it may see.  L = 3, T = 2:
    # query 0 sees positions 0..1 (mean of 1, 3 = 2), query 1 sees 0..2 (mean of 1, 3, 8 = 4)
    q = np.array([[0.7], [-1.2]])
    k = np.zeros((3, 1))
    v = np.array([[1.0], [3.0], [8.0]])
    out = attention.attend_tokens(q, k, v, 1.0)
    assert out[0, 0] == pytest.approx(2.0, abs=1e-15)
    assert out[1, 0] == pytest.approx(4.0, abs=1e-15)


def test_attend_tokens_reduces_to_attend_one():
    rng = np.random.default_rng(7)
    k, v = rng.standard_normal((40, 16)), rng.standard_normal((40, 16))
    q = rng.standard_normal((5, 16))
    out = attention.attend_tokens(q, k, v, 0.25)
    # the last draft sees the whole sequence; T = 1 is single-token decode
    np.testing.assert_allclose(out[4], attention.attend_one(q[4], k, v, 0.25), rtol=0, atol=1e-14)
    np.testing.assert_allclose(attention.attend_tokens(q[:1], k, v, 0.25)[0],
                               attention.attend_one(q[0], k, v, 0.25), rtol=0, atol=1e-14)
    # draft i equals a single-token decode of the sequence cut after position L - T + i
    for i in range(5):
        np.testing.assert_allclose(out[i], attention.attend_one(q[i], k[:36 + i], v[:36 + i], 0.25),
                                   rtol=0, atol=1e-14)


def test_attend_tokens_sequence_shorter_than_drafts():
    # L = 1, T = 3: queries 0 and 1 see nothing (zeros), query 2 sees position 0
    q = np.ones((3, 2))
    k = np.ones((1, 2))
    v = np.array([[5.0, -2.0]])
    out = attention.attend_tokens(q, k, v, 1.0)
    assert np.array_equal(out[0], [0.0, 0.0]) and np.array_equal(out[1], [0.0, 0.0])
    np.testing.assert_array_equal(out[2], [5.0, -2.0])
