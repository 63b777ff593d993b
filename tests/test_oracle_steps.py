"""Pins for the oracle's steps: Hadamard rotation, affine quantizer, INT8 query.

Each check uses something other than the oracle: the dense Sylvester matrix
built from (−1)^popcount(i&j), float64 arithmetic, numpy's fp16 decoder, and
the values the pages print (tests/golden/pages_constants.json).
"""
import json
import os

import numpy as np
import pytest

import oracle
from int8_hybrid_paged_gb300 import bytes_model

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")))
D = 128


def dense_hadamard():
    i = np.arange(D)
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0) / np.sqrt(D)


def f16v(bits):
    return np.array(bits, np.uint16).view(np.float16).astype(np.float64)


# --------------------------------------------------------------------------- rotation

def test_fwht_equals_dense_sylvester_matrix():
    H = dense_hadamard()
    cols = np.stack([oracle.fwht128(np.eye(D, dtype=np.float32)[i]) for i in range(D)], axis=1)
    np.testing.assert_allclose(cols, H, rtol=0, atol=1e-8)
    np.testing.assert_allclose(cols @ cols.T, np.eye(D), rtol=0, atol=1e-6)
    np.testing.assert_allclose(H, H.T)
    rng = np.random.default_rng(0)
    for _ in range(20):
        x = (rng.standard_normal(D) * rng.choice([1, 20], D)).astype(np.float32)
        ref = H @ x.astype(np.float64)
        np.testing.assert_allclose(oracle.fwht128(x), ref, rtol=0,
                                   atol=1e-6 * np.abs(x).sum() / np.sqrt(D))


def test_rotation_preserves_scores_and_is_an_involution():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((16, D)).astype(np.float32)
    k = (rng.standard_normal((16, D)) * np.where(np.isin(np.arange(D), [5, 37, 70, 101]), 20, 1)
         ).astype(np.float32)
    qr = np.stack([oracle.fwht128(r) for r in q]).astype(np.float64)
    kr = np.stack([oracle.fwht128(r) for r in k]).astype(np.float64)
    ref = q.astype(np.float64) @ k.astype(np.float64).T
    scale = np.linalg.norm(q, axis=1)[:, None] * np.linalg.norm(k, axis=1)[None, :]
    assert np.max(np.abs(qr @ kr.T - ref) / scale) < 1e-6
    back = np.stack([oracle.fwht128(r.astype(np.float32)) for r in qr])
    np.testing.assert_allclose(back, q, rtol=0, atol=1e-5)


# --------------------------------------------------------------------------- quantizer

def _vectors():
    rng = np.random.default_rng(2)
    out = []
    for _ in range(200):
        out.append(rng.standard_normal(D))
        out.append(rng.standard_normal(D) * np.where(rng.random(D) < 0.03, 20, 1))
        out.append(rng.uniform(-1e-3, 1e-3, D))
        out.append(rng.uniform(3, 7, D) * 10.0 ** rng.integers(-6, 3))
        out.append(rng.standard_normal(D) * 1e-6)
    out.append(np.zeros(D))
    out.append(np.full(D, 0.1))
    out.append(np.full(D, -123.456))
    return [v.astype(np.float32) for v in out]


@pytest.mark.parametrize("levels", [15, 255])
def test_affine_quantizer_bounds(levels):
    for x in _vectors():
        code, dh, mh = oracle.quant_affine(x, levels)
        delta, m = f16v(dh), f16v(mh)
        lo, hi = float(x.min()), float(x.max())
        assert code.max() <= levels
        # m is the largest fp16 value not above min x
        assert m <= lo
        assert np.nextafter(np.float16(m), np.float16(np.inf)).astype(np.float64) > lo
        # the grid covers the group
        assert m + levels * delta >= hi
        if delta == 0:
            # only a group whose values are all the same fp16 number has no spread
            assert lo == hi == m and np.all(code == 0)
            continue
        # Δ is the smallest fp16 step that covers, up to the float32 rounding before it
        prev = np.nextafter(np.float16(delta), np.float16(0)).astype(np.float64)
        assert prev * levels < (hi - m) * (1 + 2.0 ** -22)
        # reconstruction error ≤ Δ/2 (plus the float32 rounding of the quotient)
        rec = delta * code.astype(np.float64) + m
        assert np.all(np.abs(x.astype(np.float64) - rec) <= delta / 2 * (1 + 2.0 ** -20))
        # the code is the nearest grid index
        t = (x.astype(np.float64) - m) / delta
        assert np.all(np.abs(code - t) <= 0.5 + 1e-5)


def test_affine_quantizer_special_cases():
    # constant fp16-exact group: Δ = 0, every code 0, exact reconstruction
    x = np.full(D, 0.375, np.float32)
    code, dh, mh = oracle.quant_affine(x, 15)
    assert f16v(dh) == 0 and np.all(code == 0) and f16v(mh) == 0.375
    # constant group between fp16 values: m is the value rounded down, one shared
    # code, and the reconstruction error stays below one fp16 step of the value
    x = np.full(D, 0.3, np.float32)
    code, dh, mh = oracle.quant_affine(x, 15)
    assert 0 < 0.3 - f16v(mh) < np.spacing(np.float16(0.3)).astype(np.float64)
    assert np.all(code == code[0])
    rec = f16v(dh) * code.astype(np.float64) + f16v(mh)
    assert np.all(np.abs(rec - np.float32(0.3)) <= f16v(dh) / 2 * (1 + 2.0 ** -20))
    # two values one fp16-exact grid apart: endpoints reconstruct exactly
    x = np.where(np.arange(D) % 3 == 0, -1.0, 14.0).astype(np.float32)
    code, dh, mh = oracle.quant_affine(x, 15)
    assert f16v(dh) == 1.0 and f16v(mh) == -1.0
    np.testing.assert_array_equal(f16v(dh) * code + f16v(mh), x)
    x = np.where(np.arange(D) % 2 == 0, 2.0, 2.0 + 255 * 0.25).astype(np.float32)
    code, dh, mh = oracle.quant_affine(x, 255)
    np.testing.assert_array_equal(f16v(dh) * code + f16v(mh), x)


def test_bits_per_element_matches_pages():
    g = GOLDEN["group_size"]["value"]
    b = GOLDEN["code_bits_main"]["value"]
    assert bytes_model.affine_bits_per_element(g, b, 16, 2) == GOLDEN["bits_per_element"]["value"]
    # and the packed layout really stores that much per token-head and tensor
    assert (bytes_model.INT4_CODE_BYTES + bytes_model.META_BYTES) * 8 / g == 4.25


# --------------------------------------------------------------------------- query

def test_int8_query_quantization():
    rng = np.random.default_rng(4)
    for i in range(300):
        q = (rng.standard_normal(D) * 10 ** rng.uniform(-4, 2)).astype(np.float32)
        q8, sq, qs = oracle.quant_query(q)
        assert np.abs(q8.astype(np.int32)).max() == 127
        assert qs == int(q8.astype(np.int64).sum())
        assert np.isclose(sq, np.abs(q).max() / 127, rtol=2 ** -23)
        err = np.abs(q.astype(np.float64) - q8 * float(sq))
        assert np.all(err <= float(sq) / 2 * (1 + 1e-5))
    q8, sq, qs = oracle.quant_query(np.zeros(D, np.float32))
    assert sq == 0 and qs == 0 and np.all(q8 == 0)
