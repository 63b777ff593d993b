"""Pins for the oracle's RoPE (reading R11): keys rotated by RoPE at their position
before the Hadamard transform, queries at position L − 1.

References used here, none of them the oracle's own code:
  * the float64 complex rotation (x_i + i x_{i+64}) e^{iθ};
  * exact special angles (0, π/2) where the result is a permutation with a sign;
  * the float64 dense Hadamard matrix and the quantizer's Δ/2 bound;
  * the relative-position property of rotary embeddings.
"""
import math

import numpy as np
import pytest

import oracle
from int8_hybrid_paged_gb300 import inputs

D = 128


def bits_to_f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def textbook_rope(x, row):
    z = x[:64].astype(np.float64) + 1j * x[64:].astype(np.float64)
    z = z * (row[:64].astype(np.float64) + 1j * row[64:].astype(np.float64))
    return np.concatenate([z.real, z.imag])


def test_rope_is_the_complex_rotation_of_pairs_i_and_i_plus_64():
    rng = np.random.default_rng(0)
    tab = inputs.rope_table(4096)
    for p in (0, 1, 7, 100, 4095):
        x = rng.standard_normal(D).astype(np.float32) * 3
        got = oracle.rope128(x, tab[p]).astype(np.float64)
        ref = textbook_rope(x, tab[p])
        mag = np.abs(np.concatenate([x[:64] * tab[p, :64], x[64:] * tab[p, :64]])) + \
            np.abs(np.concatenate([x[64:] * tab[p, 64:], x[:64] * tab[p, 64:]]))
        assert np.all(np.abs(got - ref) <= 2.0 ** -22 * mag + 1e-30)


def test_special_angles_are_exact():
    x = np.arange(1, D + 1, dtype=np.float32)
    row = np.concatenate([np.ones(64), np.zeros(64)]).astype(np.float32)
    np.testing.assert_array_equal(oracle.rope128(x, row), x)          # angle 0: identity
    row[5], row[64 + 5] = 0.0, 1.0                                     # pair 5 by π/2
    got = oracle.rope128(x, row)
    assert got[5] == -x[69] and got[69] == x[5]
    keep = np.ones(D, bool)
    keep[[5, 69]] = False
    np.testing.assert_array_equal(got[keep], x[keep])


def test_relative_positions():
    """⟨RoPE(q, m), RoPE(k, n)⟩ depends on m − n only (to FP32 rounding)."""
    rng = np.random.default_rng(1)
    tab = inputs.rope_table(3000)
    q = rng.standard_normal(D).astype(np.float32)
    k = rng.standard_normal(D).astype(np.float32)
    for m, n in ((10, 3), (500, 17), (2000, 1999)):
        base = float(oracle.rope128(q, tab[m]).astype(np.float64) @ oracle.rope128(k, tab[n]))
        for d in (1, 250, 900):
            sh = float(oracle.rope128(q, tab[m + d]).astype(np.float64)
                       @ oracle.rope128(k, tab[n + d]))
            assert abs(sh - base) <= 2e-5 * (np.abs(q) @ np.abs(k))


def test_identity_table_changes_nothing():
    H, G, L = 2, 4, 200
    k, v = inputs.sequence_kv(0, L, H, 3)
    kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
    ident = np.tile(np.concatenate([np.ones(64), np.zeros(64)]).astype(np.float32), (L, 1))
    a = oracle.OracleCache(H, 16, 128, L)
    b = oracle.OracleCache(H, 16, 128, L, rope=ident)
    a.append(0, 0, kb, vb)
    b.append(0, 0, kb, vb)
    for n in ("k4_code", "k4_delta", "k4_min", "k8_code", "k8_delta", "k8_min"):
        np.testing.assert_array_equal(getattr(a, n), getattr(b, n))
    q = inputs.bf16_bits(inputs.queries(1, H * G, seed=2))
    oa, la, _ = a.decode(0, L, G, q[0], 0.1)
    ob, lb, _ = b.decode(0, L, G, q[0], 0.1)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(la, lb)


@pytest.mark.parametrize("kv8", [False, True])
def test_keys_are_rope_then_hadamard(kv8):
    """Stored keys reconstruct H̃·RoPE(k, p) (float64 textbook rotation, dense
    Hadamard) within the quantizer's Δ/2 bound, at every position."""
    H, L = 1, 70
    s, w = (0, 0) if kv8 else (16, 128)
    tab = inputs.rope_table(L)
    k, v = inputs.sequence_kv(0, L, H, 5)
    kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
    c = oracle.OracleCache(H, s, w, L, kv8=kv8, rope=tab)
    c.append(0, 0, kb, vb)
    i = np.arange(D)
    pop = np.vectorize(lambda x: bin(int(x)).count("1"))(i[:, None] & i[None, :])
    Hd = np.where(pop % 2 == 0, 1.0, -1.0) / math.sqrt(D)
    kf = bits_to_f32(kb)
    for p in range(L):
        x = textbook_rope(kf[p, 0], tab[p]) @ Hd
        d = np.asarray(c.k4_delta[0, p, 0], np.uint16).view(np.float16).astype(np.float64)
        m = np.asarray(c.k4_min[0, p, 0], np.uint16).view(np.float16).astype(np.float64)
        rec = d * c.k4_code[0, p, 0] + m
        assert np.all(np.abs(rec - x) <= d / 2 * (1 + 2 ** -20) + 1e-5 * np.abs(x).max())


def test_query_takes_the_position_of_the_last_token():
    H, G, L = 1, 2, 50
    tab = inputs.rope_table(64)
    k, v = inputs.sequence_kv(0, L, H, 6)
    c = oracle.OracleCache(H, 16, 128, L, rope=tab)
    c.append(0, 0, inputs.bf16_bits(k), inputs.bf16_bits(v))
    qb = inputs.bf16_bits(inputs.queries(1, H * G, seed=4))[0]
    _, _, dbg = c.decode(0, L, G, qb, 0.1, debug=True)
    for hq in range(H * G):
        q8, sq, _ = oracle.quant_query(oracle.fwht128(oracle.rope128(bits_to_f32(qb[hq]), tab[L - 1])))
        np.testing.assert_array_equal(dbg["q8"][hq], q8)
        assert dbg["q_scale"][hq] == np.float32(sq)


def test_positions_beyond_the_table_are_rejected():
    tab = inputs.rope_table(40)
    k, v = inputs.sequence_kv(0, 41, 1, 1)
    c = oracle.OracleCache(1, 16, 128, 41, rope=tab)
    with pytest.raises(ValueError):
        c.append(0, 0, inputs.bf16_bits(k), inputs.bf16_bits(v))
    c.append(0, 0, inputs.bf16_bits(k[:40]), inputs.bf16_bits(v[:40]))
    q = inputs.bf16_bits(inputs.queries(1, 2, seed=1))
    c.decode(0, 40, 2, q[0], 0.1)
    with pytest.raises(ValueError):
        c.decode(0, 41, 2, q[0], 0.1)
