"""Pins for the oracle's whole-cache 8-bit configuration (KV8, reading R10).

References used here, none of them the oracle's own code:
  * the dense Sylvester Hadamard matrix in float64 for the key rotation;
  * numpy int64 matmul for the integer dot products;
  * a textbook float64 softmax attention over the oracle's dequantized state;
  * the hybrid configuration with every position protected (L <= s + w), itself
    pinned against the textbook attention in test_oracle_attention.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from int8_hybrid_paged_gb300 import inputs

D = 128


def f16v(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def bf16_round(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16) \
        .to(torch.float32).numpy().astype(np.float64)


def hadamard():
    i = np.arange(D)
    bits = np.bitwise_and(i[:, None], i[None, :])
    pop = np.vectorize(lambda x: bin(int(x)).count("1"))(bits)
    return np.where(pop % 2 == 0, 1.0, -1.0) / math.sqrt(D)


def make(H, lens, seed=0, kv8=True, s=0, w=0):
    c = oracle.OracleCache(H, s, w, max(lens), num_slots=len(lens), kv8=kv8)
    raw = []
    for b, L in enumerate(lens):
        k, v = inputs.sequence_kv(b, L, H, seed)
        kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
        c.append(b, 0, kb, vb)
        raw.append((kb, vb))
    return c, raw


def textbook(c, slot, L, G, dbg, sm_scale):
    """float64 softmax attention over every position's dequantized 8-bit key and its
    BF16-rounded dequantized value, with the INT8 query q8·s_q (natural-log units)."""
    H = c.H
    out = np.zeros((H * G, D))
    lse = np.full(H * G, -np.inf)
    for hq in range(H * G):
        h = hq // G
        if L == 0:
            continue
        qhat = dbg["q8"][hq].astype(np.float64) * float(dbg["q_scale"][hq])
        K = f16v(c.k4_delta[slot, :L, h])[:, None] * c.k4_code[slot, :L, h] \
            + f16v(c.k4_min[slot, :L, h])[:, None]
        v32 = (f16v(c.v4_delta[slot, :L, h])[:, None] * c.v4_code[slot, :L, h].astype(np.float64)
               + f16v(c.v4_min[slot, :L, h])[:, None]).astype(np.float32)
        V = bf16_round(v32)
        sc = (K @ qhat) * sm_scale
        mx = sc.max()
        p = np.exp(sc - mx)
        out[hq] = p @ V / p.sum()
        lse[hq] = mx + math.log(p.sum())
    return out, lse


LENS = [1, 15, 16, 17, 40, 161, 300]


def test_codes_are_8bit_affine_of_rotated_keys_and_plain_values():
    """Every position: |Δc + m − x| ≤ Δ/2 (1 + 2^-20) for x = H̃k (float64 dense
    Hadamard) and for x = v (unrotated), codes spanning 0..255."""
    H = 2
    c, raw = make(H, [70])
    Hd = hadamard()
    kb, vb = raw[0]
    k = (kb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    v = (vb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(70):
        for h in range(H):
            for x, code, dl, mn in ((k[t, h] @ Hd, c.k4_code, c.k4_delta, c.k4_min),
                                    (v[t, h], c.v4_code, c.v4_delta, c.v4_min)):
                d = f16v(dl[0, t, h])
                rec = d * code[0, t, h] + f16v(mn[0, t, h])
                assert np.all(np.abs(rec - x) <= d / 2 * (1 + 2 ** -20) + 1e-6 * np.abs(x).max())
                assert code[0, t, h].max() == 255 or d == 0
    assert c.side_bytes() == 0                         # no side buffer in KV8


@pytest.mark.parametrize("G", [1, 2, 4])
def test_integer_qk_over_every_position(G):
    H = 2
    c, _ = make(H, LENS)
    q = inputs.bf16_bits(inputs.queries(len(LENS), H * G, seed=7))
    for b, L in enumerate(LENS):
        _, _, dbg = c.decode(b, L, G, q[b], 1 / math.sqrt(D), debug=True)
        for hq in range(H * G):
            ref = c.k4_code[b, :L, hq // G].astype(np.int64) @ dbg["q8"][hq].astype(np.int64)
            np.testing.assert_array_equal(dbg["qk"][hq, :L], ref)
            assert np.all(dbg["w_hat"][hq, :L] == 0)    # no u8 PV weights in KV8


@pytest.mark.parametrize("G", [1, 4])
def test_float_pv_equals_single_softmax(G):
    H = 2
    sm = 1 / math.sqrt(D)
    c, _ = make(H, LENS)
    q = inputs.bf16_bits(inputs.queries(len(LENS), H * G, seed=8))
    for b, L in enumerate(LENS):
        out, lse, dbg = c.decode(b, L, G, q[b], sm, pv_mode=oracle.PV_FLOAT, debug=True)
        ref, ref_lse = textbook(c, b, L, G, dbg, sm)
        np.testing.assert_allclose(out, ref, rtol=0, atol=2e-6 * max(1.0, np.abs(ref).max()))
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=2e-6 * max(1, np.abs(ref_lse).max()))


def test_bf16_weights_within_rounding_bound():
    """Integer mode rounds each p to BF16 (8 significant bits): each position moves
    an output element by at most 2^-8 2^(σ_t − M*) |v_tj| / den (1% slack)."""
    H, G = 1, 2
    sm = 1 / math.sqrt(D)
    c, _ = make(H, LENS)
    q = inputs.bf16_bits(inputs.queries(len(LENS), H * G, seed=9))
    for b, L in enumerate(LENS):
        o_int, lse_i, dbg = c.decode(b, L, G, q[b], sm, pv_mode=oracle.PV_INTEGER, debug=True)
        o_flt, lse_f, _ = c.decode(b, L, G, q[b], sm, pv_mode=oracle.PV_FLOAT)
        np.testing.assert_array_equal(lse_i, lse_f)
        for hq in range(H * G):
            sig = dbg["sigma"][hq, :L].astype(np.float64)
            Ms = sig.max()
            den = math.exp2(lse_i[hq] / math.log(2) - Ms)
            v32 = (f16v(c.v4_delta[b, :L, 0])[:, None] * c.v4_code[b, :L, 0].astype(np.float64)
                   + f16v(c.v4_min[b, :L, 0])[:, None]).astype(np.float32)
            bound = (2.0 ** -8 * np.exp2(sig - Ms)) @ np.abs(bf16_round(v32))
            assert np.all(np.abs(o_int[hq] - o_flt[hq]) <= bound / den * 1.01 + 1e-9)


@pytest.mark.parametrize("L", [1, 15, 16, 17, 100, 128, 129, 143, 144])
def test_equals_hybrid_when_every_position_is_protected(L):
    """With L ≤ s + w = 144 the hybrid cache holds every position in its INT8 side
    rows, one page per 16-row group: KV8 computes the same attention (group fold
    order aside) and the same integer dots."""
    H, G = 2, 4
    kv8, _ = make(H, [L], seed=2)
    hyb, _ = make(H, [L], seed=2, kv8=False, s=16, w=128)
    q = inputs.bf16_bits(inputs.queries(1, H * G, seed=10))
    for mode in (oracle.PV_INTEGER, oracle.PV_FLOAT):
        o8, l8, d8 = kv8.decode(0, L, G, q[0], 0.09, pv_mode=mode, debug=True)
        oh, lh, dh = hyb.decode(0, L, G, q[0], 0.09, pv_mode=mode, debug=True)
        np.testing.assert_array_equal(d8["qk"][:, :L], dh["qk"][:, :L])
        np.testing.assert_allclose(o8, oh, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l8, lh, rtol=0, atol=1e-12)


def test_chunked_append_and_batch_entry():
    H, G = 1, 2
    k, v = inputs.sequence_kv(0, 90, H, 4)
    kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
    a = oracle.OracleCache(H, 0, 0, 90, kv8=True)
    a.append(0, 0, kb, vb)
    b = oracle.OracleCache(H, 0, 0, 90, kv8=True)
    for lo, hi in ((0, 1), (1, 17), (17, 50), (50, 90)):
        b.append(0, lo, kb[lo:hi], vb[lo:hi])
    q = inputs.bf16_bits(inputs.queries(1, H * G, seed=11))
    oa, la, _ = a.decode(0, 90, G, q[0], 0.1)
    ob, lb, _ = b.decode(0, 90, G, q[0], 0.1)
    np.testing.assert_array_equal(oa, ob)
    ot, lt = a.decode_batch([0], [90], G, q, 0.1)
    np.testing.assert_array_equal(ot[0], oa)
    np.testing.assert_array_equal(lt[0], la)


def test_empty_context_and_rejected_protected_region():
    c = oracle.OracleCache(1, 0, 0, 4, kv8=True)
    q = inputs.bf16_bits(inputs.queries(1, 2, seed=1))
    out, lse, _ = c.decode(0, 0, 2, q[0], 0.1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    with pytest.raises(ValueError):
        oracle.OracleCache(1, 16, 128, 4, kv8=True)
