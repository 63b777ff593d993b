"""Pins for the oracle's MXFP4 configuration (reading R13).

References used here, none of them the oracle's own code:
  * the shared exponent floor(log2 amax) - 2 from Python's float64 frexp;
  * the E2M1 grid with nearest / ties-to-even chosen by brute force in float64;
  * the grid's half spacing as the error bound, 2 X for saturated values;
  * the float64 dense Sylvester Hadamard matrix for the stored keys;
  * the scores against float64 dots of the dequantized keys with the INT8 query;
  * a textbook float64 softmax attention over the exact dequantized state (float mode);
  * the fp16 rounding bound of the PV weights, checked against float mode.
"""
import math

import numpy as np
import pytest

import oracle
from int8_hybrid_paged_gb300 import inputs

D = 128
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def nearest_e2m1(v):
    """Brute force: the grid point nearest |v| (ties: the even code), held at 6."""
    a = min(abs(float(v)), 6.0)
    dist = np.abs(GRID - a)
    best = min(range(8), key=lambda k: (dist[k], k & 1))
    return -GRID[best] if (v < 0 and best) else GRID[best]


def shared_exp(block):
    amax = float(np.max(np.abs(block)))
    if amax == 0.0:
        return -127
    return min(127, max(-127, math.frexp(amax)[1] - 1 - 2))


def half_spacing(a):
    return 0.25 if a <= 2 else (0.5 if a <= 4 else 1.0)


def _decoded(codes, es):
    scale = np.repeat([2.0 ** (int(e) - 127) for e in es[:4]], 32)
    return np.array([oracle.e2m1_value(int(c)) for c in codes]) * scale, scale


def test_quantizer_scale_codes_and_bound():
    rng = np.random.default_rng(3)
    for trial in range(60):
        x = (rng.standard_normal(D) * 2.0 ** rng.uniform(-20, 20)).astype(np.float32)
        if trial % 4 == 0:
            x[rng.integers(0, D, 3)] *= 50.0                 # outliers
        if trial % 7 == 0:
            x[32:64] = 0.0                                    # an all-zero block
        codes, es = oracle.quant_mxfp4(x)
        for b in range(4):
            blk = x[32 * b:32 * b + 32].astype(np.float64)
            s = shared_exp(blk)
            assert int(es[b]) == s + 127
            X = 2.0 ** s
            for i in range(32):
                r = blk[i] / X
                assert oracle.e2m1_value(int(codes[32 * b + i])) == nearest_e2m1(r)
                err = abs(blk[i] - X * nearest_e2m1(r))
                # nearest grid point within half a spacing, saturation above 6 below 2 X
                assert err <= (X * half_spacing(abs(r)) if abs(r) <= 6 else 2 * X)
            if not blk.any():
                assert not codes[32 * b:32 * b + 32].any()
    # the block maximum lands in [4, 8) X, so the scale uses the grid's top binade
    codes, es = oracle.quant_mxfp4(np.float32([3.0] * D))
    assert all(int(e) == 127 - 1 for e in es)                # 3 = 6 * 2^-1
    assert all(oracle.e2m1_value(int(c)) == 6.0 for c in codes)


def _hadamard():
    i = np.arange(D)
    pop = np.vectorize(lambda x: bin(int(x)).count("1"))(i[:, None] & i[None, :])
    return np.where(pop % 2 == 0, 1.0, -1.0) / math.sqrt(D)


def _make(H, lens, seed=0):
    c = oracle.OracleCache(H, 0, 0, max(lens), num_slots=len(lens), mxfp4=True)
    raw = []
    for b, L in enumerate(lens):
        k, v = inputs.sequence_kv(b, L, H, seed)
        kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
        c.append(b, 0, kb, vb)
        raw.append((kb, vb))
    return c, raw


def test_cache_holds_mxfp4_of_rotated_keys_and_plain_values():
    H, L = 2, 40
    c, raw = _make(H, [L])
    Hd = _hadamard()
    kb, vb = raw[0]
    k = (kb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    v = (vb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(L):
        for h in range(H):
            for x, cd, es in ((k[t, h] @ Hd, c.k4_code, c.k_bscale), (v[t, h], c.v4_code, c.v_bscale)):
                rec, scale = _decoded(cd[0, t, h], es[0, t, h])
                # within two scale units (saturation) plus the float32 rounding of the rotation
                assert np.all(np.abs(rec - x) <= 2 * scale + 1e-5 * np.abs(x).max())
                assert not es[0, t, h, 4:].any()
    assert c.side_bytes() == 0


LENS = [1, 16, 17, 40, 161]


def test_scores_are_the_scaled_block_dots():
    H, G = 1, 2
    sm = 1 / math.sqrt(D)
    c, _ = _make(H, LENS, seed=1)
    q = inputs.bf16_bits(inputs.queries(len(LENS), H * G, seed=4))
    for b, L in enumerate(LENS):
        _, _, dbg = c.decode(b, L, G, q[b], sm, debug=True)
        for hq in range(H * G):
            qhat = dbg["q8"][hq].astype(np.float64)
            for t in range(L):
                rec, _ = _decoded(c.k4_code[b, t, 0], c.k_bscale[b, t, 0])
                exact = float(rec @ qhat) * float(dbg["q_scale"][hq]) * sm * math.log2(math.e)
                terms = float(np.abs(rec * qhat).sum()) * float(dbg["q_scale"][hq]) * sm * math.log2(math.e)
                # four fma roundings, then two products and the rounding of C
                assert abs(float(dbg["sigma"][hq, t]) - exact) <= 8 * 2.0 ** -24 * terms + 1e-30


def _textbook(c, slot, L, G, dbg, sm):
    out = np.zeros((c.H * G, D))
    lse = np.full(c.H * G, -np.inf)
    for hq in range(c.H * G):
        h = hq // G
        if L == 0:
            continue
        qhat = dbg["q8"][hq].astype(np.float64) * float(dbg["q_scale"][hq])
        K = np.stack([_decoded(c.k4_code[slot, t, h], c.k_bscale[slot, t, h])[0] for t in range(L)])
        V = np.stack([_decoded(c.v4_code[slot, t, h], c.v_bscale[slot, t, h])[0] for t in range(L)])
        sc = (K @ qhat) * sm
        mx = sc.max()
        p = np.exp(sc - mx)
        out[hq] = p @ V / p.sum()
        lse[hq] = mx + math.log(p.sum())
    return out, lse


@pytest.mark.parametrize("G", [1, 4])
def test_float_pv_equals_single_softmax(G):
    H = 2
    sm = 1 / math.sqrt(D)
    c, _ = _make(H, LENS)
    q = inputs.bf16_bits(inputs.queries(len(LENS), H * G, seed=8))
    for b, L in enumerate(LENS):
        out, lse, dbg = c.decode(b, L, G, q[b], sm, pv_mode=oracle.PV_FLOAT, debug=True)
        ref, ref_lse = _textbook(c, b, L, G, dbg, sm)
        np.testing.assert_allclose(out, ref, rtol=0, atol=2e-5 * max(1.0, np.abs(ref).max()))
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=2e-5 * max(1, np.abs(ref_lse).max()))


def test_fp16_weights_within_rounding_bound():
    """Integer mode against float mode: w = fp16(fp16(p)·2^(s_b - k)) with 2^k the
    group's largest block scale; fp16(p) is off by at most 2^-11 p (normal) or 2^-25
    (subnormal), the power-of-two scaling is exact unless the result is subnormal, where
    it adds at most 2^-25; the group's sum is scaled by 2^k and by 2^(M_group - M)."""
    H, G = 1, 2
    sm = 1 / math.sqrt(D)
    c, _ = _make(H, LENS, seed=2)
    q = inputs.bf16_bits(inputs.queries(len(LENS), H * G, seed=9))
    worst = 0.0
    for b, L in enumerate(LENS):
        o_int, lse_i, dbg = c.decode(b, L, G, q[b], sm, pv_mode=oracle.PV_INTEGER, debug=True)
        o_flt, lse_f, _ = c.decode(b, L, G, q[b], sm, pv_mode=oracle.PV_FLOAT)
        np.testing.assert_array_equal(lse_i, lse_f)
        worst = max(worst, np.abs(o_int - o_flt).max())
        for hq in range(H * G):
            sig = dbg["sigma"][hq, :L].astype(np.float64)
            Ms = sig.max()
            den = math.exp2(lse_i[hq] / math.log(2) - Ms)
            bound = np.zeros(D)
            for g0 in range(0, L, 16):
                idx = np.arange(g0, min(L, g0 + 16))
                Mg = sig[idx].max()
                p = np.exp2(sig[idx] - Mg)
                k = int(c.v_bscale[b, idx, 0, :4].max()) - 127
                for n, t in enumerate(idx):
                    sb = np.repeat([int(e) - 127 for e in c.v_bscale[b, t, 0, :4]], 32).astype(np.float64)
                    e = np.abs([oracle.e2m1_value(int(x)) for x in c.v4_code[b, t, 0]])
                    W = p[n] * 2.0 ** (sb - k)
                    bound += 2.0 ** k * e * (2 ** -11 * W + 2 ** -25 * (2.0 ** (sb - k) + 1)) * 2.0 ** (Mg - Ms)
            assert np.all(np.abs(o_int[hq] - o_flt[hq]) <= bound / den * 1.01 + 1e-12)
    assert worst > 0                                          # the rounding is there


def test_chunked_append_empty_context_and_rejections():
    H, G = 1, 2
    k, v = inputs.sequence_kv(0, 90, H, 4)
    kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
    a = oracle.OracleCache(H, 0, 0, 90, mxfp4=True)
    a.append(0, 0, kb, vb)
    b = oracle.OracleCache(H, 0, 0, 90, mxfp4=True)
    for lo, hi in ((0, 1), (1, 17), (17, 50), (50, 90)):
        b.append(0, lo, kb[lo:hi], vb[lo:hi])
    for n in ("k4_code", "v4_code", "k_bscale", "v_bscale"):
        np.testing.assert_array_equal(getattr(a, n), getattr(b, n))
    q = inputs.bf16_bits(inputs.queries(1, H * G, seed=11))
    out, lse, _ = a.decode(0, 0, G, q[0], 0.1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    with pytest.raises(ValueError):
        oracle.OracleCache(1, 16, 128, 4, mxfp4=True)
    with pytest.raises(ValueError):
        oracle.OracleCache(1, 0, 0, 4, mxfp4=True, nvfp4=True)
