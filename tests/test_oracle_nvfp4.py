"""Pins for the oracle's NVFP4 configuration (reading R12).

References used here, none of them the oracle's own code:
  * the E2M1 grid with nearest / ties-to-even chosen by brute force in float64;
  * torch's float8_e4m3fn conversion for E4M3 rounding and decoding;
  * the float64 dense Sylvester Hadamard matrix and the rounding bound of the format;
  * a textbook float64 softmax attention over the oracle's dequantized state;
  * the fp16 rounding bound of the PV weights, checked against the exact float mode.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from int8_hybrid_paged_gb300 import inputs

D = 128
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def nearest_e2m1(v):
    """Brute force: the grid point nearest |v| (ties: the even code), clamped to 6."""
    a = min(abs(float(v)), 6.0)
    dist = np.abs(GRID - a)
    best = min(range(8), key=lambda k: (dist[k], k & 1))
    return -GRID[best] if (v < 0 and best) else GRID[best]


def test_e2m1_rounding_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(0)
    vals = list(rng.uniform(-8, 8, 4000)) + [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0, 6.0,
                                             7.0, -0.25, 0.0, -0.0, 1e-8] + list(GRID) + list(-GRID)
    for v in vals:
        code = oracle.e2m1_rn(np.float32(v))
        assert oracle.e2m1_value(code) == nearest_e2m1(np.float32(v)), v
        if oracle.e2m1_value(code) == 0.0:
            assert code == 0                          # canonical zero


def test_e4m3_matches_torch():
    rng = np.random.default_rng(1)
    t = np.concatenate([rng.uniform(0, 448, 3000), rng.uniform(0, 1, 1000), 2.0 ** rng.uniform(-12, 8, 1000),
                        [0.0, 2 ** -9, 2 ** -10, 1.5 * 2 ** -9, 0.0625, 448.0, 416.0, 432.0]]).astype(np.float32)
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle.e4m3_value(oracle.e4m3_rn(float(x))) for x in t], np.float32)
    np.testing.assert_array_equal(got, ref)
    bits = np.arange(0x7F, dtype=np.uint8)                 # every finite non-negative pattern
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    np.testing.assert_array_equal(np.array([oracle.e4m3_value(int(b)) for b in bits], np.float32), ref)
    assert oracle.e4m3_value(oracle.e4m3_rn(1e6)) == 448.0


def _hadamard():
    i = np.arange(D)
    pop = np.vectorize(lambda x: bin(int(x)).count("1"))(i[:, None] & i[None, :])
    return np.where(pop % 2 == 0, 1.0, -1.0) / math.sqrt(D)


def _decoded(codes, bs, g):
    scale = np.repeat([oracle.e4m3_value(int(b)) for b in bs], 16) * float(g)
    return np.array([oracle.e2m1_value(int(c)) for c in codes]) * scale, scale


def test_quantizer_bound_special_cases_and_zeros():
    rng = np.random.default_rng(2)
    for trial in range(50):
        x = (rng.standard_normal(D) * rng.uniform(0.01, 50)).astype(np.float32)
        if trial % 5 == 0:
            x[rng.integers(0, D, 4)] *= 30.0               # outliers
        codes, bs, g = oracle.quant_nvfp4(x)
        assert g == np.float32(np.abs(x).max() / np.float32(2688.0))
        rec, scale = _decoded(codes, bs, g)
        # nearest-grid error is at most one scale unit (the 4 -> 6 gap), saturation
        # above 6 is below 0.4 units because s_b is rounded to E4M3 (3 mantissa bits)
        assert np.all(np.abs(rec - x) <= scale * (1 + 1e-6) + 1e-30)
        for b in range(8):
            blk = np.abs(x[16 * b:16 * b + 16]).max()
            assert np.abs(rec[16 * b:16 * b + 16]).max() <= blk * (1 + 1 / 6) + 1e-30
    # values on the grid times a power of two keep their grid codes (the block scale is
    # 448 g, and g = amax / 2688 carries one float rounding into the reconstruction)
    c = 2.0 ** -3
    x = np.tile(np.concatenate([GRID, -GRID]), 8).astype(np.float32) * np.float32(c)
    codes, bs, g = oracle.quant_nvfp4(x)
    assert all(oracle.e4m3_value(int(b)) == 448.0 for b in bs)
    np.testing.assert_array_equal([oracle.e2m1_value(int(cd)) for cd in codes], x / np.float32(c))
    rec, _ = _decoded(codes, bs, g)
    np.testing.assert_allclose(rec, x.astype(np.float64), rtol=1e-6, atol=0)
    codes, bs, g = oracle.quant_nvfp4(np.zeros(D, np.float32))
    assert not codes.any() and not bs.any() and g == 0.0


def _make(H, lens, seed=0, rope=None):
    c = oracle.OracleCache(H, 0, 0, max(lens), num_slots=len(lens), nvfp4=True, rope=rope)
    raw = []
    for b, L in enumerate(lens):
        k, v = inputs.sequence_kv(b, L, H, seed)
        kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
        c.append(b, 0, kb, vb)
        raw.append((kb, vb))
    return c, raw


def test_cache_holds_nvfp4_of_rotated_keys_and_plain_values():
    H, L = 2, 40
    c, raw = _make(H, [L])
    Hd = _hadamard()
    kb, vb = raw[0]
    k = (kb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    v = (vb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(L):
        for h in range(H):
            for x, cd, bs, gs in ((k[t, h] @ Hd, c.k4_code, c.k_bscale, c.k_gscale),
                                  (v[t, h], c.v4_code, c.v_bscale, c.v_gscale)):
                rec, scale = _decoded(cd[0, t, h], bs[0, t, h], gs[0, t, h])
                assert np.all(np.abs(rec - x) <= scale * (1 + 1e-5) + 1e-6 * np.abs(x).max())
    assert c.side_bytes() == 0


def _textbook(c, slot, L, G, dbg, sm):
    out = np.zeros((c.H * G, D))
    lse = np.full(c.H * G, -np.inf)
    for hq in range(c.H * G):
        h = hq // G
        if L == 0:
            continue
        qhat = dbg["q8"][hq].astype(np.float64) * float(dbg["q_scale"][hq])
        K = np.stack([_decoded(c.k4_code[slot, t, h], c.k_bscale[slot, t, h], c.k_gscale[slot, t, h])[0]
                      for t in range(L)])
        # float mode: the exact dequantized values
        V = np.stack([_decoded(c.v4_code[slot, t, h], c.v_bscale[slot, t, h], c.v_gscale[slot, t, h])[0]
                      for t in range(L)])
        sc = (K @ qhat) * sm
        mx = sc.max()
        p = np.exp(sc - mx)
        out[hq] = p @ V / p.sum()
        lse[hq] = mx + math.log(p.sum())
    return out, lse


LENS = [1, 16, 17, 40, 161]


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
    """Integer mode (fp16 weights carrying the value scales, exact E2M1 values) against
    float mode (exact values, unrounded p). Per position i and block b the weight
    W = p·g·s_b / 2^k is rounded twice to fp16: relative error at most 2^-11 each while
    normal, absolute error at most 2^-25 (times s_b + 1) in the subnormal range; the
    group's sum is scaled by 2^k and by 2^(M_group - M) in the merge."""
    H, G = 1, 2
    sm = 1 / math.sqrt(D)
    c, _ = _make(H, LENS)
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
                pg = np.exp2(sig[idx] - Mg) * c.v_gscale[b, idx, 0]
                gm = c.v_gscale[b, idx, 0].max()
                k = math.frexp(gm)[1] if gm >= 2.0 ** -126 else -126
                for n, t in enumerate(idx):
                    sb = np.repeat([oracle.e4m3_value(int(x)) for x in c.v_bscale[b, t, 0]], 16)
                    e = np.abs([oracle.e2m1_value(int(x)) for x in c.v4_code[b, t, 0]])
                    W = pg[n] * sb * 2.0 ** -k
                    bound += 2.0 ** k * e * ((2 ** -10 + 2 ** -22) * W + 2 ** -25 * (sb + 1)) \
                        * 2.0 ** (Mg - Ms)
            assert np.all(np.abs(o_int[hq] - o_flt[hq]) <= bound / den * 1.01 + 1e-12)
    assert worst > 0                                          # the rounding is there


def test_chunked_append_empty_context_and_rejections():
    H, G = 1, 2
    k, v = inputs.sequence_kv(0, 90, H, 4)
    kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
    a = oracle.OracleCache(H, 0, 0, 90, nvfp4=True)
    a.append(0, 0, kb, vb)
    b = oracle.OracleCache(H, 0, 0, 90, nvfp4=True)
    for lo, hi in ((0, 1), (1, 17), (17, 50), (50, 90)):
        b.append(0, lo, kb[lo:hi], vb[lo:hi])
    for n in ("k4_code", "v4_code", "k_bscale", "v_bscale", "k_gscale", "v_gscale"):
        np.testing.assert_array_equal(getattr(a, n), getattr(b, n))
    q = inputs.bf16_bits(inputs.queries(1, H * G, seed=11))
    out, lse, _ = a.decode(0, 0, G, q[0], 0.1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    with pytest.raises(ValueError):
        oracle.OracleCache(1, 16, 128, 4, nvfp4=True)
