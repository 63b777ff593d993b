"""Pins for the oracle's decode attention and cache state.

References used here, none of them the oracle's own code:
  * numpy int64 matmul for the integer dot products;
  * a textbook float64 softmax attention over the oracle's dequantized state;
  * exact float64 attention over the unquantized bf16 inputs (loose bound);
  * the ring/sink index rule applied by hand to per-token quantizations.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from int8_hybrid_paged_gb300 import bytes_model, inputs

D = 128
LOG2E = 1.4426950408889634


def f16v(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def bf16_round(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16) \
        .to(torch.float32).numpy().astype(np.float64)


def make_cache(H, s, w, lens, seed=0):
    c = oracle.OracleCache(H, s, w, max(lens), num_slots=len(lens))
    raw = []
    for b, L in enumerate(lens):
        k, v = inputs.sequence_kv(b, L, H, seed)
        kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
        c.append(b, 0, kb, vb)
        raw.append((kb, vb))
    return c, raw


def side_index(t, s, w):
    return t if t < s else s + (t % w)


def regions(L, s, w):
    prot = list(range(0, min(s, L))) + list(range(max(s, L - w), L))
    r4 = list(range(s, max(s, L - w)))
    return r4, prot


def textbook(c, slot, L, G, dbg, sm_scale):
    """float64 softmax attention over the oracle's own dequantized keys/values and
    its INT8 query q8·s_q (natural-log units)."""
    s, w, H = c.s, c.w, c.H
    r4, prot = regions(L, s, w)
    HG = H * G
    out = np.zeros((HG, D))
    lse = np.zeros(HG)
    for hq in range(HG):
        h = hq // G
        qhat = dbg["q8"][hq].astype(np.float64) * float(dbg["q_scale"][hq])
        keys, vals = [], []
        for t in r4:
            kd = f16v(c.k4_delta[slot, t, h]) * c.k4_code[slot, t, h] + f16v(c.k4_min[slot, t, h])
            vd = f16v(c.v4_delta[slot, t, h]) * c.v4_code[slot, t, h] + f16v(c.v4_min[slot, t, h])
            keys.append(kd)
            vals.append(vd)
        for t in prot:
            i = side_index(t, s, w)
            kd = f16v(c.k8_delta[slot, i, h]) * c.k8_code[slot, i, h] + f16v(c.k8_min[slot, i, h])
            v32 = (f16v(c.v8_delta[slot, i, h]) * c.v8_code[slot, i, h].astype(np.float64)
                   + f16v(c.v8_min[slot, i, h])).astype(np.float32)
            keys.append(kd)
            vals.append(bf16_round(v32))
        if not keys:
            lse[hq] = -np.inf
            continue
        K = np.stack(keys)
        V = np.stack(vals)
        sc = (K @ qhat) * sm_scale
        mx = sc.max()
        p = np.exp(sc - mx)
        out[hq] = p @ V / p.sum()
        lse[hq] = mx + math.log(p.sum())
    return out, lse


CASES = [
    # (H, s, w, lens, G)
    (1, 4, 8, [1, 3, 12, 13, 20, 40], 2),
    (2, 16, 128, [300, 1000], 4),
    (1, 0, 0, [37], 2),          # pure KV4: no protected positions
    (1, 16, 128, [100, 144], 2),  # L ≤ s + w: every position protected
    (1, 5, 0, [29], 1),           # sink only
    (1, 0, 7, [29], 1),           # ring only
]


@pytest.mark.parametrize("H,s,w,lens,G", CASES)
def test_region_split_and_integer_qk(H, s, w, lens, G):
    c, _ = make_cache(H, s, w, lens)
    q = inputs.bf16_bits(inputs.queries(len(lens), H * G, seed=3))
    for b, L in enumerate(lens):
        _, _, dbg = c.decode(b, L, G, q[b], 1 / math.sqrt(D), debug=True)
        r4, prot = regions(L, s, w)
        assert sorted(r4 + prot) == list(range(L))          # disjoint and covering
        assert len(prot) <= s + w                             # bounded side
        assert np.all(np.isfinite(dbg["sigma"][:, :L]))
        for hq in range(H * G):
            h = hq // G
            q8 = dbg["q8"][hq].astype(np.int64)
            if r4:
                ref4 = c.k4_code[b, r4, h].astype(np.int64) @ q8
                np.testing.assert_array_equal(dbg["qk"][hq, r4], ref4)
            if prot:
                idx = [side_index(t, s, w) for t in prot]
                ref8 = c.k8_code[b, idx, h].astype(np.int64) @ q8
                np.testing.assert_array_equal(dbg["qk"][hq, prot], ref8)
            # u8 PV weights exist only in the INT4 region
            outside = np.ones(L, bool)
            outside[r4] = False
            assert np.all(dbg["w_hat"][hq, :L][outside] == 0)


@pytest.mark.parametrize("H,s,w,lens,G", CASES[:2])
def test_scores_equal_dequantized_dot(H, s, w, lens, G):
    """σ = (q8·s_q)·(Δc+m)·sm_scale·log2e: the deferred scale/offset form of the
    dot product of the dequantized vectors."""
    sm = 0.0883883
    c, _ = make_cache(H, s, w, lens)
    q = inputs.bf16_bits(inputs.queries(len(lens), H * G, seed=4))
    for b, L in enumerate(lens):
        _, _, dbg = c.decode(b, L, G, q[b], sm, debug=True)
        r4, prot = regions(L, s, w)
        for hq in range(H * G):
            h = hq // G
            qhat = dbg["q8"][hq].astype(np.float64) * float(dbg["q_scale"][hq])
            for t in range(L):
                if t in prot:
                    i = side_index(t, s, w)
                    k = f16v(c.k8_delta[b, i, h]) * c.k8_code[b, i, h] + f16v(c.k8_min[b, i, h])
                else:
                    k = f16v(c.k4_delta[b, t, h]) * c.k4_code[b, t, h] + f16v(c.k4_min[b, t, h])
                ref = float(qhat @ k) * sm * LOG2E
                mag = float(np.abs(qhat) @ np.abs(k)) * sm * LOG2E
                assert abs(float(dbg["sigma"][hq, t]) - ref) <= 4e-6 * mag + 1e-6


@pytest.mark.parametrize("H,s,w,lens,G", CASES)
def test_float_pv_equals_single_softmax(H, s, w, lens, G):
    """Region split + exact LSE merge equals one softmax over the concatenated
    scores (FP32 page weights are the only rounding left)."""
    sm = 1 / math.sqrt(D)
    c, _ = make_cache(H, s, w, lens)
    q = inputs.bf16_bits(inputs.queries(len(lens), H * G, seed=5))
    for b, L in enumerate(lens):
        out, lse, dbg = c.decode(b, L, G, q[b], sm, pv_mode=oracle.PV_FLOAT, debug=True)
        ref, ref_lse = textbook(c, b, L, G, dbg, sm)
        np.testing.assert_allclose(out, ref, rtol=0, atol=2e-6 * max(1.0, np.abs(ref).max()))
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=2e-6 * max(1, np.abs(ref_lse).max()))


@pytest.mark.parametrize("H,s,w,lens,G", CASES)
def test_integer_pv_within_weight_rounding_bound(H, s, w, lens, G):
    """Integer PV differs from float PV only through ŵ and the BF16 rounding of the
    protected p. Per page |ŵ·s_w − p'Δ^V| ≤ s_w/2 with s_w = 2^(floor(log2 max w) − 7)
    (a weight that rounds to 256 is held at 255, at most s_w/2 further when it is
    within 1 of the top), so each output element moves by at most
    Σ_pages 2^(M_page−M*) (s_w/2) Σ_t c^V_tj / den; a protected p rounded to BF16
    (8 significant bits) moves by at most 2^-8 of itself, so each protected position
    adds at most 2^-8 2^(σ_t−M*) |v_tj| / den (all checked with 1% slack)."""
    sm = 1 / math.sqrt(D)
    c, _ = make_cache(H, s, w, lens)
    q = inputs.bf16_bits(inputs.queries(len(lens), H * G, seed=6))
    for b, L in enumerate(lens):
        o_int, lse_i, dbg = c.decode(b, L, G, q[b], sm, pv_mode=oracle.PV_INTEGER, debug=True)
        o_flt, lse_f, _ = c.decode(b, L, G, q[b], sm, pv_mode=oracle.PV_FLOAT)
        np.testing.assert_array_equal(lse_i, lse_f)          # normalisers do not use ŵ
        r4, _ = regions(L, s, w)
        for hq in range(H * G):
            h = hq // G
            sig = dbg["sigma"][hq, :L].astype(np.float64)
            Ms = sig.max()
            den = math.exp2(lse_i[hq] / math.log(2) - Ms) if np.isfinite(lse_i[hq]) else 1.0
            bound = np.zeros(D)
            for pg in sorted({t // 16 for t in r4}):
                ts = [t for t in r4 if t // 16 == pg]
                Mp = sig[ts].max()
                wts = np.exp2(sig[ts] - Mp) * f16v(c.v4_delta[b, ts, h])
                sw = 2.0 ** (np.floor(np.log2(wts.max())) - 7) if wts.max() > 0 else 0.0
                codes = c.v4_code[b, ts, h].astype(np.float64)
                csum = codes.sum(axis=0)
                held = (wts / sw >= 255.5) if sw > 0 else np.zeros(len(ts), bool)
                csum = csum + codes[held].sum(axis=0)          # held at 255: one more s_w/2
                bound += 2.0 ** (Mp - Ms) * (sw / 2) * csum
            _, prot = regions(L, s, w)
            for t_ in prot:
                i = side_index(t_, s, w)
                v32 = (f16v(c.v8_delta[b, i, h]) * c.v8_code[b, i, h].astype(np.float64)
                       + f16v(c.v8_min[b, i, h])).astype(np.float32)
                bound += 2.0 ** -8 * 2.0 ** (sig[t_] - Ms) * np.abs(bf16_round(v32))
            bound = bound / den * 1.01 + 1e-9
            assert np.all(np.abs(o_int[hq] - o_flt[hq]) <= bound)
            for pg in sorted({t // 16 for t in r4}):
                ts = [t for t in r4 if t // 16 == pg]
                assert 128 <= dbg["w_hat"][hq, ts].max() <= 255    # each page's largest weight


def test_close_to_exact_attention_on_unquantized_inputs():
    """Against exact float64 attention on the raw bf16 q, K, V (no rotation, no
    quantization): the INT4 error is visible but bounded, and the protected
    positions make the result much closer than INT4 everywhere."""
    H, G, L = 2, 4, 256
    sm = 1 / math.sqrt(D)
    q = inputs.bf16_bits(inputs.queries(1, H * G, seed=7))[0]
    errs = {}
    for s, w in ((16, 128), (0, 0), (256, 0)):
        c, raw = make_cache(H, s, w, [L])
        kb, vb = raw[0]
        out, _, _ = c.decode(0, L, G, q, sm)
        K = oracle.bf16_to_f32(kb).astype(np.float64)
        V = oracle.bf16_to_f32(vb).astype(np.float64)
        Q = oracle.bf16_to_f32(q).astype(np.float64)
        rel = []
        for hq in range(H * G):
            sc = K[:, hq // G] @ Q[hq] * sm
            p = np.exp(sc - sc.max())
            ref = p @ V[:, hq // G] / p.sum()
            rel.append(np.linalg.norm(out[hq] - ref) / np.linalg.norm(ref))
        errs[(s, w)] = float(np.mean(rel))
    print(errs)
    assert errs[(256, 0)] < 0.03           # all positions INT8
    assert errs[(16, 128)] < 0.25
    assert errs[(0, 0)] < 0.4
    assert errs[(256, 0)] < errs[(16, 128)] < errs[(0, 0)]


def test_side_buffer_size_is_independent_of_context_length():
    s, w, H = 16, 128, 8
    sizes = {oracle.OracleCache(H, s, w, L, num_slots=1).side_bytes() for L in (1, 144, 5000, 16640)}
    assert sizes == {(s + w) * H * bytes_model.SIDE_POSITION_HEAD_BYTES}


def test_ring_and_sink_hold_the_right_positions():
    H, s, w, L = 2, 16, 128, 333
    c, raw = make_cache(H, s, w, [L])
    kb, vb = raw[0]
    K = oracle.bf16_to_f32(kb)
    V = oracle.bf16_to_f32(vb)
    expect = list(range(min(s, L))) + list(range(max(0, L - w), L))
    for t in expect:
        i = side_index(t, s, w) if t < s and t < L - w else s + (t % w)
        if t < s and t >= L - w:
            idxs = [t, s + (t % w)]
        elif t < s:
            idxs = [t]
        else:
            idxs = [s + (t % w)]
        for i in idxs:
            for h in range(H):
                kc, kd, km = oracle.quant_affine(oracle.fwht128(K[t, h]), 255)
                vc, vd, vm = oracle.quant_affine(V[t, h], 255)
                np.testing.assert_array_equal(c.k8_code[0, i, h], kc)
                np.testing.assert_array_equal(c.v8_code[0, i, h], vc)
                assert (c.k8_delta[0, i, h], c.k8_min[0, i, h]) == (kd, km)
                assert (c.v8_delta[0, i, h], c.v8_min[0, i, h]) == (vd, vm)
    # the INT4 entries exist for every position (nothing rewritten when a position
    # leaves the ring)
    for t in (0, 17, L - w - 1, L - 1):
        for h in range(H):
            kc, kd, km = oracle.quant_affine(oracle.fwht128(K[t, h]), 15)
            np.testing.assert_array_equal(c.k4_code[0, t, h], kc)
    assert c.length[0] == L


def test_chunked_append_equals_one_call():
    H, s, w = 2, 16, 128
    k, v = inputs.sequence_kv(0, 400, H, 11)
    kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
    a = oracle.OracleCache(H, s, w, 400)
    a.append(0, 0, kb, vb)
    b = oracle.OracleCache(H, s, w, 400)
    for lo, hi in ((0, 1), (1, 150), (150, 151), (151, 400)):
        b.append(0, lo, kb[lo:hi], vb[lo:hi])
    for n in ("k4_code", "v4_code", "k4_delta", "k8_code", "v8_code", "v8_min", "length"):
        np.testing.assert_array_equal(getattr(a, n), getattr(b, n))


def test_empty_context():
    c = oracle.OracleCache(1, 16, 128, 4)
    q = inputs.bf16_bits(inputs.queries(1, 2, seed=1))[0]
    out, lse, _ = c.decode(0, 0, 2, q, 0.1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_batch_entry_equals_per_sequence_calls():
    H, G, lens = 2, 4, [300, 77, 1000, 1]
    c, _ = make_cache(H, 16, 128, lens)
    q = inputs.bf16_bits(inputs.queries(len(lens), H * G, seed=8))
    o, l = c.decode_batch(np.arange(len(lens)), np.array(lens), G, q, 1 / math.sqrt(D), threads=3)
    for b, L in enumerate(lens):
        o1, l1, _ = c.decode(b, L, G, q[b], 1 / math.sqrt(D))
        np.testing.assert_array_equal(o1, o[b])
        np.testing.assert_array_equal(l1, l[b])
