"""Pins for the grouping of the oracle's protected-path weights (reading R7).

The protected positions [0, min(s, L)) ∪ [max(s, L − w), L) form their softmax
weights per 16-position page of the paged cache, in position order: each weight
is p = 2^(σ − M) with M the largest score among the protected positions of the
same page. Where a side row sits in the ring buffer must not matter.

References used here, none of them the oracle's grouping code:
  * the page of a position (pos // 16) and the region rule, applied by hand in
    numpy to the oracle's own per-position scores;
  * the whole-cache 8-bit configuration (reading R10), whose groups are whole
    pages by construction: with the INT4 region's scores pushed out of range, the
    hybrid cache must give exactly KV8's attention, window straddling a page or not.
"""
import numpy as np
import pytest
import torch

import oracle
from int8_hybrid_paged_gb300 import inputs

D = 128
P = 16


def protected_positions(L, s, w):
    return [t for t in range(L) if t < s or t >= max(s, L - w)]


def expected_p_bits(sig, prot):
    """BF16 bits of 2^(σ − page max) for each protected position, the page max taken
    over the protected positions of that page only."""
    prot = np.asarray(prot)
    out = {}
    for pg in np.unique(prot // P):
        members = prot[prot // P == pg]
        m = np.max(sig[members])
        p = oracle.exp2f(sig[members] - m)
        bits = oracle.f32_to_bf16_rn(p)
        out.update(zip(members.tolist(), bits.tolist()))
    return out


@pytest.mark.parametrize("s,w", [(16, 128), (5, 7), (33, 40), (0, 64), (16, 0)])
@pytest.mark.parametrize("L", [1, 17, 100, 145, 150, 161, 200, 333, 1000])
def test_protected_weights_use_their_page_max(s, w, L):
    H, G = 2, 2
    c = oracle.OracleCache(H, s, w, L)
    k, v = inputs.sequence_kv(0, L, H, seed=L + s)
    c.append(0, 0, inputs.bf16_bits(k), inputs.bf16_bits(v))
    q = inputs.bf16_bits(inputs.queries(1, H * G, seed=L))
    _, _, d = c.decode(0, L, G, q[0], 1 / np.sqrt(D), debug=True)
    prot = protected_positions(L, s, w)
    r4 = [t for t in range(L) if t not in set(prot)]
    for hq in range(H * G):
        want = expected_p_bits(d["sigma"][hq], prot)
        got = {t: int(d["p_bits"][hq, t]) for t in prot}
        assert got == want
        assert np.all(d["p_bits"][hq, r4] == 0)


def adversarial_kv(L, H, G, s, w, q, seed):
    """K, V with every key of the INT4 region [s, L − w) pointed against all G queries
    of its KV head, so that its scores sit far below 2^-126 of any protected score."""
    k, v = inputs.sequence_kv(0, L, H, seed)
    k = k.float()
    qf = q.float()[0].reshape(H, G, D)
    for t in range(s, max(s, L - w)):
        for h in range(H):
            k[t, h] = -16.0 * qf[h].sum(0)
    return k.to(torch.bfloat16), v


@pytest.mark.parametrize("s,w", [(16, 128), (0, 128), (16, 64), (5, 7), (33, 40)])
@pytest.mark.parametrize("L", [145, 150, 161, 200, 263, 333, 1000])
def test_protected_region_equals_kv8_on_its_positions(s, w, L):
    """Past L = s + w the window [L − w, L) straddles pages whenever L − w is not a
    multiple of 16, and its ring rows then share side-row groups with positions one
    window older or with sink rows. The page grouping makes the protected region's
    result that of KV8 over the same positions; any grouping by side-row order, or by
    one region-wide max, gives other BF16 weights and fails."""
    H, G = 2, 4
    qt = inputs.queries(1, H * G, seed=L + 7)
    q = inputs.bf16_bits(qt)
    k, v = adversarial_kv(L, H, G, s, w, qt, seed=3)
    kb, vb = inputs.bf16_bits(k), inputs.bf16_bits(v)
    hyb = oracle.OracleCache(H, s, w, L)
    hyb.append(0, 0, kb, vb)
    kv8 = oracle.OracleCache(H, 0, 0, L, kv8=True)
    kv8.append(0, 0, kb, vb)
    oh, lh, dh = hyb.decode(0, L, G, q[0], 1 / np.sqrt(D), debug=True)
    o8, l8, d8 = kv8.decode(0, L, G, q[0], 1 / np.sqrt(D), debug=True)
    prot = protected_positions(L, s, w)
    r4 = sorted(set(range(L)) - set(prot))
    # the INT4 region really is out of range: its scores lie more than 126 below
    # every protected score
    for hq in range(H * G):
        assert np.max(dh["sigma"][hq, r4]) < np.min(dh["sigma"][hq, prot]) - 130
    # same integer dots and scores on the protected positions, same BF16 weights
    np.testing.assert_array_equal(dh["qk"][:, prot], d8["qk"][:, prot])
    np.testing.assert_array_equal(dh["p_bits"][:, prot], d8["p_bits"][:, prot])
    np.testing.assert_allclose(oh, o8, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lh, l8, rtol=1e-12, atol=1e-12)
