"""Pins for the oracle's number formats, against numpy / torch conversions and
libm (independent implementations), never against the oracle itself."""
import numpy as np
import pytest
import torch

import oracle


def _f32_samples(n=1 << 18, seed=0):
    rng = np.random.default_rng(seed)
    raw = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    scaled = (rng.standard_normal(n) * np.exp2(rng.integers(-27, 17, n))).astype(np.float32)
    # every fp16 value, its float32 neighbours and the midpoints between fp16 values
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    h = h[np.isfinite(h)].astype(np.float32)
    hs = np.sort(np.unique(h))
    mids = ((hs[:-1].astype(np.float64) + hs[1:].astype(np.float64)) / 2).astype(np.float32)
    pts = np.concatenate([h, mids])
    near = np.concatenate([np.nextafter(pts, np.float32(np.inf)),
                           np.nextafter(pts, np.float32(-np.inf))])
    special = np.array([0.0, -0.0, np.inf, -np.inf, 65504, 65519.99, 65520, -65520, 7e4, -7e4,
                        1e-8, -1e-8, 2.0 ** -25, -(2.0 ** -25), 2.0 ** -24, 3 * 2.0 ** -26],
                       np.float32)
    return np.concatenate([raw, scaled, pts, near, special]).astype(np.float32)


def test_f16_round_to_nearest_matches_numpy():
    x = _f32_samples()
    x = x[~np.isnan(x)]
    got = oracle.f32_to_f16(x, oracle.RN)
    ref = x.astype(np.float16).view(np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("mode", [oracle.RD, oracle.RU])
def test_f16_directed_rounding_brackets(mode):
    x = _f32_samples(seed=1)
    x = x[~np.isnan(x)]
    got = oracle.f32_to_f16(x, mode).view(np.float16)
    xv = x.astype(np.float64)
    gv = got.astype(np.float64)
    if mode == oracle.RD:
        assert np.all(gv <= xv)
        nxt = np.nextafter(got, np.float16(np.inf)).astype(np.float64)
        ok = (nxt > xv) | (got == np.float16(np.inf))
    else:
        assert np.all(gv >= xv)
        nxt = np.nextafter(got, np.float16(-np.inf)).astype(np.float64)
        ok = (nxt < xv) | (got == np.float16(-np.inf))
    # exact fp16 values map to themselves; everything else to the adjacent grid point
    assert np.all(ok)
    exact = x.astype(np.float16).astype(np.float32) == x
    assert np.all(got[exact].astype(np.float32) == x[exact])


def test_f16_nan_stays_nan():
    x = np.array([np.nan, -np.nan], np.float32)
    for mode in (oracle.RN, oracle.RD, oracle.RU):
        assert np.all(np.isnan(oracle.f32_to_f16(x, mode).view(np.float16)))


def test_f16_decoder_matches_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    sel = bits[::37]
    got = oracle.f16_bits_to_f64(sel)
    ref = sel.view(np.float16).astype(np.float64)
    both_nan = np.isnan(got) & np.isnan(ref)
    assert np.all((got == ref) | both_nan)


def test_bf16_round_to_nearest_matches_torch():
    x = _f32_samples(seed=2)
    x = x[~np.isnan(x)]
    got = oracle.f32_to_bf16_rn(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_exp2_within_one_ulp_of_libm():
    rng = np.random.default_rng(3)
    x = np.concatenate([-rng.uniform(0, 125, 1 << 20), -np.linspace(0, 1, 20001),
                        -np.arange(0, 126)]).astype(np.float32)
    got = oracle.exp2f(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(got - ref) / ulp) <= 1.0
    # integers are exact powers of two; below −125 the result is 0
    ints = -np.arange(0, 126).astype(np.float32)
    assert np.all(oracle.exp2f(ints) == np.exp2(ints.astype(np.float64)).astype(np.float32))
    assert np.all(oracle.exp2f(np.array([-125.5, -300, -np.inf], np.float32)) == 0)
