"""GPU parity of the MXFP4 format (KV4_FORMAT_MXFP4) against the oracle's reading R13.

Bit-exact: E2M1 codes, E8M0 block scales, slot lengths, the INT8 query and its scale, and
every position's FP32 score (the fma chain of exact 32-value block dots over the block
powers of two, times s_q and C) and every fp16 PV weight fp16(p). Floating point: outputs and log-normalizers
within abs 2e-3 / rel 1e-2 (the PV weights are formed identically on both sides, so the
observed worst case is asserted below 1e-4).
"""
import numpy as np
import pytest
import torch

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import inputs, kv4
from kv4_testlib import Setup, check_decode, unpack_mxfp4_pages

pytestmark = pytest.mark.gpu
D = 128
EDGE_LENS = [1, 15, 16, 17, 143, 144, 145, 300, 1000]
DECODE_LENS = [1, 15, 16, 17, 143, 144, 145, 160, 161, 300, 1000, 2049]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    kbuild.build()
    kv4.load()


def check_state(st, bs):
    pages, _, _, lens = st.cache.raw_pools()
    for b in bs:
        oc = st.oracle_for(b)
        L = st.lens[b]
        pos = np.arange(L)
        pids = st.bt[b][pos // 16]
        for h in range(st.H):
            kc, ke, vc, ve = unpack_mxfp4_pages(pages, st.H, pids, pos % 16, h)
            np.testing.assert_array_equal(kc, oc.k4_code[0, :L, h])
            np.testing.assert_array_equal(vc, oc.v4_code[0, :L, h])
            np.testing.assert_array_equal(ke, oc.k_bscale[0, :L, h, :4])
            np.testing.assert_array_equal(ve, oc.v_bscale[0, :L, h, :4])
        assert lens[b] == L


@pytest.mark.parametrize("rope", [False, True])
def test_append_matches_oracle(rope):
    tab = inputs.rope_table(1001) if rope else None
    st = Setup(2, 4, 0, 0, EDGE_LENS, seed=51, mxfp4=True, rope=tab, chunks=[1, 17, 100, 299])
    try:
        check_state(st, range(st.B))
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_large_append_all_heads_per_warp():
    st = Setup(8, 4, 0, 0, [16384, 3000], seed=52, mxfp4=True, kv_device="cuda")
    try:
        check_state(st, [0, 1])
        assert st.cache.device_error() == 0
    finally:
        st.close()


@pytest.mark.parametrize("H,G", [(2, 4), (1, 1), (3, 2)])
def test_decode_matches_oracle(H, G):
    st = Setup(H, G, 0, 0, DECODE_LENS, seed=H * 100 + G * 10 + 9, mxfp4=True)
    try:
        q = inputs.queries(st.B, H * G, seed=6).cuda()
        assert check_decode(st, q, range(st.B)) < 1e-4
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_decode_with_rope_and_chunked_appends():
    lens = [300, 1000, 129, 5]
    tab = inputs.rope_table(1001)
    st = Setup(2, 4, 0, 0, lens, seed=54, mxfp4=True, rope=tab,
               chunks=[1, 17, 100, 250, 600] + [L - 1 for L in lens])
    try:
        q = inputs.queries(st.B, 8, seed=10).cuda()
        check_decode(st, q, range(st.B))
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_decode_empty_context():
    st = Setup(1, 4, 0, 0, [1, 400], seed=55, mxfp4=True)
    try:
        q = inputs.queries(2, 4, seed=3).cuda()
        check_decode(st, q, [1], lens=[0, 400])
        st.cache.device_error()              # slot 0 holds 1 position: the mismatch is reported
        check_decode(st, q, [0, 1], lens=[1, 400])
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_decode_workload_sampled():
    wl = inputs.workload("qwen3-8b")
    st = Setup(wl.num_kv_heads, wl.group, 0, 0, wl.context_lens, seed=wl.seed, kv_device="cuda",
               spare_pages=1000, mxfp4=True)
    try:
        order = np.argsort(wl.context_lens)
        bs = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
        check_state(st, bs)
        q = inputs.queries(st.B, wl.num_q_heads, seed=wl.seed, device="cuda")
        check_decode(st, q, bs)
        assert st.cache.device_error() == 0
    finally:
        st.close()
