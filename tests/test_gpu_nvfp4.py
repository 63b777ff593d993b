"""GPU parity of the NVFP4 format (KV4_FORMAT_NVFP4) against the oracle's reading R12:
E2M1 codes, E4M3 block scales, FP32 vector scales and slot lengths bit for bit."""
import numpy as np
import pytest
import torch

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import inputs, kv4
from kv4_testlib import Setup, unpack_nvfp4_pages

pytestmark = pytest.mark.gpu
EDGE_LENS = [1, 15, 16, 17, 143, 144, 145, 300, 1000]


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
            kc, kbs, kg, vc, vbs, vg = unpack_nvfp4_pages(pages, st.H, pids, pos % 16, h)
            np.testing.assert_array_equal(kc, oc.k4_code[0, :L, h])
            np.testing.assert_array_equal(vc, oc.v4_code[0, :L, h])
            np.testing.assert_array_equal(kbs, oc.k_bscale[0, :L, h])
            np.testing.assert_array_equal(vbs, oc.v_bscale[0, :L, h])
            np.testing.assert_array_equal(kg.view(np.uint32), oc.k_gscale[0, :L, h].view(np.uint32))
            np.testing.assert_array_equal(vg.view(np.uint32), oc.v_gscale[0, :L, h].view(np.uint32))
        assert lens[b] == L


@pytest.mark.parametrize("rope", [False, True])
def test_append_matches_oracle(rope):
    tab = inputs.rope_table(1001) if rope else None
    st = Setup(2, 4, 0, 0, EDGE_LENS, seed=51, nvfp4=True, rope=tab, chunks=[1, 17, 100, 299])
    try:
        check_state(st, range(st.B))
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_large_append_all_heads_per_warp():
    st = Setup(8, 4, 0, 0, [16384, 3000], seed=52, nvfp4=True, kv_device="cuda")
    try:
        check_state(st, [0, 1])
        assert st.cache.device_error() == 0
    finally:
        st.close()
