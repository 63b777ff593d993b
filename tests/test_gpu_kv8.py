"""GPU parity of the whole-cache 8-bit format (KV4_FORMAT_INT8) against the oracle's
KV8 configuration, through the C ABI, on the same seeded inputs.

Bit-exact: 8-bit codes, fp16 Δ/m, slot lengths, INT8 query and its scale, integer QK
accumulators. Floating point: outputs and log-normalizers within abs 2e-3 / rel 1e-2.
"""

import numpy as np
import pytest
import torch

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import inputs, kv4
from kv4_testlib import Setup, check_decode, unpack_kv8_pages

pytestmark = pytest.mark.gpu
D = 128
EDGE_LENS = [1, 15, 16, 17, 143, 144, 145, 160, 161, 300, 1000, 2049]


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
            k8, v8, kd, km, vd, vm = unpack_kv8_pages(pages, st.H, pids, pos % 16, h)
            np.testing.assert_array_equal(k8, oc.k4_code[0, :L, h])
            np.testing.assert_array_equal(v8, oc.v4_code[0, :L, h])
            np.testing.assert_array_equal(kd, oc.k4_delta[0, :L, h])
            np.testing.assert_array_equal(km, oc.k4_min[0, :L, h])
            np.testing.assert_array_equal(vd, oc.v4_delta[0, :L, h])
            np.testing.assert_array_equal(vm, oc.v4_min[0, :L, h])
        assert lens[b] == L


@pytest.mark.parametrize("H,G", [(2, 4), (1, 1), (3, 2)])
def test_append_and_decode_match_oracle(H, G):
    st = Setup(H, G, 0, 0, EDGE_LENS, seed=H * 100 + G * 10 + 7, kv8=True)
    try:
        check_state(st, range(st.B))
        q = inputs.queries(st.B, H * G, seed=5).cuda()
        assert check_decode(st, q, range(st.B)) < 1e-4
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_chunked_and_single_token_appends():
    lens = [300, 1000, 129, 5]
    cuts = [1, 17, 100, 250, 600] + [L - 1 for L in lens]
    st = Setup(2, 4, 0, 0, lens, seed=3, chunks=cuts, kv8=True)
    try:
        check_state(st, range(st.B))
        q = inputs.queries(st.B, 8, seed=9).cuda()
        check_decode(st, q, range(st.B))
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_empty_context_and_bad_page_reported():
    st = Setup(1, 4, 0, 0, [1, 400], seed=8, kv8=True)
    try:
        q = inputs.queries(2, 4, seed=2).cuda()
        st.cache.device_error()
        check_decode(st, q, [1], lens=[0, 400])
        st.cache.device_error()              # slot 0 holds 1 position: the mismatch is reported
        out = torch.empty((2, 4, D), device="cuda")
        bt = st.bt_dev.clone()
        bt[1, 7] = st.num_pages + 100
        kv4.kv4_decode_attention(st.cache.handle, q, torch.tensor([0, 1], dtype=torch.int32,
                                                                  device="cuda"),
                                 torch.tensor([1, 400], dtype=torch.int32, device="cuda"), bt, out)
        assert st.cache.device_error() == 2
        check_decode(st, q, [0, 1], lens=[1, 400])
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_workload_sampled():
    wl = inputs.workload("qwen3-8b")
    st = Setup(wl.num_kv_heads, wl.group, 0, 0, wl.context_lens, seed=wl.seed, kv_device="cuda",
               spare_pages=1000, kv8=True)
    try:
        order = np.argsort(wl.context_lens)
        bs = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
        check_state(st, bs)
        q = inputs.queries(st.B, wl.num_q_heads, seed=wl.seed, device="cuda")
        check_decode(st, q, bs)
        assert st.cache.device_error() == 0
    finally:
        st.close()
