"""GPU parity with RoPE fused into the append and the query preparation
(kv4_cache_set_rope), against the oracle's reading R11, for both cache formats.

Bit-exact: codes, fp16 Δ/m, side entries, INT8 query, integer QK accumulators and
u8 weights; outputs within abs 2e-3 / rel 1e-2 (helpers of the plain parity tests).
"""
import numpy as np
import pytest
import torch

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import inputs, kv4
from kv4_testlib import Setup
import test_gpu_kv8 as kv8_checks
import test_gpu_parity as checks

pytestmark = pytest.mark.gpu
EDGE_LENS = [1, 15, 16, 17, 143, 144, 145, 160, 161, 300, 1000, 2049]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    kbuild.build()
    kv4.load()


@pytest.mark.parametrize("H,G,s,w", [(2, 4, 16, 128), (1, 2, 0, 0), (3, 1, 32, 32)])
def test_hybrid_with_rope_matches_oracle(H, G, s, w):
    st = Setup(H, G, s, w, EDGE_LENS, seed=31 + H, rope=inputs.rope_table(2100))
    try:
        checks.check_state(st, range(st.B))
        q = inputs.queries(st.B, H * G, seed=8).cuda()
        assert checks.check_decode(st, q, range(st.B)) < 1e-4
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_kv8_with_rope_matches_oracle():
    st = Setup(2, 4, 0, 0, EDGE_LENS, seed=41, kv8=True, rope=inputs.rope_table(2049))
    try:
        kv8_checks.check_state(st, range(st.B))
        q = inputs.queries(st.B, 8, seed=9).cuda()
        assert kv8_checks.check_decode(st, q, range(st.B)) < 1e-4
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_chunked_appends_with_rope():
    lens = [300, 1000, 129, 5]
    st = Setup(2, 4, 16, 128, lens, seed=3, chunks=[1, 17, 100, 250, 600] + [L - 1 for L in lens],
               rope=inputs.rope_table(1000))
    try:
        checks.check_state(st, range(st.B))
        q = inputs.queries(st.B, 8, seed=10).cuda()
        checks.check_decode(st, q, range(st.B))
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_positions_beyond_the_table_are_reported():
    st = Setup(1, 2, 16, 128, [40], seed=5, rope=inputs.rope_table(40))
    try:
        assert st.cache.device_error() == 0
        k, v = inputs.sequence_kv(0, 1, 1, 99)
        one = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
        st.cache.append(k.cuda(), v.cuda(), one, torch.zeros(1, dtype=torch.int32, device="cuda"),
                        torch.tensor([40], dtype=torch.int32, device="cuda"), st.bt_dev)
        torch.cuda.synchronize()
        assert st.cache.device_error() == 3            # position 40 is past the table
        q = inputs.queries(1, 2, seed=3).cuda()
        out = torch.empty((1, 2, 128), device="cuda")
        kv4.kv4_decode_attention(st.cache.handle, q, torch.zeros(1, dtype=torch.int32, device="cuda"),
                                 torch.tensor([41], dtype=torch.int32, device="cuda"), st.bt_dev, out)
        torch.cuda.synchronize()
        assert st.cache.device_error() == 3
        checks.check_decode(st, q, [0])                # the 40 stored positions are intact
        assert st.cache.device_error() == 0
    finally:
        st.close()
