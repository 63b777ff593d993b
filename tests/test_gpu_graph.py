"""The decode call (prep, split and merge, the latter two as programmatic dependent
launches) and the append can be captured in a CUDA graph and replayed: the replay
gives the same bits as direct calls."""
import math

import pytest
import torch

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import inputs, kv4
from kv4_testlib import Setup

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    kbuild.build()
    kv4.load()


def test_decode_layers_replay_from_a_graph():
    st = Setup(2, 4, 16, 128, [300, 1000, 129, 5], seed=21)
    try:
        B, Hq = st.B, 8
        q = inputs.queries(B, Hq, seed=3).cuda()
        slots = torch.arange(B, dtype=torch.int32, device="cuda")
        cl = torch.tensor(st.lens, dtype=torch.int32, device="cuda")
        ref = torch.empty((B, Hq, 128), device="cuda")
        ref_lse = torch.empty((B, Hq), device="cuda")
        kv4.kv4_decode_attention(st.cache.handle, q, slots, cl, st.bt_dev, ref, ref_lse,
                                 sm_scale=1 / math.sqrt(128))
        torch.cuda.synchronize()
        layers = 4
        outs = [torch.zeros((B, Hq, 128), device="cuda") for _ in range(layers)]
        lses = [torch.zeros((B, Hq), device="cuda") for _ in range(layers)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(layers):
                kv4.kv4_decode_attention(st.cache.handle, q, slots, cl, st.bt_dev, outs[i],
                                         lses[i], sm_scale=1 / math.sqrt(128))
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        for i in range(layers):
            assert torch.equal(outs[i], ref)
            assert torch.equal(lses[i], ref_lse)
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_append_replays_from_a_graph():
    lens = [40, 77]
    a = Setup(1, 2, 16, 128, lens, seed=5)                 # appended directly
    b = kv4.KV4Cache(1, a.num_pages, max_slots=a.B + 1, max_batch=a.B, max_q_heads=2)
    try:
        k = torch.cat([a.kv[i][0] for i in range(2)]).cuda()
        v = torch.cat([a.kv[i][1] for i in range(2)]).cuda()
        cu = torch.tensor([0, 40, 117], dtype=torch.int32, device="cuda")
        slots = torch.arange(2, dtype=torch.int32, device="cuda")
        start = torch.zeros(2, dtype=torch.int32, device="cuda")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            b.append(k, v, cu, slots, start, a.bt_dev)
        g.replay()
        torch.cuda.synchronize()
        pa, sa, _, la = a.cache.raw_pools()
        pb, sb, _, lb = b.raw_pools()
        assert (pa == pb).all() and (sa == sb).all() and list(lb[:2]) == lens
        assert b.device_error() == 0
    finally:
        a.close()
        b.close()
