"""kv4_decode_attention_noalloc against kv4_decode_attention.

Some callers of libkv4 cannot allocate device memory when they decode: their
host framework's allocator has already reserved the GPU for its own arena, or
they are a plugin handed device buffers with no right to call cudaMalloc. The
allocation-free entry point serves them: it reads the pools through plain
pointers and keeps its split-K scratch in a fixed array inside libkv4. This
test calls it through the C ABI twice in a row (different queries and batch
sizes, so the second call runs over the first call's leftover scratch) and
checks each result against the regular entry point on the same inputs.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import math

import numpy as np
import pytest
import torch

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import inputs, kv4
from kv4_testlib import Setup

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    kbuild.build()
    kv4.load()


def _config(st):
    return kv4.kv4_cache_config(st.H, 128, 16, st.s, st.w, st.num_pages, st.B + 1, st.B,
                                st.H * st.G, 0)


def _regular(st, q, lens, rows):
    B, Hq = q.shape[0], q.shape[1]
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    kv4.kv4_decode_attention(st.cache.handle, q, torch.tensor(rows, dtype=torch.int32,
                                                              device="cuda"),
                             torch.tensor(lens, dtype=torch.int32, device="cuda"),
                             st.bt_dev[rows].contiguous(), out, lse, sm_scale=1 / math.sqrt(128))
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def _noalloc(st, q, lens, rows):
    info = st.cache.info()
    B, Hq = q.shape[0], q.shape[1]
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    kv4.kv4_decode_attention_noalloc(
        _config(st), info.page_pool_dev, info.side_pool_dev, info.seq_len_dev, q,
        torch.tensor(rows, dtype=torch.int32, device="cuda"),
        torch.tensor(lens, dtype=torch.int32, device="cuda"), st.bt_dev[rows].contiguous(),
        out, lse, sm_scale=1 / math.sqrt(128))
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def test_noalloc_matches_regular_decode_on_two_calls_in_a_row():
    lens = [5000, 1, 144, 145, 300, 1000, 2049, 16, 17, 777, 3100, 12000]
    st = Setup(8, 4, 16, 128, lens, seed=21, kv_device="cuda")
    try:
        # first call: the whole batch
        rows = list(range(st.B))
        q1 = inputs.queries(st.B, 32, seed=31, device="cuda")
        ref1 = _regular(st, q1, lens, rows)
        got1 = _noalloc(st, q1, lens, rows)
        np.testing.assert_allclose(got1[0], ref1[0], atol=ATOL, rtol=RTOL)
        np.testing.assert_allclose(got1[1], ref1[1], atol=ATOL, rtol=RTOL)
        # second call: a smaller batch and other queries, over the first call's scratch
        rows2 = [11, 3, 0, 6]
        lens2 = [lens[r] for r in rows2]
        q2 = inputs.queries(len(rows2), 32, seed=32, device="cuda")
        ref2 = _regular(st, q2, lens2, rows2)
        got2 = _noalloc(st, q2, lens2, rows2)
        np.testing.assert_allclose(got2[0], ref2[0], atol=ATOL, rtol=RTOL)
        np.testing.assert_allclose(got2[1], ref2[1], atol=ATOL, rtol=RTOL)
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_noalloc_refuses_batches_beyond_its_scratch():
    st = Setup(8, 4, 16, 128, [40], seed=22)
    try:
        info = st.cache.info()
        B = 600                                  # the workspace of 600 x 32 heads exceeds 16 MiB
        q = torch.zeros((B, 32, 128), dtype=torch.bfloat16, device="cuda")
        out = torch.zeros((B, 32, 128), dtype=torch.float32, device="cuda")
        z = torch.zeros(B, dtype=torch.int32, device="cuda")
        bt = st.bt_dev[[0] * B].contiguous()
        with pytest.raises(kv4.KV4Error) as e:
            kv4.kv4_decode_attention_noalloc(_config(st), info.page_pool_dev, info.side_pool_dev,
                                             info.seq_len_dev, q, z, z, bt, out)
        assert e.value.status == -5
        assert torch.count_nonzero(out).item() == 0     # nothing was enqueued
    finally:
        st.close()
