"""kv4_decode_attention_noalloc against kv4_decode_attention.

Some callers of libkv4 cannot allocate device memory when they decode: their
host framework's allocator has already reserved the GPU for its own arena, or
they are a plugin handed device buffers with no right to call cudaMalloc. The
allocation-free entry point serves them: it reads the pools through plain
pointers and keeps its split-K scratch in a fixed array inside libkv4. These
tests call it through the C ABI twice in a row (different queries and batch
sizes, so the second call runs over the first call's leftover scratch) and
check each result against the regular entry point on the same inputs: within
the parity tolerance, and in fact bit for bit, since both launch the same
kernels on the same grid. The cases cover the three cache formats (the
whole-cache ones without a side pool) and the three group sizes, and the
error word that the allocation-free path reports device-side errors through.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import math

import numpy as np
import pytest
import torch

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import inputs, kv4
from kv4_testlib import Guarded, Setup

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    kbuild.build()
    kv4.load()
    kv4.kv4_noalloc_device_error(clear=True)      # start from a clear error word


def _fmt(st):
    if st.mxfp4:
        return kv4.FORMAT_MXFP4
    return kv4.FORMAT_NVFP4 if st.nvfp4 else (kv4.FORMAT_INT8 if st.kv8 else kv4.FORMAT_INT4_HYBRID)


def _config(st):
    return kv4.kv4_cache_config(st.H, 128, 16, st.s, st.w, st.num_pages, st.B + 1, st.B,
                                st.H * st.G, 0, _fmt(st))


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


def _noalloc(st, q, lens, rows, side=True, block_table=None):
    info = st.cache.info()
    B, Hq = q.shape[0], q.shape[1]
    out = Guarded((B, Hq, 128), torch.float32, float("nan"))
    lse = Guarded((B, Hq), torch.float32, float("nan"))
    bt = st.bt_dev[rows].contiguous() if block_table is None else block_table
    kv4.kv4_decode_attention_noalloc(
        _config(st), info.page_pool_dev, info.side_pool_dev if side else 0, info.seq_len_dev, q,
        torch.tensor(rows, dtype=torch.int32, device="cuda"),
        torch.tensor(lens, dtype=torch.int32, device="cuda"), bt,
        out.t, lse.t, sm_scale=1 / math.sqrt(128))
    torch.cuda.synchronize()
    assert out.intact() and lse.intact()
    return out.t.cpu().numpy(), lse.t.cpu().numpy()


def _same(got, ref):
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, atol=ATOL, rtol=RTOL)
        np.testing.assert_array_equal(g, r)


def _two_calls(st, lens, side=True):
    Hq = st.H * st.G
    # first call: the whole batch
    rows = list(range(st.B))
    q1 = inputs.queries(st.B, Hq, seed=31, device="cuda")
    _same(_noalloc(st, q1, lens, rows, side), _regular(st, q1, lens, rows))
    # second call: a smaller batch and other queries, over the first call's scratch
    rows2 = [st.B - 1, 3, 0, 6]
    lens2 = [lens[r] for r in rows2]
    q2 = inputs.queries(len(rows2), Hq, seed=32, device="cuda")
    _same(_noalloc(st, q2, lens2, rows2, side), _regular(st, q2, lens2, rows2))
    assert st.cache.device_error() == 0
    assert kv4.kv4_noalloc_device_error() == 0


LENS = [5000, 1, 144, 145, 300, 1000, 2049, 16, 17, 777, 3100, 12000]


def test_noalloc_matches_regular_decode_on_two_calls_in_a_row():
    st = Setup(8, 4, 16, 128, LENS, seed=21, kv_device="cuda")
    try:
        _two_calls(st, LENS)
    finally:
        st.close()


@pytest.mark.parametrize("H,G", [(4, 1), (2, 2)])
def test_noalloc_other_group_sizes(H, G):
    st = Setup(H, G, 16, 128, LENS, seed=23, kv_device="cuda")
    try:
        _two_calls(st, LENS)
    finally:
        st.close()


@pytest.mark.parametrize("fmt", ["kv8", "nvfp4", "mxfp4"])
def test_noalloc_whole_cache_formats_without_a_side_pool(fmt):
    st = Setup(8, 4, 0, 0, LENS, seed=24, kv_device="cuda", kv8=fmt == "kv8", nvfp4=fmt == "nvfp4",
               mxfp4=fmt == "mxfp4")
    try:
        _two_calls(st, LENS, side=False)
    finally:
        st.close()


def test_noalloc_reports_device_errors_through_its_error_word():
    st = Setup(2, 4, 16, 128, [400, 50], seed=25)
    try:
        q = inputs.queries(2, 8, seed=3, device="cuda")
        bt = st.bt_dev.clone()
        bt[0, 5] = st.num_pages + 100                   # a page outside the pool
        _noalloc(st, q, [400, 50], [0, 1], block_table=bt)
        assert kv4.kv4_noalloc_device_error(clear=False) == 2      # KV4_DEVERR_BAD_PAGE
        assert kv4.kv4_noalloc_device_error(clear=True) == 2
        assert kv4.kv4_noalloc_device_error() == 0
        # a correct call afterwards still equals the regular path and reports nothing
        _same(_noalloc(st, q, [400, 50], [0, 1]), _regular(st, q, [400, 50], [0, 1]))
        assert kv4.kv4_noalloc_device_error() == 0
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
