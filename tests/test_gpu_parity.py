"""GPU parity: libkv4 (through the C ABI) against the CPU oracle on the same seeded inputs.

Bit-exact: INT4 codes, fp16 Δ/m, INT8 side entries, slot lengths, INT8 query and
its scale, integer QK accumulators, u8 PV weights. Floating point: outputs and
log-normalizers within abs 2e-3 / rel 1e-2.
"""

import numpy as np
import pytest
import torch

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import inputs, kv4
from kv4_testlib import Setup, check_decode, unpack_page_tokens, unpack_side

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    kbuild.build()
    kv4.load()


def check_state(st: Setup, bs):
    pages, side, side_block, lens = st.cache.raw_pools()
    S = st.s + st.w
    for b in bs:
        oc = st.oracle_for(b)
        L = st.lens[b]
        pos = np.arange(L)
        pids = st.bt[b][pos // 16]
        for h in range(st.H):
            k, v, kd, km, vd, vm = unpack_page_tokens(pages, st.H, pids, pos % 16, h)
            np.testing.assert_array_equal(k, oc.k4_code[0, :L, h])
            np.testing.assert_array_equal(v, oc.v4_code[0, :L, h])
            np.testing.assert_array_equal(kd, oc.k4_delta[0, :L, h])
            np.testing.assert_array_equal(km, oc.k4_min[0, :L, h])
            np.testing.assert_array_equal(vd, oc.v4_delta[0, :L, h])
            np.testing.assert_array_equal(vm, oc.v4_min[0, :L, h])
            if S:
                k8, v8, k8d, k8m, v8d, v8m = unpack_side(side, side_block, st.H, S, b, h)
                np.testing.assert_array_equal(k8, oc.k8_code[0, :, h])
                np.testing.assert_array_equal(v8, oc.v8_code[0, :, h])
                np.testing.assert_array_equal(k8d, oc.k8_delta[0, :, h])
                np.testing.assert_array_equal(k8m, oc.k8_min[0, :, h])
                np.testing.assert_array_equal(v8d, oc.v8_delta[0, :, h])
                np.testing.assert_array_equal(v8m, oc.v8_min[0, :, h])
        assert lens[b] == L


# --------------------------------------------------------------------------- small cases

EDGE_LENS = [1, 15, 16, 17, 143, 144, 145, 160, 161, 300, 1000, 2049]


@pytest.mark.parametrize("H,G,s,w", [(2, 4, 16, 128), (1, 1, 16, 128), (3, 2, 16, 128),
                                     (2, 4, 0, 0), (1, 4, 32, 48), (2, 2, 0, 64), (1, 4, 16, 0),
                                     (1, 2, 48, 16)])
def test_append_and_decode_match_oracle(H, G, s, w):
    st = Setup(H, G, s, w, EDGE_LENS, seed=H * 100 + G * 10 + s + w)
    try:
        check_state(st, range(st.B))
        q = inputs.queries(st.B, H * G, seed=5).cuda()
        worst = check_decode(st, q, range(st.B))
        assert worst < 1e-4
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_tiny_workload():
    wl = inputs.workload("tiny")
    st = Setup(wl.num_kv_heads, wl.group, wl.sink, wl.window, wl.context_lens, seed=wl.seed)
    try:
        check_state(st, range(st.B))
        q = inputs.queries(st.B, wl.num_q_heads, seed=wl.seed).cuda()
        check_decode(st, q, range(st.B))
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_chunked_appends_equal_one_sequential_append():
    st = Setup(2, 4, 16, 128, [300, 1000, 129, 5], seed=3, chunks=[1, 17, 100, 250, 600])
    try:
        check_state(st, range(st.B))
        q = inputs.queries(st.B, 8, seed=9).cuda()
        check_decode(st, q, range(st.B))
    finally:
        st.close()


def test_decode_steps_with_single_token_appends():
    """Prefill, then three decode-style steps that append one token per sequence."""
    lens = [200, 513, 144, 1]
    cuts = sorted(set([L + i for L in lens for i in range(3)]))
    st = Setup(2, 4, 16, 128, [L + 3 for L in lens], seed=4, chunks=cuts)
    try:
        check_state(st, range(st.B))
        q = inputs.queries(st.B, 8, seed=11).cuda()
        check_decode(st, q, range(st.B))
    finally:
        st.close()


def test_empty_context_and_repeatability():
    st = Setup(1, 2, 16, 128, [0 + 1, 700], seed=6)
    try:
        q = inputs.queries(2, 2, seed=2).cuda()
        lens = [0, 700]
        st.cache.device_error()
        check_decode(st, q, [0, 1], lens=lens)
        st.cache.device_error()            # slot 0 holds 1 position: the mismatch is reported
        a, _, _ = st.decode(q)
        b, _, _ = st.decode(q)
        assert torch.equal(a, b)
    finally:
        st.close()


def test_device_errors_are_reported_without_faulting():
    st = Setup(1, 4, 16, 128, [400, 50], seed=8)
    try:
        q = inputs.queries(2, 4, seed=1).cuda()
        out = torch.empty((2, 4, D), device="cuda")
        cl = torch.tensor([400, 50], dtype=torch.int32, device="cuda")
        bad_slot = torch.tensor([0, 7], dtype=torch.int32, device="cuda")
        kv4.kv4_decode_attention(st.cache.handle, q, bad_slot, cl, st.bt_dev, out)
        assert st.cache.device_error() == 1
        bt = st.bt_dev.clone()
        bt[0, 5] = st.num_pages + 100
        kv4.kv4_decode_attention(st.cache.handle, q, torch.tensor([0, 1], dtype=torch.int32,
                                                                  device="cuda"), cl, bt, out)
        assert st.cache.device_error() == 2
        kv4.kv4_decode_attention(st.cache.handle, q, torch.tensor([0, 1], dtype=torch.int32,
                                                                  device="cuda"),
                                 torch.tensor([399, 50], dtype=torch.int32, device="cuda"),
                                 st.bt_dev, out)
        assert st.cache.device_error() == 4
        # the context is intact: a correct call still matches the oracle
        check_decode(st, q, [0, 1])
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_host_validation_on_device():
    st = Setup(2, 4, 16, 128, [40], seed=1)
    try:
        q = inputs.queries(1, 6, seed=1).cuda()                 # 6 q heads over 2 KV heads
        out = torch.empty((1, 6, D), device="cuda")
        with pytest.raises(kv4.KV4Error):
            kv4.kv4_decode_attention(st.cache.handle, q, torch.zeros(1, dtype=torch.int32,
                                                                     device="cuda"),
                                     torch.tensor([40], dtype=torch.int32, device="cuda"),
                                     st.bt_dev, out)
        q2 = inputs.queries(2, 8, seed=1).cuda()                # batch above max_batch
        out2 = torch.empty((2, 8, D), device="cuda")
        with pytest.raises(kv4.KV4Error):
            kv4.kv4_decode_attention(st.cache.handle, q2, torch.zeros(2, dtype=torch.int32,
                                                                      device="cuda"),
                                     torch.tensor([40, 40], dtype=torch.int32, device="cuda"),
                                     st.bt_dev.repeat(2, 1), out2)
    finally:
        st.close()


# --------------------------------------------------------------------------- full-size workloads

def _sampled(lens, k=3):
    order = np.argsort(lens)
    return sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})[:k]


@pytest.mark.parametrize("name", ["qwen3-4b", "qwen3-8b"])
def test_workload_sampled(name):
    wl = inputs.workload(name)
    st = Setup(wl.num_kv_heads, wl.group, wl.sink, wl.window, wl.context_lens, seed=wl.seed,
               kv_device="cuda", spare_pages=1000)
    try:
        bs = _sampled(np.array(wl.context_lens))
        check_state(st, bs)
        q = inputs.queries(st.B, wl.num_q_heads, seed=wl.seed, device="cuda")
        check_decode(st, q, bs)
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_long_tail_layer_sampled():
    wl = inputs.workload("long-tail")
    st = Setup(wl.num_kv_heads, wl.group, wl.sink, wl.window, wl.context_lens, seed=wl.seed,
               kv_device="cuda", spare_pages=5000)
    try:
        bs = _sampled(np.array(wl.context_lens))
        q = inputs.queries(st.B, wl.num_q_heads, seed=wl.seed, device="cuda")
        check_decode(st, q, bs)
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_large_batch_of_short_contexts():
    """1300 sequences of 0..200 tokens: more sequences than threads in the plan kernel and
    in the split kernel's own plan (several sequences per thread), 2600 units."""
    rng = np.random.default_rng(31)
    lens = [int(x) for x in rng.integers(1, 201, size=1300)]
    lens[7] = 1
    st = Setup(2, 4, 16, 128, lens, seed=31)
    try:
        q = inputs.queries(st.B, 8, seed=31).cuda()
        bs = [0, 7, 511, 512, 513, 1023, 1024, 1299] + sorted(int(b) for b in np.argsort(lens)[-2:])
        check_decode(st, q, bs)
        zl = list(lens)
        zl[3] = 0                                             # an empty context inside the batch
        check_decode(st, q, [2, 3, 4], lens=zl)
        st.cache.device_error()                               # slot 3 holds more than 0 positions
    finally:
        st.close()


def test_one_very_long_context():
    """One 120,000-token sequence among short ones: its units are cut into hundreds of
    pieces, so the merge takes more than 32 partials per q head."""
    lens = [120000, 5, 3000]
    st = Setup(1, 4, 16, 128, lens, seed=32, kv_device="cuda", spare_pages=16)
    try:
        q = inputs.queries(st.B, 4, seed=32).cuda()
        check_decode(st, q, [0, 1, 2])
        assert st.cache.device_error() == 0
    finally:
        st.close()


def test_append_stress_sampled():
    # (a) 512 sequences, one new token each after a short prefix
    lens = [33 + (i % 7) for i in range(512)]
    st = Setup(8, 4, 16, 128, lens, seed=12, kv_device="cuda",
               chunks=[L - 1 for L in set(lens)])
    try:
        check_state(st, [0, 255, 511])
    finally:
        st.close()
    # (b) 8 sequences, one 16384-token re-prefill chunk each
    st = Setup(8, 4, 16, 128, [16384] * 8, seed=13, kv_device="cuda")
    try:
        check_state(st, [0, 7])
    finally:
        st.close()
