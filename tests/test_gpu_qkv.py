"""The fused projection + append (kv4_qkv_append) against the same two steps done
apart: kv4_linear_bf16 (pinned against a float32 matmul) followed by kv4_append
(pinned against the oracle). Pages, side buffers, slot lengths and the projected
queries must agree byte for byte, for all four cache formats, with and without RoPE,
over chunked appends that start at unaligned positions."""
import numpy as np
import pytest
import torch

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import inputs, kv4

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    kbuild.build()
    kv4.load()


def _case(H, Hq, d_model, lens, cuts, fmt, s, w, rope, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    wq = (torch.randn(((Hq + 2 * H) * D, d_model), generator=g, device="cuda") / d_model ** 0.5).to(torch.bfloat16)
    xs = [torch.randn((L, d_model), generator=g, device="cuda").to(torch.bfloat16) for L in lens]
    need = sum((L + 15) // 16 for L in lens) + 5
    bt = torch.from_numpy(inputs.block_tables(lens, 16, need, seed)).cuda()
    mk = lambda: kv4.KV4Cache(H, need, len(lens) + 1, len(lens), Hq, s, w, fmt=fmt)
    ca, cb = mk(), mk()
    tab = None
    if rope:
        tab = torch.from_numpy(inputs.rope_table(max(lens) + 1)).cuda()
        ca.set_rope(tab)
        cb.set_rope(tab)
    qa_all, qb_all = [], []
    try:
        edges = sorted(set([0] + list(cuts) + [max(lens)]))
        for lo, hi in zip(edges[:-1], edges[1:]):
            rows, cu, slots, starts, btr = [], [0], [], [], []
            for b, L in enumerate(lens):
                a_, z_ = min(lo, L), min(hi, L)
                if z_ <= a_:
                    continue
                rows.append(xs[b][a_:z_])
                cu.append(cu[-1] + z_ - a_)
                slots.append(b)
                starts.append(a_)
                btr.append(b)
            if not rows:
                continue
            x = torch.cat(rows).contiguous()
            cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
            sl_t = torch.tensor(slots, dtype=torch.int32, device="cuda")
            st_t = torch.tensor(starts, dtype=torch.int32, device="cuda")
            bt_t = bt[btr].contiguous()
            # apart: the projection, then the append of its K and V columns
            y = kv4.kv4_linear_bf16(x, wq)
            kvp = y[:, Hq * D:].reshape(x.shape[0], H, 2, D)
            ca.append(kvp[:, :, 0].contiguous(), kvp[:, :, 1].contiguous(), cu_t, sl_t, st_t, bt_t)
            qa_all.append(y[:, :Hq * D].reshape(x.shape[0], Hq, D).clone())
            # fused
            qb_all.append(cb.qkv_append(x, wq, Hq, cu_t, sl_t, st_t, bt_t))
        torch.cuda.synchronize()
        for qa, qb in zip(qa_all, qb_all):
            assert torch.equal(qa, qb)
        pa, sa, _, la = ca.raw_pools()
        pb, sb, _, lb = cb.raw_pools()
        diff = np.flatnonzero(pa != pb)
        assert diff.size == 0, f"{diff.size} page bytes differ, first at {diff[:8]}"
        assert np.array_equal(sa, sb)
        assert np.array_equal(la, lb) and list(la[:len(lens)]) == list(lens)
        assert ca.device_error() == 0 and cb.device_error() == 0
    finally:
        ca.close()
        cb.close()


LENS = [300, 1000, 129, 5, 17]
FORMATS = [(kv4.FORMAT_INT4_HYBRID, 16, 128), (kv4.FORMAT_INT8, 0, 0), (kv4.FORMAT_NVFP4, 0, 0),
           (kv4.FORMAT_MXFP4, 0, 0)]


@pytest.mark.parametrize("fmt,s,w", FORMATS)
@pytest.mark.parametrize("rope", [False, True])
def test_fused_equals_projection_then_append(fmt, s, w, rope):
    _case(2, 8, 256, LENS, [], fmt, s, w, rope, seed=11)


@pytest.mark.parametrize("fmt,s,w", FORMATS)
def test_fused_chunked_appends(fmt, s, w):
    cuts = [1, 3, 17, 100, 250, 600] + [L - 1 for L in LENS]
    _case(2, 8, 256, LENS, cuts, fmt, s, w, True, seed=12)


@pytest.mark.parametrize("fmt,s,w", FORMATS)
def test_fused_wide_tiles(fmt, s, w):
    """Enough tokens for 256-wide tiles (K and V of a head in one tile); the cases above
    take 128-wide tiles (K or V alone)."""
    _case(2, 8, 256, [1500, 2000, 333], [700], fmt, s, w, True, seed=14)


def test_fused_qwen3_8b_shapes():
    """Qwen3-8B attention shapes (32 q heads, 8 KV heads, d_model 4096): a decode step of
    256 single tokens after a 600-token prefill."""
    lens = [600 + (b % 3) for b in range(256)]
    _case(8, 32, 4096, lens, [599, 600, 601], kv4.FORMAT_INT4_HYBRID, 16, 128, True, seed=13)
