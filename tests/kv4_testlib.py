"""Test helpers: read libkv4's documented page/side layout back into the oracle's
logical form, and set up matching GPU and oracle caches from the seeded inputs."""
import math

import numpy as np
import torch

import oracle
from int8_hybrid_paged_gb300 import inputs
from int8_hybrid_paged_gb300.kv4 import (FORMAT_INT4_HYBRID, FORMAT_INT8, FORMAT_MXFP4, FORMAT_NVFP4,
                                          KV4Cache)

D = 128
P = 16
BLOCK = 2176


def unpack_page_tokens(pages, H, page_ids, slots_in_page, h):
    """K/V INT4 codes and metadata of positions (page_ids[i], slots_in_page[i]) of head h,
    following the page-block layout declared in include/kv4.h."""
    n = len(page_ids)
    base = (np.asarray(page_ids, np.int64) * H + h) * BLOCK
    ts = np.asarray(slots_in_page, np.int64)
    dd = np.arange(D)
    lane = dd // 4
    i, c = lane % 8, lane // 8
    kbyte = (i // 4) * 512 + (4 * (ts[:, None] % 8) + c[None, :]) * 16 + (i % 4 * 4)[None, :] \
        + np.array([0, 2, 1, 3])[dd % 4][None, :]
    kb = pages[base[:, None] + kbyte]
    k = np.where((ts[:, None] // 8) == 0, kb & 15, kb >> 4).astype(np.uint8)
    j = np.arange(64)[None, :]
    t = ts[:, None]
    voff = 4 * (8 * (4 * (j % 8) + t % 4) + j // 8) + t // 4
    vbytes = pages[base[:, None] + 1024 + voff]
    v = np.empty((n, D), np.uint8)
    v[:, 0::2] = vbytes & 15
    v[:, 1::2] = vbytes >> 4
    mrow = base + 2048 + 16 * (ts % 8) + 4 * (ts // 8)
    km = pages[mrow[:, None] + np.arange(4)[None, :]].copy().view(np.uint16)
    vm = pages[(mrow + 8)[:, None] + np.arange(4)[None, :]].copy().view(np.uint16)
    return k, v, km[:, 0], km[:, 1], vm[:, 0], vm[:, 1]


def side_k_offset(r, d):
    """Byte of (side row r, dim d) in a group's K block, as declared in include/kv4.h."""
    word = d % 32 // 4
    return 1024 * (word // 4) + 64 * r + 16 * (d // 32) + 4 * (word % 4) + d % 4


def side_v_byte(r):
    return (r // 8) % 2 + 2 * ((r // 4) % 2)


def side_v_offset(r, d):
    """Byte of (side row r, dim d) in a group's V block, as declared in include/kv4.h."""
    n = 4 * (d % 8) + r % 4
    word = 2 * (d // 16) + (d // 8) % 2
    return 16 * (32 * (word // 4) + n) + 4 * (word % 4) + side_v_byte(r)


def unpack_int8_rows(blk, gbase, rr):
    """8-bit codes and metadata of rows rr of the 16-row groups starting at byte
    offsets gbase of blk (side groups, or pages of the 8-bit format)."""
    d = np.arange(128)
    koff = np.array([[side_k_offset(x, y) for y in d] for x in range(16)])
    voff = np.array([[side_v_offset(x, y) for y in d] for x in range(16)])
    k8 = blk[gbase[:, None] + koff[rr]]
    v8 = blk[gbase[:, None] + 2176 + voff[rr]]
    kmo = gbase + 2048 + 8 * (rr % 8) + 4 * (rr // 8)
    vmo = gbase + 2176 + 2048 + 16 * (rr % 4) + 4 * np.array([side_v_byte(x) for x in rr], dtype=np.int64)
    km = blk[kmo[:, None] + np.arange(4)[None, :]].copy().view(np.uint16)
    vm = blk[vmo[:, None] + np.arange(4)[None, :]].copy().view(np.uint16)
    return k8, v8, km[:, 0], km[:, 1], vm[:, 0], vm[:, 1]


def unpack_kv8_pages(pages, H, page_ids, slots_in_page, h):
    """8-bit codes and metadata of positions (page_ids[i], slots_in_page[i]) of head h in
    a KV4_FORMAT_INT8 page pool: one 4352-byte group per (page, head), row = slot."""
    base = (np.asarray(page_ids, np.int64) * H + h) * 4352
    return unpack_int8_rows(pages, base, np.asarray(slots_in_page, np.int64))


def unpack_nvfp4_pages(pages, H, page_ids, slots_in_page, h):
    """E2M1 codes [n][128], E4M3 block scale bits [n][8] and FP32 vector scales [n] of K and
    of V at positions (page_ids[i], slots_in_page[i]) of head h in a KV4_FORMAT_NVFP4
    pool, following the layout declared in include/kv4.h."""
    base = (np.asarray(page_ids, np.int64) * H + h) * 2432
    t = np.asarray(slots_in_page, np.int64)[:, None]
    d = np.arange(128)[None, :]
    # K: dims (2j, 2j+1), j = 8b + jj
    j = d // 2
    b, jj = j // 8, j % 8
    koff = 16 * (32 * (b // 4) + 4 * (t % 8) + jj % 4) + 4 * (b % 4) + t // 8 + 2 * (jj // 4)
    kbyte = pages[base[:, None] + koff]
    kc = np.where(d % 2 == 0, kbyte & 15, kbyte >> 4).astype(np.uint8)
    # V: a byte holds dim 16m + r of tokens t (low nibble) and t + 8 (high nibble);
    # the word of (16m + r mod 8, t mod 4) has dims r < 8, r >= 8 of tokens {t, t+8} in
    # bytes 0, 1 and of tokens {t+4, t+12} in bytes 2, 3
    m, r = d // 16, d % 16
    g = r % 8
    voff = 16 * (32 * (m // 4) + 4 * g + t % 4) + 4 * (m % 4) + 2 * ((t // 4) % 2) + (r >= 8)
    vbyte = pages[base[:, None] + 1216 + voff]
    vc = np.where(t < 8, vbyte & 15, vbyte >> 4).astype(np.uint8)
    ts = np.asarray(slots_in_page, np.int64)
    bb = np.arange(8)[None, :]
    tt = ts[:, None]
    kbs = pages[base[:, None] + 1024 + 16 * (tt % 8) + 2 * bb + tt // 8]
    vbs = pages[base[:, None] + 1216 + 1024 + 32 * (tt % 4) + 4 * bb + np.array([0, 2, 1, 3])[tt // 4]]
    goff = 1152 + 8 * (ts % 8) + 4 * (ts // 8)
    kg = pages[(base + goff)[:, None] + np.arange(4)[None, :]].copy().view(np.float32)[:, 0]
    vg = pages[(base + 1216 + goff)[:, None] + np.arange(4)[None, :]].copy().view(np.float32)[:, 0]
    return kc, kbs, kg, vc, vbs, vg


def unpack_mxfp4_pages(pages, H, page_ids, slots_in_page, h):
    """E2M1 codes [n][128] and E8M0 scale bytes [n][4] of K and of V at positions
    (page_ids[i], slots_in_page[i]) of head h in a KV4_FORMAT_MXFP4 pool (2176-byte blocks,
    halves of 1088 bytes), following the layout declared in include/kv4.h."""
    base = (np.asarray(page_ids, np.int64) * H + h) * 2176
    t = np.asarray(slots_in_page, np.int64)[:, None]
    d = np.arange(128)[None, :]
    j = d // 2
    b, jj = j // 8, j % 8
    koff = 16 * (32 * (b // 4) + 4 * (t % 8) + jj % 4) + 4 * (b % 4) + t // 8 + 2 * (jj // 4)
    kbyte = pages[base[:, None] + koff]
    kc = np.where(d % 2 == 0, kbyte & 15, kbyte >> 4).astype(np.uint8)
    m, r = d // 16, d % 16
    g = r % 8
    kb = np.array([0, 2, 1, 3])[t // 4]
    voff = 16 * (32 * (m // 4) + 4 * g + t % 4) + 4 * (m % 4) + 2 * ((t // 4) % 2) + (r >= 8)
    vbyte = pages[base[:, None] + 1088 + voff]
    vc = np.where(t < 8, vbyte & 15, vbyte >> 4).astype(np.uint8)
    bb = np.arange(4)[None, :]
    ke = pages[base[:, None] + 1024 + 8 * (t % 8) + 2 * bb + t // 8]
    ve = pages[base[:, None] + 1088 + 1024 + 16 * (t % 4) + 4 * bb + kb]
    return kc, ke, vc, ve


def unpack_side(side, side_block, H, S, slot, h):
    """INT8 side rows 0..S-1 of (slot, head h): 16-row groups of a K block and a V block
    in tensor-core fragment order, as declared in include/kv4.h."""
    blk = side[(slot * H + h) * side_block:(slot * H + h + 1) * side_block]
    r = np.arange(S)
    g = (r // 16) * 4352
    rr = r % 16
    d = np.arange(128)
    koff = np.array([[side_k_offset(x, y) for y in d] for x in range(16)])
    voff = np.array([[side_v_offset(x, y) for y in d] for x in range(16)])
    k8 = blk[g[:, None] + koff[rr]]
    v8 = blk[g[:, None] + 2176 + voff[rr]]
    kmo = g + 2048 + 8 * (rr % 8) + 4 * (rr // 8)
    vmo = g + 2176 + 2048 + 16 * (rr % 4) + 4 * np.array([side_v_byte(x) for x in rr], dtype=np.int64)
    km = blk[kmo[:, None] + np.arange(4)[None, :]].copy().view(np.uint16)
    vm = blk[vmo[:, None] + np.arange(4)[None, :]].copy().view(np.uint16)
    return k8, v8, km[:, 0], km[:, 1], vm[:, 0], vm[:, 1]


class Guarded:
    """A device tensor between two 256-byte guard bands of a known byte pattern; the
    tensor starts 256 bytes into its allocation, so its alignment is kept."""
    CANARY = 0xA5
    GUARD = 256

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((n + 2 * self.GUARD,), self.CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[self.GUARD:self.GUARD + n].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    @classmethod
    def of(cls, src):
        g = cls(tuple(src.shape), src.dtype)
        g.t.copy_(src)
        return g

    def intact(self):
        raw = self.raw.cpu().numpy()
        return bool(np.all(raw[:self.GUARD] == self.CANARY) and np.all(raw[-self.GUARD:] == self.CANARY))


class Setup:
    """A GPU cache and (for the sampled sequences) oracle caches over the same inputs."""

    def __init__(self, H, G, s, w, lens, seed=0, spare_pages=7, kv_device="cpu",
                 chunks=None, max_work_items=0, kv8=False, rope=None, nvfp4=False, mxfp4=False):
        self.H, self.G, self.s, self.w, self.kv8, self.nvfp4 = H, G, s, w, kv8, nvfp4
        self.mxfp4 = mxfp4
        self.rope = rope                     # float32 numpy table [max_pos][128] or None
        self.lens = [int(L) for L in lens]
        self.B = len(lens)
        self.seed = seed
        need = sum((L + P - 1) // P for L in self.lens)
        self.num_pages = need + spare_pages
        self.bt = inputs.block_tables(self.lens, P, self.num_pages, seed)
        self.cache = KV4Cache(H, self.num_pages, max_slots=self.B + 1, max_batch=self.B,
                              max_q_heads=H * G, sink=s, window=w, max_work_items=max_work_items,
                              fmt=(FORMAT_MXFP4 if mxfp4 else FORMAT_NVFP4 if nvfp4 else
                                   (FORMAT_INT8 if kv8 else FORMAT_INT4_HYBRID)))
        self.kv = []
        for b, L in enumerate(self.lens):
            k, v = inputs.sequence_kv(b, L, H, seed, device=kv_device)
            self.kv.append((k, v))
        self.bt_dev = torch.from_numpy(self.bt).cuda()
        if rope is not None:
            self.cache.set_rope(torch.from_numpy(rope).cuda())
        self._append(chunks)

    def _append(self, chunks):
        """chunks: list of position cut points applied to every sequence; default one call."""
        cuts = sorted(set([0] + list(chunks or []) + [max(self.lens)]))
        for lo, hi in zip(cuts[:-1], cuts[1:]):
            ks, vs, cu, slots, starts, rows = [], [], [0], [], [], []
            for b, L in enumerate(self.lens):
                a, z = min(lo, L), min(hi, L)
                if z <= a:
                    continue
                ks.append(self.kv[b][0][a:z])
                vs.append(self.kv[b][1][a:z])
                cu.append(cu[-1] + z - a)
                slots.append(b)
                starts.append(a)
                rows.append(b)
            if not slots:
                continue
            k = torch.cat(ks).cuda().contiguous()
            v = torch.cat(vs).cuda().contiguous()
            self.cache.append(k, v, torch.tensor(cu, dtype=torch.int32).cuda(),
                              torch.tensor(slots, dtype=torch.int32).cuda(),
                              torch.tensor(starts, dtype=torch.int32).cuda(),
                              self.bt_dev[rows].contiguous())

    def oracle_for(self, b):
        oc = oracle.OracleCache(self.H, self.s, self.w, self.lens[b], num_slots=1, kv8=self.kv8,
                                rope=self.rope, nvfp4=self.nvfp4, mxfp4=self.mxfp4)
        k, v = self.kv[b]
        oc.append(0, 0, inputs.bf16_bits(k), inputs.bf16_bits(v))
        return oc

    def decode(self, q, debug_stride=0, lens=None):
        """One decode call: through the debug entry point when debug_stride > 0 (also
        returning its records), else through plain kv4_decode_attention, the kernels
        bench.py times. Every input and output sits between guard bands of a known byte
        pattern that must come back intact, and the outputs start as NaN, so a stray
        write or a missed one fails the test."""
        lens = self.lens if lens is None else lens
        B, Hq = q.shape[0], q.shape[1]
        bufs = {
            "q": Guarded.of(q), "slots": Guarded.of(torch.arange(B, dtype=torch.int32, device="cuda")),
            "lens": Guarded.of(torch.tensor(lens, dtype=torch.int32, device="cuda")),
            "block_table": Guarded.of(self.bt_dev),
            "out": Guarded((B, Hq, D), torch.float32, float("nan")),
            "lse": Guarded((B, Hq), torch.float32, float("nan")),
        }
        args = (bufs["q"].t, bufs["slots"].t, bufs["lens"].t, bufs["block_table"].t,
                bufs["out"].t, bufs["lse"].t)
        dbg = None
        if debug_stride:
            from int8_hybrid_paged_gb300.kv4 import kv4_decode_attention_debug
            bufs.update(q8=Guarded((B, Hq, D), torch.int8, 0), q_scale=Guarded((B, Hq), torch.float32, 0),
                        qk=Guarded((B, Hq, debug_stride), torch.int32, -(2 ** 31)),
                        w_hat=Guarded((B, Hq, debug_stride), torch.uint8, 0),
                        p_bits=Guarded((B, Hq, debug_stride), torch.int16, 0))
            kv4_decode_attention_debug(self.cache.handle, *args[:4], args[4], args[5],
                                       bufs["q8"].t, bufs["q_scale"].t, bufs["qk"].t, bufs["w_hat"].t,
                                       bufs["p_bits"].t, sm_scale=1 / math.sqrt(D))
        else:
            self.cache.decode(*args[:4], args[4], args[5], sm_scale=1 / math.sqrt(D))
        torch.cuda.synchronize()
        for name, g in bufs.items():
            assert g.intact(), f"decode wrote outside its {name} buffer"
        if debug_stride:
            dbg = {k: bufs[k].t.cpu().numpy() for k in ("q8", "q_scale", "qk", "w_hat")}
            dbg["p_bits"] = bufs["p_bits"].t.cpu().numpy().view(np.uint16)
        return bufs["out"].t, bufs["lse"].t, dbg

    def close(self):
        self.cache.close()


ATOL, RTOL = 2e-3, 1e-2


def protected_positions(L, s, w, whole_cache):
    """Positions whose PV weight the protected arithmetic forms: every position in the
    whole-cache formats, else [0, min(s, L)) ∪ [max(s, L − w), L)."""
    if whole_cache:
        return np.arange(L)
    return np.array([t for t in range(L) if t < s or t >= max(s, L - w)], dtype=np.int64)


def check_decode(st, q, bs, lens=None):
    """Decode the whole batch through the debug entry point and through plain
    kv4_decode_attention (the kernels bench.py times) and compare sequences bs with the
    oracle: q8 and s_q, the QK record (integer dots, or the FP32 score bits of NVFP4),
    the u8 INT4 weights and every protected weight bit for bit; outputs and
    log-normalizers of both calls within 2e-3 abs / 1e-2 rel. Returns the worst output
    difference."""
    lens = st.lens if lens is None else lens
    whole = st.kv8 or st.nvfp4 or st.mxfp4
    out, lse, dbg = st.decode(q, debug_stride=max(max(lens), 1), lens=lens)
    pout, plse, _ = st.decode(q, lens=lens)
    outs = [(out.cpu().numpy(), lse.cpu().numpy()), (pout.cpu().numpy(), plse.cpu().numpy())]
    qb = inputs.bf16_bits(q)
    worst = 0.0
    for b in bs:
        L = lens[b]
        o_ref, lse_ref, d = st.oracle_for(b).decode(0, L, st.G, qb[b], 1 / math.sqrt(D), debug=True)
        np.testing.assert_array_equal(dbg["q8"][b], d["q8"])
        np.testing.assert_array_equal(dbg["q_scale"][b].view(np.uint32), d["q_scale"].view(np.uint32))
        if L:
            if st.nvfp4 or st.mxfp4:     # no single integer dot: the record holds the score's bits
                np.testing.assert_array_equal(dbg["qk"][b][:, :L], d["sigma"][:, :L].view(np.int32))
            else:
                np.testing.assert_array_equal(dbg["qk"][b][:, :L], d["qk"][:, :L])
            r4 = np.setdiff1d(np.arange(L), protected_positions(L, st.s, st.w, whole))
            np.testing.assert_array_equal(dbg["w_hat"][b][:, r4], d["w_hat"][:, r4])
            prot = protected_positions(L, st.s, st.w, whole)
            np.testing.assert_array_equal(dbg["p_bits"][b][:, prot], d["p_bits"][:, prot])
        for o, l in outs:
            np.testing.assert_allclose(o[b], o_ref, atol=ATOL, rtol=RTOL)
            if L:
                np.testing.assert_allclose(l[b], lse_ref, atol=ATOL, rtol=RTOL)
                worst = max(worst, float(np.max(np.abs(o[b] - o_ref))))
            else:
                assert np.all(o[b] == 0) and np.all(np.isneginf(l[b]))
    return worst
