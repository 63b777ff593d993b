"""ctypes wrapper over ``liboracle_kv4.so`` (see ``kv4_oracle.c``).

TEST INFRASTRUCTURE ONLY. Arrays are numpy; bf16 and fp16 values travel as
their uint16 bit patterns. The logical cache state lives in numpy arrays owned
by :class:`OracleCache`.
"""
import ctypes as C

import numpy as np

from . import build as _build

D = 128
RN, RD, RU = 0, 1, 2
PV_INTEGER, PV_FLOAT = 0, 1

_lib = None


def load():
    """Build (if stale) and load the oracle library."""
    global _lib
    if _lib is None:
        path = _build.build()
        lib = C.CDLL(path)
        P = C.c_void_p
        lib.orc_f16_to_f64.argtypes = [C.c_uint16]
        lib.orc_f16_to_f64.restype = C.c_double
        lib.orc_f32_to_f16.argtypes = [C.c_float, C.c_int]
        lib.orc_f32_to_f16.restype = C.c_uint16
        lib.orc_exp2f.argtypes = [C.c_float]
        lib.orc_exp2f.restype = C.c_float
        lib.orc_fwht128.argtypes = [P, P]
        lib.orc_rope128.argtypes = [P, P, P]
        lib.orc_e4m3_rn.argtypes = [C.c_float]
        lib.orc_e4m3_rn.restype = C.c_uint8
        lib.orc_e4m3_value.argtypes = [C.c_uint8]
        lib.orc_e4m3_value.restype = C.c_float
        lib.orc_e2m1_rn.argtypes = [C.c_float]
        lib.orc_e2m1_rn.restype = C.c_uint8
        lib.orc_e2m1_value.argtypes = [C.c_uint8]
        lib.orc_e2m1_value.restype = C.c_float
        lib.orc_quant_nvfp4.argtypes = [P, P, P, P]
        lib.orc_quant_mxfp4.argtypes = [P, P, P]
        lib.orc_quant_affine.argtypes = [P, C.c_int, C.c_int, P, P, P]
        lib.orc_quant_query.argtypes = [P, P, P, P]
        lib.orc_append.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
        lib.orc_append.restype = C.c_int
        lib.orc_decode.argtypes = [P, C.c_int, C.c_int, C.c_int, P, C.c_float, C.c_int, P, P, P]
        lib.orc_decode.restype = C.c_int
        lib.orc_decode_batch.argtypes = [P, C.c_int, P, P, C.c_int, P, C.c_float, C.c_int, P, P,
                                         C.c_int]
        lib.orc_decode_batch.restype = C.c_int
        lib.orc_num_threads.restype = C.c_int
        lib.orc_f32_to_f16_array.argtypes = [P, P, C.c_int64, C.c_int]
        lib.orc_f32_to_bf16_array.argtypes = [P, P, C.c_int64]
        lib.orc_exp2f_array.argtypes = [P, P, C.c_int64]
        _lib = lib
    return _lib


def _p(a):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- formats

def f16_bits_to_f64(bits):
    """fp16 bit patterns -> float64 values, by the oracle's own decoder."""
    lib = load()
    bits = np.asarray(bits, dtype=np.uint16)
    flat = [lib.orc_f16_to_f64(int(b)) for b in bits.ravel()]
    return np.array(flat, dtype=np.float64).reshape(bits.shape)


def f32_to_f16(x, mode=RN):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    load().orc_f32_to_f16_array(_p(x), _p(out), x.size, mode)
    return out


def f32_to_bf16_rn(x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    load().orc_f32_to_bf16_array(_p(x), _p(out), x.size)
    return out


def bf16_to_f32(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def exp2f(x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.float32)
    load().orc_exp2f_array(_p(x), _p(out), x.size)
    return out


# --------------------------------------------------------------------------- steps

def fwht128(x):
    x = _c(x, np.float32)
    assert x.shape == (D,)
    out = np.empty(D, np.float32)
    load().orc_fwht128(_p(x), _p(out))
    return out


def rope128(x, cos_sin_row):
    """RoPE of one 128-dim vector with one table row (cos at [i], sin at [64+i])."""
    x = _c(x, np.float32)
    row = _c(cos_sin_row, np.float32)
    assert x.shape == (D,) and row.shape == (D,)
    out = np.empty(D, np.float32)
    load().orc_rope128(_p(x), _p(row), _p(out))
    return out


def e4m3_rn(t):
    """E4M3 bits of t >= 0 (nearest, ties even, held at 448)."""
    return int(load().orc_e4m3_rn(C.c_float(t)))


def e4m3_value(bits):
    return float(load().orc_e4m3_value(C.c_uint8(bits)))


def e2m1_rn(v):
    """E2M1 code (sign in bit 3) of v (nearest, ties to the even code, held at 6)."""
    return int(load().orc_e2m1_rn(C.c_float(v)))


def e2m1_value(code):
    return float(load().orc_e2m1_value(C.c_uint8(code)))


def quant_nvfp4(x):
    """(codes uint8[128], block scales uint8[8] E4M3 bits, vector scale float32)."""
    x = _c(x, np.float32)
    assert x.shape == (D,)
    codes = np.empty(D, np.uint8)
    bs = np.empty(8, np.uint8)
    g = np.zeros(1, np.float32)
    load().orc_quant_nvfp4(_p(x), _p(codes), _p(bs), _p(g))
    return codes, bs, np.float32(g[0])


def quant_mxfp4(x):
    """(codes uint8[128], E8M0 scale bytes uint8[4] = shared exponent + 127), reading R13."""
    x = _c(x, np.float32)
    assert x.shape == (D,)
    codes = np.empty(D, np.uint8)
    es = np.empty(4, np.uint8)
    load().orc_quant_mxfp4(_p(x), _p(codes), _p(es))
    return codes, es


def quant_affine(x, levels):
    """Returns (codes uint8[n], delta fp16 bits, min fp16 bits)."""
    x = _c(x, np.float32)
    code = np.empty(x.size, np.uint8)
    dh = np.zeros(1, np.uint16)
    mh = np.zeros(1, np.uint16)
    load().orc_quant_affine(_p(x), x.size, levels, _p(code), _p(dh), _p(mh))
    return code, int(dh[0]), int(mh[0])


def quant_query(q_rot):
    """Returns (q8 int8[128], s_q float32, Σq8 int)."""
    q_rot = _c(q_rot, np.float32)
    q8 = np.empty(D, np.int8)
    sq = np.zeros(1, np.float32)
    qs = np.zeros(1, np.int32)
    load().orc_quant_query(_p(q_rot), _p(q8), _p(sq), _p(qs))
    return q8, np.float32(sq[0]), int(qs[0])


def num_threads():
    return int(load().orc_num_threads())


# --------------------------------------------------------------------------- cache

_STATE_ARRAYS = ("k4_code", "v4_code", "k4_delta", "k4_min", "v4_delta", "v4_min",
                 "k8_code", "v8_code", "k8_delta", "k8_min", "v8_delta", "v8_min", "length")


class _State(C.Structure):
    _fields_ = [("num_heads", C.c_int32), ("sink", C.c_int32), ("window", C.c_int32),
                ("max_len", C.c_int32), ("num_slots", C.c_int32), ("format", C.c_int32)] + \
               [(n, C.c_void_p) for n in _STATE_ARRAYS] + \
               [("rope", C.c_void_p), ("rope_max_pos", C.c_int32)] + \
               [(n, C.c_void_p) for n in ("k_bscale", "v_bscale", "k_gscale", "v_gscale")]


class _Debug(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("q8", "q_scale", "q_sum", "qk", "sigma", "w_hat", "p_bits")]


class OracleCache:
    """Logical KV4 cache state: INT4 main cache for every position plus the
    bounded INT8 side buffer (s sink + w recent positions) per slot. With
    kv8=True, the whole-cache 8-bit configuration (reading R10): 8-bit codes for
    every position, no side buffer (sink = window = 0). With nvfp4=True or mxfp4=True,
    the whole-cache 4-bit floating-point configurations of readings R12 and R13."""

    def __init__(self, num_heads, sink, window, max_len, num_slots=1, kv8=False, rope=None,
                 nvfp4=False, mxfp4=False):
        if (kv8 or nvfp4 or mxfp4) and (sink or window):
            raise ValueError("the KV8, NVFP4 and MXFP4 configurations have no protected region")
        if int(bool(kv8)) + int(bool(nvfp4)) + int(bool(mxfp4)) > 1:
            raise ValueError("one cache format at a time")
        H, S = num_heads, sink + window
        self.kv8 = bool(kv8)
        self.nvfp4 = bool(nvfp4)
        self.mxfp4 = bool(mxfp4)
        self.format = 3 if mxfp4 else (2 if nvfp4 else (1 if kv8 else 0))
        self.H, self.s, self.w, self.max_len, self.num_slots = H, sink, window, max_len, num_slots
        z = np.zeros
        self.k4_code = z((num_slots, max_len, H, D), np.uint8)
        self.v4_code = z((num_slots, max_len, H, D), np.uint8)
        self.k4_delta = z((num_slots, max_len, H), np.uint16)
        self.k4_min = z((num_slots, max_len, H), np.uint16)
        self.v4_delta = z((num_slots, max_len, H), np.uint16)
        self.v4_min = z((num_slots, max_len, H), np.uint16)
        self.k8_code = z((num_slots, S, H, D), np.uint8)
        self.v8_code = z((num_slots, S, H, D), np.uint8)
        self.k8_delta = z((num_slots, S, H), np.uint16)
        self.k8_min = z((num_slots, S, H), np.uint16)
        self.v8_delta = z((num_slots, S, H), np.uint16)
        self.v8_min = z((num_slots, S, H), np.uint16)
        self.length = z((num_slots,), np.int32)
        # reading R12 (NVFP4): E4M3 block scales and the FP32 vector scale per token-head;
        # reading R13 (MXFP4): E8M0 scales of the four 32-value blocks in bytes 0..3
        self.k_bscale = z((num_slots, max_len, H, 8), np.uint8)
        self.v_bscale = z((num_slots, max_len, H, 8), np.uint8)
        self.k_gscale = z((num_slots, max_len, H), np.float32)
        self.v_gscale = z((num_slots, max_len, H), np.float32)
        st = _State(H, sink, window, max_len, num_slots, self.format)
        for n in ("k_bscale", "v_bscale", "k_gscale", "v_gscale"):
            setattr(st, n, getattr(self, n).ctypes.data)
        for n in _STATE_ARRAYS:
            setattr(st, n, getattr(self, n).ctypes.data)
        # reading R11: with a RoPE table [max_pos][128] (cos at [p][i], sin at [p][64+i]),
        # appended keys and decode queries are pre-RoPE
        self.rope = None if rope is None else _c(rope, np.float32)
        if self.rope is not None:
            assert self.rope.ndim == 2 and self.rope.shape[1] == D
            st.rope = self.rope.ctypes.data
            st.rope_max_pos = self.rope.shape[0]
        self._st = st

    def append(self, slot, start, k_bits, v_bits):
        """k_bits, v_bits: uint16 bf16 patterns [T][H][128]."""
        k = _c(k_bits, np.uint16)
        v = _c(v_bits, np.uint16)
        T = k.shape[0]
        assert k.shape == (T, self.H, D) and v.shape == k.shape
        rc = load().orc_append(C.byref(self._st), slot, start, T, _p(k), _p(v))
        if rc != 0:
            raise ValueError("oracle append rejected its arguments")

    def decode(self, slot, L, G, q_bits, sm_scale, pv_mode=PV_INTEGER, debug=False):
        """q_bits: uint16 bf16 patterns [H*G][128].
        Returns (out f64 [HG][128], lse f64 [HG], debug dict or None)."""
        q = _c(q_bits, np.uint16)
        HG = self.H * G
        assert q.shape == (HG, D)
        out = np.empty((HG, D), np.float64)
        lse = np.empty(HG, np.float64)
        dbg = None
        dptr = None
        if debug:
            n = max(L, 1)
            dbg = dict(q8=np.zeros((HG, D), np.int8), q_scale=np.zeros(HG, np.float32),
                       q_sum=np.zeros(HG, np.int32), qk=np.zeros((HG, n), np.int32),
                       sigma=np.full((HG, n), np.nan, np.float32),
                       w_hat=np.zeros((HG, n), np.uint8), p_bits=np.zeros((HG, n), np.uint16))
            dptr = _Debug(*[dbg[k].ctypes.data for k in ("q8", "q_scale", "q_sum", "qk",
                                                         "sigma", "w_hat", "p_bits")])
        rc = load().orc_decode(C.byref(self._st), slot, L, G, _p(q), C.c_float(sm_scale),
                               pv_mode, _p(out), _p(lse),
                               C.byref(dptr) if dptr is not None else None)
        if rc != 0:
            raise ValueError("oracle decode rejected its arguments")
        return out, lse, dbg

    def decode_batch(self, slots, lens, G, q_bits, sm_scale, pv_mode=PV_INTEGER, threads=0):
        """q_bits: [B][H*G][128]. Sequences spread over host threads (OpenMP)."""
        slots = _c(slots, np.int32)
        lens = _c(lens, np.int32)
        q = _c(q_bits, np.uint16)
        B, HG = len(slots), self.H * G
        out = np.empty((B, HG, D), np.float64)
        lse = np.empty((B, HG), np.float64)
        rc = load().orc_decode_batch(C.byref(self._st), B, _p(slots), _p(lens), G, _p(q),
                                     C.c_float(sm_scale), pv_mode, _p(out), _p(lse), threads)
        if rc != 0:
            raise ValueError("oracle decode_batch rejected its arguments")
        return out, lse

    def side_bytes(self):
        """Bytes held by the INT8 side buffer (codes + FP16 metadata), all slots."""
        return sum(getattr(self, n).nbytes for n in ("k8_code", "v8_code", "k8_delta", "k8_min",
                                                     "v8_delta", "v8_min"))
