"""Python binding of libkv4 (include/kv4.h): argument marshalling only.

Every function here has the name of the C entry point it calls. Tensors are
torch CUDA tensors; their device pointers and the current torch stream are
passed through unchanged. The compute happens in libkv4's kernels; there is no
fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkv4.so")

KV4_OK = 0
STATUS = {0: "KV4_OK", -1: "KV4_ERR_INVALID_ARG", -2: "KV4_ERR_UNSUPPORTED",
          -3: "KV4_ERR_OUT_OF_MEMORY", -4: "KV4_ERR_CUDA", -5: "KV4_ERR_OUT_OF_RANGE",
          -6: "KV4_ERR_DEVICE_FAULT"}
DEVICE_ERRORS = {0: "none", 1: "bad slot", 2: "bad page", 3: "bad position",
                 4: "context length mismatch", 5: "staging wait timeout", 6: "bad token layout"}
PAGE_BLOCK_BYTES = 2176
HEAD_DIM = 128
PAGE_SIZE = 16

EXPORTED = ("kv4_cache_create", "kv4_cache_free", "kv4_cache_get_info", "kv4_append",
            "kv4_decode_attention", "kv4_decode_attention_debug", "kv4_get_device_error",
            "kv4_status_string", "kv4_profile_start", "kv4_profile_stop",
            "kv4_decode_attention_noalloc", "kv4_cache_set_rope", "kv4_linear_bf16",
            "kv4_qkv_append")


class KV4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_status_text(status)})")


class kv4_cache_config(C.Structure):
    _fields_ = [("num_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("page_size", C.c_int32),
                ("sink", C.c_int32), ("window", C.c_int32), ("num_pages", C.c_int64),
                ("max_slots", C.c_int32), ("max_batch", C.c_int32), ("max_q_heads", C.c_int32),
                ("max_work_items", C.c_int32), ("format", C.c_int32)]


FORMAT_INT4_HYBRID = 0     # INT4 pages + bounded INT8 side buffer (the method)
FORMAT_INT8 = 1            # whole-cache 8-bit codes in pages, no side buffer (KV8)
FORMAT_NVFP4 = 2           # whole-cache NVFP4 (E2M1, E4M3 block scales, FP32 vector scales)
FORMAT_MXFP4 = 3           # whole-cache MXFP4 (E2M1, E8M0 scale per 32 values)


class kv4_cache_info(C.Structure):
    _fields_ = [("page_pool_dev", C.c_void_p), ("page_pool_bytes", C.c_size_t),
                ("side_pool_dev", C.c_void_p), ("side_pool_bytes", C.c_size_t),
                ("side_block_bytes", C.c_size_t), ("seq_len_dev", C.c_void_p),
                ("num_sms", C.c_int32), ("decode_grid", C.c_int32), ("device", C.c_int32)]


class kv4_profile(C.Structure):
    _fields_ = [("calls", C.c_int32), ("plan_ms", C.c_float), ("split_ms", C.c_float),
                ("merge_ms", C.c_float)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libkv4. Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libkv4 is not built ({path} missing); run "
                           "`python -m int8_hybrid_paged_gb300.build` first")
    lib = C.CDLL(path)
    P, I, F = C.c_void_p, C.c_int, C.c_float
    lib.kv4_status_string.argtypes = [I]
    lib.kv4_status_string.restype = C.c_char_p
    lib.kv4_cache_create.argtypes = [C.POINTER(kv4_cache_config), C.POINTER(P)]
    lib.kv4_cache_free.argtypes = [P]
    lib.kv4_cache_get_info.argtypes = [P, C.POINTER(kv4_cache_info)]
    lib.kv4_append.argtypes = [P, P, P, P, P, P, P, I, I, I, P]
    lib.kv4_decode_attention.argtypes = [P, P, I, P, P, P, I, I, F, P, P, P]
    lib.kv4_decode_attention_debug.argtypes = [P, P, I, P, P, P, I, I, F, P, P, P, P, P, P, P, I, P]
    lib.kv4_get_device_error.argtypes = [P, C.POINTER(C.c_int32), I]
    lib.kv4_profile_start.argtypes = [P, I]
    lib.kv4_decode_attention_noalloc.argtypes = [C.POINTER(kv4_cache_config), P, P, P, P, I, P,
                                                 P, P, I, I, F, P, P, P]
    lib.kv4_profile_stop.argtypes = [P, C.POINTER(kv4_profile)]
    lib.kv4_cache_set_rope.argtypes = [P, P, I]
    lib.kv4_linear_bf16.argtypes = [P, P, P, I, I, I, P, P]
    lib.kv4_qkv_append.argtypes = [P, P, P, I, I, P, P, P, P, P, I, I, I, P]
    for name in EXPORTED:
        getattr(lib, name).restype = C.c_int if name != "kv4_status_string" else C.c_char_p
    _lib = lib
    return lib


def _status_text(status: int) -> str:
    try:
        return load().kv4_status_string(status).decode()
    except Exception:  # noqa: BLE001 - only for message text
        return "?"


def _check(status: int, where: str):
    if status != KV4_OK:
        raise KV4Error(status, where)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


# --------------------------------------------------------------------------- entry points

def kv4_status_string(status: int) -> str:
    return load().kv4_status_string(status).decode()


def kv4_cache_create(num_kv_heads, num_pages, max_slots, max_batch, max_q_heads, sink=16,
                     window=128, head_dim=HEAD_DIM, page_size=PAGE_SIZE, max_work_items=0,
                     fmt=FORMAT_INT4_HYBRID):
    cfg = kv4_cache_config(num_kv_heads, head_dim, page_size, sink, window, num_pages, max_slots,
                           max_batch, max_q_heads, max_work_items, fmt)
    h = C.c_void_p()
    _check(load().kv4_cache_create(C.byref(cfg), C.byref(h)), "kv4_cache_create")
    return h


def kv4_cache_set_rope(handle, cos_sin=None):
    """RoPE table for the cache's appends and decodes: a float32 CUDA tensor
    [max_pos][128] (cos of pair i at [p][i], sin at [p][64+i]), or None to clear.
    The tensor must outlive the setting."""
    if cos_sin is None:
        _check(load().kv4_cache_set_rope(handle, None, 0), "kv4_cache_set_rope")
        return
    assert cos_sin.dim() == 2 and cos_sin.shape[1] == HEAD_DIM
    _check(load().kv4_cache_set_rope(handle, _ptr(cos_sin, torch.float32, "cos_sin"),
                                     int(cos_sin.shape[0])), "kv4_cache_set_rope")


def kv4_linear_bf16(x, w, y=None, err=None, stream=None):
    """y = x @ w.T on the tcgen05 tensor cores: x [M][K], w [N][K] bf16 CUDA tensors
    (N % 128 == 0, K % 64 == 0); returns y [M][N] bf16. err: optional int32 device word."""
    M, K = x.shape
    N = w.shape[0]
    assert w.shape[1] == K
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(load().kv4_linear_bf16(_ptr(x, torch.bfloat16, "x"), _ptr(w, torch.bfloat16, "w"),
                                  _ptr(y, torch.bfloat16, "y"), M, N, K,
                                  _ptr(err, torch.int32, "err"), _stream(stream)),
           "kv4_linear_bf16")
    return y


def kv4_qkv_append(handle, x, w_qkv, num_q_heads, cu_tokens, slot_ids, start_pos, block_table,
                   q_out=None, stream=None):
    """Projection + fused append: x [T][d_model], w_qkv [(Hq + 2 H_kv) * 128][d_model] (rows:
    Q heads, then K0, V0, K1, V1, ...) bf16 CUDA tensors; appends K/V to the cache and
    returns q_out [T][Hq][128] bf16."""
    T, d_model = x.shape
    if q_out is None:
        q_out = torch.empty((T, num_q_heads, HEAD_DIM), dtype=torch.bfloat16, device=x.device)
    _check(load().kv4_qkv_append(
        handle, _ptr(x, torch.bfloat16, "x"), _ptr(w_qkv, torch.bfloat16, "w_qkv"), num_q_heads, d_model,
        _ptr(q_out, torch.bfloat16, "q_out"), _ptr(cu_tokens, torch.int32, "cu_tokens"),
        _ptr(slot_ids, torch.int32, "slot_ids"), _ptr(start_pos, torch.int32, "start_pos"),
        _ptr(block_table, torch.int32, "block_table"), block_table.shape[-1], slot_ids.shape[0], T,
        _stream(stream)), "kv4_qkv_append")
    return q_out


def kv4_cache_free(handle):
    _check(load().kv4_cache_free(handle), "kv4_cache_free")


def kv4_cache_get_info(handle) -> kv4_cache_info:
    info = kv4_cache_info()
    _check(load().kv4_cache_get_info(handle, C.byref(info)), "kv4_cache_get_info")
    return info


def kv4_append(handle, k, v, cu_tokens, slot_ids, start_pos, block_table, stream=None):
    """k, v: bf16 [T][H_kv][128]; cu_tokens int32 [n+1]; slot_ids, start_pos int32 [n];
    block_table int32 [n][stride]."""
    n = slot_ids.numel()
    _check(load().kv4_append(handle, _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"),
                             _ptr(cu_tokens, torch.int32, "cu_tokens"),
                             _ptr(slot_ids, torch.int32, "slot_ids"),
                             _ptr(start_pos, torch.int32, "start_pos"),
                             _ptr(block_table, torch.int32, "block_table"),
                             block_table.shape[-1], n, k.shape[0], _stream(stream)), "kv4_append")


def kv4_decode_attention(handle, q, slot_ids, context_lens, block_table, out, lse=None,
                         sm_scale=None, stream=None):
    """q: bf16 [B][H_q][128]; out: fp32 [B][H_q][128]; lse: fp32 [B][H_q] or None."""
    B, Hq = q.shape[0], q.shape[1]
    scale = float(HEAD_DIM ** -0.5 if sm_scale is None else sm_scale)
    _check(load().kv4_decode_attention(handle, _ptr(q, torch.bfloat16, "q"), Hq,
                                       _ptr(slot_ids, torch.int32, "slot_ids"),
                                       _ptr(context_lens, torch.int32, "context_lens"),
                                       _ptr(block_table, torch.int32, "block_table"),
                                       block_table.shape[-1], B, scale,
                                       _ptr(out, torch.float32, "out"),
                                       _ptr(lse, torch.float32, "lse"), _stream(stream)),
           "kv4_decode_attention")


def kv4_decode_attention_debug(handle, q, slot_ids, context_lens, block_table, out, lse=None,
                               q8=None, q_scale=None, qk=None, w_hat=None, p_bits=None,
                               sm_scale=None, stream=None):
    B, Hq = q.shape[0], q.shape[1]
    scale = float(HEAD_DIM ** -0.5 if sm_scale is None else sm_scale)
    dstride = next((t.shape[-1] for t in (qk, w_hat, p_bits) if t is not None), 0)
    _check(load().kv4_decode_attention_debug(
        handle, _ptr(q, torch.bfloat16, "q"), Hq, _ptr(slot_ids, torch.int32, "slot_ids"),
        _ptr(context_lens, torch.int32, "context_lens"),
        _ptr(block_table, torch.int32, "block_table"), block_table.shape[-1], B, scale,
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(q8, torch.int8, "q8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(qk, torch.int32, "qk"), _ptr(w_hat, torch.uint8, "w_hat"),
        _ptr(p_bits, torch.int16, "p_bits"), dstride,
        _stream(stream)), "kv4_decode_attention_debug")


def kv4_get_device_error(handle, clear=True) -> int:
    code = C.c_int32(0)
    _check(load().kv4_get_device_error(handle, C.byref(code), 1 if clear else 0),
           "kv4_get_device_error")
    return int(code.value)


def kv4_decode_attention_noalloc(config, page_pool_dev, side_pool_dev, seq_len_dev, q, slot_ids,
                                 context_lens, block_table, out, lse=None, sm_scale=None,
                                 stream=None):
    """Decode attention that allocates nothing (scratch in libkv4's static device array).
    config: kv4_cache_config; the pool arguments are device addresses (ints)."""
    B, Hq = q.shape[0], q.shape[1]
    scale = float(HEAD_DIM ** -0.5 if sm_scale is None else sm_scale)
    _check(load().kv4_decode_attention_noalloc(
        C.byref(config), C.c_void_p(page_pool_dev), C.c_void_p(side_pool_dev),
        C.c_void_p(seq_len_dev), _ptr(q, torch.bfloat16, "q"), Hq,
        _ptr(slot_ids, torch.int32, "slot_ids"), _ptr(context_lens, torch.int32, "context_lens"),
        _ptr(block_table, torch.int32, "block_table"), block_table.shape[-1], B, scale,
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"), _stream(stream)),
        "kv4_decode_attention_noalloc")


def kv4_noalloc_device_error(clear=True) -> int:
    """Error word of kv4_decode_attention_noalloc on the current device (kv4_device_error
    code, 0 = none); waits for the device."""
    code = C.c_int32(0)
    _check(load().kv4_get_device_error(None, C.byref(code), 1 if clear else 0),
           "kv4_get_device_error")
    return int(code.value)


def kv4_profile_start(handle, max_calls):
    _check(load().kv4_profile_start(handle, int(max_calls)), "kv4_profile_start")


def kv4_profile_stop(handle) -> dict:
    prof = kv4_profile()
    _check(load().kv4_profile_stop(handle, C.byref(prof)), "kv4_profile_stop")
    return dict(calls=prof.calls, plan_ms=prof.plan_ms, split_ms=prof.split_ms,
                merge_ms=prof.merge_ms)


# --------------------------------------------------------------------------- convenience

class KV4Cache:
    """Owning wrapper: creates the cache on construction, frees it on close()."""

    def __init__(self, num_kv_heads, num_pages, max_slots, max_batch, max_q_heads, sink=16,
                 window=128, max_work_items=0, fmt=FORMAT_INT4_HYBRID):
        self.num_kv_heads, self.sink, self.window = num_kv_heads, sink, window
        self.num_pages, self.max_slots, self.fmt = num_pages, max_slots, fmt
        self.handle = kv4_cache_create(num_kv_heads, num_pages, max_slots, max_batch, max_q_heads,
                                       sink, window, max_work_items=max_work_items, fmt=fmt)

    def close(self):
        if self.handle is not None:
            kv4_cache_free(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass

    def info(self):
        return kv4_cache_get_info(self.handle)

    def qkv_append(self, x, w_qkv, num_q_heads, cu_tokens, slot_ids, start_pos, block_table,
                   q_out=None, stream=None):
        return kv4_qkv_append(self.handle, x, w_qkv, num_q_heads, cu_tokens, slot_ids, start_pos,
                              block_table, q_out, stream)

    def set_rope(self, cos_sin=None):
        """Fuse RoPE into appends and decodes (pre-RoPE K and q from now on); None clears."""
        self._rope = cos_sin                 # keep the table alive while it is set
        kv4_cache_set_rope(self.handle, cos_sin)

    def append(self, k, v, cu_tokens, slot_ids, start_pos, block_table, stream=None):
        kv4_append(self.handle, k, v, cu_tokens, slot_ids, start_pos, block_table, stream)

    def decode(self, q, slot_ids, context_lens, block_table, out=None, lse=None, sm_scale=None,
               stream=None):
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        kv4_decode_attention(self.handle, q, slot_ids, context_lens, block_table, out, lse,
                             sm_scale, stream)
        return out

    def device_error(self, clear=True):
        return kv4_get_device_error(self.handle, clear)

    def raw_pools(self):
        """Host copies of the page pool (uint8), the side pool (uint8) and the slot
        lengths (int32), read through views of the cache's device memory."""
        info = self.info()
        dev = torch.device("cuda", info.device)

        def view(ptr, nbytes, typestr, itemsize):
            class _Mem:
                __cuda_array_interface__ = {"shape": (nbytes // itemsize,), "typestr": typestr,
                                            "data": (ptr, False), "version": 3}
            return torch.as_tensor(_Mem(), device=dev)

        torch.cuda.synchronize(dev)
        pages = view(info.page_pool_dev, info.page_pool_bytes, "|u1", 1).cpu().numpy()
        side = view(info.side_pool_dev, info.side_pool_bytes, "|u1", 1).cpu().numpy()
        lens = view(info.seq_len_dev, 4 * self.max_slots, "<i4", 4).cpu().numpy()
        return pages, side, int(info.side_block_bytes), lens
