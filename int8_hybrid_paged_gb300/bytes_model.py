"""Byte accounting for the KV4 cache and the algorithmic bytes of one call.

Pages cited (title, then section):
  [zh] "KV4-RL:用 INT4 KV 缓存量化为 RLVR 异步 Rollout 提速" — 方法步骤详情 step 2
       (per-128-dim group, INT4 codes, FP16 Δ and m: 4.25 bits per element).
  [kvq] "KV 캐시 양자화 — 가중치보다 이쪽이 먼저 넘친다" — 얼마나 자라는지 먼저 세어 본다
       (KV bytes = 2 · layers · H_kv · d_h · bytes/element · batch · seq).
"""
from __future__ import annotations

HEAD_DIM = 128
INT4_CODE_BYTES = HEAD_DIM // 2          # 64 B of packed codes per token-head per tensor
INT8_CODE_BYTES = HEAD_DIM               # 128 B per side position-head per tensor
META_BYTES = 4                           # FP16 Δ + FP16 m
INT4_TOKEN_HEAD_BYTES = 2 * (INT4_CODE_BYTES + META_BYTES)   # K + V: 136 B
SIDE_POSITION_HEAD_BYTES = 2 * (INT8_CODE_BYTES + META_BYTES)  # K + V: 264 B
BF16_TOKEN_HEAD_BYTES = 2 * HEAD_DIM * 2                     # K + V: 512 B
# NVFP4: E2M1 codes (64 B), one E4M3 scale per 16 dims (8 B) and an FP32 vector scale
NVFP4_POSITION_HEAD_BYTES = 2 * (HEAD_DIM // 2 + HEAD_DIM // 16 + 4)   # K + V: 152 B
# MXFP4: E2M1 codes (64 B) and one E8M0 scale per 32 dims (4 B)
MXFP4_POSITION_HEAD_BYTES = 2 * (HEAD_DIM // 2 + HEAD_DIM // 32)        # K + V: 136 B


def kv_cache_bytes(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: float,
                   batch: int, seq: int) -> float:
    """Dense KV cache size ([kvq] formula): 2 · L · H_kv · d_h · p · B · S."""
    return 2 * layers * kv_heads * head_dim * bytes_per_elem * batch * seq


def affine_bits_per_element(group: int = HEAD_DIM, code_bits: int = 4, meta_bits: int = 16,
                            meta_values: int = 2) -> float:
    """Storage per element of a group-affine code: (g·b + (Δ, m) bits) / g ([zh] step 2)."""
    return (group * code_bits + meta_values * meta_bits) / group


def regions(L: int, sink: int, window: int):
    """(INT4-region length, protected length) for a context of L positions:
    INT4 = [s, L−w), protected = [0, min(s, L)) ∪ [max(s, L−w), L)."""
    n4 = max(0, L - window - sink)
    return n4, L - n4


def decode_call_bytes(context_lens, num_q_heads: int, num_kv_heads: int, sink: int,
                      window: int, page_size: int = 16, with_lse: bool = False) -> int:
    """Algorithmic HBM bytes of one decode-attention call: INT4 codes + metadata of
    the INT4 region, INT8 side entries + metadata of the protected region, bf16
    queries, fp32 outputs, context lengths and slot ids, and the block-table
    entries of the pages read."""
    total = 0
    for L in context_lens:
        L = int(L)
        n4, npr = regions(L, sink, window)
        total += num_kv_heads * (n4 * INT4_TOKEN_HEAD_BYTES + npr * SIDE_POSITION_HEAD_BYTES)
        if n4 > 0:
            first = sink // page_size
            last = (L - window - 1) // page_size
            total += 4 * (last - first + 1)
        total += 8
    B = len(context_lens)
    total += B * num_q_heads * HEAD_DIM * (2 + 4)
    if with_lse:
        total += B * num_q_heads * 4
    return total


def decode_call_bytes_kv8(context_lens, num_q_heads: int, num_kv_heads: int,
                          page_size: int = 16, with_lse: bool = False) -> int:
    """Algorithmic HBM bytes of one decode-attention call on the whole-cache 8-bit
    format: 8-bit codes + metadata of every position (264 B per position-head), bf16
    queries, fp32 outputs, context lengths and slot ids, and the block-table entries
    of the pages read."""
    total = 0
    for L in context_lens:
        L = int(L)
        total += num_kv_heads * L * SIDE_POSITION_HEAD_BYTES + 4 * ((L + page_size - 1) // page_size) + 8
    B = len(context_lens)
    total += B * num_q_heads * HEAD_DIM * (2 + 4)
    if with_lse:
        total += B * num_q_heads * 4
    return total


def decode_call_bytes_nvfp4(context_lens, num_q_heads: int, num_kv_heads: int,
                            page_size: int = 16, with_lse: bool = False,
                            per_position: int = NVFP4_POSITION_HEAD_BYTES) -> int:
    """Algorithmic HBM bytes of one decode-attention call on the NVFP4 format (or, with
    per_position = MXFP4_POSITION_HEAD_BYTES, MXFP4): codes and scales of every position
    (152 B, or 136 B, per position-head), bf16 queries, fp32 outputs, context lengths and
    slot ids, and the block-table entries of the pages read."""
    total = 0
    for L in context_lens:
        L = int(L)
        total += num_kv_heads * L * per_position + 4 * ((L + page_size - 1) // page_size) + 8
    B = len(context_lens)
    total += B * num_q_heads * HEAD_DIM * (2 + 4)
    if with_lse:
        total += B * num_q_heads * 4
    return total


def append_call_bytes(num_tokens: int, num_kv_heads: int, side_writes: int) -> int:
    """Algorithmic bytes of one append: bf16 K and V read, INT4 codes and metadata
    written, and ``side_writes`` INT8 side position-heads written."""
    read = num_tokens * num_kv_heads * BF16_TOKEN_HEAD_BYTES
    written = num_tokens * num_kv_heads * INT4_TOKEN_HEAD_BYTES
    written += side_writes * SIDE_POSITION_HEAD_BYTES
    return read + written
