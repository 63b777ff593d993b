"""Seeded synthetic inputs for the KV4 decode hot path.

This module holds no arithmetic of the method: it draws random numbers and
shapes workloads. The CUDA path and the CPU oracle both receive what it makes.

Stand-in for the pages' workload: decode-forward replay of Qwen3-4B/8B-Base
rollout traces (DAPO-Math-17k prompts, 16,384-token response cap). Neither the
traces nor the weights are available, so K, V and q are bf16 draws from N(0, 1)
with four fixed K channels scaled ×20 as outliers (before rotation), and
context lengths are a prompt of 256 tokens plus a lognormal response length.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

HEAD_DIM = 128
PAGE_SIZE = 16
OUTLIER_CHANNELS = (5, 37, 70, 101)
OUTLIER_SCALE = 20.0
PROMPT_LEN = 256
RESPONSE_CAP = 16384


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload (single layer unless ``layers`` > 1)."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    context_lens: tuple
    layers: int = 1
    sink: int = 16
    window: int = 128
    page_size: int = PAGE_SIZE
    seed: int = 0

    @property
    def batch(self) -> int:
        return len(self.context_lens)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def lognormal_context_lengths(batch: int, mean_response: float, sigma_log: float,
                              seed: int) -> list:
    """Prompt 256 + lognormal response (arithmetic mean ``mean_response``) capped at 16,384."""
    rng = np.random.default_rng(seed)
    mu = math.log(mean_response) - sigma_log * sigma_log / 2.0
    x = rng.lognormal(mean=mu, sigma=sigma_log, size=batch)
    resp = np.clip(np.rint(x), 1, RESPONSE_CAP).astype(np.int64)
    return [int(PROMPT_LEN + r) for r in resp]


def long_tail_context_lengths(batch: int, seed: int, frac_long: float = 0.10,
                              long_len: int = 16384, lo: int = 512, hi: int = 4096) -> list:
    """A fixed share of sequences at ``long_len``, the rest uniform on [lo, hi]."""
    rng = np.random.default_rng(seed)
    n_long = int(round(frac_long * batch))
    rest = rng.integers(lo, hi + 1, size=batch - n_long)
    lens = [long_len] * n_long + [int(v) for v in rest]
    perm = rng.permutation(batch)
    return [lens[i] for i in perm]


def workload(name: str, seed: int = 0) -> Workload:
    """The named workloads: tiny, qwen3-4b, qwen3-8b, long-tail."""
    if name == "tiny":
        return Workload("tiny: B=2 L={300,1000} Hq=8 Hkv=2", 8, 2, (300, 1000), seed=seed)
    if name == "qwen3-4b":
        lens = lognormal_context_lengths(64, 1450.0, 0.9, seed)
        return Workload("Qwen3-4B-shaped layer: B=64 Hq=32 Hkv=8 D=128 P=16, "
                        "L=256+lognormal(mean 1.45k, sigma 0.9)", 32, 8, tuple(lens), seed=seed)
    if name == "qwen3-8b":
        lens = lognormal_context_lengths(256, 4000.0, 1.0, seed)
        return Workload("Qwen3-8B-shaped layer: B=256 Hq=32 Hkv=8 D=128 P=16, "
                        "L=256+lognormal(mean 4k, sigma 1.0)", 32, 8, tuple(lens), seed=seed)
    if name == "long-tail":
        lens = long_tail_context_lengths(128, seed)
        return Workload("long tail: 36 layers B=128 Hq=32 Hkv=8, 10% at 16384, rest U[512,4096]",
                        32, 8, tuple(lens), layers=36, seed=seed)
    raise KeyError(name)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def kv_tokens(num_tokens: int, num_kv_heads: int, seed: int, device="cpu"):
    """bf16 K, V of shape [T][H_kv][128] ~ N(0,1); K channels 5, 37, 70, 101 scaled ×20."""
    g = _gen(seed, device)
    k = torch.randn((num_tokens, num_kv_heads, HEAD_DIM), generator=g, device=device,
                    dtype=torch.float32)
    v = torch.randn((num_tokens, num_kv_heads, HEAD_DIM), generator=g, device=device,
                    dtype=torch.float32)
    k[:, :, list(OUTLIER_CHANNELS)] *= OUTLIER_SCALE
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def sequence_kv(seq_index: int, length: int, num_kv_heads: int, seed: int, device="cpu"):
    """K, V for one sequence, drawn from its own stream (seed, seq_index), so any
    sequence can be regenerated alone."""
    return kv_tokens(length, num_kv_heads, seed * 1_000_003 + 7919 * (seq_index + 1), device)


def queries(batch: int, num_q_heads: int, seed: int, device="cpu"):
    """bf16 q of shape [B][H_q][128] ~ N(0,1)."""
    g = _gen(seed * 1_000_003 + 104729, device)
    q = torch.randn((batch, num_q_heads, HEAD_DIM), generator=g, device=device,
                    dtype=torch.float32)
    return q.to(torch.bfloat16)


def rope_table(max_pos: int, base: float = 1_000_000.0) -> np.ndarray:
    """The model's RoPE constants as a float32 table [max_pos][128]: for position p and
    pair i < 64 (dims i and i + 64), cos(p·base^(−i/64)) at [p][i] and its sin at
    [p][64 + i], evaluated in float64 and rounded once. base = 1e6 is Qwen3's."""
    p = np.arange(max_pos, dtype=np.float64)[:, None]
    inv_freq = base ** (-np.arange(HEAD_DIM // 2, dtype=np.float64) / (HEAD_DIM // 2))
    ang = p * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def block_tables(context_lens, page_size: int, num_pages: int, seed: int,
                 stride: int | None = None) -> np.ndarray:
    """int32 [B][stride] block tables: a seeded random choice of distinct physical
    pages (scattered over the pool), -1 past each sequence's last page."""
    need = [(int(L) + page_size - 1) // page_size for L in context_lens]
    total = sum(need)
    if total > num_pages:
        raise ValueError(f"pool of {num_pages} pages cannot hold {total}")
    if stride is None:
        stride = max(need) if need else 1
    rng = np.random.default_rng(seed + 1)
    pages = rng.permutation(num_pages)[:total].astype(np.int32)
    bt = np.full((len(need), max(stride, 1)), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = pages[o:o + n]
        o += n
    return bt


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
