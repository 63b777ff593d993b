"""The byte model used for the roofline, pinned to the numbers the pages print."""
import json
import os

from int8_hybrid_paged_gb300 import bytes_model as bm

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")))


def test_dense_kv_bytes_match_the_printed_example():
    e = G["kv_bytes_per_token_fp16"]
    assert bm.kv_cache_bytes(e["layers"], e["kv_heads"], e["head_dim"], e["bytes_per_elem"],
                             1, 1) == e["value"]
    r = G["kv_bytes_per_request_32k_fp16"]
    assert bm.kv_cache_bytes(32, 8, 128, 2, 1, r["seq"]) == r["value"]
    m = G["kv_bytes_16_requests_32k_fp16"]
    assert bm.kv_cache_bytes(32, 8, 128, 2, m["batch"], m["seq"]) == m["value"]


def test_int4_token_head_bytes_follow_the_bit_budget():
    bits = G["bits_per_element"]["value"]
    # K and V, 128 elements each, at 4.25 bits
    assert bm.INT4_TOKEN_HEAD_BYTES == 2 * 128 * bits / 8 == 136
    assert bm.BF16_TOKEN_HEAD_BYTES == bm.kv_cache_bytes(1, 1, 128, 2, 1, 1) == 512
    # INT8 side entry: 8-bit codes + the same FP16 pair
    assert bm.SIDE_POSITION_HEAD_BYTES == 2 * (128 + 4) == 264


def test_regions_and_decode_bytes():
    s, w = G["sink_positions"]["value"], G["recent_positions"]["value"]
    assert s + w == G["protected_budget"]["value"]
    assert bm.regions(100, s, w) == (0, 100)
    assert bm.regions(144, s, w) == (0, 144)
    assert bm.regions(1000, s, w) == (856, 144)
    # one sequence of 1000 positions, one KV head, one q head
    n4, npr = 856, 144
    pages = (1000 - 128 - 1) // 16 - 16 // 16 + 1
    expect = n4 * 136 + npr * 264 + 4 * pages + 8 + 128 * 6
    assert bm.decode_call_bytes([1000], 1, 1, s, w) == expect


def test_kv8_decode_bytes():
    """Every position at 264 B per head (8-bit codes of K and V plus two FP16 pairs):
    a length-1000 context over 8 heads reads 2,112,000 KV bytes, 63 block-table
    entries, and the query/output bytes of 32 q heads."""
    got = bm.decode_call_bytes_kv8([1000], 32, 8)
    assert got == 8 * 1000 * 264 + 4 * 63 + 8 + 32 * 128 * 6
    assert bm.decode_call_bytes_kv8([0], 4, 1) == 8 + 4 * 128 * 6
    # KV8 reads 264 / 136 of the INT4 bytes per token-head
    assert bm.SIDE_POSITION_HEAD_BYTES / bm.INT4_TOKEN_HEAD_BYTES == 264 / 136


def test_nvfp4_decode_bytes():
    """NVFP4 holds 4.75 bits per element (4-bit codes, an 8-bit scale per 16 values, a
    32-bit scale per 128): 152 B per position-head for K and V, the page block size of
    include/kv4.h over 16 positions."""
    assert bm.NVFP4_POSITION_HEAD_BYTES == 152
    assert bm.NVFP4_POSITION_HEAD_BYTES * 8 / (2 * 128) == 4.75
    assert 16 * bm.NVFP4_POSITION_HEAD_BYTES == 2432
    got = bm.decode_call_bytes_nvfp4([1000], 32, 8)
    assert got == 8 * 1000 * 152 + 4 * 63 + 8 + 32 * 128 * 6


def test_mxfp4_decode_bytes():
    """MXFP4 holds 4.25 bits per element (4-bit codes and an 8-bit scale per 32 values), the
    storage of the method's INT4 codes with their fp16 (delta, min) per 128: 136 B per
    position-head, and a 2176-byte page block of 16 positions."""
    assert bm.MXFP4_POSITION_HEAD_BYTES == bm.INT4_TOKEN_HEAD_BYTES == 136
    assert 16 * bm.MXFP4_POSITION_HEAD_BYTES == 2176
    got = bm.decode_call_bytes_nvfp4([1000], 32, 8, per_position=bm.MXFP4_POSITION_HEAD_BYTES)
    assert got == 8 * 1000 * 136 + 4 * 63 + 8 + 32 * 128 * 6
