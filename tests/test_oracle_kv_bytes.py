"""Pins of the oracle's per-token KV byte accounting against the figures the
pages print (tests/golden/kv_bytes_pins.json): 64 KiB per token for the bf16
cache of 16 full-attention layers x 4 KV heads x 256 dims, and 16.5 KiB per
token per device (a 16.50 GiB pool at 1,048,576 tokens) for the INT8 group-64
cache of the two-device engine, scale planes included."""
import json
import os

from oracle import paged as PG

HERE = os.path.dirname(os.path.abspath(__file__))
with open(os.path.join(HERE, "golden", "kv_bytes_pins.json")) as f:
    PINS = {p["name"]: p for p in json.load(f)["pins"]}


def _per_token(dtype, heads, layers, head_dim=256):
    # a page-head record holds 16 tokens' K and V (and their scales)
    return PG.page_head_bytes(dtype, head_dim) // PG.PAGE * heads * layers


def test_bf16_per_token():
    p = PINS["bf16_kv_per_token_16_layers"]
    got = _per_token(PG.BF16, p["kv_heads"], p["layers"], p["head_dim"])
    assert got == p["value_kib"] * 1024
    # the page's size formula: layers * tokens * batch * 2 * kv_heads * head_dim * bytes
    assert got == p["layers"] * 1 * 1 * 2 * p["kv_heads"] * p["head_dim"] * p["bytes_per_elem"]


def test_int8_group64_per_token_per_device():
    p = PINS["int8_group64_kv_per_token_per_device_tp2"]
    got = _per_token(PG.INT8, p["kv_heads_per_device"], p["layers"], p["head_dim"])
    assert got == p["value_kib"] * 1024                     # 16,896 B
    assert got * 1048576 == p["pool_gib_at_1048576_tokens"] * 2 ** 30


def test_nvfp4_and_fp8_per_token():
    # the same accounting for this library's own formats (one layer, 4 KV heads)
    assert _per_token(PG.NVFP4, 4, 1) == 4 * 2 * (128 + 16)    # 1,152 B
    assert _per_token(PG.FP8, 4, 1) == 4 * 2 * 256             # 2,048 B
