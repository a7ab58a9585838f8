"""bench.py host logic: byte accounting and the roofline bookkeeping."""
import json
import os

import bench
from int4_weight_only_w4_gb300 import synthetic as syn


def test_canonical_bytes_formula():
    # packed nibbles + fp16 scales + uint8 zeros + bf16 x + bf16 y
    assert bench.canonical_bytes(1, 3584, 37888) == 37888 * 1792 + 3 * 37888 * 28 + 7168 + 75776
    assert bench.canonical_bytes(8, 3584, 152064) == (152064 * 3584 // 2 + 3 * 152064 * 28
                                                      + 2 * 8 * 3584 + 2 * 8 * 152064)


def test_chain_bytes_matches_layer_shapes():
    per_layer = sum(bench.canonical_bytes(1, K, N) for _, K, N in syn.LAYER_7B)
    assert bench.chain_bytes() == 28 * per_layer
    assert abs(bench.chain_bytes() / 1e9 - 3.420) < 0.001


def test_small_chain_shapes_and_bytes():
    # 0.5B shape: hidden 896, intermediate 4864, 14 query + 2 key/value heads of 64
    assert syn.LAYER_05B == [("qkv", 896, (14 + 2 * 2) * 64), ("o", 896, 896),
                             ("gate_up", 896, 2 * 4864), ("down", 4864, 896)]
    per_layer = sum(bench.canonical_bytes(1, K, N) for _, K, N in syn.LAYER_05B)
    assert syn.LAYERS_05B * per_layer == 188270592     # the bytes per step it reports


def test_traffic_record_is_consistent():
    with open(os.path.join(bench.ROOT, "profiles", "gemv_traffic.json")) as f:
        rec = json.load(f)
    assert rec["traffic_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert rec["algorithmic_bytes_per_launch"] == bench.canonical_bytes(1, 3584, 37888)
    t = bench.gemv_traffic()
    assert t is None or t == rec["traffic_bytes_per_launch"]


def test_peaks_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_peaks() == (6800.0, "fallback")
