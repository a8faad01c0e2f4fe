"""Pins of the block-pool policy and of the step byte model (numbers the pages print)."""
import json
import os

import pytest

import oracle
import synth
from graph_replayed_decode_gb300 import roofline

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))


def test_pool_fifo_policy_hand_worked():
    p = oracle.BlockPool(8)
    assert p.alloc(3) == [0, 1, 2]
    assert p.alloc(2) == [3, 4]
    p.free([1, 3])
    assert p.alloc(3) == [5, 6, 7]
    assert p.alloc(2) == [1, 3]                 # freed blocks come back in the order they were freed
    assert p.free_count == 0 and p.scratch == 8
    with pytest.raises(oracle.PoolExhausted):
        p.alloc(1)
    with pytest.raises(ValueError):
        p.free([99])


def test_blocks_needed_reserve_on_admit():
    assert oracle.blocks_needed(16) == 1 and oracle.blocks_needed(17) == 2 and oracle.blocks_needed(0) == 0
    assert oracle.blocks_needed(512 + 256) == 48


def test_byte_model_reproduces_the_decode_ceiling():
    g = GOLDEN["decode_ceiling_qwen3_0p6b"]
    s = synth.shape("qwen3_0p6b")
    gb = roofline.weight_bytes(s) / 1e9
    assert abs(gb - g["weight_gb_per_token"]) < 0.005
    tok_s = roofline.decode_ceiling_tokens_per_s(s, g["bandwidth_gb_s"] * 1e9)
    assert abs(tok_s - g["tokens_per_s_about"]) / g["tokens_per_s_about"] < 0.02


def test_byte_model_reproduces_the_weight_read_time():
    g = GOLDEN["weight_read_qwen2p5_1p5b"]
    s = synth.shape("qwen2p5_1p5b")
    ms = roofline.weight_bytes(s) / (g["assumed_bandwidth_gb_s"] * 1e9) * 1e3
    assert abs(ms - g["weight_read_ms"]) < 0.01


def test_step_bytes_counts_kv_read_and_write():
    s = synth.shape("qwen3_0p6b")
    base = roofline.step_bytes(s, 1, [0])
    assert roofline.step_bytes(s, 1, [512]) - base == 512 * 114_688
    assert roofline.kv_bytes_per_token(s) == 114_688
    assert roofline.kv_bytes_per_token(synth.shape("dense_8b")) == 147_456
