"""The benchmark's algorithmic byte model against the byte and budget
arithmetic the pages print (Fathom opening paragraphs; OasisKV core method and
method details)."""
import json
import os

import numpy as np

from top_sparse_decode_gb300 import roofline as rl

GOLD = os.path.join(os.path.dirname(__file__), "golden", "byte_model.json")


def test_136_bit_scan_and_dense_bytes():
    g = json.load(open(GOLD))
    L, H = g["layers"], g["kv_heads"]
    per_tok = rl.fixed_scan_bytes_per_token(32)  # 32 channels x 4 bits + scales
    assert per_tok * 8 == g["scan_bits"]
    assert round(per_tok * 32768 * L * H / 1e6) == g["scan_32k_MB"]
    assert round(per_tok * (1 << 20) * L * H / 1e9, 1) == g["scan_1M_GB"]
    assert round(rl.dense_kv_bytes(32768, H, layers=L) / 1e9, 1) == g["dense_32k_GB"]


def test_fixed_plan_bytes_match_per_token_rate():
    plan = np.zeros((1, 8, 128), np.uint8)
    plan[..., :32] = 4
    n = 1 << 20
    assert rl.plane_scan_bytes(plan, n) == 8 * n * rl.fixed_scan_bytes_per_token(32)
    assert rl.plane_scan_bits_per_token(plan) == 128


def test_summary_fraction_and_block_budget():
    g = json.load(open(GOLD))
    n = 16 * 1024
    frac = rl.quest_scan_bytes(1, 1, n) / rl.dense_kv_bytes(n, 1)
    assert frac == g["summary_fraction"]
    assert g["blocks"] * g["block_tokens"] == g["tokens_per_head"]
    assert rl.gather_bytes([g["tokens_per_head"]]) == g["tokens_per_head"] * 512


def test_sparq_bit_counts_match_the_results_table():
    """SparQ r channels at full depth cost r x (4 plane bits + a quarter bit of fp16
    scale per 64 tokens): 68 bits at r = 16 and 136 at r = 32, as the table prints."""
    g = json.load(open(GOLD))
    assert rl.fixed_scan_bytes_per_token(16) * 8 == g["sparq_r16_bits"]
    assert rl.fixed_scan_bytes_per_token(32) * 8 == g["sparq_r32_bits"]


def test_landmark_and_resident_bytes():
    # 8-token landmarks: 32 B (256 bits) per token per KV head
    assert rl.landmark_scan_bytes(1, 8, 1 << 20) == 8 * (1 << 20) * 32
    assert rl.landmark_scan_bytes(1, 1, 9) == 2 * 256  # a short last block is a full row
    # an admitted 16-token block moves 16 K rows and 16 V rows of 256 B
    assert rl.resident_transfer_bytes(3584) == 3584 * 16 * 512
