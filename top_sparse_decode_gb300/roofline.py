"""Algorithmic byte and operation counts of the hot path (host logic only).

Bytes are what the method must move, not what a kernel happens to move:
  * Hamming scan: 4 B per token per KV head (one 32-bit signature;
    HashAttention: Semantic Sparsity for Faster Inference, 2.5).
  * Bit-plane scan: t_j * n / 8 B for each channel with t_j planned planes, plus
    that channel's fp16 scales (2 B per 64 tokens) (Fathom, bit planes).  A
    fixed 32-channel, 4-bit scan is 17 B per token per KV head -- the "136-bit"
    class the Fathom page prices at 160 MB per step at 32k over 36 layers and
    8 KV heads.
  * Quest scan: 512 B per 16-token block per KV head (min and max rows of
    128 bf16), 1/16 of the K+V bytes (OasisKV, core method).
  * Gather-attend: 512 B (one K and one V bf16 row of 128) per selected token
    per KV head (HashAttention 2.5: 256-byte rows read by index).
The score buffer (4 B per unit written by the scan, read by top-k) is
implementation traffic and is reported apart.
"""
from __future__ import annotations

import numpy as np

ROW_BYTES = 2 * 128          # one bf16 row of d = 128
KV_ROW_BYTES = 2 * ROW_BYTES  # K and V


def hamming_scan_bytes(B: int, Hkv: int, n: int) -> int:
    return 4 * B * Hkv * n


def plane_scan_bytes(plan: np.ndarray, n: int) -> int:
    """plan: uint8 [B][Hkv][d] bits per channel."""
    t = plan.astype(np.int64)
    active = (t > 0).sum()
    return int(t.sum() * (n // 8) + active * (n // 64) * 2)


def plane_scan_bits_per_token(plan: np.ndarray) -> float:
    """Average planned bits per token per KV head (the budget B)."""
    return float(plan.astype(np.int64).sum(axis=-1).mean())


def fixed_scan_bytes_per_token(channels: int, bits: int = 4) -> float:
    """Bytes per token per KV head of a fixed-channel full-depth scan."""
    return channels * bits / 8 + channels * 2 / 64


def quest_scan_bytes(B: int, Hkv: int, n: int) -> int:
    return B * Hkv * ((n + 15) // 16) * 2 * ROW_BYTES


def landmark_scan_bytes(B: int, Hkv: int, n: int, block: int = 8) -> int:
    """One bf16 landmark row (256 B) per `block` tokens per KV head."""
    return B * Hkv * ((n + block - 1) // block) * ROW_BYTES


def resident_transfer_bytes(admitted_units: int, block: int = 16) -> int:
    """K and V rows of the units admitted into a resident set (512 B per token)."""
    return int(admitted_units) * block * KV_ROW_BYTES


def gather_bytes(counts: np.ndarray) -> int:
    return int(np.asarray(counts, np.int64).clip(min=0).sum() * KV_ROW_BYTES)


def dense_kv_bytes(n: int, Hkv: int, layers: int = 1, B: int = 1) -> int:
    return B * layers * Hkv * n * KV_ROW_BYTES


def score_buffer_bytes(B: int, Hkv: int, n_units: int) -> int:
    """Write by the scan plus read by top-k (implementation traffic)."""
    return 2 * 4 * B * Hkv * n_units


def plane_scan_alu_ops(plan: np.ndarray, n: int) -> int:
    """Planned token-planes: each costs one bit test and one predicated FP32 add
    per token per KV head (the in-HBM bit-plane scan is bound by these, as the
    Fathom page notes); counted once, against the FP32 pipe's one add per lane
    per clock."""
    return int(plan.astype(np.int64).sum() * n)
