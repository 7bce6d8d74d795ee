"""The benchmark's algorithmic work per step (CPU only): the FLOPs and bytes that every
roofline fraction in its JSON line divides by.

GEMM FLOPs are 2·M·N·K per projection; attention is 4·d FLOPs per visible (query, key)
pair per query head (q·k and p·v); the visible pairs of a causal block of T queries are
T(T + 1)/2, and with a window W the queries past the first W see W keys each. The
windowed and cached counts are also checked against the visible set of the oracle's
attention on small shapes, so that "visible" means what the oracle masks.
"""
import dataclasses

import numpy as np
import pytest

import bench
import oracle
from llama_family_decoder_gb300.synth import WORKLOADS


def _gemm_flops(B, T, D, H, Hkv, d, F, gated):
    M = B * T
    return {"qkv": 2.0 * M * D * (H + 2 * Hkv) * d, "o": 2.0 * M * (H * d) * D,
            "up": 2.0 * M * D * (2 * F if gated else F), "down": 2.0 * M * F * D}


@pytest.mark.parametrize("name, gated", [("llama7b_bf16_B1_T2048", True), ("arcee_gqa_bf16_B4_T2048", False),
                                         ("apertus_qknorm_bf16_B2_T4096", False)])
def test_prefill_flops_closed_form(name, gated):
    wl = WORKLOADS[name]
    g, weight_bytes, kv_bytes = bench.work_counts(wl)
    B, T, D, H, Hkv, d, F = (wl.batch, wl.seq, wl.hidden_size, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                             wl.intermediate_size)
    want = _gemm_flops(B, T, D, H, Hkv, d, F, gated)
    for k, v in want.items():
        assert g[k] == v, k
    assert g["attn"] == 4.0 * B * H * d * (T * (T + 1) // 2)
    assert kv_bytes == 0.0
    # weights in bf16: the four projections and the two norm gains
    assert weight_bytes == 2 * (D * (H + 2 * Hkv) * d + H * d * D + (2 * F if gated else F) * D + F * D + 2 * D)


def test_headline_and_decode_totals():
    # 3161.2 GFLOP for the Apertus-shape block; 1.4275 GB per decode step (the weights,
    # the K/V cache with the new token's key, x in and out)
    g, _, _ = bench.work_counts(WORKLOADS["apertus_qknorm_bf16_B2_T4096"])
    assert sum(g.values()) / 1e9 == pytest.approx(3161.16, abs=0.01)
    wl = WORKLOADS["llama7b_decode_bf16_B64_L4096"]
    g, weight_bytes, kv_bytes = bench.work_counts(wl)
    L = wl.cache_len + 1
    assert kv_bytes == 2.0 * wl.batch * wl.num_kv_heads * L * wl.head_dim * 2
    assert g["attn"] == 4.0 * wl.batch * wl.num_heads * wl.head_dim * L
    step_bytes = weight_bytes + kv_bytes + 2.0 * wl.batch * wl.hidden_size * 2
    assert step_bytes / 1e9 == pytest.approx(1.4275, abs=2e-4)


def _oracle_visible_pairs(q_pos, k_pos, window):
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, len(q_pos), 4))
    k = rng.standard_normal((1, len(k_pos), 4))
    _, scores, _ = oracle.causal_gqa_attention(q, k, k, np.asarray(q_pos), np.asarray(k_pos), return_pattern=True,
                                               window=window)
    return int(np.isfinite(scores).sum())


@pytest.mark.parametrize("T, W", [(16, 0), (16, 5), (16, 16), (9, 12)])
def test_windowed_prefill_pairs_match_the_oracle_mask(T, W):
    wl = WORKLOADS["afmoe_nano_sliding_bf16_B8_T4096_W2048"]
    small = dataclasses.replace(wl, batch=1, seq=T, num_heads=1, num_kv_heads=1, head_dim=1, sliding_window=W)
    g, _, _ = bench.work_counts(small)
    pairs = _oracle_visible_pairs(np.arange(T), np.arange(T), W)
    assert g["attn"] == 4.0 * pairs
    if W and T >= W:  # closed form: W(W + 1)/2 for the first W queries, W for each after
        assert pairs == W * (W + 1) // 2 + (T - W) * W


@pytest.mark.parametrize("cache_len, T, W", [(7, 5, 0), (7, 1, 0), (12, 4, 6), (3, 1, 8)])
def test_cached_pairs_and_bytes_match_the_oracle_mask(cache_len, T, W):
    wl = WORKLOADS["llama7b_chunk_bf16_B4_T512_L1536"]
    small = dataclasses.replace(wl, batch=1, seq=T, cache_len=cache_len, num_heads=1, num_kv_heads=1, head_dim=1,
                                sliding_window=W)
    g, _, kv_bytes = bench.work_counts(small)
    q_pos = np.arange(cache_len, cache_len + T)
    k_pos = np.arange(cache_len + T)
    pairs = _oracle_visible_pairs(q_pos, k_pos, W)
    assert g["attn"] == 4.0 * pairs
    # K and V bytes: every cached or new key that some query of the step can see
    _, scores, _ = oracle.causal_gqa_attention(np.zeros((1, T, 1)), np.zeros((1, cache_len + T, 1)),
                                               np.zeros((1, cache_len + T, 1)), q_pos, k_pos, return_pattern=True,
                                               window=W)
    keys_read = int(np.isfinite(scores[0]).any(axis=0).sum())
    assert kv_bytes == 2.0 * keys_read * 2
