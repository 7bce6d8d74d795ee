"""Seeded synthetic inputs for the decoder block (weights, residual stream, KV cache).

This module holds the workload shapes and the seeded random draws only: no step
of the block's arithmetic lives here. Both the CUDA path's tests/benchmark and
the fp64 oracle take their inputs from it.

Recipe: a CPU ``torch.Generator`` seeded per workload; every tensor is drawn in
fp32 in a fixed order and then cast to the workload's storage dtype (bf16 or
fp32). Projection weights ~ N(0, 0.02), residual input ~ N(0, 1), RMSNorm gains
1 (optionally 1 + N(0, gain_std)), KV cache ~ N(0, 1). The oracle reads the same
(bf16-rounded) values upcast exactly to float64.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    """One block shape plus the batch it runs on.

    Field names follow the pages' config keys (hidden_size, num_heads,
    num_kv_heads, head_dim, intermediate_size, hidden_act, rms_norm_eps,
    rope_theta) plus the batch geometry.
    """

    name: str
    dtype: str  # "f32" or "bf16"
    batch: int
    seq: int  # tokens per sequence in this call (1 for a decode step)
    hidden_size: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    intermediate_size: int
    hidden_act: str  # "silu" | "relu2" | "xielu"
    qk_norm: bool = False
    cache_len: int = 0  # positions already in the KV cache (seq == 1: a decode step; seq > 1: a prefill chunk)
    rms_norm_eps: float = 1e-5
    rope_theta: float = 10000.0
    rope_scaling: tuple | None = None  # (kind, factor, original positions, low, high) of a stretched rotary
    xielu_alpha_p: float = 0.8
    xielu_alpha_n: float = 0.8
    seed: int = 0
    n_layers: int = 0  # > 0: the model around the block (embeddings, n_layers blocks, norm, lm_head)
    vocab: int = 0
    # the "afmoe" block options
    sliding_window: int = 0  # > 0: attention over the last sliding_window positions
    use_rope: bool = True
    attn_gate: bool = False
    sandwich_norm: bool = False

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_f32_T64_D256", "f32", 1, 64, 256, 4, 2, 64, 1024, "relu2", seed=0),
        Workload("llama7b_bf16_B1_T2048", "bf16", 1, 2048, 4096, 32, 32, 128, 10928, "silu", seed=1),
        Workload("arcee_gqa_bf16_B4_T2048", "bf16", 4, 2048, 4096, 32, 8, 128, 14336, "relu2", seed=2),
        Workload("apertus_qknorm_bf16_B2_T4096", "bf16", 2, 4096, 4096, 32, 8, 128, 16384, "xielu",
                 qk_norm=True, seed=3),
        Workload("llama7b_decode_bf16_B64_L4096", "bf16", 64, 1, 4096, 32, 8, 128, 10928, "silu",
                 cache_len=4096, seed=4),
        Workload("llama7b_chunk_bf16_B4_T512_L1536", "bf16", 4, 512, 4096, 32, 8, 128, 10928, "silu",
                 cache_len=1536, seed=5),
        Workload("llama7b_model_bf16_B1_T2048_L32", "bf16", 1, 2048, 4096, 32, 32, 128, 10928, "silu", seed=6,
                 n_layers=32, vocab=32000),
        # Trinity Nano's dense block ("afmoe" Config: hidden 1024, 8 heads over 2 KV heads,
        # head_dim 128, intermediate 3072, silu, window 2048), a sliding-window block with its
        # rotary and a whole-prefix block without, both with q/k norms, head gate and sandwich norms
        Workload("afmoe_nano_sliding_bf16_B8_T4096_W2048", "bf16", 8, 4096, 1024, 8, 2, 128, 3072, "silu",
                 qk_norm=True, seed=7, sliding_window=2048, attn_gate=True, sandwich_norm=True),
        Workload("afmoe_nano_global_bf16_B8_T4096", "bf16", 8, 4096, 1024, 8, 2, 128, 3072, "silu",
                 qk_norm=True, seed=8, use_rope=False, attn_gate=True, sandwich_norm=True),
        Workload("afmoe_nano_decode_bf16_B64_L8192_W2048", "bf16", 64, 1, 1024, 8, 2, 128, 3072, "silu",
                 qk_norm=True, cache_len=8192, seed=9, sliding_window=2048, attn_gate=True, sandwich_norm=True),
    ]
}


def torch_dtype(w: Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def _normal(gen, shape, std, dtype):
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * std).to(dtype)


def make_weights(w: Workload, seed: int | None = None, gain_std: float = 0.0,
                 weight_std: float = 0.02) -> dict:
    """Block weights as CPU tensors in the workload's dtype, [out, in] layout."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    dt = torch_dtype(w)
    D, H, Hkv, d, F = w.hidden_size, w.num_heads, w.num_kv_heads, w.head_dim, w.intermediate_size

    def gain(n):
        if gain_std == 0.0:
            return torch.ones(n, dtype=dt)
        return (1.0 + torch.randn(n, generator=gen) * gain_std).to(dt)

    out = {
        "input_layernorm": gain(D),
        "q_proj": _normal(gen, (H * d, D), weight_std, dt),
        "k_proj": _normal(gen, (Hkv * d, D), weight_std, dt),
        "v_proj": _normal(gen, (Hkv * d, D), weight_std, dt),
        "o_proj": _normal(gen, (D, H * d), weight_std, dt),
        "post_attention_layernorm": gain(D),
        "up_proj": _normal(gen, (F, D), weight_std, dt),
        "down_proj": _normal(gen, (D, F), weight_std, dt),
    }
    if w.hidden_act == "silu":
        out["gate_proj"] = _normal(gen, (F, D), weight_std, dt)
    if w.qk_norm:
        out["q_norm"] = gain(d)
        out["k_norm"] = gain(d)
    if w.attn_gate:
        out["attn_gate_proj"] = _normal(gen, (H * d, D), weight_std, dt)
    if w.sandwich_norm:
        out["post_attn_norm"] = gain(D)
        out["post_mlp_norm"] = gain(D)
    return out


def make_input(w: Workload, seed: int | None = None, std: float = 1.0) -> torch.Tensor:
    """Residual stream entering the block: [batch, seq, hidden] ~ N(0, std)."""
    gen = torch.Generator().manual_seed((w.seed if seed is None else seed) + 1000)
    return _normal(gen, (w.batch, w.seq, w.hidden_size), std, torch_dtype(w))


def make_kv_cache(w: Workload, capacity: int | None = None, seed: int | None = None):
    """Decode KV cache [batch, num_kv_heads, capacity, head_dim] ~ N(0, 1).

    The first cache_len slots hold values; the rest are zero. Returns (k, v).
    """
    cap = capacity if capacity is not None else w.cache_len + w.seq  # room for this call's new tokens
    gen = torch.Generator().manual_seed((w.seed if seed is None else seed) + 2000)
    dt = torch_dtype(w)
    shape = (w.batch, w.num_kv_heads, cap, w.head_dim)
    k = torch.zeros(shape, dtype=dt)
    v = torch.zeros(shape, dtype=dt)
    L = w.cache_len
    k[:, :, :L] = _normal(gen, (w.batch, w.num_kv_heads, L, w.head_dim), 1.0, dt)
    v[:, :, :L] = _normal(gen, (w.batch, w.num_kv_heads, L, w.head_dim), 1.0, dt)
    return k, v


def make_model(w: Workload, n_layers: int, vocab: int, seed: int | None = None):
    """A synthetic model around the block: per-layer weights (make_weights, one seed per
    layer), embeddings ~ N(0, 1), lm_head ~ N(0, 0.02), final gain 1, and token ids
    uniform over the vocabulary, [batch, seq]. Returns (layers, embed, norm_g, lm_head, tokens)."""
    s = w.seed if seed is None else seed
    layers = [make_weights(w, seed=s + 101 * (l + 1)) for l in range(n_layers)]
    gen = torch.Generator().manual_seed(s + 3000)
    dt = torch_dtype(w)
    embed = torch.randn(vocab, w.hidden_size, generator=gen).to(dt)
    lm_head = (torch.randn(vocab, w.hidden_size, generator=gen) * 0.02).to(dt)
    norm_g = torch.ones(w.hidden_size, dtype=dt)
    tokens = torch.randint(0, vocab, (w.batch, w.seq), generator=gen, dtype=torch.int32)
    return layers, embed, norm_g, lm_head, tokens
