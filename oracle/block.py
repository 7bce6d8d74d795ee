"""Plain, slow, fp64 CPU oracle of the Llama-style decoder block forward pass.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module; the
tests, the smoke check and the CPU-baseline leg of the benchmark do. It shares
no code, table or constant generator with the CUDA library.

Every step is written the way the pages state it, in float64, with no blocking,
fusion or reordering. NumPy's matmul is the only library primitive used (for
the projections and the per-head score/value products).

Sources (page title, section):
  * "LlamaForCausalLM-32L-4096d" sheet, "Implementing it": the block pseudo-code
    (rmsnorm -> q/k/v projections -> rope(theta=10000) -> softmax(q k^T / sqrt(128),
    causal) v -> o_proj -> residual -> rmsnorm -> silu(gate) * up -> down ->
    residual).
  * nnterp encyclopedia "arcee", "The block, in order": the two pre-norm
    sublayers and the ungated squared-ReLU MLP ``down_proj(relu(up_proj(z)) ** 2)``;
    "Grouped-query attention, 128-wide heads": key/value head j serves a
    contiguous group of query heads (repeat_kv); "The API": tap names/layouts.
  * nnterp encyclopedia "apertus", "The MLP has no gate, and its activation is
    learned per block": xIELU and its parameter transform; "Queries and keys are
    normed per head, before the rotary": q_norm/k_norm over head_dim, one gain for
    every head, applied before RoPE.
  * nnterp encyclopedia "afmoe", "The block, in order": the sandwich block, each
    sublayer's output RMSNormed before the residual add; "Attention: per-head q/k
    norms and a sigmoid gate on every head": o_proj reads the head outputs times
    sigmoid(gate_proj(normed input)), one gate value per channel of every head;
    "Rotary runs on the sliding-window blocks only": a window of the last
    sliding_window tokens, and no rotary on the whole-prefix blocks.

Readings where the pages leave a step open:
  * RMSNorm is x / sqrt(mean(x^2) + eps) * g over the last axis (eps inside the
    square root, no mean-centering, no bias).
  * RoPE pairs element i with element i + d/2 ("rotate half"), with
    inv_freq_i = theta^(-2i/d) for i < d/2 and angle = position * inv_freq_i.
  * Key j is visible to query i iff position(j) <= position(i), and, with a
    sliding window W, position(i) - position(j) < W (the last W tokens, the
    query's own included).
  * The attention gate is projected from the attention's input, i.e. the
    input_layernorm output, the same rows q/k/v are projected from.
  * xIELU at exactly x = 0 takes the negative branch (the positive one is
    written for x > 0 only).

Every function here is pinned by the not-gpu tests (closed forms, page-printed
values, invariants, brute force on tiny inputs); SwiGLU's silu is pinned by its
textbook properties only.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

F64 = np.float64


@dataclass(frozen=True)
class RopeScaling:
    """A stretched rotary (the pages name the settings, not the formulas; these are
    the published definitions).

    kind "yarn": YaRN's by-parts interpolation, "arcee" page ("Loading and
    positions": YaRN, factor 20 over 4096 original positions, the model loaded
    through transformers). low / high are the turn counts over the original
    context that bound the blend (beta_slow 1 and beta_fast 32); the blend runs
    linearly over the pair index between the indices where those turn counts
    fall, as the published YaRN implementation builds it.
    kind "llama3": the frequency-dependent rule of Llama 3.1's rope_type llama3,
    "apertus" page ("The default load runs the same attention as eager": factor 8
    over 8192 original positions, rope_theta 12,000,000). low / high are its
    low_freq_factor / high_freq_factor (1 and 4).
    """

    kind: str
    factor: float
    original_max_position: float
    low: float
    high: float

    def __post_init__(self):
        if self.kind not in ("yarn", "llama3"):
            raise ValueError(f"unknown rope scaling {self.kind!r}")
        if not (self.factor >= 1.0 and self.original_max_position > 0 and self.high > self.low > 0):
            raise ValueError("rope scaling needs factor >= 1, original positions > 0 and high > low > 0")


@dataclass(frozen=True)
class BlockConfig:
    """The block's configuration, in the pages' config-key vocabulary.

    Keys follow the "Config" tables of the nnterp encyclopedia pages
    (hidden_size, num_attention_heads, num_key_value_heads, head_dim,
    intermediate_size, hidden_act, rms_norm_eps, rope_theta).
    """

    hidden_size: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    intermediate_size: int
    hidden_act: str  # "silu" (gated SwiGLU), "relu2", "xielu"
    rms_norm_eps: float = 1e-5
    rope_theta: float = 10000.0
    qk_norm: bool = False
    xielu_alpha_p: float = 0.8  # effective value (after the softplus transform)
    xielu_alpha_n: float = 0.8  # effective value (after beta + softplus)
    xielu_beta: float = 0.5
    xielu_eps: float = -1e-6
    rope_scaling: "RopeScaling | None" = None  # a stretched rotary, or None for the plain one
    # "afmoe" block variant
    sliding_window: int = 0       # 0: the whole prefix; W > 0: the last W tokens
    use_rope: bool = True         # False on afmoe's whole-prefix blocks
    attn_gate: bool = False       # o_proj input = heads * sigmoid(attn_gate_proj(normed input))
    sandwich_norm: bool = False   # RMSNorm of each sublayer's output before its residual add

    def __post_init__(self):
        if self.hidden_act not in ("silu", "relu2", "xielu"):
            raise ValueError(f"unknown hidden_act {self.hidden_act!r}")
        if self.num_heads % self.num_kv_heads:
            raise ValueError("num_heads must be a multiple of num_kv_heads")
        if self.head_dim % 2:
            raise ValueError("head_dim must be even for the rotary")
        if self.sliding_window < 0:
            raise ValueError("sliding_window must be >= 0")


# --------------------------------------------------------------------------
# Elementary operations
# --------------------------------------------------------------------------

def rms_norm(x, gain, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gain.

    Pages: "arcee" printout ``ArceeRMSNorm((2560,), eps=1e-05)``; the
    "LlamaForCausalLM-32L-4096d" pseudo-code ``rmsnorm(x, ..., eps=1e-05)``;
    "afmoe", "The contributions are the post-norms' outputs" (scale-invariant up
    to eps).
    """
    x = np.asarray(x, dtype=F64)
    mean_sq = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(mean_sq + eps) * np.asarray(gain, dtype=F64)


def rope_inv_freq(head_dim, theta, scaling=None):
    """inv_freq_i = theta^(-2i/head_dim), i = 0 .. head_dim/2 - 1, then stretched.

    With a scaling of factor s over L original positions, a frequency f has the
    wavelength lam = 2 pi / f and makes r = L / lam turns over the original
    context. Both published rules keep fast components, divide slow ones by s,
    and blend in between; they differ in what the blend is linear in:
      llama3 (Llama 3.1's rule, "apertus"): kept when lam < L / high, divided
              when lam > L / low, otherwise (1 - g) f / s + g f with
              g = (L / lam - low) / (high - low), linear in the turn count;
      yarn (the published YaRN implementation, which transformers runs for
              "arcee"): the pair index where a component makes R turns is
              i(R) = d ln(L / (2 pi R)) / (2 ln theta); with a = floor(i(high))
              and b = ceil(i(low)) (clamped to [0, d - 1]), the weight of f / s is
              clip((i - a) / (b - a), 0, 1), linear in the pair index.
    """
    i = np.arange(head_dim // 2, dtype=F64)
    f = np.power(F64(theta), -2.0 * i / head_dim)
    if scaling is None:
        return f
    s, L, lo, hi = scaling.factor, scaling.original_max_position, scaling.low, scaling.high
    lam = 2.0 * np.pi / f
    if scaling.kind == "llama3":
        g = (L / lam - lo) / (hi - lo)
        out = (1.0 - g) * f / s + g * f
        out = np.where(lam < L / hi, f, out)
        return np.where(lam > L / lo, f / s, out)

    def index_of_turns(r):
        return head_dim * np.log(L / (2.0 * np.pi * r)) / (2.0 * np.log(F64(theta)))

    a = max(np.floor(index_of_turns(hi)), 0.0)
    b = min(np.ceil(index_of_turns(lo)), head_dim - 1.0)
    if b == a:
        b = a + 0.001
    w = np.clip((i - a) / (b - a), 0.0, 1.0)  # weight of the interpolated frequency
    return (1.0 - w) * f + w * f / s


def rope_attention_factor(scaling):
    """YaRN scales cos and sin (so q.k by its square) by 0.1 ln(s) + 1, the paper's
    sqrt(1/t); the llama3 rule and the plain rotary by 1."""
    if scaling is None or scaling.kind != "yarn":
        return 1.0
    return 0.1 * np.log(scaling.factor) + 1.0


def rope(x, positions, theta, scaling=None):
    """Rotary embedding of x[..., T, d] at the given positions (length T).

    Pages: "LlamaForCausalLM-32L-4096d" ``q, k = rope(q, k, theta=10000)``;
    "apertus" ("at position 0, where the rotation is the identity").
    Element i is rotated together with element i + d/2 by the angle
    position * inv_freq_i (stretched by `scaling`, whose attention factor then
    multiplies the rotated vector).
    """
    x = np.asarray(x, dtype=F64)
    d = x.shape[-1]
    half = d // 2
    pos = np.asarray(positions, dtype=F64)
    ang = pos[:, None] * rope_inv_freq(d, theta, scaling)[None, :]  # [T, d/2]
    m = rope_attention_factor(scaling)
    c, s = m * np.cos(ang), m * np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def causal_gqa_attention(q, k, v, q_positions, k_positions, return_pattern=False, window=0, key_valid=None):
    """softmax(q k^T / sqrt(d), causal) v per query head, grouped over KV heads.

    q: [H, Tq, d], k, v: [Hkv, Tk, d] (one sequence). Query head h reads KV head
    h // (H / Hkv) ("arcee": "an edit to key/value head j reaches query heads 5j
    to 5j + 4"). Key j is visible to query i iff k_positions[j] <= q_positions[i]
    and, when window > 0, q_positions[i] - k_positions[j] < window ("afmoe",
    "Rotary runs on the sliding-window blocks only": the last sliding_window
    tokens). key_valid (bool [Tk], optional) hides the padding keys of an
    attention_mask ("arcee", "The API": zeros are padding); a query that sees no
    key at all gets a zero output. Returns head outputs [H, Tq, d] (and the
    masked scores and probabilities).
    """
    q = np.asarray(q, dtype=F64)
    k = np.asarray(k, dtype=F64)
    v = np.asarray(v, dtype=F64)
    H, Tq, d = q.shape
    Hkv = k.shape[0]
    group = H // Hkv
    gap = np.asarray(q_positions)[:, None] - np.asarray(k_positions)[None, :]
    visible = gap >= 0
    if window > 0:
        visible &= gap < window
    if key_valid is not None:
        visible &= np.asarray(key_valid, dtype=bool)[None, :]
    seen = np.any(visible, axis=-1)  # [Tq]: queries with at least one visible key
    out = np.empty((H, Tq, d), dtype=F64)
    scores_all, probs_all = [], []
    for h in range(H):
        j = h // group
        s = (q[h] @ k[j].T) / np.sqrt(F64(d))
        s = np.where(visible, s, -np.inf)
        m = np.where(seen[:, None], np.max(s, axis=-1, keepdims=True), 0.0)
        e = np.exp(s - m)
        z = np.sum(e, axis=-1, keepdims=True)
        p = e / np.where(z > 0, z, 1.0)
        out[h] = p @ v[j]
        if return_pattern:
            scores_all.append(s)
            probs_all.append(p)
    if return_pattern:
        return out, np.stack(scores_all), np.stack(probs_all)
    return out


def silu(u):
    """silu(u) = u / (1 + exp(-u)) (the gated MLP's act_fn)."""
    u = np.asarray(u, dtype=F64)
    with np.errstate(over="ignore"):
        return u / (1.0 + np.exp(-u))


def relu2(u):
    """relu(u) ** 2 ("arcee": ``down_proj(relu(up_proj(z)) ** 2)``)."""
    u = np.asarray(u, dtype=F64)
    r = np.maximum(u, 0.0)
    return r * r


def softplus(t):
    """softplus(t) = log(1 + exp(t)), evaluated without overflow."""
    t = np.asarray(t, dtype=F64)
    return np.logaddexp(0.0, t)


def xielu_effective(raw_alpha_p, raw_alpha_n, beta=0.5):
    """Stored xIELU parameters -> the values the formula uses.

    "apertus": the effective alpha_p is softplus(alpha_p) and the effective
    alpha_n is beta + softplus(alpha_n).
    """
    return float(softplus(raw_alpha_p)), float(beta + softplus(raw_alpha_n))


def xielu(u, alpha_p, alpha_n, beta=0.5, eps=-1e-6):
    """xIELU with effective parameters.

    "apertus": alpha_p * x^2 + beta * x for x > 0, and
    alpha_n * (expm1(min(x, eps)) - x) + beta * x otherwise.
    """
    u = np.asarray(u, dtype=F64)
    pos = alpha_p * u * u + beta * u
    neg = alpha_n * (np.expm1(np.minimum(u, eps)) - u) + beta * u
    return np.where(u > 0, pos, neg)


# --------------------------------------------------------------------------
# The block
# --------------------------------------------------------------------------

def _act(cfg, up, gate=None):
    if cfg.hidden_act == "silu":
        return silu(gate)
    if cfg.hidden_act == "relu2":
        return relu2(up)
    return xielu(up, cfg.xielu_alpha_p, cfg.xielu_alpha_n, cfg.xielu_beta, cfg.xielu_eps)


def _heads(t, n, d):
    """[T, n*d] -> [n, T, d]."""
    return t.reshape(t.shape[0], n, d).transpose(1, 0, 2)


def _project_kv(cfg, w, h_norm, positions):
    """Keys and values of every row: k_proj/v_proj, optional k_norm, RoPE on k."""
    d = cfg.head_dim
    k = _heads(h_norm @ w["k_proj"].T, cfg.num_kv_heads, d)
    v = _heads(h_norm @ w["v_proj"].T, cfg.num_kv_heads, d)
    if cfg.qk_norm:
        k = rms_norm(k, w["k_norm"], cfg.rms_norm_eps)
    if cfg.use_rope:
        k = rope(k, positions, cfg.rope_theta, cfg.rope_scaling)
    return k, v


def _project_q(cfg, w, h_norm_rows, positions_rows):
    d = cfg.head_dim
    q = _heads(h_norm_rows @ w["q_proj"].T, cfg.num_heads, d)
    if cfg.qk_norm:
        q = rms_norm(q, w["q_norm"], cfg.rms_norm_eps)
    if not cfg.use_rope:  # "afmoe": the whole-prefix blocks order tokens by the causal mask alone
        return q
    return rope(q, positions_rows, cfg.rope_theta, cfg.rope_scaling)


def mlp(cfg, w, h):
    """The MLP sublayer on normed rows h [..., D] (no residual).

    "LlamaForCausalLM-32L-4096d": (silu(h gate^T) * (h up^T)) down^T; "arcee":
    down_proj(relu(up_proj(z)) ** 2); "apertus": down_proj(xielu(up_proj(z))).
    Returns mlp_up_output, (mlp_gate_output), mlp_activation, mlp_neurons, mlp_output.
    """
    h = np.asarray(h, dtype=F64)
    taps = {}
    up = h @ w["up_proj"].T
    if cfg.hidden_act == "silu":
        gate = h @ w["gate_proj"].T
        act = _act(cfg, up, gate)
        neurons = act * up
        taps["mlp_gate_output"] = gate
    else:
        act = _act(cfg, up)
        neurons = act
    taps.update(mlp_up_output=up, mlp_activation=act, mlp_neurons=neurons, mlp_output=neurons @ w["down_proj"].T)
    return taps


def sigmoid(u):
    """1 / (1 + exp(-u)) (the attention gate of "afmoe")."""
    u = np.asarray(u, dtype=F64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-u))


def _finish_rows(cfg, w, x_rows, heads_out, h_rows):
    """o_proj, residual, second norm, MLP and residual for a set of rows.

    heads_out: [H, R, d] per-head outputs of those rows; h_rows: [R, D] their
    input_layernorm outputs (the attention gate's input).

    With cfg.attn_gate ("afmoe", "Attention: per-head q/k norms and a sigmoid
    gate on every head") o_proj reads heads * sigmoid(h_rows attn_gate_proj^T);
    attention_head_outputs stay ungated. With cfg.sandwich_norm ("afmoe", "The
    block, in order") each sublayer's output passes an RMSNorm before its
    residual add: "post_attn_norm" (afmoe's post_attention_layernorm) after
    o_proj and "post_mlp_norm" after down_proj; the MLP's input norm keeps the
    key "post_attention_layernorm" (afmoe's pre_mlp_layernorm). attention_output
    and mlp_output are then the post-norms' outputs ("The contributions are the
    post-norms' outputs").
    """
    R = x_rows.shape[0]
    premix = heads_out.transpose(1, 0, 2).reshape(R, -1)  # [R, H*d]
    taps = {}
    if cfg.attn_gate:
        gate = np.asarray(h_rows, dtype=F64) @ w["attn_gate_proj"].T  # [R, H*d]
        taps["attention_gate"] = gate
        premix = premix * sigmoid(gate)
    attn_out = premix @ w["o_proj"].T
    if cfg.sandwich_norm:
        attn_out = rms_norm(attn_out, w["post_attn_norm"], cfg.rms_norm_eps)
    mid = x_rows + attn_out
    h2 = rms_norm(mid, w["post_attention_layernorm"], cfg.rms_norm_eps)
    taps.update(mlp(cfg, w, h2))
    if cfg.sandwich_norm:
        taps["mlp_output"] = rms_norm(taps["mlp_output"], w["post_mlp_norm"], cfg.rms_norm_eps)
    taps.update(
        o_proj_input=premix,
        attention_head_outputs=heads_out.transpose(1, 0, 2),  # [R, H, d]
        attention_output=attn_out,
        layer_mid=mid,
        mlp_norm_output=h2,
        layer_output=mid + taps["mlp_output"],
    )
    return taps


def padding_run(mask_row):
    """[lo, hi): the contiguous run of ones of one attention_mask row (left
    padding, right padding or both); (T, T) for a row of zeros. Other patterns
    are refused."""
    m = np.asarray(mask_row) != 0
    T = m.shape[0]
    ones = np.flatnonzero(m)
    if ones.size == 0:
        return T, T
    lo, hi = int(ones[0]), int(ones[-1]) + 1
    if ones.size != hi - lo:
        raise ValueError("attention_mask rows must hold one contiguous run of ones")
    return lo, hi


def block_forward(cfg, w, x, rows=None, positions=None, return_pattern=False, attention_mask=None):
    """Forward pass of one decoder block over x[B, T, D] (fp64).

    Follows the "LlamaForCausalLM-32L-4096d" pseudo-code, with the MLP variant
    chosen by cfg.hidden_act ("arcee": relu2, "apertus": xielu) and the
    optional per-head q/k RMSNorm before RoPE ("apertus").

    rows: optional sorted list of sequence positions whose outputs are wanted
    (keys/values are still formed for every position, as attention needs them).
    positions: optional rotary positions of the T rows (default 0 .. T-1).
    attention_mask: optional [B, T] of 0/1 ("arcee", "The API": zeros are
    padding), each row one contiguous run of ones [lo, hi): padding keys are
    hidden and row t takes position t - lo, so a real row equals the unpadded
    sequence's row; rows before lo see no key (zero head outputs).

    Returns a dict of taps, each with a leading batch axis, named as the nnterp
    pages name them: attention_norm_output, attention_queries [B,H,R,d],
    attention_keys [B,Hkv,T,d], attention_values, attention_head_outputs
    [B,R,H,d], (attention_gate), o_proj_input, attention_output, layer_mid,
    mlp_norm_output, mlp_up_output, (mlp_gate_output), mlp_activation,
    mlp_neurons, mlp_output, layer_output.
    """
    x = np.asarray(x, dtype=F64)
    B, T, D = x.shape
    assert D == cfg.hidden_size
    if rows is None:
        rows = np.arange(T)
    rows = np.asarray(rows)
    if positions is None:
        positions = np.arange(T)
    positions = np.asarray(positions)
    if attention_mask is not None and positions is not None and not np.array_equal(positions, np.arange(T)):
        raise ValueError("attention_mask sets the positions itself")
    per_batch = []
    for b in range(B):
        taps = {}
        pos_b, valid = positions, None
        if attention_mask is not None:
            lo, _ = padding_run(attention_mask[b])
            pos_b = np.arange(T) - lo
            valid = np.asarray(attention_mask[b]) != 0
        h = rms_norm(x[b], w["input_layernorm"], cfg.rms_norm_eps)  # [T, D]
        k, v = _project_kv(cfg, w, h, pos_b)
        q = _project_q(cfg, w, h[rows], pos_b[rows])
        res = causal_gqa_attention(q, k, v, pos_b[rows], pos_b, return_pattern, cfg.sliding_window, valid)
        if return_pattern:
            heads, scores, probs = res
            taps["attention_scores"] = scores
            taps["attention_probabilities"] = probs
        else:
            heads = res
        taps.update(_finish_rows(cfg, w, x[b][rows], heads, h[rows]))
        taps.update(
            layer_input=x[b][rows],
            attention_norm_output=h[rows],
            attention_queries=q,
            attention_keys=k,
            attention_values=v,
        )
        per_batch.append(taps)
    return {key: np.stack([t[key] for t in per_batch]) for key in per_batch[0]}


def prefill_with_cache(cfg, w, x, cache_k, cache_v, lens):
    """T new tokens per sequence after lens[b] cached positions (a prefill chunk).

    x: [B, T, D]; cache_k, cache_v: [B, Hkv, capacity, d] holding keys (after
    k_norm and RoPE) and values for positions 0 .. lens[b]-1. Token t of
    sequence b sits at position lens[b] + t; its key and value join the cache at
    slot lens[b] + t, and it attends causally over slots 0 .. lens[b] + t. The
    pages define no cache: this is the prefill block on the whole sequence,
    restricted to the new rows, with the earlier keys read from the cache.

    Returns the taps of the new rows ([B, T, ...]) plus new_keys / new_values
    [B, Hkv, T, d].
    """
    x = np.asarray(x, dtype=F64)
    B, T, D = x.shape
    per_batch = []
    for b in range(B):
        L = int(lens[b])
        pos = np.arange(L, L + T)
        h = rms_norm(x[b], w["input_layernorm"], cfg.rms_norm_eps)  # [T, D]
        k_new, v_new = _project_kv(cfg, w, h, pos)  # [Hkv, T, d]
        q = _project_q(cfg, w, h, pos)  # [H, T, d]
        k_all = np.concatenate([np.asarray(cache_k[b, :, :L], dtype=F64), k_new], axis=1)
        v_all = np.concatenate([np.asarray(cache_v[b, :, :L], dtype=F64), v_new], axis=1)
        heads = causal_gqa_attention(q, k_all, v_all, pos, np.arange(L + T), window=cfg.sliding_window)
        taps = _finish_rows(cfg, w, x[b], heads, h)
        taps.update(attention_norm_output=h, attention_queries=q, new_keys=k_new, new_values=v_new)
        per_batch.append(taps)
    return {key: np.stack([t[key] for t in per_batch]) for key in per_batch[0]}


def decode_step(cfg, w, x, cache_k, cache_v, lens):
    """One decode step: one new token per sequence attends to its KV cache.

    x: [B, D] new tokens; cache_k, cache_v: [B, Hkv, capacity, d] holding keys
    (after k_norm and RoPE) and values for positions 0 .. lens[b]-1; lens: [B].
    The new token sits at position lens[b]; its key/value join the cache at slot
    lens[b] and it attends over lens[b] + 1 keys. The pages define no cache;
    this is the prefill block restricted to its last row, with earlier keys
    read from the cache instead of recomputed.

    Returns the taps of the new rows ([B, ...], row axis dropped) plus
    new_key [B, Hkv, d] and new_value [B, Hkv, d].
    """
    x = np.asarray(x, dtype=F64)
    B, D = x.shape
    per_batch = []
    for b in range(B):
        L = int(lens[b])
        pos = np.array([L])
        h = rms_norm(x[b:b + 1], w["input_layernorm"], cfg.rms_norm_eps)  # [1, D]
        k_new, v_new = _project_kv(cfg, w, h, pos)  # [Hkv, 1, d]
        q = _project_q(cfg, w, h, pos)  # [H, 1, d]
        k_all = np.concatenate([np.asarray(cache_k[b, :, :L], dtype=F64), k_new], axis=1)
        v_all = np.concatenate([np.asarray(cache_v[b, :, :L], dtype=F64), v_new], axis=1)
        heads = causal_gqa_attention(q, k_all, v_all, pos, np.arange(L + 1), window=cfg.sliding_window)
        taps = _finish_rows(cfg, w, x[b:b + 1], heads, h)
        taps = {key: val[0] for key, val in taps.items()}
        taps.update(
            attention_norm_output=h[0],
            attention_queries=q[:, 0],
            new_key=k_new[:, 0],
            new_value=v_new[:, 0],
        )
        per_batch.append(taps)
    return {key: np.stack([t[key] for t in per_batch]) for key in per_batch[0]}


def model_forward(cfg, layers, embed, norm_g, lm_head, tokens):
    """Logits of the model around the block ("LlamaForCausalLM-32L-4096d" sheet,
    "Implementing it": embed_tokens, the decoder layers in order, norm, lm_head).

    tokens: int [B, T]; layers: a list of block weight dicts; embed and lm_head
    [vocab, D]; norm_g [D]. Returns logits [B, T, vocab].
    """
    x = np.asarray(embed, dtype=F64)[np.asarray(tokens)]
    for w in layers:
        x = block_forward(cfg, w, x)["layer_output"]
    h = rms_norm(x, norm_g, cfg.rms_norm_eps)
    return h @ np.asarray(lm_head, dtype=F64).T
