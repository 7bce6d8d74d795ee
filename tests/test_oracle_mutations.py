"""Plants plausible mistakes in the oracle (CPU only) and checks a pin catches each.

This guards the pins themselves: a dropped term, a wrong sign or index, or a
misread pairing in any oracle step must make at least one pin test fail.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import oracle.block as ob
from tests import test_oracle_pins as pins

F64 = np.float64


def _rms_eps_outside(x, gain, eps):
    x = np.asarray(x, dtype=F64)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * gain


def _rms_sum(x, gain, eps):
    x = np.asarray(x, dtype=F64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * gain


def _rope_interleaved(x, positions, theta, scaling=None):
    x = np.asarray(x, dtype=F64)
    d = x.shape[-1]
    ang = np.asarray(positions, dtype=F64)[:, None] * ob.rope_inv_freq(d, theta)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x1 * c - x2 * s
    out[..., 1::2] = x2 * c + x1 * s
    return out


def _inv_freq_wrong(head_dim, theta, scaling=None):
    i = np.arange(head_dim // 2, dtype=F64)
    return np.power(F64(theta), -i / head_dim)


def _rope_sign(x, positions, theta, scaling=None):
    x = np.asarray(x, dtype=F64)
    d = x.shape[-1]
    ang = np.asarray(positions, dtype=F64)[:, None] * ob.rope_inv_freq(d, theta)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], axis=-1)


def _attn_factory(scale=True, gqa="div", strict=False, window_slack=0, use_key_valid=True):
    def attn(q, k, v, q_positions, k_positions, return_pattern=False, window=0, key_valid=None):
        q, k, v = (np.asarray(a, dtype=F64) for a in (q, k, v))
        H, Tq, d = q.shape
        Hkv = k.shape[0]
        qp, kp = np.asarray(q_positions), np.asarray(k_positions)
        vis = (kp[None, :] < qp[:, None]) | (kp[None, :] == 0) if strict else kp[None, :] <= qp[:, None]
        if window > 0:
            vis = vis & (qp[:, None] - kp[None, :] < window + window_slack)
        if key_valid is not None and use_key_valid:
            vis = vis & np.asarray(key_valid, dtype=bool)[None, :]
        out = np.empty((H, Tq, d))
        ss, pp = [], []
        for h in range(H):
            j = h // (H // Hkv) if gqa == "div" else h % Hkv
            s = q[h] @ k[j].T / (np.sqrt(F64(d)) if scale else 1.0)
            s = np.where(vis, s, -np.inf)
            mx = s.max(-1, keepdims=True)
            e = np.exp(s - np.where(np.isfinite(mx), mx, 0.0))
            p = e / np.maximum(e.sum(-1, keepdims=True), 1e-300)
            out[h] = p @ v[j]
            ss.append(s)
            pp.append(p)
        return (out, np.stack(ss), np.stack(pp)) if return_pattern else out
    return attn


def _xielu_beta_sign(u, alpha_p, alpha_n, beta=0.5, eps=-1e-6):
    u = np.asarray(u, dtype=F64)
    return np.where(u > 0, alpha_p * u * u + beta * u, alpha_n * (np.expm1(np.minimum(u, eps)) - u) - beta * u)


def _xielu_no_min(u, alpha_p, alpha_n, beta=0.5, eps=-1e-6):
    u = np.asarray(u, dtype=F64)
    return np.where(u > 0, alpha_p * u * u + beta * u, alpha_n * (np.expm1(u) + u) + beta * u)


def _silu_wrong(u):
    u = np.asarray(u, dtype=F64)
    return u / (1.0 + np.exp(u))


_orig_inv_freq = ob.rope_inv_freq


def _scaling_ramp_reversed(head_dim, theta, scaling=None):
    # the blend weight turned around: fast components divided, slow ones kept
    if scaling is None:
        return _orig_inv_freq(head_dim, theta)
    f = _orig_inv_freq(head_dim, theta)
    s = _orig_inv_freq(head_dim, theta, scaling)
    return f * (f / s) / scaling.factor


def _yarn_ramp_over_turns(head_dim, theta, scaling=None):
    # YaRN's blend taken linear in the turn count r = L / lam (the paper's gamma(r))
    # instead of the published implementation's ramp over the pair index
    if scaling is None or scaling.kind != "yarn":
        return _orig_inv_freq(head_dim, theta, scaling)
    f = _orig_inv_freq(head_dim, theta)
    r = scaling.original_max_position * f / (2 * np.pi)
    g = np.clip((r - scaling.low) / (scaling.high - scaling.low), 0.0, 1.0)
    return (1 - g) * f / scaling.factor + g * f


def _yarn_unrounded_indices(head_dim, theta, scaling=None):
    # the correction indices used as computed, without the floor / ceil
    if scaling is None or scaling.kind != "yarn":
        return _orig_inv_freq(head_dim, theta, scaling)
    f = _orig_inv_freq(head_dim, theta)
    L = scaling.original_max_position
    idx = lambda r: head_dim * np.log(L / (2 * np.pi * r)) / (2 * np.log(theta))
    a, b = idx(scaling.high), idx(scaling.low)
    w = np.clip((np.arange(head_dim // 2) - a) / (b - a), 0.0, 1.0)
    return (1 - w) * f + w * f / scaling.factor


def _llama3_ramp_over_index(head_dim, theta, scaling=None):
    # llama3's blend taken linear in the pair index between the band's edges
    if scaling is None or scaling.kind != "llama3":
        return _orig_inv_freq(head_dim, theta, scaling)
    f = _orig_inv_freq(head_dim, theta)
    L, s, lo, hi = scaling.original_max_position, scaling.factor, scaling.low, scaling.high
    idx = lambda r: head_dim * np.log(L / (2 * np.pi * r)) / (2 * np.log(theta))
    g = np.clip(1 - (np.arange(head_dim // 2) - idx(hi)) / (idx(lo) - idx(hi)), 0.0, 1.0)
    return (1 - g) * f / s + g * f


def _llama3_ramp_over_wavelength(head_dim, theta, scaling=None):
    # llama3's blend taken linear in the wavelength instead of the turn count
    if scaling is None or scaling.kind != "llama3":
        return _orig_inv_freq(head_dim, theta, scaling)
    f = _orig_inv_freq(head_dim, theta)
    L, s, lo, hi = scaling.original_max_position, scaling.factor, scaling.low, scaling.high
    lam = 2 * np.pi / f
    g = np.clip(1 - (lam - L / hi) / (L / lo - L / hi), 0.0, 1.0)
    return (1 - g) * f / s + g * f


def _relu_not_squared(u):
    return np.maximum(np.asarray(u, dtype=F64), 0.0)


def _mlp_swapped(cfg, w, h):
    # silu applied to up instead of gate
    w2 = dict(w)
    if cfg.hidden_act == "silu":
        w2["gate_proj"], w2["up_proj"] = w["up_proj"], w["gate_proj"]
    return _orig_mlp(cfg, w2, h)


def _finish_no_residual(cfg, w, x_rows, heads_out, h_rows):
    taps = _orig_finish(cfg, w, x_rows, heads_out, h_rows)
    taps["layer_output"] = taps["layer_output"] - x_rows
    return taps


def _finish_gate_from_raw_input(cfg, w, x_rows, heads_out, h_rows):
    # the gate projected from the block's input instead of the normed rows
    return _orig_finish(cfg, w, x_rows, heads_out, x_rows)


def _sigmoid_sign(u):
    u = np.asarray(u, dtype=F64)
    return 1.0 / (1.0 + np.exp(u))


def _finish_norm_after_residual(cfg, w, x_rows, heads_out, h_rows):
    # the sandwich post-norms applied to the residual sums instead of the sublayer outputs
    if not cfg.sandwich_norm:
        return _orig_finish(cfg, w, x_rows, heads_out, h_rows)
    plain = dataclasses.replace(cfg, sandwich_norm=False)
    taps = _orig_finish(plain, w, x_rows, heads_out, h_rows)
    mid = ob.rms_norm(taps["layer_mid"], w["post_attn_norm"], cfg.rms_norm_eps)
    h2 = ob.rms_norm(mid, w["post_attention_layernorm"], cfg.rms_norm_eps)
    m = ob.mlp(plain, w, h2)
    taps.update(layer_mid=mid, attention_output=mid - x_rows, mlp_output=m["mlp_output"],
                layer_output=ob.rms_norm(mid + m["mlp_output"], w["post_mlp_norm"], cfg.rms_norm_eps))
    return taps


def _finish_no_mlp_post_norm(cfg, w, x_rows, heads_out, h_rows):
    taps = _orig_finish(cfg, w, x_rows, heads_out, h_rows)
    if cfg.sandwich_norm:
        raw = taps["mlp_neurons"] @ w["down_proj"].T
        taps.update(mlp_output=raw, layer_output=taps["layer_mid"] + raw)
    return taps


def _project_q_rope_always(cfg, w, h_norm_rows, positions_rows):
    return _orig_project_q(dataclasses.replace(cfg, use_rope=True), w, h_norm_rows, positions_rows)


def _project_kv_rope_always(cfg, w, h_norm, positions):
    return _orig_project_kv(dataclasses.replace(cfg, use_rope=True), w, h_norm, positions)


def _padding_run_unshifted(mask_row):
    # the padding keys hidden, but the real tokens' positions left unshifted
    lo, hi = _orig_padding_run(mask_row)
    return 0, hi


def _yarn_attention_factor_dropped(scaling):
    return 1.0


def _xielu_alpha_n_without_beta(raw_alpha_p, raw_alpha_n, beta=0.5):
    return float(ob.softplus(raw_alpha_p)), float(ob.softplus(raw_alpha_n))


def _xielu_raw_parameters(raw_alpha_p, raw_alpha_n, beta=0.5):
    return float(raw_alpha_p), float(beta + raw_alpha_n)


def _decode_factory(shift=0, own_key=True):
    # decode_step with the new token's rotary position shifted, or without its own key
    def decode_step(cfg, w, x, cache_k, cache_v, lens):
        x = np.asarray(x, dtype=F64)
        outs = []
        for b in range(x.shape[0]):
            L = int(lens[b])
            pos = np.array([L + shift])
            h = ob.rms_norm(x[b:b + 1], w["input_layernorm"], cfg.rms_norm_eps)
            k_new, v_new = ob._project_kv(cfg, w, h, pos)
            q = ob._project_q(cfg, w, h, pos)
            k_all = np.asarray(cache_k[b, :, :L], dtype=F64)
            v_all = np.asarray(cache_v[b, :, :L], dtype=F64)
            if own_key:
                k_all = np.concatenate([k_all, k_new], axis=1)
                v_all = np.concatenate([v_all, v_new], axis=1)
            heads = ob.causal_gqa_attention(q, k_all, v_all, np.array([L]), np.arange(k_all.shape[1]),
                                            window=cfg.sliding_window)
            taps = {key: val[0] for key, val in ob._finish_rows(cfg, w, x[b:b + 1], heads, h).items()}
            taps.update(new_key=k_new[:, 0], new_value=v_new[:, 0])
            outs.append(taps)
        return {key: np.stack([t[key] for t in outs]) for key in outs[0]}
    return decode_step


def _prefill_chunk_positions_from_zero(cfg, w, x, cache_k, cache_v, lens):
    # the chunk's rotary positions restart at 0 instead of following the cache
    x = np.asarray(x, dtype=F64)
    B, T, _ = x.shape
    outs = []
    for b in range(B):
        L = int(lens[b])
        h = ob.rms_norm(x[b], w["input_layernorm"], cfg.rms_norm_eps)
        k_new, v_new = ob._project_kv(cfg, w, h, np.arange(T))
        q = ob._project_q(cfg, w, h, np.arange(T))
        k_all = np.concatenate([np.asarray(cache_k[b, :, :L], dtype=F64), k_new], axis=1)
        v_all = np.concatenate([np.asarray(cache_v[b, :, :L], dtype=F64), v_new], axis=1)
        heads = ob.causal_gqa_attention(q, k_all, v_all, np.arange(L, L + T), np.arange(L + T),
                                        window=cfg.sliding_window)
        taps = ob._finish_rows(cfg, w, x[b], heads, h)
        taps.update(new_keys=k_new, new_values=v_new)
        outs.append(taps)
    return {key: np.stack([t[key] for t in outs]) for key in outs[0]}


def _model_without_final_norm(cfg, layers, embed, norm_g, lm_head, tokens):
    x = np.asarray(embed, dtype=F64)[np.asarray(tokens)]
    for w in layers:
        x = ob.block_forward(cfg, w, x)["layer_output"]
    return (x * np.asarray(norm_g, dtype=F64)) @ np.asarray(lm_head, dtype=F64).T


_orig_padding_run = ob.padding_run
_orig_finish = ob._finish_rows
_orig_mlp = ob.mlp
_orig_project_q = ob._project_q
_orig_project_kv = ob._project_kv

MUTATIONS = {
    "rms_eps_outside_sqrt": [("rms_norm", _rms_eps_outside)],
    "rms_sum_not_mean": [("rms_norm", _rms_sum)],
    "rope_interleaved_pairs": [("rope", _rope_interleaved)],
    "rope_inv_freq_exponent": [("rope_inv_freq", _inv_freq_wrong)],
    "rope_rotation_sign": [("rope", _rope_sign)],
    "attn_no_scale": [("causal_gqa_attention", _attn_factory(scale=False))],
    "attn_gqa_modulo": [("causal_gqa_attention", _attn_factory(gqa="mod"))],
    "attn_mask_off_by_one": [("causal_gqa_attention", _attn_factory(strict=True))],
    "xielu_beta_sign": [("xielu", _xielu_beta_sign)],
    "xielu_dropped_min_and_sign": [("xielu", _xielu_no_min)],
    "silu_sign": [("silu", _silu_wrong)],
    "relu_not_squared": [("relu2", _relu_not_squared)],
    "swiglu_gate_up_swapped": [("mlp", _mlp_swapped)],
    "missing_residual": [("_finish_rows", _finish_no_residual)],
    "rope_scaling_ramp_reversed": [("rope_inv_freq", _scaling_ramp_reversed)],
    "yarn_ramp_over_turns": [("rope_inv_freq", _yarn_ramp_over_turns)],
    "yarn_correction_indices_unrounded": [("rope_inv_freq", _yarn_unrounded_indices)],
    "llama3_ramp_over_pair_index": [("rope_inv_freq", _llama3_ramp_over_index)],
    "llama3_ramp_over_wavelength": [("rope_inv_freq", _llama3_ramp_over_wavelength)],
    "attn_window_one_too_wide": [("causal_gqa_attention", _attn_factory(window_slack=1))],
    "attn_window_one_too_narrow": [("causal_gqa_attention", _attn_factory(window_slack=-1))],
    "gate_from_raw_input": [("_finish_rows", _finish_gate_from_raw_input)],
    "gate_sigmoid_sign": [("sigmoid", _sigmoid_sign)],
    "sandwich_norm_after_residual": [("_finish_rows", _finish_norm_after_residual)],
    "sandwich_mlp_post_norm_dropped": [("_finish_rows", _finish_no_mlp_post_norm)],
    "rotary_on_whole_prefix_blocks": [("_project_q", _project_q_rope_always),
                                      ("_project_kv", _project_kv_rope_always)],
    "padding_keys_visible": [("causal_gqa_attention", _attn_factory(use_key_valid=False))],
    "padding_positions_unshifted": [("padding_run", _padding_run_unshifted)],
    "yarn_attention_factor_dropped": [("rope_attention_factor", _yarn_attention_factor_dropped)],
    "xielu_alpha_n_without_beta": [("xielu_effective", _xielu_alpha_n_without_beta)],
    "xielu_parameters_without_softplus": [("xielu_effective", _xielu_raw_parameters)],
    "decode_rotary_one_position_early": [("decode_step", _decode_factory(shift=-1))],
    "decode_without_its_own_key": [("decode_step", _decode_factory(own_key=False))],
    "prefill_chunk_positions_from_zero": [("prefill_with_cache", _prefill_chunk_positions_from_zero)],
    "model_without_final_norm": [("model_forward", _model_without_final_norm)],
}

PIN_TESTS = [
    pins.test_rmsnorm_worked_example,
    pins.test_rmsnorm_eps_inside_sqrt,
    pins.test_rope_worked_values,
    pins.test_rope_matches_complex_rotation,
    pins.test_attention_brute_force,
    pins.test_attention_special_cases,
    pins.test_attention_gqa_reach,
    pins.test_relu2_exact_zeros,
    pins.test_xielu_page_values,
    pins.test_silu_textbook_properties,
    lambda: pins.test_block_brute_force("silu", False, 2, 2),
    lambda: pins.test_block_brute_force("relu2", False, 4, 2),
    lambda: pins.test_block_brute_force("xielu", True, 4, 1),
    pins.test_block_identity_and_taps,
    pins.test_llama3_scaling_keeps_fast_divides_slow_and_blends_between,
    pins.test_yarn_scaling_keeps_fast_divides_slow_and_scales_attention,
    pins.test_rope_scaling_golden_values,
    lambda: pins.test_attention_window_brute_force(3),
    pins.test_attention_window_special_cases,
    lambda: pins.test_afmoe_block_brute_force(3, True, True, True),
    lambda: pins.test_afmoe_block_brute_force(0, False, True, True),
    pins.test_afmoe_identity_and_post_norm_taps,
    pins.test_afmoe_sandwich_scale_invariance,
    pins.test_afmoe_gate_taps_and_half_gate,
    pins.test_afmoe_whole_prefix_block_queries_are_q_norm_output,
    pins.test_padded_batch_real_rows_equal_the_unpadded_rows,
    pins.test_xielu_parameter_transform,
    pins.test_decode_equals_last_prefill_row,
    pins.test_prefill_chunk_equals_the_full_prefill_rows,
    pins.test_prefill_chunk_of_one_token_is_a_decode_step,
    pins.test_model_with_identity_blocks_and_tied_embeddings_reads_its_own_token,
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    for attr, fn in MUTATIONS[name]:
        monkeypatch.setattr(ob, attr, fn)
        if hasattr(oracle, attr):
            monkeypatch.setattr(oracle, attr, fn)
    caught = []
    for t in PIN_TESTS:
        try:
            t()
        except AssertionError:
            caught.append(getattr(t, "__name__", "block"))
    assert caught, f"no pin caught mutation {name}"
