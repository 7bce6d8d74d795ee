"""Pins of the fp64 oracle to facts fixed outside it (runs without a GPU).

Each test checks the oracle against something other than its own code: values
printed on the pages, closed forms, invariants the pages state, special cases
with a textbook answer, or a pure-Python brute-force restatement on tiny inputs.
"""
import cmath
import dataclasses
import json
import math
import os
import zlib

from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import BlockConfig

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_worked_example():
    # mean(3^2, 4^2) = 12.5; 1/sqrt(12.5) = 0.28284271247461906
    y = oracle.rms_norm(np.array([3.0, 4.0]), np.array([1.0, 1.0]), 0.0)
    np.testing.assert_allclose(y, [0.848528137423857, 1.131370849898476], rtol=1e-14)
    y = oracle.rms_norm(np.array([3.0, 4.0]), np.array([2.0, -1.0]), 0.0)
    np.testing.assert_allclose(y, [1.697056274847714, -1.131370849898476], rtol=1e-14)


def test_rmsnorm_eps_inside_sqrt():
    # x = (1, 1), eps = 1: 1/sqrt(1 + 1); eps outside the root would give 1/2.
    y = oracle.rms_norm(np.array([1.0, 1.0]), np.ones(2), 1.0)
    np.testing.assert_allclose(y, [0.7071067811865476] * 2, rtol=1e-15)
    # an all-zero row stays zero (no NaN)
    assert np.all(oracle.rms_norm(np.zeros(8), np.ones(8), 1e-5) == 0.0)


def test_rmsnorm_scale_invariant_and_sink_row():
    # "afmoe": RMSNorm is scale-invariant up to eps.
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 64))
    g = 1 + 0.1 * rng.standard_normal(64)
    np.testing.assert_allclose(oracle.rms_norm(7.5 * x, g, 0.0), oracle.rms_norm(x, g, 0.0), rtol=1e-13)
    # "apertus": the position-0 sink has a norm ~100x the others; a row scaled
    # by 1e4 normalises to the same direction with unit RMS.
    y = oracle.rms_norm(1e4 * x[0], np.ones(64), 1e-5)
    assert np.all(np.isfinite(y))
    np.testing.assert_allclose(np.sqrt(np.mean(y * y)), 1.0, rtol=1e-12)


# ---------------------------------------------------------------- RoPE

def _rope_complex(x, pos, theta):
    """Rotary as a complex rotation: z_i = x_i + i x_{i+d/2}, z_i * exp(i pos theta^(-2i/d))."""
    d = len(x)
    out = [0.0] * d
    for i in range(d // 2):
        z = complex(x[i], x[i + d // 2]) * cmath.exp(1j * pos * theta ** (-2.0 * i / d))
        out[i], out[i + d // 2] = z.real, z.imag
    return out


def test_rope_worked_values():
    # d = 2: inv_freq = 1, so (1, 0) at position p becomes (cos p, sin p).
    for p in (0, 1, 3, 17):
        np.testing.assert_allclose(oracle.rope(np.array([[1.0, 0.0]]), [p], 10000.0)[0],
                                   [math.cos(p), math.sin(p)], rtol=0, atol=1e-15)
    # d = 4, theta = 1e4: inv_freq = (1, 0.01); pairs (x0, x2) and (x1, x3).
    got = oracle.rope(np.array([[1.0, 2.0, 3.0, 4.0]]), [1], 10000.0)[0]
    np.testing.assert_allclose(got, [-1.9841106484, 1.9599006750, 2.4623778975, 4.0197997033], atol=1e-9)


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 16))
    pos = [0, 1, 7, 100, 4095]
    got = oracle.rope(x, pos, 10000.0)
    for t in range(5):
        np.testing.assert_allclose(got[t], _rope_complex(list(x[t]), pos[t], 10000.0), atol=1e-12)


def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))
    # "apertus": at position 0 the rotation is the identity (bitwise).
    assert np.array_equal(oracle.rope(q, [0], 1e4), q)
    # rotations preserve the norm
    for p in (1, 2048, 4096):
        np.testing.assert_allclose(np.linalg.norm(oracle.rope(q, [p], 1e4)), np.linalg.norm(q), rtol=1e-13)
    # rope(q, m) . rope(k, n) depends only on m - n
    def dot(m, n):
        return float(oracle.rope(q, [m], 1e4)[0] @ oracle.rope(k, [n], 1e4)[0])
    np.testing.assert_allclose(dot(10, 3), dot(107, 100), rtol=1e-10)
    np.testing.assert_allclose(dot(5, 5), float(q[0] @ k[0]), rtol=1e-12)


# ---------------------------------------------------------------- attention

def _attention_loops(q, k, v, group, window=0):
    """Pure-Python triple loop: softmax over visible keys, then the value mix.

    window > 0: query i sees keys i - window + 1 .. i only ("afmoe": the last
    sliding_window tokens)."""
    H, T, d = len(q), len(q[0]), len(q[0][0])
    out = [[[0.0] * d for _ in range(T)] for _ in range(H)]
    for h in range(H):
        j = h // group
        for i in range(T):
            keys = list(range(max(0, i - window + 1) if window else 0, i + 1))
            s = [sum(q[h][i][c] * k[j][t][c] for c in range(d)) / math.sqrt(d) for t in keys]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = sum(e)
            for c in range(d):
                out[h][i][c] = sum(e[n] / z * v[j][t][c] for n, t in enumerate(keys))
    return out


def test_attention_brute_force():
    rng = np.random.default_rng(3)
    H, Hkv, T, d = 4, 2, 6, 4
    q, k, v = (rng.standard_normal((n, T, d)) for n in (H, Hkv, Hkv))
    got = oracle.causal_gqa_attention(q, k, v, np.arange(T), np.arange(T))
    want = _attention_loops(q.tolist(), k.tolist(), v.tolist(), H // Hkv)
    np.testing.assert_allclose(got, np.array(want), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("window", [1, 2, 3, 5])
def test_attention_window_brute_force(window):
    rng = np.random.default_rng(30 + window)
    H, Hkv, T, d = 4, 2, 7, 4
    q, k, v = (rng.standard_normal((n, T, d)) for n in (H, Hkv, Hkv))
    got = oracle.causal_gqa_attention(q, k, v, np.arange(T), np.arange(T), window=window)
    want = _attention_loops(q.tolist(), k.tolist(), v.tolist(), H // Hkv, window)
    np.testing.assert_allclose(got, np.array(want), rtol=1e-12, atol=1e-14)


def test_attention_window_special_cases():
    rng = np.random.default_rng(31)
    H, T, d = 2, 8, 4
    q, k, v = (rng.standard_normal((n, T, d)) for n in (H, 1, 1))
    # a window of one token: every query reads its own value
    o = oracle.causal_gqa_attention(q, k, v, np.arange(T), np.arange(T), window=1)
    np.testing.assert_array_equal(o, np.broadcast_to(v[0], (H, T, d)))
    # a window as long as the sequence is the plain causal mask
    full = oracle.causal_gqa_attention(q, k, v, np.arange(T), np.arange(T))
    np.testing.assert_array_equal(oracle.causal_gqa_attention(q, k, v, np.arange(T), np.arange(T), window=T), full)
    # a window of two: query i mixes v[i-1] and v[i] by the softmax of their two scores
    o = oracle.causal_gqa_attention(q, k, v, np.arange(T), np.arange(T), window=2)
    for i in range(1, T):
        s0, s1 = q[0, i] @ k[0, i - 1] / math.sqrt(d), q[0, i] @ k[0, i] / math.sqrt(d)
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        np.testing.assert_allclose(o[0, i], (1 - w1) * v[0, i - 1] + w1 * v[0, i], rtol=1e-12)
    # positions, not indices, decide: queries at 10..13 over keys at 0..13 with a window of 3
    qp, kp = np.arange(10, 14), np.arange(14)
    k2, v2 = rng.standard_normal((1, 14, d)), rng.standard_normal((1, 14, d))
    o = oracle.causal_gqa_attention(q[:, :4], k2, v2, qp, kp, window=3)
    want = oracle.causal_gqa_attention(q[:, :4], k2[:, 8:], v2[:, 8:], qp, kp[8:], window=3)
    np.testing.assert_allclose(o, want, rtol=1e-14)


def test_attention_special_cases():
    rng = np.random.default_rng(4)
    T, d = 9, 8
    q = rng.standard_normal((2, T, d))
    v = rng.standard_normal((1, T, d))
    # all keys equal: every visible key gets the same weight -> prefix mean of v
    k = np.repeat(rng.standard_normal((1, 1, d)), T, axis=1)
    o = oracle.causal_gqa_attention(q, k, v, np.arange(T), np.arange(T))
    for i in range(T):
        np.testing.assert_allclose(o[0, i], v[0, : i + 1].mean(axis=0), rtol=1e-12)
    # query 0 sees only key 0
    k = rng.standard_normal((1, T, d))
    o = oracle.causal_gqa_attention(q, k, v, np.arange(T), np.arange(T))
    np.testing.assert_array_equal(o[:, 0], np.broadcast_to(v[0, 0], (2, d)))
    # two keys, closed form: softmax of the two scaled scores
    s0, s1 = q[0, 1] @ k[0, 0] / math.sqrt(d), q[0, 1] @ k[0, 1] / math.sqrt(d)
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    np.testing.assert_allclose(o[0, 1], (1 - w1) * v[0, 0] + w1 * v[0, 1], rtol=1e-12)


def test_attention_gqa_reach():
    # "arcee": an edit to key/value head j reaches query heads 5j .. 5j+4 only.
    rng = np.random.default_rng(5)
    H, Hkv, T, d = 20, 4, 5, 4
    q, k, v = (rng.standard_normal((n, T, d)) for n in (H, Hkv, Hkv))
    base = oracle.causal_gqa_attention(q, k, v, np.arange(T), np.arange(T))
    for j in range(Hkv):
        v2 = v.copy()
        v2[j] += 1.0
        o = oracle.causal_gqa_attention(q, k, v2, np.arange(T), np.arange(T))
        changed = [h for h in range(H) if not np.array_equal(o[h], base[h])]
        assert changed == list(range(5 * j, 5 * j + 5))


def test_attention_pattern_rows():
    rng = np.random.default_rng(6)
    q, k, v = (rng.standard_normal((2, 7, 4)) for _ in range(3))
    _, s, p = oracle.causal_gqa_attention(q, k, v, np.arange(7), np.arange(7), return_pattern=True)
    assert np.all(np.isneginf(s[:, np.triu_indices(7, 1)[0], np.triu_indices(7, 1)[1]]))
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-14)


# ---------------------------------------------------------------- activations

def test_relu2_exact_zeros():
    # "arcee": torch.equal(acts, relu(pre) ** 2); zero wherever pre < 0.
    rng = np.random.default_rng(7)
    u = rng.standard_normal(10000)
    a = oracle.relu2(u)
    assert np.all(a[u <= 0] == 0.0)
    assert np.count_nonzero(a == 0.0) == np.count_nonzero(u <= 0)
    np.testing.assert_array_equal(oracle.relu2(np.array([3.0, -2.0, 0.5])), [9.0, 0.0, 0.25])


def test_xielu_page_values():
    g = json.load(open(os.path.join(GOLDEN, "xielu_apertus_block8.json")))
    beta, eps = g["beta"], g["eps"]
    # fit block 8's effective alpha_n from the x = -20 value (expm1(-20) + 20 = 19 to 1e-8)
    x20, y20, _ = g["values"][2]
    alpha_n = (y20 - beta * x20) / (math.expm1(x20) - x20)
    for x, want, dec in g["values"]:
        got = float(oracle.xielu(np.array(x), 1.0, alpha_n, beta, eps))
        assert round(got, dec) == pytest.approx(want, abs=1e-12), (x, got, want)
    xs = np.linspace(-3, 0, 300001)
    ys = oracle.xielu(xs, 1.0, alpha_n, beta, eps)
    i = int(np.argmin(ys))
    assert round(xs[i], g["minimum"]["x_decimals"]) == pytest.approx(g["minimum"]["x"])
    assert round(ys[i], g["minimum"]["value_decimals"]) == pytest.approx(g["minimum"]["value"])
    # far out it grows like (alpha_n - beta) |x|
    slope = (oracle.xielu(np.array(-200.0), 1.0, alpha_n, beta, eps)
             - oracle.xielu(np.array(-100.0), 1.0, alpha_n, beta, eps)) / 100.0
    np.testing.assert_allclose(slope, alpha_n - beta, rtol=1e-12)


def test_xielu_positive_branch_and_joint():
    # x > 0: alpha_p x^2 + beta x; worked: alpha_p = 0.8, x = 2 -> 3.2 + 1.0
    assert float(oracle.xielu(np.array(2.0), 0.8, 0.8)) == pytest.approx(4.2, abs=1e-15)
    # continuous at 0 (both branches tend to 0), x = 0 takes the eps branch
    for a_p, a_n in ((0.8, 0.8), (17.75, 6.28)):
        left = float(oracle.xielu(np.array(-1e-9), a_p, a_n))
        right = float(oracle.xielu(np.array(1e-9), a_p, a_n))
        assert abs(left - right) < 1e-5
    np.testing.assert_allclose(oracle.xielu(np.array(0.0), 0.8, 0.8), 0.8 * math.expm1(-1e-6), rtol=1e-12)


def test_xielu_parameter_transform():
    # "apertus": effective alpha_p = softplus(raw), alpha_n = beta + softplus(raw)
    a_p, a_n = oracle.xielu_effective(0.0, 0.0)
    assert a_p == pytest.approx(math.log(2.0), rel=1e-15)
    assert a_n == pytest.approx(0.5 + math.log(2.0), rel=1e-15)
    a_p, a_n = oracle.xielu_effective(50.0, -50.0)
    assert a_p == pytest.approx(50.0, rel=1e-15)
    assert a_n == pytest.approx(0.5, abs=1e-20)


def test_silu_textbook_properties():
    assert float(oracle.silu(np.array(0.0))) == 0.0
    assert float(oracle.silu(np.array(1.0))) == pytest.approx(0.7310585786300049, rel=1e-15)
    x = np.linspace(-30, 30, 601)
    # silu(x) - silu(-x) = x
    np.testing.assert_allclose(oracle.silu(x) - oracle.silu(-x), x, atol=1e-12)
    # slope 1/2 at the origin; -> x for large x, -> 0 for very negative x
    h = 1e-6
    assert (oracle.silu(np.array(h)) - oracle.silu(np.array(-h))) / (2 * h) == pytest.approx(0.5, rel=1e-9)
    assert float(oracle.silu(np.array(800.0))) == 800.0
    assert abs(float(oracle.silu(np.array(-800.0)))) < 1e-300


# ---------------------------------------------------------------- the block

def _tiny(act, qk_norm=False, H=2, Hkv=1, d=4, D=6, F=5):
    return BlockConfig(hidden_size=D, num_heads=H, num_kv_heads=Hkv, head_dim=d, intermediate_size=F,
                       hidden_act=act, qk_norm=qk_norm, xielu_alpha_p=0.9, xielu_alpha_n=1.3)


def _weights(cfg, rng, gain_std=0.3):
    D, H, Hkv, d, F = cfg.hidden_size, cfg.num_heads, cfg.num_kv_heads, cfg.head_dim, cfg.intermediate_size
    w = {
        "input_layernorm": 1 + gain_std * rng.standard_normal(D),
        "q_proj": 0.4 * rng.standard_normal((H * d, D)),
        "k_proj": 0.4 * rng.standard_normal((Hkv * d, D)),
        "v_proj": 0.4 * rng.standard_normal((Hkv * d, D)),
        "o_proj": 0.4 * rng.standard_normal((D, H * d)),
        "post_attention_layernorm": 1 + gain_std * rng.standard_normal(D),
        "up_proj": 0.4 * rng.standard_normal((F, D)),
        "gate_proj": 0.4 * rng.standard_normal((F, D)),
        "down_proj": 0.4 * rng.standard_normal((D, F)),
        "q_norm": 1 + gain_std * rng.standard_normal(d),
        "k_norm": 1 + gain_std * rng.standard_normal(d),
        # "afmoe": the attention gate and the two sandwich post-norms
        "attn_gate_proj": 0.4 * rng.standard_normal((H * d, D)),
        "post_attn_norm": 1 + gain_std * rng.standard_normal(D),
        "post_mlp_norm": 1 + gain_std * rng.standard_normal(D),
    }
    return w


def _block_loops(cfg, w, x):
    """Pure-Python restatement of one sequence's block, element by element.

    Written from the "LlamaForCausalLM-32L-4096d" pseudo-code with the "arcee" /
    "apertus" MLP variants and q/k norms; RoPE as a complex rotation. The
    "afmoe" options: a window of the last sliding_window keys, no rotary, the
    sigmoid head gate projected from the normed input, and the sandwich
    post-norms of both sublayers.
    """
    T, D = len(x), len(x[0])
    H, Hkv, d, F = cfg.num_heads, cfg.num_kv_heads, cfg.head_dim, cfg.intermediate_size
    eps = cfg.rms_norm_eps
    W = cfg.sliding_window

    def norm(row, g):
        r = 1.0 / math.sqrt(sum(a * a for a in row) / len(row) + eps)
        return [a * r * gg for a, gg in zip(row, g)]

    def lin(row, Wm):
        return [sum(Wm[o][i] * row[i] for i in range(len(row))) for o in range(len(Wm))]

    def rot(a, t):
        return _rope_complex(a, t, cfg.rope_theta) if cfg.use_rope else list(a)

    g1, g2 = list(w["input_layernorm"]), list(w["post_attention_layernorm"])
    Wq, Wk, Wv = (w[n].tolist() for n in ("q_proj", "k_proj", "v_proj"))
    h = [norm(r, g1) for r in x]
    Q, K, V = [], [], []
    for t in range(T):
        q, k, v = lin(h[t], Wq), lin(h[t], Wk), lin(h[t], Wv)
        qh = [q[n * d:(n + 1) * d] for n in range(H)]
        kh = [k[n * d:(n + 1) * d] for n in range(Hkv)]
        vh = [v[n * d:(n + 1) * d] for n in range(Hkv)]
        if cfg.qk_norm:
            qh = [norm(a, list(w["q_norm"])) for a in qh]
            kh = [norm(a, list(w["k_norm"])) for a in kh]
        Q.append([rot(a, t) for a in qh])
        K.append([rot(a, t) for a in kh])
        V.append(vh)
    outs = []
    for t in range(T):
        first = max(0, t - W + 1) if W > 0 else 0  # the last W keys, this one included
        keys = range(first, t + 1)
        heads = []
        for n in range(H):
            j = n // (H // Hkv)
            s = [sum(Q[t][n][c] * K[u][j][c] for c in range(d)) / math.sqrt(d) for u in keys]
            m = max(s)
            e = [math.exp(a - m) for a in s]
            z = sum(e)
            heads += [sum(e[i] / z * V[u][j][c] for i, u in enumerate(keys)) for c in range(d)]
        if cfg.attn_gate:
            gate = lin(h[t], w["attn_gate_proj"].tolist())
            heads = [a / (1.0 + math.exp(-gg)) for a, gg in zip(heads, gate)]
        attn = lin(heads, w["o_proj"].tolist())
        if cfg.sandwich_norm:
            attn = norm(attn, list(w["post_attn_norm"]))
        mid = [a + b for a, b in zip(x[t], attn)]
        h2 = norm(mid, g2)
        up = lin(h2, w["up_proj"].tolist())
        if cfg.hidden_act == "silu":
            gate = lin(h2, w["gate_proj"].tolist())
            neu = [gg / (1.0 + math.exp(-gg)) * uu for gg, uu in zip(gate, up)]
        elif cfg.hidden_act == "relu2":
            neu = [max(uu, 0.0) ** 2 for uu in up]
        else:
            ap, an, b, ep = cfg.xielu_alpha_p, cfg.xielu_alpha_n, cfg.xielu_beta, cfg.xielu_eps
            neu = [ap * uu * uu + b * uu if uu > 0 else an * (math.expm1(min(uu, ep)) - uu) + b * uu
                   for uu in up]
        mlp = lin(neu, w["down_proj"].tolist())
        if cfg.sandwich_norm:
            mlp = norm(mlp, list(w["post_mlp_norm"]))
        outs.append([a + b for a, b in zip(mid, mlp)])
    return outs


@pytest.mark.parametrize("act,qk_norm,H,Hkv", [("silu", False, 2, 2), ("relu2", False, 4, 2),
                                               ("xielu", True, 4, 1), ("silu", True, 2, 1)])
def test_block_brute_force(act, qk_norm, H, Hkv):
    rng = np.random.default_rng(zlib.crc32(f"{act}-{qk_norm}-{H}".encode()))
    cfg = _tiny(act, qk_norm, H=H, Hkv=Hkv)
    w = _weights(cfg, rng)
    x = rng.standard_normal((2, 5, cfg.hidden_size))
    taps = oracle.block_forward(cfg, w, x)
    for b in range(2):
        np.testing.assert_allclose(taps["layer_output"][b], _block_loops(cfg, w, x[b].tolist()),
                                   rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- the afmoe block variant

def _afmoe(window=0, use_rope=True, gate=True, sandwich=True, act="silu", H=4, Hkv=2, eps=1e-5):
    """A tiny "afmoe"-style block: q/k norms, and the options under test."""
    return dataclasses.replace(_tiny(act, True, H=H, Hkv=Hkv), sliding_window=window, use_rope=use_rope,
                               attn_gate=gate, sandwich_norm=sandwich, rms_norm_eps=eps)


@pytest.mark.parametrize("window,use_rope,gate,sandwich", [(3, True, True, True), (0, False, True, True),
                                                          (2, True, False, False), (0, True, True, False),
                                                          (0, True, False, True), (4, False, False, False)])
def test_afmoe_block_brute_force(window, use_rope, gate, sandwich):
    rng = np.random.default_rng(zlib.crc32(f"afmoe-{window}-{use_rope}-{gate}-{sandwich}".encode()))
    cfg = _afmoe(window, use_rope, gate, sandwich)
    w = _weights(cfg, rng)
    x = rng.standard_normal((2, 7, cfg.hidden_size))
    taps = oracle.block_forward(cfg, w, x)
    for b in range(2):
        np.testing.assert_allclose(taps["layer_output"][b], _block_loops(cfg, w, x[b].tolist()),
                                   rtol=1e-11, atol=1e-12)


def test_afmoe_identity_and_post_norm_taps():
    # "afmoe", "The block, in order": layer input + attention_output + mlp_output
    # == layer_output, the contributions being the post-norms' outputs: with unit
    # gains every row of each has mean square m / (m + eps), m the mean square of
    # the tensor entering the norm.
    rng = np.random.default_rng(40)
    cfg = _afmoe(window=3)
    w = _weights(cfg, rng)
    w["post_attn_norm"] = np.ones(cfg.hidden_size)
    w["post_mlp_norm"] = np.ones(cfg.hidden_size)
    x = rng.standard_normal((2, 6, cfg.hidden_size))
    t = oracle.block_forward(cfg, w, x)
    np.testing.assert_allclose(x + t["attention_output"] + t["mlp_output"], t["layer_output"], rtol=0, atol=1e-14)
    raw_attn = t["o_proj_input"] @ w["o_proj"].T
    raw_mlp = t["mlp_neurons"] @ w["down_proj"].T
    for out, raw in ((t["attention_output"], raw_attn), (t["mlp_output"], raw_mlp)):
        m = np.mean(raw * raw, axis=-1)
        np.testing.assert_allclose(np.mean(out * out, axis=-1), m / (m + cfg.rms_norm_eps), rtol=1e-12)


def test_afmoe_sandwich_scale_invariance():
    # "afmoe", "The contributions are the post-norms' outputs": RMSNorm is
    # scale-invariant up to eps, so scaling o_proj or down_proj leaves the stream
    # unchanged; without the post-norms it does not.
    rng = np.random.default_rng(41)
    x = rng.standard_normal((1, 5, 6))
    for sandwich in (True, False):
        cfg = _afmoe(sandwich=sandwich, eps=1e-300)
        w = _weights(cfg, rng)
        base = oracle.block_forward(cfg, w, x)["layer_output"]
        w2 = dict(w, o_proj=7.0 * w["o_proj"], down_proj=0.25 * w["down_proj"])
        scaled = oracle.block_forward(cfg, w2, x)["layer_output"]
        if sandwich:
            np.testing.assert_allclose(scaled, base, rtol=1e-12, atol=1e-13)
        else:
            assert np.max(np.abs(scaled - base)) > 1e-2


def test_afmoe_gate_taps_and_half_gate():
    # "afmoe", "Attention: per-head q/k norms and a sigmoid gate on every head":
    # o_proj's input is heads.flatten(-2) * sigmoid(gate), the gate projected from
    # the attention's input (the normed rows) and attention_head_outputs ungated.
    rng = np.random.default_rng(42)
    cfg = _afmoe(sandwich=False)
    w = _weights(cfg, rng)
    x = rng.standard_normal((2, 5, cfg.hidden_size))
    t = oracle.block_forward(cfg, w, x)
    gate = t["attention_norm_output"] @ w["attn_gate_proj"].T
    np.testing.assert_allclose(t["attention_gate"], gate, rtol=1e-13, atol=1e-14)
    sig = np.vectorize(lambda g: 1.0 / (1.0 + math.exp(-g)))(gate)
    heads = t["attention_head_outputs"].reshape(2, 5, -1)
    np.testing.assert_allclose(t["o_proj_input"], heads * sig, rtol=1e-13, atol=1e-15)
    # zero gate weights: sigmoid(0) = 1/2 halves the attention's contribution
    w0 = dict(w, attn_gate_proj=np.zeros_like(w["attn_gate_proj"]))
    half = oracle.block_forward(cfg, w0, x)["attention_output"]
    ungated = oracle.block_forward(dataclasses.replace(cfg, attn_gate=False), w, x)
    np.testing.assert_allclose(half, 0.5 * ungated["attention_output"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(t["attention_head_outputs"], ungated["attention_head_outputs"], rtol=0, atol=0)


def test_afmoe_whole_prefix_block_queries_are_q_norm_output():
    # "afmoe", "Rotary runs on the sliding-window blocks only": on a full block
    # attention_queries is q_norm's output unchanged, at every position.
    rng = np.random.default_rng(43)
    cfg = _afmoe(use_rope=False)
    w = _weights(cfg, rng)
    x = rng.standard_normal((1, 6, cfg.hidden_size))
    t = oracle.block_forward(cfg, w, x)
    for pos in range(6):
        qn = oracle.rms_norm((t["attention_norm_output"][0, pos] @ w["q_proj"].T).reshape(4, 4), w["q_norm"], 1e-5)
        np.testing.assert_allclose(t["attention_queries"][0, :, pos], qn, rtol=1e-13, atol=1e-15)
    # with the rotary the queries past position 0 differ
    tr = oracle.block_forward(dataclasses.replace(cfg, use_rope=True), w, x)
    assert np.max(np.abs(tr["attention_queries"][0, :, 1:] - t["attention_queries"][0, :, 1:])) > 1e-3


def test_afmoe_window_decode_and_chunk_match_the_prefill():
    # The cache forms of a windowed block (a decode step, a prefill chunk) give
    # the windowed prefill's rows.
    rng = np.random.default_rng(44)
    cfg = _afmoe(window=3)
    w = _weights(cfg, rng)
    B, T = 2, 9
    x = rng.standard_normal((B, T, cfg.hidden_size))
    full = oracle.block_forward(cfg, w, x)
    cap = T + 1
    ck = np.zeros((B, 2, cap, 4))
    cv = np.zeros((B, 2, cap, 4))
    ck[:, :, :T] = full["attention_keys"]
    cv[:, :, :T] = full["attention_values"]
    dec = oracle.decode_step(cfg, w, x[:, T - 1], ck, cv, np.full(B, T - 1))
    np.testing.assert_allclose(dec["layer_output"], full["layer_output"][:, T - 1], rtol=1e-12, atol=1e-13)
    lens = np.array([2, 5])
    ch = oracle.prefill_with_cache(cfg, w, np.stack([x[0, 2:6], x[1, 5:9]]), ck, cv, lens)
    np.testing.assert_allclose(ch["layer_output"][0], full["layer_output"][0, 2:6], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ch["layer_output"][1], full["layer_output"][1, 5:9], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- padded batches

def test_padded_batch_real_rows_equal_the_unpadded_rows():
    # "arcee", "The API": attention_mask [batch seq], zeros are padding. Left, right and
    # two-sided padding: every real row equals the block over the unpadded sequence,
    # for the plain block and for a windowed afmoe block.
    rng = np.random.default_rng(70)
    for cfg in (_tiny("silu", True, H=4, Hkv=2), _afmoe(window=3)):
        w = _weights(cfg, rng)
        T = 9
        x = rng.standard_normal((4, T, cfg.hidden_size))
        runs = [(3, 9), (0, 6), (2, 7), (0, 9)]
        mask = np.zeros((4, T), dtype=np.int32)
        for b, (lo, hi) in enumerate(runs):
            mask[b, lo:hi] = 1
        t = oracle.block_forward(cfg, w, x, attention_mask=mask)
        for b, (lo, hi) in enumerate(runs):
            ref = oracle.block_forward(cfg, w, x[b:b + 1, lo:hi])
            np.testing.assert_allclose(t["layer_output"][b, lo:hi], ref["layer_output"][0], rtol=1e-12, atol=1e-12)
            # the real tokens' rotary positions restart at 0 (the rotary is relative, so only the
            # query/key values, not the output, show the shift)
            np.testing.assert_allclose(t["attention_queries"][b, :, lo:hi], ref["attention_queries"][0], rtol=1e-12,
                                       atol=1e-12)
            np.testing.assert_allclose(t["attention_keys"][b, :, lo:hi], ref["attention_keys"][0], rtol=1e-12,
                                       atol=1e-12)
            # rows before the run see no key: zero head outputs
            np.testing.assert_array_equal(t["attention_head_outputs"][b, :lo], 0.0)
            assert np.all(np.isfinite(t["layer_output"][b]))


def test_padding_run_shapes():
    assert oracle.padding_run([0, 0, 1, 1, 1]) == (2, 5)
    assert oracle.padding_run([1, 1, 0]) == (0, 2)
    assert oracle.padding_run([0, 0, 0]) == (3, 3)
    with pytest.raises(ValueError):
        oracle.padding_run([1, 0, 1])


def test_block_identity_and_taps():
    # "arcee"/"apertus": layer_input + attention_output + mlp_output == layer_output
    rng = np.random.default_rng(8)
    cfg = _tiny("xielu", True, H=4, Hkv=2)
    w = _weights(cfg, rng)
    x = rng.standard_normal((1, 7, cfg.hidden_size))
    t = oracle.block_forward(cfg, w, x)
    np.testing.assert_allclose(x + t["attention_output"] + t["mlp_output"], t["layer_output"], rtol=0, atol=1e-14)
    assert t["attention_queries"].shape == (1, 4, 7, 4)
    assert t["attention_keys"].shape == (1, 2, 7, 4)
    assert t["attention_head_outputs"].shape == (1, 7, 4, 4)
    # "apertus": at position 0 the queries equal q_norm's output
    qn = oracle.rms_norm((t["attention_norm_output"][0, 0] @ w["q_proj"].T).reshape(4, 4), w["q_norm"], 1e-5)
    np.testing.assert_allclose(t["attention_queries"][0, :, 0], qn, rtol=1e-13, atol=1e-15)


def test_block_relu2_neurons_zero_where_pre_negative():
    rng = np.random.default_rng(9)
    cfg = _tiny("relu2", F=64)
    w = _weights(cfg, rng)
    t = oracle.block_forward(cfg, w, rng.standard_normal((1, 6, cfg.hidden_size)))
    pre, acts = t["mlp_up_output"], t["mlp_neurons"]
    assert np.array_equal(acts, np.maximum(pre, 0.0) ** 2)
    assert np.all(acts[pre < 0] == 0.0)


def test_block_qk_norm_scale_invariance():
    # "apertus": scaling one head's slice of q_proj.output is renormalised away.
    # (eps taken tiny so that "up to eps" is sharp)
    rng = np.random.default_rng(10)
    cfg = dataclasses.replace(_tiny("silu", True, H=4, Hkv=2), rms_norm_eps=1e-14)
    w = _weights(cfg, rng)
    x = rng.standard_normal((1, 5, cfg.hidden_size))
    w2 = dict(w)
    w2["q_proj"] = w["q_proj"].copy()
    w2["q_proj"][4:8] *= 3.0  # head 1
    a, b = oracle.block_forward(cfg, w, x), oracle.block_forward(cfg, w2, x)
    np.testing.assert_allclose(a["attention_queries"], b["attention_queries"], rtol=1e-12, atol=1e-13)


def test_block_causal_padding():
    # alpha-er docstring: padding after the prompt cannot influence it (causal).
    rng = np.random.default_rng(11)
    cfg = _tiny("relu2", H=4, Hkv=2)
    w = _weights(cfg, rng)
    x = rng.standard_normal((1, 6, cfg.hidden_size))
    xp = np.concatenate([x, 50.0 * rng.standard_normal((1, 5, cfg.hidden_size))], axis=1)
    a, b = oracle.block_forward(cfg, w, x), oracle.block_forward(cfg, w, xp)
    # exact in real arithmetic; BLAS blocking may differ with the row count
    np.testing.assert_allclose(a["layer_output"], b["layer_output"][:, :6], rtol=1e-13, atol=1e-13)


def test_block_rows_subset_matches_full():
    rng = np.random.default_rng(12)
    cfg = _tiny("silu", True, H=4, Hkv=2)
    w = _weights(cfg, rng)
    x = rng.standard_normal((2, 9, cfg.hidden_size))
    full = oracle.block_forward(cfg, w, x)
    rows = [0, 3, 8]
    sub = oracle.block_forward(cfg, w, x, rows=rows)
    np.testing.assert_allclose(sub["layer_output"], full["layer_output"][:, rows], rtol=1e-13, atol=1e-14)


def test_block_single_token_and_zero_projections():
    rng = np.random.default_rng(13)
    cfg = _tiny("silu", H=2, Hkv=1)
    w = _weights(cfg, rng)
    x = rng.standard_normal((1, 1, cfg.hidden_size))
    t = oracle.block_forward(cfg, w, x)
    # one token: each head's output is its KV head's value row
    v = t["attention_values"][0, 0, 0]
    np.testing.assert_allclose(t["attention_head_outputs"][0, 0], np.stack([v, v]), rtol=1e-14)
    w0 = dict(w, o_proj=np.zeros_like(w["o_proj"]), down_proj=np.zeros_like(w["down_proj"]))
    t0 = oracle.block_forward(cfg, w0, x)
    np.testing.assert_array_equal(t0["layer_mid"], x)
    np.testing.assert_array_equal(t0["layer_output"], x)


def test_decode_equals_last_prefill_row():
    # A decode step over a cache holding the prefill's keys/values is the
    # prefill's last row.
    rng = np.random.default_rng(14)
    cfg = _tiny("xielu", True, H=4, Hkv=2)
    w = _weights(cfg, rng)
    B, T = 3, 8
    x = rng.standard_normal((B, T, cfg.hidden_size))
    full = oracle.block_forward(cfg, w, x)
    cap = T + 2
    ck = np.zeros((B, 2, cap, 4))
    cv = np.zeros((B, 2, cap, 4))
    ck[:, :, : T - 1] = full["attention_keys"][:, :, : T - 1]
    cv[:, :, : T - 1] = full["attention_values"][:, :, : T - 1]
    dec = oracle.decode_step(cfg, w, x[:, T - 1], ck, cv, np.full(B, T - 1))
    np.testing.assert_allclose(dec["layer_output"], full["layer_output"][:, T - 1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dec["new_key"], full["attention_keys"][:, :, T - 1], rtol=1e-12, atol=1e-14)
    # per-sequence lengths differ: sequence b uses only its own prefix
    lens = np.array([2, 5, 7])
    dec = oracle.decode_step(cfg, w, x[np.arange(B), lens], ck, cv, lens)
    for b in range(B):
        fb = oracle.block_forward(cfg, w, x[b:b + 1, : lens[b] + 1])
        np.testing.assert_allclose(dec["layer_output"][b], fb["layer_output"][0, -1], rtol=1e-12, atol=1e-13)


def test_prefill_chunk_equals_the_full_prefill_rows():
    # A prefill chunk over a cache that holds the keys/values of the sequence's
    # earlier tokens gives the full prefill's rows for the chunk's tokens.
    rng = np.random.default_rng(15)
    cfg = _tiny("silu", True, H=4, Hkv=2)
    w = _weights(cfg, rng)
    B, T, cap = 3, 5, 16
    lens = np.array([0, 3, 9])
    xs = rng.standard_normal((B, cap, cfg.hidden_size))
    ck = np.zeros((B, 2, cap, 4))
    cv = np.zeros((B, 2, cap, 4))
    fulls = []
    for b in range(B):
        fb = oracle.block_forward(cfg, w, xs[b:b + 1, : lens[b] + T])
        fulls.append(fb)
        ck[b, :, : lens[b]] = fb["attention_keys"][0, :, : lens[b]]
        cv[b, :, : lens[b]] = fb["attention_values"][0, :, : lens[b]]
    x = np.stack([xs[b, lens[b]: lens[b] + T] for b in range(B)])
    ch = oracle.prefill_with_cache(cfg, w, x, ck, cv, lens)
    for b in range(B):
        rows = slice(lens[b], lens[b] + T)
        np.testing.assert_allclose(ch["layer_output"][b], fulls[b]["layer_output"][0, rows], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(ch["new_keys"][b], fulls[b]["attention_keys"][0, :, rows], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(ch["new_values"][b], fulls[b]["attention_values"][0, :, rows], rtol=1e-12,
                                   atol=1e-14)


def test_prefill_chunk_of_one_token_is_a_decode_step():
    rng = np.random.default_rng(16)
    cfg = _tiny("xielu", False, H=2, Hkv=1)
    w = _weights(cfg, rng)
    B, cap = 2, 7
    lens = np.array([4, 1])
    ck = rng.standard_normal((B, 1, cap, 4))
    cv = rng.standard_normal((B, 1, cap, 4))
    x = rng.standard_normal((B, 1, cfg.hidden_size))
    ch = oracle.prefill_with_cache(cfg, w, x, ck, cv, lens)
    dec = oracle.decode_step(cfg, w, x[:, 0], ck, cv, lens)
    np.testing.assert_allclose(ch["layer_output"][:, 0], dec["layer_output"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(ch["new_keys"][:, :, 0], dec["new_key"], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- stretched rotary

LLAMA3_APERTUS = oracle.RopeScaling("llama3", 8.0, 8192, 1.0, 4.0)  # "apertus": factor 8 over 8192, theta 12M
YARN_ARCEE = oracle.RopeScaling("yarn", 20.0, 4096, 1.0, 32.0)  # "arcee": factor 20 over 4096, theta 10000


def test_rope_scaling_of_factor_one_is_the_plain_rotary():
    for kind, lo, hi in (("llama3", 1.0, 4.0), ("yarn", 1.0, 32.0)):
        sc = oracle.RopeScaling(kind, 1.0, 4096, lo, hi)
        np.testing.assert_allclose(oracle.rope_inv_freq(128, 10000.0, sc), oracle.rope_inv_freq(128, 10000.0),
                                   rtol=4e-16)  # the blend of f and f / 1 rounds once
        assert oracle.rope_attention_factor(sc) == 1.0


def _regimes(theta, sc):
    base = oracle.rope_inv_freq(128, theta)
    lam = 2 * np.pi / base
    return base, lam, oracle.rope_inv_freq(128, theta, sc)


def test_llama3_scaling_keeps_fast_divides_slow_and_blends_between():
    base, lam, f = _regimes(12_000_000.0, LLAMA3_APERTUS)
    fast, slow = lam < 8192 / 4.0, lam > 8192 / 1.0
    mid = ~fast & ~slow
    assert fast.sum() > 0 and slow.sum() > 0 and mid.sum() > 0
    np.testing.assert_array_equal(f[fast], base[fast])
    np.testing.assert_allclose(f[slow], base[slow] / 8.0, rtol=1e-15)
    assert np.all(f[mid] < base[mid]) and np.all(f[mid] > base[mid] / 8.0)
    assert np.all(np.diff(f) < 0)  # still strictly decreasing with the dimension


def _golden_rope_cases():
    with open(os.path.join(GOLDEN, "rope_scaling.json")) as fh:
        return json.load(fh)["cases"]


def test_rope_scaling_golden_values():
    # hand-derived inverse frequencies of both published rules (tests/golden/rope_scaling.json):
    # two small settings whose blend weights are exact fractions, YaRN at the "arcee"
    # setting (pair indices 20 .. 46 of 64, from its floored and ceiled correction
    # indices 20.94 and 45.03), and the llama3 band at the "apertus" setting
    for c in _golden_rope_cases():
        L = c["original_positions"] if "original_positions" in c else 2 * np.pi * c["original_positions_over_2pi"]
        sc = oracle.RopeScaling(c["kind"], c["factor"], L, c["low"], c["high"])
        d, theta = c["head_dim"], c["theta"]
        got = oracle.rope_inv_freq(d, theta, sc)
        if "multiplier_of_f" in c:
            idx = c.get("indices", list(range(d // 2)))
            for i, frac in zip(idx, c["multiplier_of_f"]):
                want = float(Fraction(frac)) * theta ** (-2.0 * i / d)
                assert abs(got[i] - want) <= 1e-14 * want, (c["name"], i, got[i], want)
        else:
            plain = theta ** (-2.0 * np.arange(d // 2) / d)
            lo, hi = c["kept_below"], c["divided_from"]
            np.testing.assert_array_equal(got[:lo], plain[:lo])
            np.testing.assert_allclose(got[hi:], plain[hi:] / c["factor"], rtol=1e-15)
            assert np.all(got[lo:hi] < plain[lo:hi] * (1 - 1e-12))
            assert np.all(got[lo:hi] > plain[lo:hi] / c["factor"] * (1 + 1e-12))


def test_yarn_scaling_keeps_fast_divides_slow_and_scales_attention():
    base, lam, f = _regimes(10000.0, YARN_ARCEE)
    turns = 4096 / lam
    fast, slow = turns > 32.0, turns < 1.0
    mid = ~fast & ~slow
    assert fast.sum() > 0 and slow.sum() > 0 and mid.sum() > 0
    np.testing.assert_array_equal(f[fast], base[fast])
    np.testing.assert_allclose(f[slow], base[slow] / 20.0, rtol=1e-15)
    assert np.all(f[mid] < base[mid]) and np.all(f[mid] > base[mid] / 20.0)
    assert abs(oracle.rope_attention_factor(YARN_ARCEE) - (1.0 + 0.1 * np.log(20.0))) < 1e-15
    # the factor multiplies the rotated vector: its norm grows by exactly that much
    x = np.random.default_rng(17).standard_normal((3, 5, 128))
    y = oracle.rope(x, np.arange(5) * 1000, 10000.0, YARN_ARCEE)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1) * (1 + 0.1 * np.log(20.0)),
                               rtol=1e-13)


def test_model_with_identity_blocks_and_tied_embeddings_reads_its_own_token():
    # Blocks whose o_proj and down_proj are zero pass the stream through unchanged, so
    # the logits are rmsnorm(e_t) . e_v; with tied, nearly orthogonal embeddings the
    # largest is the token's own id, and its value is |e_t| sqrt(D) exactly.
    rng = np.random.default_rng(18)
    cfg = _tiny("relu2", False, H=2, Hkv=1, d=4, D=64, F=5)
    V, D = 40, 64
    embed = rng.standard_normal((V, D))
    layers = []
    for _ in range(2):
        w = _weights(cfg, rng)
        w["o_proj"] = np.zeros_like(w["o_proj"])
        w["down_proj"] = np.zeros_like(w["down_proj"])
        layers.append(w)
    tokens = rng.integers(0, V, size=(2, 7))
    logits = oracle.model_forward(cfg, layers, embed, np.ones(D), embed, tokens)
    assert logits.shape == (2, 7, V)
    np.testing.assert_array_equal(logits.argmax(-1), tokens)
    e = embed[tokens]
    want = np.sqrt((e * e).sum(-1)) * np.sqrt(D) / np.sqrt(1 + cfg.rms_norm_eps / np.mean(e * e, -1))
    np.testing.assert_allclose(np.take_along_axis(logits, tokens[..., None], -1)[..., 0], want, rtol=1e-12)
    # and one real layer is block_forward's output, normed and projected
    out1 = oracle.block_forward(cfg, layers[0], e)["layer_output"]
    np.testing.assert_allclose(out1, e, rtol=0, atol=0)
