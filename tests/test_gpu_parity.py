"""GPU parity of the CUDA path against the fp64 oracle, on seeded inputs at sizes
the oracle finishes in seconds (several tiles plus ragged tails), through the
C ABI. Bounds: max|err| / RMS(oracle) <= 1e-4 (fp32 path), <= 2e-2 (bf16 path).
"""
import numpy as np
import pytest
import torch

import oracle
from llama_family_decoder_gb300 import DecoderBlock, rmsnorm
from llama_family_decoder_gb300.synth import WORKLOADS, Workload, make_input, make_kv_cache, make_weights
from tests.helpers import TOL, bf16_floor, cfg_of, check_relu2_zeros, np64, rel_err, to_dev, weights_np

pytestmark = pytest.mark.gpu

DEV = "cuda"

SMALL_BF16 = [
    # several 128-row tiles with a ragged tail; ffn not a multiple of 64/128 (K and N tails)
    Workload("small_swiglu_mha", "bf16", 2, 200, 512, 4, 4, 128, 1000, "silu", seed=11),
    Workload("small_relu2_gqa", "bf16", 1, 320, 1024, 8, 2, 128, 1536, "relu2", seed=12),
    Workload("small_xielu_qknorm", "bf16", 3, 130, 512, 4, 1, 128, 776, "xielu", qk_norm=True, seed=13),
    Workload("small_swiglu_gqa_qknorm", "bf16", 1, 64, 256, 4, 2, 128, 512, "silu", qk_norm=True, seed=14),
    # hidden not a multiple of 32: the o_proj's last N tile and its last 32-column output box are ragged
    Workload("small_relu2_odd_hidden", "bf16", 2, 150, 1000, 4, 2, 128, 1000, "relu2", seed=16),
    # enough tiles x k-blocks that every GEMM splits tiles across CTAs (stream-K)
    Workload("medium_streamk_swiglu", "bf16", 2, 600, 2048, 16, 4, 128, 2000, "silu", seed=15),
]

TAPS = ["attention_queries", "attention_keys", "attention_values", "attention_head_outputs", "attention_output",
        "layer_mid", "mlp_neurons", "mlp_output"]


def _tap_buffers(wl, dt):
    B, T, D, H, Hkv, d, F = wl.batch, wl.seq, wl.hidden_size, wl.num_heads, wl.num_kv_heads, wl.head_dim, \
        wl.intermediate_size
    shapes = {"attention_queries": (B, H, T, d), "attention_keys": (B, Hkv, T, d),
              "attention_values": (B, Hkv, T, d), "attention_head_outputs": (B, T, H, d),
              "attention_output": (B, T, D), "layer_mid": (B, T, D), "mlp_neurons": (B, T, F),
              "mlp_output": (B, T, D)}
    return {k: torch.empty(s, dtype=dt, device=DEV) for k, s in shapes.items()}


def _run(wl, gain_std=0.0, taps=False, prepared=False):
    w = make_weights(wl, gain_std=gain_std)
    x = make_input(wl)
    blk = DecoderBlock.from_workload(wl)
    xd = x.to(DEV)
    tb = _tap_buffers(wl, xd.dtype) if taps else None
    wd = to_dev(w)
    if prepared:
        wd = blk.prepare(wd)
    out = blk.forward(xd, wd, taps=tb)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    ref = oracle.block_forward(cfg_of(wl), weights_np(w), np64(x))
    return out, tb, ref, x


# ------------------------------------------------------------------ RMSNorm stage

@pytest.mark.parametrize("n", [4096, 1000, 12288])  # 128 threads x 4 chunks, a ragged chunk count, 256 threads
@pytest.mark.parametrize("dt,tol", [(torch.float32, 1e-6), (torch.bfloat16, None)])
def test_rmsnorm_stage(dt, tol, n):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(37, n, generator=g)
    x[3] *= 1e4  # a sink-like row
    gain = 1 + 0.1 * torch.randn(n, generator=g)
    x, gain = x.to(dt), gain.to(dt)
    y = rmsnorm(x.to(DEV), gain.to(DEV), 1e-5)
    torch.cuda.synchronize()
    ref = oracle.rms_norm(np64(x), np64(gain), 1e-5)
    assert np.all(np.isfinite(np64(y)))
    if tol is None:  # bf16 output: within the error of storing the exact result in bf16
        tol = bf16_floor(ref) * 1.01 + 1e-5
    assert rel_err(y, ref) <= tol


# ------------------------------------------------------------------ fp32 path

@pytest.mark.parametrize("gain_std", [0.0, 0.1])
def test_tiny_f32_block(gain_std):
    wl = WORKLOADS["tiny_f32_T64_D256"]
    out, tb, ref, x = _run(wl, gain_std, taps=True)
    errs = {name: rel_err(tb[name], ref[name]) for name in TAPS}
    assert rel_err(out, ref["layer_output"]) <= TOL["f32"], errs
    assert all(e <= TOL["f32"] * 10 for e in errs.values()), errs
    # the block identity holds exactly (each contribution rounded, then added)
    xd = x.to(DEV)
    assert torch.equal(xd + tb["attention_output"] + tb["mlp_output"], out)


# ------------------------------------------------------------------ bf16 prefill

@pytest.mark.parametrize("prepared", [False, True], ids=["bf16_weights", "prepared_fp16"])
@pytest.mark.parametrize("wl", SMALL_BF16, ids=lambda w: w.name)
def test_bf16_block_small(wl, prepared):
    out, tb, ref, x = _run(wl, gain_std=0.1 if wl.qk_norm else 0.0, taps=True, prepared=prepared)
    err = rel_err(out, ref["layer_output"])
    floor = bf16_floor(ref["layer_output"])
    print(f"{wl.name}: layer_output {err:.4f} (bf16 storage floor {floor:.4f})")
    assert err <= TOL["bf16"], (err, floor)
    # intermediate taps: each within the tolerance or 1.5x its own bf16 storage floor
    # (max|err|/RMS of a tap whose RMS is far below its max, e.g. head outputs that
    # average many values, is dominated by the rounding of its largest entries)
    for name in TAPS:
        e, f = rel_err(tb[name], ref[name]), bf16_floor(ref[name])
        print(f"  {name}: {e:.4f} (floor {f:.4f})")
        assert e <= max(TOL["bf16"], 2.0 * f + 5e-3), (name, e, f)
    # "arcee"/"apertus" identity: layer_input + attention_output + mlp_output == layer_output;
    # the bf16 taps are rounded contributions of an fp32 residual stream, so it
    # holds to the rounding of the stored values
    ident = np64(x) + np64(tb["attention_output"]) + np64(tb["mlp_output"])
    assert rel_err(out, ident) <= TOL["bf16"]
    if wl.hidden_act == "relu2":
        zeros, du = check_relu2_zeros(tb["mlp_neurons"], ref["mlp_up_output"])
        print(f"  relu2: {zeros:.3f} exact zeros, pre-activation max|du|/RMS {du:.4f}")


def test_bf16_padding_after_prompt_is_invisible():
    # alpha-er docstring: padding after the prompt cannot influence it (causal).
    wl = SMALL_BF16[1]
    w = to_dev(make_weights(wl))
    x = make_input(wl).to(DEV)
    pad = torch.randn(1, 64, wl.hidden_size, generator=torch.Generator().manual_seed(3)).to(x.dtype).to(DEV) * 30
    blk = DecoderBlock.from_workload(wl, max_seq=wl.seq + 64)
    a = blk.forward(x, w)
    b = blk.forward(torch.cat([x, pad], dim=1), w)
    torch.cuda.synchronize()
    assert torch.equal(a, b[:, : wl.seq])


# ------------------------------------------------------------------ stages

@pytest.mark.parametrize("wl", [SMALL_BF16[2], WORKLOADS["tiny_f32_T64_D256"]], ids=lambda w: w.name)
def test_stage_qkv_attn_mlp(wl):
    w = make_weights(wl, gain_std=0.1)
    x = make_input(wl)
    cfg = cfg_of(wl)
    ref = oracle.block_forward(cfg, weights_np(w), np64(x))
    blk = DecoderBlock.from_workload(wl)
    wd = to_dev(w)
    dt = x.dtype
    B, T, H, Hkv, d = wl.batch, wl.seq, wl.num_heads, wl.num_kv_heads, wl.head_dim
    y = rmsnorm(x.to(DEV), wd["input_layernorm"], wl.rms_norm_eps)
    q = torch.empty(B, H, T, d, dtype=dt, device=DEV)
    k = torch.empty(B, Hkv, T, d, dtype=dt, device=DEV)
    v = torch.empty(B, Hkv, T, d, dtype=dt, device=DEV)
    blk.qkv_rope(y, wd, B, T, q, k, v)
    o = torch.empty(B, T, H, d, dtype=dt, device=DEV)
    blk.attn_gqa(q, k, v, o)
    # MLP stage on the oracle's own layer_mid / mlp_norm_output (cast to the storage type)
    mid = torch.from_numpy(ref["layer_mid"]).to(dt).to(DEV)
    h2 = torch.from_numpy(ref["mlp_norm_output"]).to(dt).to(DEV)
    out = torch.empty_like(mid)
    blk.mlp(mid, h2, wd, out)
    torch.cuda.synchronize()
    tol = TOL[wl.dtype] * (10 if wl.dtype == "f32" else 1)
    assert rel_err(q, ref["attention_queries"]) <= tol
    assert rel_err(k, ref["attention_keys"]) <= tol
    assert rel_err(v, ref["attention_values"]) <= tol
    # attention stage alone: the oracle's attention over the GPU's own q/k/v
    o_ref = np.stack([oracle.causal_gqa_attention(np64(q[b]), np64(k[b]), np64(v[b]), np.arange(T), np.arange(T))
                      for b in range(B)]).transpose(0, 2, 1, 3)
    f = bf16_floor(o_ref) if wl.dtype == "bf16" else 0.0
    print(f"attention stage: {rel_err(o, o_ref):.4f} (bf16 storage floor {f:.4f})")
    assert rel_err(o, o_ref) <= max(tol, 1.5 * f + 2e-3)
    # MLP stage alone: the oracle's MLP on the same (storage-rounded) inputs
    out_ref = np64(mid) + oracle.mlp(cfg, weights_np(w), np64(h2))["mlp_output"]
    f = bf16_floor(out_ref) if wl.dtype == "bf16" else 0.0
    print(f"mlp stage: {rel_err(out, out_ref):.4f} (bf16 storage floor {f:.4f})")
    assert rel_err(out, out_ref) <= max(tol, 1.5 * f + 2e-3)


# ------------------------------------------------------------------ decode

def _decode_case(wl, lens):
    w = make_weights(wl, gain_std=0.1 if wl.qk_norm else 0.0)
    x = make_input(wl)[:, 0]  # [B, D]
    cap = int(max(lens)) + 9
    kc, vc = make_kv_cache(wl.scaled(cache_len=int(max(lens))), capacity=cap)
    for b, L in enumerate(lens):  # only the first lens[b] slots are in use
        kc[b, :, L:] = 0
        vc[b, :, L:] = 0
    return w, x, kc, vc


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_step_small(dtype):
    if dtype == "bf16":
        wl = Workload("small_decode", "bf16", 5, 1, 512, 8, 2, 128, 1000, "silu", seed=21)
    else:
        wl = Workload("small_decode_f32", "f32", 3, 1, 256, 4, 2, 64, 512, "xielu", qk_norm=True, seed=22)
    lens = [17, 200, 63, 64, 1][: wl.batch]
    w, x, kc, vc = _decode_case(wl, lens)
    blk = DecoderBlock.from_workload(wl, max_seq=kc.shape[2] + 1)
    kd, vd = kc.to(DEV), vc.to(DEV)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = blk.forward(x[:, None].to(DEV), to_dev(w), cache={"k": kd, "v": vd, "lens": lens_d},
                      host_lens_max=max(lens))
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    ref = oracle.decode_step(cfg_of(wl), weights_np(w), np64(x), np64(kc), np64(vc), np.array(lens))
    tol = TOL[wl.dtype]
    assert rel_err(out[:, 0], ref["layer_output"]) <= tol
    assert lens_d.tolist() == [L + 1 for L in lens]
    for b, L in enumerate(lens):  # the new key/value landed in slot lens[b]
        assert rel_err(kd[b, :, L], ref["new_key"][b]) <= tol
        assert rel_err(vd[b, :, L], ref["new_value"][b]) <= tol
        assert torch.equal(kd[b, :, :L].cpu(), kc[b, :, :L])


@pytest.mark.parametrize("prepared", [False, True], ids=["bf16_weights", "prepared_fp16"])
@pytest.mark.parametrize("act,qk_norm,batch,ffn", [("relu2", False, 7, 1000), ("xielu", True, 3, 1024),
                                                   ("silu", True, 70, 968), ("silu", False, 5, 968)])
def test_decode_step_bf16_variants_and_taps(act, qk_norm, batch, ffn, prepared):
    # every activation, q/k-norm with non-unit gains, a token tile wider than 64
    # (the MLP-up GEMM then leaves the activation to a post kernel), ragged MLP
    # tiles (968 = 15 paired tiles of 64 and 8 features), and the per-stage taps
    # of the decode path (fp16 operands with prepared weights)
    wl = Workload(f"decode_{act}", "bf16", batch, 1, 512, 8, 2, 128, ffn, act, qk_norm=qk_norm, seed=25)
    lens = [(37 * b + 11) % 190 + 1 for b in range(batch)]
    w, x, kc, vc = _decode_case(wl, lens)
    blk = DecoderBlock.from_workload(wl, max_seq=kc.shape[2] + 1)
    kd, vd = kc.to(DEV), vc.to(DEV)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    tb = _tap_buffers(wl, torch.bfloat16)
    wd = to_dev(w)
    if prepared:
        wd = blk.prepare(wd)
    out = blk.forward(x[:, None].to(DEV), wd, cache={"k": kd, "v": vd, "lens": lens_d},
                      host_lens_max=max(lens), taps=tb)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    ref = oracle.decode_step(cfg_of(wl), weights_np(w), np64(x), np64(kc), np64(vc), np.array(lens))
    assert rel_err(out[:, 0], ref["layer_output"]) <= TOL["bf16"]
    assert lens_d.tolist() == [L + 1 for L in lens]
    idx = torch.arange(batch)
    got_k = kd[idx, :, torch.tensor(lens)]  # [B, Hkv, d]
    got_v = vd[idx, :, torch.tensor(lens)]
    assert rel_err(got_k, ref["new_key"]) <= TOL["bf16"]
    assert rel_err(got_v, ref["new_value"]) <= TOL["bf16"]
    for name, key, sl in [("attention_queries", "attention_queries", lambda t: t[:, :, 0]),
                          ("attention_output", "attention_output", lambda t: t[:, 0]),
                          ("attention_head_outputs", "attention_head_outputs", lambda t: t[:, 0]),
                          ("layer_mid", "layer_mid", lambda t: t[:, 0]),
                          ("mlp_neurons", "mlp_neurons", lambda t: t[:, 0]),
                          ("mlp_output", "mlp_output", lambda t: t[:, 0])]:
        r = ref[key]
        err, floor = rel_err(sl(tb[name]), r), bf16_floor(r)
        print(f"decode {act} tap {name}: {err:.4f} (floor {floor:.4f})")
        assert err <= max(TOL["bf16"], 2 * floor + 5e-3), (name, err, floor)


@pytest.mark.parametrize("act,qk_norm,prepared", [("silu", False, False), ("xielu", True, False),
                                                  ("silu", False, True)])
def test_prefill_chunk_over_the_cache(act, qk_norm, prepared):
    # T new tokens per sequence after ragged cached lengths: one chunk within a tile, one across
    # tiles, one from an empty cache. Unused cache slots hold NaN: nothing of them may leak.
    wl = Workload(f"chunk_{act}", "bf16", 3, 150, 512, 8, 2, 128, 1000, act, qk_norm=qk_norm, seed=26)
    lens = [0, 37, 200]
    cap = 400
    w = make_weights(wl, gain_std=0.1 if qk_norm else 0.0)
    x = make_input(wl)
    g = torch.Generator().manual_seed(27)
    kc = torch.full((wl.batch, wl.num_kv_heads, cap, wl.head_dim), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    for b, L in enumerate(lens):
        kc[b, :, :L] = torch.randn(wl.num_kv_heads, L, wl.head_dim, generator=g).to(torch.bfloat16)
        vc[b, :, :L] = torch.randn(wl.num_kv_heads, L, wl.head_dim, generator=g).to(torch.bfloat16)
    blk = DecoderBlock.from_workload(wl, max_seq=cap + 1)
    wd = to_dev(w)
    if prepared:
        wd = blk.prepare(wd)
    kd, vd = kc.to(DEV), vc.to(DEV)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    tb = _tap_buffers(wl, torch.bfloat16)
    tb.pop("attention_keys")
    tb.pop("attention_values")
    out = blk.forward(x.to(DEV), wd, cache={"k": kd, "v": vd, "lens": lens_d}, host_lens_max=max(lens), taps=tb)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    ref = oracle.prefill_with_cache(cfg_of(wl), weights_np(w), np64(x), np64(kc), np64(vc), np.array(lens))
    err, floor = rel_err(out, ref["layer_output"]), bf16_floor(ref["layer_output"])
    print(f"chunk {act}: max|err|/RMS {err:.4f} (bf16 floor {floor:.4f})")
    assert err <= TOL["bf16"]
    assert lens_d.tolist() == [L + wl.seq for L in lens]
    T = wl.seq
    kd_c, vd_c = kd.cpu(), vd.cpu()
    for b, L in enumerate(lens):
        assert rel_err(kd_c[b, :, L:L + T], ref["new_keys"][b]) <= TOL["bf16"]
        assert rel_err(vd_c[b, :, L:L + T], ref["new_values"][b]) <= TOL["bf16"]
        assert torch.equal(kd_c[b, :, :L], kc[b, :, :L])  # the cached prefix is untouched
        assert torch.isnan(kd_c[b, :, L + T:].float()).all()  # nothing written past the chunk
    for name in ("attention_output", "layer_mid", "mlp_neurons", "mlp_output"):
        r = ref[name]
        e2, f2 = rel_err(tb[name], r), bf16_floor(r)
        assert e2 <= max(TOL["bf16"], 2 * f2 + 5e-3), (name, e2, f2)
    assert rel_err(tb["attention_queries"], ref["attention_queries"]) <= TOL["bf16"]


def test_prefill_chunk_needs_the_host_lengths():
    wl = Workload("chunk_refused", "bf16", 1, 4, 512, 8, 2, 128, 1000, "silu", seed=28)
    blk = DecoderBlock.from_workload(wl, max_seq=64)
    kd = torch.zeros(1, 2, 32, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(RuntimeError):
        blk.forward(make_input(wl).to(DEV), to_dev(make_weights(wl)),
                    cache={"k": kd, "v": kd.clone(), "lens": torch.zeros(1, dtype=torch.int32, device=DEV)})


YARN_ARCEE = ("yarn", 20.0, 4096, 1.0, 32.0)          # "arcee": YaRN, factor 20 over 4096, theta 10000
LLAMA3_APERTUS = ("llama3", 8.0, 8192, 1.0, 4.0)      # "apertus": llama3, factor 8 over 8192, theta 12M


@pytest.mark.parametrize("scaling,theta,qk_norm", [(YARN_ARCEE, 10000.0, True), (LLAMA3_APERTUS, 12_000_000.0, False)])
def test_stretched_rotary_prefill_and_decode(scaling, theta, qk_norm):
    wl = Workload(f"rope_{scaling[0]}", "bf16", 2, 256, 512, 8, 2, 128, 1000, "silu", qk_norm=qk_norm, seed=29,
                  rope_theta=theta, rope_scaling=scaling)
    w = make_weights(wl, gain_std=0.1 if qk_norm else 0.0)
    x = make_input(wl)
    blk = DecoderBlock.from_workload(wl, max_seq=600)
    wd = to_dev(w)
    out = blk.forward(x.to(DEV), wd)
    torch.cuda.synchronize()
    ref = oracle.block_forward(cfg_of(wl), weights_np(w), np64(x))
    assert rel_err(out, ref["layer_output"]) <= TOL["bf16"]
    # a decode step at positions past the prefill's, over a random cache
    lens = [300, 517]
    dw = wl.scaled(batch=2, seq=1)
    kc, vc = make_kv_cache(dw.scaled(cache_len=max(lens)), capacity=max(lens) + 8)
    xd = make_input(dw)[:, 0]
    kd, vd = kc.to(DEV), vc.to(DEV)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o1 = blk.forward(xd[:, None].to(DEV), wd, cache={"k": kd, "v": vd, "lens": lens_d}, host_lens_max=max(lens))
    torch.cuda.synchronize()
    r1 = oracle.decode_step(cfg_of(dw), weights_np(w), np64(xd), np64(kc), np64(vc), np.array(lens))
    assert rel_err(o1[:, 0], r1["layer_output"]) <= TOL["bf16"]
    assert rel_err(kd[[0, 1], :, lens].cpu(), r1["new_key"]) <= TOL["bf16"]


def test_decode_matches_prefill_last_row():
    wl = Workload("small_prefill_decode", "bf16", 2, 96, 512, 4, 2, 128, 1000, "silu", seed=23)
    w = to_dev(make_weights(wl))
    x = make_input(wl).to(DEV)
    blk = DecoderBlock.from_workload(wl, max_seq=128)
    B, T, Hkv, d = wl.batch, wl.seq, wl.num_kv_heads, wl.head_dim
    tb = _tap_buffers(wl, x.dtype)
    full = blk.forward(x, w, taps=tb)
    cap = T + 4
    kc = torch.zeros(B, Hkv, cap, d, dtype=x.dtype, device=DEV)
    vc = torch.zeros_like(kc)
    kc[:, :, : T - 1] = tb["attention_keys"][:, :, : T - 1]
    vc[:, :, : T - 1] = tb["attention_values"][:, :, : T - 1]
    lens = torch.full((B,), T - 1, dtype=torch.int32, device=DEV)
    dec = blk.forward(x[:, T - 1: T].contiguous(), w, cache={"k": kc, "v": vc, "lens": lens}, host_lens_max=T - 1)
    torch.cuda.synchronize()
    assert rel_err(dec[:, 0], np64(full[:, T - 1])) <= TOL["bf16"]
    assert rel_err(kc[:, :, T - 1], np64(tb["attention_keys"][:, :, T - 1])) <= TOL["bf16"]


# ------------------------------------------------------------------ recorded forward (CUDA graph)

def test_forward_graph_replay_matches_direct_call():
    wl = SMALL_BF16[1]
    w = to_dev(make_weights(wl))
    x = make_input(wl).to(DEV)
    blk = DecoderBlock.from_workload(wl)
    direct = blk.forward(x, w)
    out = torch.empty_like(x)
    ws = torch.empty(blk.workspace_bytes(wl.batch, wl.seq), dtype=torch.uint8, device=DEV)
    g = blk.forward_graph(x, w, out, ws)
    g.launch()
    torch.cuda.synchronize()
    assert torch.equal(out, direct)
    x.mul_(0.5)  # inputs are refreshed in place between replays
    g.launch()
    direct2 = blk.forward(x, w)
    torch.cuda.synchronize()
    assert torch.equal(out, direct2)
    g.close()


def test_forward_graph_decode_bumps_lens_each_replay():
    wl = Workload("graph_decode", "bf16", 4, 1, 512, 8, 2, 128, 1000, "silu", seed=24)
    lens = [5, 9, 60, 33]
    w, x, kc, vc = _decode_case(wl, lens)
    blk = DecoderBlock.from_workload(wl, max_seq=kc.shape[2] + 4)
    kd, vd = kc.to(DEV), vc.to(DEV)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    cache = {"k": kd, "v": vd, "lens": lens_d}
    xd = x[:, None].to(DEV).contiguous()
    out = torch.empty_like(xd)
    ws = torch.empty(blk.workspace_bytes(wl.batch, 1, True), dtype=torch.uint8, device=DEV)
    g = blk.forward_graph(xd, to_dev(w), out, ws, cache=cache, host_lens_max=max(lens) + 1)
    g.launch()
    g.launch()
    torch.cuda.synchronize()
    assert lens_d.tolist() == [L + 2 for L in lens]
    ref = oracle.decode_step(cfg_of(wl), weights_np(w), np64(x), np64(kd.cpu()), np64(vd.cpu()),
                             np.array([L + 1 for L in lens]))
    # the second replay decoded the same token at position lens + 1
    assert rel_err(out[:, 0], ref["layer_output"]) <= TOL["bf16"]
    g.close()


def test_prepare_rejects_weights_outside_fp16():
    from llama_family_decoder_gb300 import BlkError
    wl = SMALL_BF16[0]
    w = to_dev(make_weights(wl))
    w["up_proj"][3, 7] = 1e5  # beyond fp16's 65504
    blk = DecoderBlock.from_workload(wl)
    with pytest.raises(BlkError, match="fp16 range"):
        blk.prepare(w)
