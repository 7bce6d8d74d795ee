"""GPU parity of the "afmoe" block variant (dense MLP) against the fp64 oracle:
a sliding window over the last W positions, no rotary on whole-prefix blocks, a
sigmoid gate on every head's channels before o_proj, and the sandwich post-norms
("afmoe", "The block, in order"; "Attention: per-head q/k norms and a sigmoid
gate on every head"; "Rotary runs on the sliding-window blocks only").

Prefill, prefill chunks over a KV cache, decode steps (fused and unfused QKV
finishers), the fp32 path and the attention stage, at sizes the oracle finishes in
seconds (several tiles and ragged tails, windows shorter and longer than a key
tile, windows reaching into the cache), plus the full-size workloads checked on
sampled rows. Bounds: max|err| / RMS(oracle) <= 2e-2 on the bf16 path, 1e-4 on
the fp32 path, for every case.

With bf16 weights left unprepared, every GEMM operand that meets a weight is bf16
(one operand type per tensor-core product), so each sublayer's output carries a
relative error of order 2^-9; the sandwich post-norms rescale that output to the
size of the residual stream, which would spend the whole bf16 tolerance there.
The library therefore refuses sandwich blocks on unprepared bf16 weights
(BLK_ERR_UNSUPPORTED, checked here); the unprepared cases below run the same
window, rotary and gate options without the post-norms.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from llama_family_decoder_gb300 import DecoderBlock
from llama_family_decoder_gb300.synth import WORKLOADS, Workload, make_input, make_kv_cache, make_weights
from tests.helpers import TOL, bf16_floor, cfg_of, np64, rel_err, to_dev, weights_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _afmoe(name, dtype, B, T, D, H, Hkv, d, F, window=0, rope=True, gate=True, sandwich=True, seed=0, **kw):
    return Workload(name, dtype, B, T, D, H, Hkv, d, F, "silu", qk_norm=True, seed=seed, sliding_window=window,
                    use_rope=rope, attn_gate=gate, sandwich_norm=sandwich, **kw)


def _taps(wl, dt, kv=True):
    B, T, D, H, Hkv, d, F = wl.batch, wl.seq, wl.hidden_size, wl.num_heads, wl.num_kv_heads, wl.head_dim, \
        wl.intermediate_size
    shapes = {"attention_queries": (B, H, T, d), "attention_head_outputs": (B, T, H, d),
              "attention_output": (B, T, D), "layer_mid": (B, T, D), "mlp_neurons": (B, T, F),
              "mlp_output": (B, T, D)}
    if kv:
        shapes.update(attention_keys=(B, Hkv, T, d), attention_values=(B, Hkv, T, d))
    return {k: torch.empty(s, dtype=dt, device=DEV) for k, s in shapes.items()}


def _bound(wl, prepared, ref_out):
    """The layer-output bound of a case."""
    return TOL["f32"] if wl.dtype == "f32" else TOL["bf16"]


def _tap_bound(wl, prepared, floor):
    """An intermediate tap's bound: the tolerance, or twice its own bf16 storage floor
    plus 5e-3 (max|err|/RMS of a tap whose RMS is far below its largest entries is set by
    the rounding of those entries, as in the other suites)."""
    return max(TOL["bf16"], 2.0 * floor + 5e-3)


def _runnable(wl, prepared):
    """Sandwich blocks need prepared weights on the bf16 path; an unprepared case runs
    the same options without the post-norms."""
    if wl.dtype == "bf16" and wl.sandwich_norm and not prepared:
        return wl.scaled(name=wl.name + "_nosandwich", sandwich_norm=False)
    return wl


def _check_taps(tb, ref, wl, prepared, prefix=""):
    errs = {}
    for name, t in tb.items():
        r = ref[name]
        e, f = rel_err(t, r), bf16_floor(r)
        errs[name] = e
        print(f"  {prefix}{name}: {e:.4f} (bf16 floor {f:.4f})")
        assert e <= _tap_bound(wl, prepared, f), (name, e, f)
    return errs


def _check_identity(x, out, tb, ref):
    """"afmoe", "The block, in order": layer input + attention_output + mlp_output ==
    layer_output. The output and both taps are bf16 roundings of fp32 values, so the
    identity holds to the sum of their measured errors (the triangle inequality)."""
    ident = np64(x) + np64(tb["attention_output"]) + np64(tb["mlp_output"])
    rms = lambda a: float(np.sqrt(np.mean(np.asarray(a, dtype=np.float64) ** 2)))
    slack = sum(rel_err(tb[n], ref[n]) * rms(ref[n]) for n in ("attention_output", "mlp_output"))
    bound = rel_err(out, ref["layer_output"]) + slack / rms(ref["layer_output"]) + 1e-3
    assert rel_err(out, ident) <= bound


PREFILL = [
    # window shorter than a key tile and not a multiple of it; several query tiles, ragged tail
    (_afmoe("sliding_w200", "bf16", 2, 520, 512, 4, 2, 128, 1000, window=200, seed=51), True),
    (_afmoe("sliding_w200", "bf16", 2, 520, 512, 4, 2, 128, 1000, window=200, seed=51), False),
    (_afmoe("sliding_w128", "bf16", 1, 700, 1024, 8, 2, 128, 1536, window=128, seed=52), True),
    # a window of one position: each query reads its own value
    (_afmoe("sliding_w1_plain", "bf16", 2, 300, 512, 4, 1, 128, 776, window=1, gate=False, sandwich=False,
            seed=53), False),
    (_afmoe("sliding_w1_plain", "bf16", 2, 300, 512, 4, 1, 128, 776, window=1, gate=False, sandwich=False,
            seed=53), True),
    # a whole-prefix block: no window, no rotary
    (_afmoe("global_norope", "bf16", 2, 400, 512, 8, 2, 128, 1000, rope=False, seed=54), True),
    (_afmoe("global_norope", "bf16", 1, 260, 512, 4, 2, 128, 1000, rope=False, seed=55), False),
    # a window longer than the sequence is the plain causal mask
    (_afmoe("sliding_w700_gate_only", "bf16", 1, 333, 512, 4, 2, 128, 1000, window=700, sandwich=False,
            seed=56), False),
    (_afmoe("sandwich_only", "bf16", 2, 200, 512, 4, 2, 128, 1000, gate=False, seed=57), True),
]


@pytest.mark.parametrize("wl,prepared", PREFILL,
                         ids=lambda v: v.name if isinstance(v, Workload) else ("prepared" if v else "bf16_weights"))
def test_afmoe_prefill_small(wl, prepared):
    wl = _runnable(wl, prepared)
    w = make_weights(wl, gain_std=0.1)
    x = make_input(wl)
    blk = DecoderBlock.from_workload(wl)
    wd = to_dev(w)
    if prepared:
        wd = blk.prepare(wd)
    tb = _taps(wl, torch.bfloat16)
    out = blk.forward(x.to(DEV), wd, taps=tb)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    ref = oracle.block_forward(cfg_of(wl), weights_np(w), np64(x))
    err, floor = rel_err(out, ref["layer_output"]), bf16_floor(ref["layer_output"])
    bound = _bound(wl, prepared, ref["layer_output"])
    print(f"{wl.name} prepared={prepared}: layer_output {err:.4f} (bf16 floor {floor:.4f}, bound {bound:.4f})")
    _check_taps(tb, ref, wl, prepared)
    assert err <= bound, (err, floor)
    _check_identity(x, out, tb, ref)
    if not wl.use_rope:
        # "Rotary runs on the sliding-window blocks only": the queries are q_norm's output
        qp = (ref["attention_norm_output"] @ weights_np(w)["q_proj"].T).reshape(wl.batch, wl.seq, wl.num_heads,
                                                                                wl.head_dim)
        qn = oracle.rms_norm(qp, weights_np(w)["q_norm"], wl.rms_norm_eps).transpose(0, 2, 1, 3)
        assert rel_err(tb["attention_queries"], qn) <= TOL["bf16"]
    if wl.sandwich_norm:
        # the post-norms' outputs have RMS gain-shaped rows: with the norm's own gain removed, mean square ~ 1
        g = np64(w["post_mlp_norm"])
        ms = np.mean((np64(tb["mlp_output"]) / g) ** 2, axis=-1)
        assert np.all(np.abs(ms - 1.0) < 0.05), (ms.min(), ms.max())


@pytest.mark.parametrize("prepared", [True, False], ids=["prepared", "bf16_weights"])
@pytest.mark.parametrize("window", [100, 260])
def test_afmoe_chunk_over_the_cache_with_window(window, prepared):
    # T new tokens after ragged cached lengths; the window reaches back into the cache
    # (or not, for the empty one). Unused slots hold NaN: nothing of them may leak.
    wl = _runnable(_afmoe(f"chunk_w{window}", "bf16", 3, 150, 512, 8, 2, 128, 1000, window=window, seed=58),
                   prepared)
    lens = [0, 37, 300]
    cap = 500
    w = make_weights(wl, gain_std=0.1)
    x = make_input(wl)
    g = torch.Generator().manual_seed(59)
    kc = torch.full((wl.batch, wl.num_kv_heads, cap, wl.head_dim), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    for b, L in enumerate(lens):
        kc[b, :, :L] = torch.randn(wl.num_kv_heads, L, wl.head_dim, generator=g).to(torch.bfloat16)
        vc[b, :, :L] = torch.randn(wl.num_kv_heads, L, wl.head_dim, generator=g).to(torch.bfloat16)
    blk = DecoderBlock.from_workload(wl, max_seq=cap + 1)
    kd, vd = kc.to(DEV), vc.to(DEV)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    tb = _taps(wl, torch.bfloat16, kv=False)
    wd = to_dev(w)
    if prepared:
        wd = blk.prepare(wd)
    out = blk.forward(x.to(DEV), wd, cache={"k": kd, "v": vd, "lens": lens_d}, host_lens_max=max(lens), taps=tb)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    ref = oracle.prefill_with_cache(cfg_of(wl), weights_np(w), np64(x), np64(kc), np64(vc), np.array(lens))
    err, floor = rel_err(out, ref["layer_output"]), bf16_floor(ref["layer_output"])
    bound = _bound(wl, prepared, ref["layer_output"])
    print(f"chunk window {window} prepared={prepared}: {err:.4f} (bf16 floor {floor:.4f}, bound {bound:.4f})")
    _check_taps(tb, ref, wl, prepared, "chunk ")
    assert err <= bound
    assert lens_d.tolist() == [L + wl.seq for L in lens]
    kd_c = kd.cpu()
    for b, L in enumerate(lens):
        assert rel_err(kd_c[b, :, L:L + wl.seq], ref["new_keys"][b]) <= TOL["bf16"]
        assert torch.isnan(kd_c[b, :, L + wl.seq:].float()).all()


def _decode(wl, lens, taps=True, gain_std=0.1, prepared=False):
    w = make_weights(wl, gain_std=gain_std)
    x = make_input(wl)[:, 0]
    cap = int(max(lens)) + 9
    kc, vc = make_kv_cache(wl.scaled(cache_len=int(max(lens))), capacity=cap)
    for b, L in enumerate(lens):
        kc[b, :, L:] = float("nan")  # unused slots: nothing may leak from them
        vc[b, :, L:] = float("nan")
    blk = DecoderBlock.from_workload(wl, max_seq=cap + 1)
    kd, vd = kc.to(DEV), vc.to(DEV)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    tb = None
    if taps:
        tb = {k: v[:, :1] if k != "attention_queries" else v[:, :, :1]
              for k, v in _taps(wl.scaled(seq=1), torch.float32 if wl.dtype == "f32" else torch.bfloat16,
                                kv=False).items()}
    wd = to_dev(w)
    if prepared:
        wd = blk.prepare(wd)
    out = blk.forward(x[:, None].to(DEV), wd, cache={"k": kd, "v": vd, "lens": lens_d},
                      host_lens_max=max(lens), taps=tb)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    ref = oracle.decode_step(cfg_of(wl), weights_np(w), np64(x), np64(kc), np64(vc), np.array(lens))
    assert lens_d.tolist() == [L + 1 for L in lens]
    idx = torch.arange(wl.batch)
    assert rel_err(kd[idx, :, torch.tensor(lens)], ref["new_key"]) <= TOL[wl.dtype]
    return out[:, 0], tb, ref


@pytest.mark.parametrize("prepared", [True, False], ids=["prepared", "bf16_weights"])
@pytest.mark.parametrize("window,rope", [(64, True), (200, True), (0, False)])
def test_afmoe_decode_small(window, rope, prepared):
    # sequences shorter and longer than the window (the split-KV units start at the window)
    wl = _runnable(_afmoe(f"decode_w{window}", "bf16", 7, 1, 512, 8, 2, 128, 1000, window=window, rope=rope,
                          seed=60), prepared)
    lens = [1, 30, 63, 64, 65, 190, 400]
    out, tb, ref = _decode(wl, lens, prepared=prepared)
    err, bound = rel_err(out, ref["layer_output"]), _bound(wl, prepared, ref["layer_output"])
    print(f"decode window {window} prepared={prepared}: {err:.4f} (bound {bound:.4f})")
    for name, t in tb.items():
        r = ref[name]
        t = t[:, :, 0] if name == "attention_queries" else t[:, 0]
        e, f = rel_err(t, r), bf16_floor(r)
        print(f"  decode {name}: {e:.4f} (floor {f:.4f})")
        assert e <= _tap_bound(wl, prepared, f), (name, e, f)
    assert err <= bound


@pytest.mark.parametrize("prepared", [True, False], ids=["prepared", "bf16_weights"])
def test_afmoe_decode_unfused_qkv(prepared):
    # 80 weight tiles (q, k, v, gate) x 2 token tiles exceed the SMs: the QKV partials are
    # summed by the post kernel, which also forms the gate
    wl = _runnable(_afmoe("decode_wide", "bf16", 260, 1, 4096, 32, 8, 128, 1024, window=48, seed=61), prepared)
    lens = [(53 * b + 7) % 120 + 1 for b in range(wl.batch)]
    out, _, ref = _decode(wl, lens, taps=False, gain_std=0.0, prepared=prepared)
    err, bound = rel_err(out, ref["layer_output"]), _bound(wl, prepared, ref["layer_output"])
    print(f"decode wide prepared={prepared}: {err:.4f} (floor {bf16_floor(ref['layer_output']):.4f}, "
          f"bound {bound:.4f})")
    assert err <= bound


def test_afmoe_sandwich_refused_on_unprepared_bf16_weights():
    # prefill, prefill chunk, decode and the MLP stage: refused on the host, nothing launched
    from llama_family_decoder_gb300.binding import BlkError
    wl = _afmoe("refused", "bf16", 2, 64, 512, 4, 2, 128, 1000, window=32, seed=65)
    w = to_dev(make_weights(wl))
    x = make_input(wl).to(DEV)
    blk = DecoderBlock.from_workload(wl, max_seq=200)
    kc = torch.zeros(2, 2, 160, 128, dtype=torch.bfloat16, device=DEV)
    lens = torch.tensor([3, 9], dtype=torch.int32, device=DEV)
    calls = [lambda: blk.forward(x, w),
             lambda: blk.forward(x, w, cache={"k": kc, "v": kc.clone(), "lens": lens}, host_lens_max=9),
             lambda: blk.forward(x[:, :1].contiguous(), w, cache={"k": kc, "v": kc.clone(), "lens": lens},
                                 host_lens_max=9),
             lambda: blk.mlp(x.view(-1, 512), x.view(-1, 512), w, torch.empty_like(x).view(-1, 512))]
    for call in calls:
        with pytest.raises(BlkError) as e:
            call()
        assert e.value.status == 2  # BLK_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert lens.tolist() == [3, 9]  # no launch touched the cache
    out = blk.forward(x, blk.prepare(w))  # the same block on prepared weights runs
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("window,rope,gate,sandwich", [(5, True, True, True), (0, False, True, True),
                                                      (3, True, False, True), (9, True, True, False)])
def test_afmoe_f32_prefill_and_decode(window, rope, gate, sandwich):
    wl = _afmoe("f32", "f32", 2, 40, 256, 4, 2, 64, 512, window=window, rope=rope, gate=gate, sandwich=sandwich,
                seed=62)
    w = make_weights(wl, gain_std=0.1)
    x = make_input(wl)
    blk = DecoderBlock.from_workload(wl)
    tb = _taps(wl, torch.float32)
    out = blk.forward(x.to(DEV), to_dev(w), taps=tb)
    torch.cuda.synchronize()
    ref = oracle.block_forward(cfg_of(wl), weights_np(w), np64(x))
    assert rel_err(out, ref["layer_output"]) <= TOL["f32"]
    for name, t in tb.items():
        assert rel_err(t, ref[name]) <= 10 * TOL["f32"], name
    dl = wl.scaled(batch=3, seq=1)
    out, tb, ref = _decode(dl, [2, 7, 30])
    assert rel_err(out, ref["layer_output"]) <= TOL["f32"]


@pytest.mark.parametrize("dtype,decode", [("bf16", False), ("bf16", True), ("f32", False)])
def test_attention_stage_with_window(dtype, decode):
    # blk_attn_gqa honours the handle's window (the head outputs: no gate)
    B, H, Hkv, d, T, W = 2, 8, 2, (128 if dtype == "bf16" else 64), (1 if decode else 300), 70
    wl = _afmoe("stage", dtype, B, T, 512, H, Hkv, d, 512, window=W, seed=63)
    blk = DecoderBlock.from_workload(wl, max_seq=400)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(64)
    S = 300
    q = torch.randn(B, H, T, d, generator=g).to(dt)
    k = torch.randn(B, Hkv, S, d, generator=g).to(dt)
    v = torch.randn(B, Hkv, S, d, generator=g).to(dt)
    o = torch.empty(B, T, H, d, dtype=dt, device=DEV)
    lens = [150, 300] if decode else None
    blk.attn_gqa(q.to(DEV), k.to(DEV), v.to(DEV), o,
                 kv_lens=torch.tensor(lens, dtype=torch.int32, device=DEV) if decode else None)
    torch.cuda.synchronize()
    for b in range(B):
        n = lens[b] if decode else T
        ref = oracle.causal_gqa_attention(np64(q[b]), np64(k[b, :, :n]), np64(v[b, :, :n]), np.arange(n - T, n),
                                          np.arange(n), window=W)
        err = rel_err(o[b].transpose(0, 1), ref)
        floor = bf16_floor(ref) if dtype == "bf16" else 0.0
        print(f"attention stage {dtype} decode={decode} sequence {b}: {err:.4f} (bf16 floor {floor:.4f})")
        assert err <= max(TOL[dtype], 1.5 * floor + 2e-3), (b, err, floor)  # as the other stage tests


# ------------------------------------------------------------------ full size, sampled

@pytest.mark.parametrize("name", ["afmoe_nano_sliding_bf16_B8_T4096_W2048", "afmoe_nano_global_bf16_B8_T4096"])
def test_afmoe_prefill_full_size_sampled_rows(name):
    wl = WORKLOADS[name]
    w = make_weights(wl)
    x = make_input(wl)
    blk = DecoderBlock.from_workload(wl)
    wd = blk.prepare({k: v.cuda() for k, v in w.items()})  # as bench.py runs it
    out = blk.forward(x.cuda(), wd)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    out = out.cpu()
    T = wl.seq
    rows = sorted({0, 1, 127, 128, 2046, 2047, 2048, 2049, 3000, T - 129, T - 1})
    wn = weights_np(w)
    for b in sorted({0, wl.batch - 1}):
        ref = oracle.block_forward(cfg_of(wl), wn, np64(x[b:b + 1]), rows=rows)["layer_output"][0]
        err, floor = rel_err(out[b, rows], ref), bf16_floor(ref)
        print(f"{name} batch {b}: {err:.4f} (bf16 floor {floor:.4f})")
        assert err <= TOL["bf16"], (err, floor)
        assert torch.isfinite(out[b]).all()


def test_afmoe_decode_full_size_sampled_sequences():
    wl = WORKLOADS["afmoe_nano_decode_bf16_B64_L8192_W2048"]
    w = make_weights(wl)
    x = make_input(wl)[:, 0]
    kc, vc = make_kv_cache(wl)
    blk = DecoderBlock.from_workload(wl)
    lens = torch.full((wl.batch,), wl.cache_len, dtype=torch.int32, device="cuda")
    kd, vd = kc.cuda(), vc.cuda()
    wd = blk.prepare({k: v.cuda() for k, v in w.items()})  # as bench.py runs it
    out = blk.forward(x[:, None].cuda(), wd, cache={"k": kd, "v": vd, "lens": lens}, host_lens_max=wl.cache_len)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    seqs = [0, 31, 63]
    ref = oracle.decode_step(cfg_of(wl), weights_np(w), np64(x[seqs]), np64(kc[seqs]), np64(vc[seqs]),
                             np.full(len(seqs), wl.cache_len))
    err = rel_err(out[seqs, 0].cpu(), ref["layer_output"])
    print(f"afmoe decode: {err:.4f}")
    assert err <= TOL["bf16"]
