"""Full-size parity: the pages' workload shapes, run exactly as bench.py runs them
(one blk_forward over the whole batch), checked on sampled output rows that the
fp64 oracle computes one by one (keys/values of the whole prefix included)."""
import numpy as np
import pytest
import torch

import oracle
from llama_family_decoder_gb300 import DecoderBlock
from llama_family_decoder_gb300.synth import WORKLOADS, make_input, make_kv_cache, make_weights
from tests.helpers import TOL, bf16_floor, cfg_of, check_relu2_zeros, np64, rel_err, weights_np

pytestmark = pytest.mark.gpu

PREFILL = ["llama7b_bf16_B1_T2048", "arcee_gqa_bf16_B4_T2048", "apertus_qknorm_bf16_B2_T4096"]


@pytest.mark.parametrize("name", PREFILL)
def test_prefill_full_size_sampled_rows(name):
    wl = WORKLOADS[name]
    w = make_weights(wl)
    x = make_input(wl)
    blk = DecoderBlock.from_workload(wl)
    wd = blk.prepare({k: v.cuda() for k, v in w.items()})  # as bench.py runs it
    relu2 = wl.hidden_act == "relu2"
    taps = {"mlp_neurons": torch.empty(wl.batch, wl.seq, wl.intermediate_size, dtype=torch.bfloat16,
                                       device="cuda")} if relu2 else None
    out = blk.forward(x.cuda(), wd, taps=taps)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    out = out.cpu()
    del blk, wd
    wn = weights_np(w)
    T = wl.seq
    rows = sorted({0, 1, 63, 64, 127, 128, 129, 1000, T // 2 + 3, T - 129, T - 2, T - 1})
    for b in sorted({0, wl.batch - 1}):
        ref = oracle.block_forward(cfg_of(wl), wn, np64(x[b:b + 1]), rows=rows)
        got = out[b, rows]
        err, floor = rel_err(got, ref["layer_output"][0]), bf16_floor(ref["layer_output"][0])
        print(f"{name} batch {b}: max|err|/RMS {err:.4f} (bf16 floor {floor:.4f})")
        assert err <= TOL["bf16"], (err, floor)
        assert torch.isfinite(out[b]).all()
        if relu2:  # the sampled rows' neurons, element by element
            zeros, du = check_relu2_zeros(taps["mlp_neurons"][b, rows].cpu(), ref["mlp_up_output"][0])
            print(f"  relu2: {zeros:.3f} exact zeros, pre-activation max|du|/RMS {du:.4f}")


def test_decode_full_size_sampled_sequences():
    wl = WORKLOADS["llama7b_decode_bf16_B64_L4096"]
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
    assert (lens == wl.cache_len + 1).all()
    seqs = [0, 31, 63]
    ref = oracle.decode_step(cfg_of(wl), weights_np(w), np64(x[seqs]), np64(kc[seqs]), np64(vc[seqs]),
                             np.full(len(seqs), wl.cache_len))
    got = out[seqs, 0].cpu()
    err, floor = rel_err(got, ref["layer_output"]), bf16_floor(ref["layer_output"])
    print(f"decode: max|err|/RMS {err:.4f} (bf16 floor {floor:.4f})")
    assert err <= TOL["bf16"], (err, floor)
    assert rel_err(kd[seqs, :, wl.cache_len].cpu(), ref["new_key"]) <= TOL["bf16"]
    assert rel_err(vd[seqs, :, wl.cache_len].cpu(), ref["new_value"]) <= TOL["bf16"]


def test_prefill_full_size_every_row():
    # every output of the Llama-7B-shape workload (1 x 2048 x 4096) against the oracle
    wl = WORKLOADS["llama7b_bf16_B1_T2048"]
    w = make_weights(wl)
    x = make_input(wl)
    blk = DecoderBlock.from_workload(wl)
    wd = blk.prepare({k: v.cuda() for k, v in w.items()})
    out = blk.forward(x.cuda(), wd).cpu()
    ref = oracle.block_forward(cfg_of(wl), weights_np(w), np64(x))["layer_output"]
    e = np.abs(np64(out) - ref) / np.sqrt(np.mean(ref * ref))
    print(f"llama7b every row: max {e.max():.4f}, 99.99th pct {np.quantile(e, 0.9999):.4f}, "
          f"bf16 floor {bf16_floor(ref):.4f}")
    assert e.max() <= TOL["bf16"]


def test_full_size_runs_are_bitwise_repeatable():
    """Every reduction on the path has a fixed order (split partials summed in split order,
    per-tile sums of squares in tile order, persistent work lists whose per-unit results do
    not depend on the CTA that computes them), so two runs of the same step agree to the bit:
    the Apertus-shape prefill (CTA pairs, persistent attention) and the decode step (units
    taken from an atomic counter, splits combined afterwards)."""
    wl = WORKLOADS["apertus_qknorm_bf16_B2_T4096"]
    x = make_input(wl).cuda()
    blk = DecoderBlock.from_workload(wl)
    wd = blk.prepare({k: v.cuda() for k, v in make_weights(wl).items()})
    first = blk.forward(x, wd)
    second = blk.forward(x, wd)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    assert torch.equal(first, second)
    del blk, wd, first, second, x

    wl = WORKLOADS["llama7b_decode_bf16_B64_L4096"]
    x = make_input(wl)[:, 0][:, None].cuda()
    kc, vc = make_kv_cache(wl)
    kd, vd = kc.cuda(), vc.cuda()
    blk = DecoderBlock.from_workload(wl)
    wd = blk.prepare({k: v.cuda() for k, v in make_weights(wl).items()})
    outs = []
    for _ in range(2):
        lens = torch.full((wl.batch,), wl.cache_len, dtype=torch.int32, device="cuda")  # the same slot each time
        outs.append(blk.forward(x, wd, cache={"k": kd, "v": vd, "lens": lens}, host_lens_max=wl.cache_len))
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    assert torch.equal(outs[0], outs[1])
