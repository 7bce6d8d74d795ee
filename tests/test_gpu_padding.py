"""GPU parity of padded prefill batches (nnterp's attention_mask, "arcee", "The API":
[batch seq], zeros are padding) against the fp64 oracle, through blk_forward_masked.

Each row's ones form one run [lo, hi): padding keys are hidden, row t takes rotary
position t - lo, rows before lo see no key. Every output row is compared (the
padding rows are defined the same way on both sides); the query values only on the
real rows, since a left-padding row's negative position is clamped on the GPU and
no key of such a row is ever visible. Bounds as in the other suites.
"""
import numpy as np
import pytest
import torch

import oracle
from llama_family_decoder_gb300 import DecoderBlock
from llama_family_decoder_gb300.binding import BlkError
from llama_family_decoder_gb300.synth import Workload, make_input, make_weights
from tests.helpers import TOL, bf16_floor, cfg_of, np64, rel_err, to_dev, weights_np

pytestmark = pytest.mark.gpu

DEV = "cuda"
RUNS = [(100, 300), (0, 250), (37, 201), (0, 300), (300, 300)]  # left, right, both, none, all padding


def _mask(B, T, runs):
    m = torch.zeros(B, T, dtype=torch.int32)
    for b, (lo, hi) in enumerate(runs):
        m[b, lo:hi] = 1
    return m


CASES = [
    (Workload("pad_swiglu_gqa", "bf16", 5, 300, 512, 8, 2, 128, 1000, "silu", seed=81), False),
    (Workload("pad_swiglu_gqa", "bf16", 5, 300, 512, 8, 2, 128, 1000, "silu", seed=81), True),
    (Workload("pad_afmoe_window", "bf16", 5, 300, 512, 4, 2, 128, 1000, "silu", qk_norm=True, seed=82,
              sliding_window=90, attn_gate=True, sandwich_norm=True), True),
    (Workload("pad_f32", "f32", 5, 300, 256, 4, 2, 64, 512, "xielu", qk_norm=True, seed=83), False),
]


@pytest.mark.parametrize("wl,prepared", CASES, ids=lambda v: v.name if isinstance(v, Workload) else str(v))
def test_padded_prefill_batch(wl, prepared):
    w = make_weights(wl, gain_std=0.1)
    x = make_input(wl)
    mask = _mask(wl.batch, wl.seq, RUNS)
    blk = DecoderBlock.from_workload(wl)
    wd = to_dev(w)
    if prepared:
        wd = blk.prepare(wd)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    tb = {"attention_queries": torch.empty(wl.batch, wl.num_heads, wl.seq, wl.head_dim, dtype=dt, device=DEV),
          "attention_head_outputs": torch.empty(wl.batch, wl.seq, wl.num_heads, wl.head_dim, dtype=dt, device=DEV)}
    out = blk.forward(x.to(DEV), wd, taps=tb, attention_mask=mask.to(DEV))
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    ref = oracle.block_forward(cfg_of(wl), weights_np(w), np64(x), attention_mask=mask.numpy())
    tol = TOL[wl.dtype]
    if wl.sandwich_norm and not prepared:
        tol = max(tol, 2 * bf16_floor(ref["layer_output"]) + 5e-3)
    err = rel_err(out, ref["layer_output"])
    print(f"{wl.name} prepared={prepared}: layer_output {err:.4f}")
    assert err <= tol
    assert torch.isfinite(out.float()).all()
    for b, (lo, hi) in enumerate(RUNS):
        if hi > lo:
            e = rel_err(tb["attention_queries"][b, :, lo:hi], ref["attention_queries"][b, :, lo:hi])
            assert e <= max(tol, 2 * bf16_floor(ref["attention_queries"][b, :, lo:hi]) + 5e-3), (b, e)
        # rows before the run see no key: zero head outputs
        assert (tb["attention_head_outputs"][b, :lo] == 0).all()
    # each real row equals the block over its unpadded sequence
    for b in (0, 2):
        lo, hi = RUNS[b]
        solo = blk.forward(x[b:b + 1, lo:hi].contiguous().to(DEV), wd)
        torch.cuda.synchronize()
        assert rel_err(out[b, lo:hi], np64(solo[0])) <= tol


def test_mask_with_a_hole_is_flagged():
    wl = Workload("pad_hole", "bf16", 2, 64, 512, 4, 2, 128, 512, "silu", seed=84)
    blk = DecoderBlock.from_workload(wl)
    mask = torch.ones(2, 64, dtype=torch.int32)
    mask[1, 10] = 0  # ones on both sides of a zero: not a padding run
    out = blk.forward(make_input(wl).to(DEV), to_dev(make_weights(wl)), attention_mask=mask.to(DEV))
    torch.cuda.synchronize()
    assert blk.last_status() == 1  # BLK_ERR_INVALID_ARG, recorded on the device
    assert torch.isfinite(out.float()).all()


def test_mask_refused_with_a_cache():
    wl = Workload("pad_cache", "bf16", 1, 4, 512, 4, 2, 128, 512, "silu", seed=85)
    blk = DecoderBlock.from_workload(wl, max_seq=64)
    kd = torch.zeros(1, 2, 32, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises((BlkError, ValueError)):
        blk.forward(make_input(wl).to(DEV), to_dev(make_weights(wl)),
                    cache={"k": kd, "v": kd.clone(), "lens": torch.zeros(1, dtype=torch.int32, device=DEV)},
                    host_lens_max=0, attention_mask=torch.ones(1, 4, dtype=torch.int32, device=DEV))
