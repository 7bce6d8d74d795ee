"""The model around the block (blk_model_forward): embed_tokens, the decoder layers,
the final norm and lm_head ("LlamaForCausalLM-32L-4096d" sheet, "Implementing it"),
against the oracle's model_forward, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from llama_family_decoder_gb300 import DecoderBlock
from llama_family_decoder_gb300.binding import BlkError
from llama_family_decoder_gb300.synth import Workload, make_model
from tests.helpers import TOL, bf16_floor, cfg_of, np64, rel_err, to_dev, weights_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
# The block's bar (max|err|/RMS <= 2e-2) composed over the layers: each block adds an independent
# rounding error of the same size, so the stream's error grows as sqrt(layers).
TOL_MODEL_2 = TOL["bf16"] * np.sqrt(2)


def _dev_model(parts):
    layers, embed, norm_g, lm_head, tokens = parts
    return [to_dev(w) for w in layers], embed.to(DEV), norm_g.to(DEV), lm_head.to(DEV), tokens.to(DEV)


@pytest.mark.parametrize("act,qk_norm", [("silu", False), ("xielu", True)])
def test_model_prefill_logits(act, qk_norm):
    wl = Workload(f"model_{act}", "bf16", 2, 96, 512, 8, 2, 128, 1000, act, qk_norm=qk_norm, seed=31)
    parts = make_model(wl, n_layers=2, vocab=1024)
    layers, embed, norm_g, lm_head, tokens = parts
    blk = DecoderBlock.from_workload(wl)
    dl, de, dn, dh, dt = _dev_model(parts)
    logits = blk.model_forward(dt, dl, de, dn, dh)
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    ref = oracle.model_forward(cfg_of(wl), [weights_np(w) for w in layers], np64(embed), np64(norm_g),
                               np64(lm_head), tokens.numpy())
    err, floor = rel_err(logits, ref), bf16_floor(ref)
    print(f"model {act}: logits max|err|/RMS {err:.4f} (bf16 floor {floor:.4f})")
    assert err <= TOL_MODEL_2


def test_model_prompt_then_decode_through_the_caches():
    wl = Workload("model_decode", "bf16", 2, 65, 512, 8, 2, 128, 1000, "silu", seed=32)
    parts = make_model(wl, n_layers=2, vocab=1024)
    layers, embed, norm_g, lm_head, tokens = parts
    blk = DecoderBlock.from_workload(wl, max_seq=128)
    dl, de, dn, dh, dt = _dev_model(parts)
    T = wl.seq - 1
    caches = [{"k": torch.zeros(wl.batch, wl.num_kv_heads, 96, wl.head_dim, dtype=torch.bfloat16, device=DEV),
               "v": torch.zeros(wl.batch, wl.num_kv_heads, 96, wl.head_dim, dtype=torch.bfloat16, device=DEV),
               "lens": torch.zeros(wl.batch, dtype=torch.int32, device=DEV)} for _ in layers]
    blk.model_forward(dt[:, :T].contiguous(), dl, de, dn, dh, caches=caches, host_lens_max=0)  # the prompt
    last = blk.model_forward(dt[:, T:].contiguous(), dl, de, dn, dh, caches=caches, host_lens_max=T)  # one step
    torch.cuda.synchronize()
    assert blk.last_status() == 0
    for c in caches:
        assert c["lens"].tolist() == [wl.seq] * wl.batch
    ref = oracle.model_forward(cfg_of(wl), [weights_np(w) for w in layers], np64(embed), np64(norm_g),
                               np64(lm_head), tokens.numpy())
    err = rel_err(last[:, 0], ref[:, -1])
    print(f"model decode step: logits max|err|/RMS {err:.4f}")
    assert err <= TOL_MODEL_2


def test_model_flags_token_ids_outside_the_vocabulary():
    wl = Workload("model_bad_ids", "bf16", 1, 8, 512, 8, 2, 128, 1000, "silu", seed=33)
    parts = make_model(wl, n_layers=1, vocab=256)
    blk = DecoderBlock.from_workload(wl)
    dl, de, dn, dh, dt = _dev_model(parts)
    dt[0, 3] = 256
    blk.model_forward(dt, dl, de, dn, dh)
    torch.cuda.synchronize()
    assert blk.last_status() == 1  # BLK_ERR_INVALID_ARG, read and cleared
    assert blk.last_status() == 0
