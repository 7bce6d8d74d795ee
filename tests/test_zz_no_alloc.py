"""Allocation-free decode attention (blk_attn_decode_noalloc), through the C ABI.

Some callers cannot call cudaMalloc: a plugin interface that is handed only
input and output pointers, a runtime whose memory pool already owns all device
memory, or a latency-critical loop that cannot take cudaMalloc's implicit device
synchronisation. For them the library offers a decode-attention entry point
that keeps its split partials in a fixed device array instead of a caller
workspace. Its results must match the workspace-taking path (blk_attn_gqa with
kv_lens), call after call, whatever the previous call left in that array.
This file is collected last, so a failure here comes after every other test.
"""
import ctypes

import pytest
import torch

from llama_family_decoder_gb300 import DecoderBlock
from llama_family_decoder_gb300.binding import attn_decode_noalloc, lib
from tests.helpers import TOL, np64, rel_err

pytestmark = pytest.mark.gpu

B, H, HKV, D, CAP = 6, 16, 4, 128, 700


def _inputs(seed, lens):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, 1, D, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, HKV, CAP, D, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, HKV, CAP, D, generator=g).to(torch.bfloat16).cuda()
    return q, k, v, torch.tensor(lens, dtype=torch.int32).cuda()


def test_noalloc_decode_attention_matches_workspace_path():
    blk = DecoderBlock(hidden=H * D, n_heads=H, n_kv_heads=HKV, head_dim=D, ffn=1024, act="silu", dtype="bf16",
                       max_batch=B, max_seq=CAP + 1)
    cases = [(41, [1, 64, 65, 300, 699, 700]), (42, [700, 2, 129, 511, 37, 640])]
    for seed, lens in cases:  # two calls in a row, different inputs and lengths
        q, k, v, kl = _inputs(seed, lens)
        want = torch.empty(B, 1, H, D, dtype=torch.bfloat16, device="cuda")
        blk.attn_gqa(q, k, v, want, kv_lens=kl)
        got = torch.empty_like(want)
        attn_decode_noalloc(q, k, v, kl, got)
        torch.cuda.synchronize()
        err = rel_err(got, np64(want))
        assert err <= TOL["bf16"], (seed, err)
        assert torch.isfinite(got).all()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 2048 x 32 heads x (128 + 2) x 4 bytes > 16 MiB: refused on the host before any launch
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = lib().blk_attn_decode_noalloc(p, p, p, ctypes.c_void_p(lens.data_ptr()), 2048, 32, 8, 128, 16, p, None)
    assert st == 2  # BLK_ERR_UNSUPPORTED
    assert b"16 MiB" in lib().blk_last_error_message()
