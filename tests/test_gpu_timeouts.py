"""Bounded device waits: a wait limit far below a kernel's own latency makes waits run
out; the kernels must record BLK_ERR_TIMEOUT, stop, drain their copies and MMAs, free
their tensor memory and return, leaving the context usable for the next, correct call.

The limit is the library's debug knob (blk_debug_set_wait_timeout_ns, 1 us here). The
shapes are chosen so that some wait certainly outlasts it: the bare GEMM's epilogue
waits for a 256-k-block main loop (tens of microseconds), and the small block's GEMMs
and attention wait microseconds per tile. Every shape keeps K below 2048, so that no
CTA pair is involved (one CTA per tile, whose drain is complete). No wait is removed
and nothing is left hanging: every wait in these kernels is bounded either way.
"""
import numpy as np
import pytest
import torch

import oracle
from llama_family_decoder_gb300 import DecoderBlock
from llama_family_decoder_gb300.binding import debug_gemm_bf16, lib, set_wait_timeout_ns
from llama_family_decoder_gb300.synth import Workload, make_input, make_weights
from tests.helpers import TOL, cfg_of, np64, rel_err, to_dev, weights_np

pytestmark = pytest.mark.gpu

TIMEOUT = 6  # BLK_ERR_TIMEOUT
SHORT_NS = 1000


@pytest.fixture
def short_waits():
    set_wait_timeout_ns(SHORT_NS)
    try:
        yield
    finally:
        set_wait_timeout_ns(0)  # back to the default limit, whatever happened


def _gemm_inputs():
    g = torch.Generator().manual_seed(71)
    M, N, K = 256, 384, 16384
    a = (torch.randn(M, K, generator=g) * 0.05).to(torch.bfloat16)
    b = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    return a, b


def _gemm_bound(a, b):
    # fp32 accumulation of bf16 products: |err| <= K * 2^-23 * sum|a||b| elementwise, far
    # above the real error; the bf16 store adds half an ulp of the result
    aa, bb = np64(a), np64(b)
    ref = aa @ bb.T
    bound = aa.shape[1] * 2.0 ** -23 * (np.abs(aa) @ np.abs(bb).T) + np.abs(ref) * 2.0 ** -8
    return ref, bound


def test_gemm_wait_runs_out_then_recovers(short_waits):
    a, b = _gemm_inputs()
    ad, bd = a.cuda(), b.cuda()
    c = torch.full((a.shape[0], b.shape[0]), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert lib().blk_debug_last_status() == 0
    debug_gemm_bf16(ad, bd, bn=128, out=c)
    torch.cuda.synchronize()  # every CTA returned: no wait was left hanging
    assert lib().blk_debug_last_status() == TIMEOUT
    assert lib().blk_debug_last_status() == 0  # reading it clears it
    set_wait_timeout_ns(0)
    debug_gemm_bf16(ad, bd, bn=128, out=c)
    torch.cuda.synchronize()
    assert lib().blk_debug_last_status() == 0
    ref, bound = _gemm_bound(a, b)
    assert np.all(np.abs(np64(c) - ref) <= bound)


SMALL = Workload("timeout_small", "bf16", 1, 512, 1536, 12, 4, 128, 2040, "silu", seed=72)


def test_block_forward_wait_runs_out_then_recovers(short_waits):
    wl = SMALL
    w = make_weights(wl)
    x = make_input(wl)
    blk = DecoderBlock.from_workload(wl)
    wd, xd = to_dev(w), x.cuda()
    blk.forward(xd, wd)
    torch.cuda.synchronize()  # the forward's kernels all returned
    assert blk.last_status() == TIMEOUT
    assert blk.last_status() == 0
    set_wait_timeout_ns(0)
    for _ in range(2):  # the context, the handle and its workspace stay usable
        out = blk.forward(xd, wd)
        torch.cuda.synchronize()
        assert blk.last_status() == 0
        ref = oracle.block_forward(cfg_of(wl), weights_np(w), np64(x))["layer_output"]
        assert rel_err(out, ref) <= TOL["bf16"]
