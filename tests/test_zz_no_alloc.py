"""Allocation-free decode attention (blk_attn_decode_noalloc), through the C ABI.

Some callers cannot call cudaMalloc: a plugin interface that is handed only
input and output pointers, a runtime whose memory pool already owns all device
memory, or a latency-critical loop that cannot take cudaMalloc's implicit device
synchronisation. For them the library offers a decode-attention entry point
that keeps its split partials in a fixed device array instead of a caller
workspace. Its results must match the fp64 oracle's attention and the
workspace-taking path (blk_attn_gqa with kv_lens), call after call, whatever the
previous call left in that array: with one split per sequence, with many splits
over ragged lengths, and at the size where the array holds fewer splits than the
workspace path would use (its split count is then capped). A wait that runs out
must turn the whole output into NaN, since such a caller has no status word to read.
This file is collected last, so a failure here comes after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from llama_family_decoder_gb300 import DecoderBlock
from llama_family_decoder_gb300.binding import attn_decode_noalloc, lib, set_wait_timeout_ns
from tests.helpers import TOL, bf16_floor, np64, rel_err

pytestmark = pytest.mark.gpu

D = 128
SCRATCH = 16 << 20


def _inputs(seed, B, H, Hkv, cap, lens):
    """Seeded q, k, v on the device (bf16) and the int32 lengths; unused cache slots hold NaN."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(B, H, 1, D, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, Hkv, cap, D, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Hkv, cap, D, generator=g, device="cuda").to(torch.bfloat16)
    for b, n in enumerate(lens):  # nothing past kv_lens[b] may reach the result
        k[b, :, n:] = float("nan")
        v[b, :, n:] = float("nan")
    return q, k, v, torch.tensor(lens, dtype=torch.int32, device="cuda")


def _oracle(q, k, v, lens, seqs):
    """[len(seqs), H, d]: the oracle's attention of the last query of each sampled sequence."""
    out = []
    for b in seqs:
        n = int(lens[b])
        out.append(oracle.causal_gqa_attention(np64(q[b]), np64(k[b, :, :n]), np64(v[b, :, :n]),
                                               np.array([n - 1]), np.arange(n))[:, 0])
    return np.stack(out)


def _splits(B, H, cap):
    """Splits of this entry point: 512-key units (at most 64), then what the fixed array holds."""
    ws = min(64, max(1, cap // 512))
    fit = (SCRATCH - 256) // (B * H * (D + 2) * 4)
    return ws, min(ws, fit)


def _stage_bound(ref):
    """The bound of the other attention-stage tests, per sequence: the tolerance, or 1.5x
    the error of storing the exact output in bf16 plus 2e-3 (an attention output whose
    RMS is far below its largest entries has max|err|/RMS set by their rounding)."""
    return max(TOL["bf16"], 1.5 * bf16_floor(ref) + 2e-3)


def _check(B, H, Hkv, cap, cases, seqs):
    blk = DecoderBlock(hidden=H * D, n_heads=H, n_kv_heads=Hkv, head_dim=D, ffn=1024, act="silu", dtype="bf16",
                       max_batch=B, max_seq=cap + 1)
    got = torch.empty(B, 1, H, D, dtype=torch.bfloat16, device="cuda")
    for seed, lens in cases:  # calls in a row, different inputs and lengths
        q, k, v, kl = _inputs(seed, B, H, Hkv, cap, lens)
        attn_decode_noalloc(q, k, v, kl, got)
        want = torch.empty_like(got)
        blk.attn_gqa(q, k, v, want, kv_lens=kl)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        ref = _oracle(q, k, v, lens, seqs)
        for j, b in enumerate(seqs):  # each sequence on its own scale
            err, bound = rel_err(got[b, 0], ref[j]), _stage_bound(ref[j])
            print(f"B{B} H{H} cap {cap} seed {seed} sequence {b} ({lens[b]} keys): oracle {err:.4f} "
                  f"(bound {bound:.4f})")
            assert err <= bound, (seed, b, err, bound)
            # the workspace path (its own split count) against this one: both within the
            # bound of the oracle, so within twice it of each other
            assert rel_err(got[b, 0], np64(want[b, 0])) <= 2 * bound, (seed, b)
    blk.close()


def test_noalloc_one_split_matches_oracle():
    B, H, Hkv, cap = 6, 16, 4, 700
    assert _splits(B, H, cap) == (1, 1)
    _check(B, H, Hkv, cap, [(41, [1, 64, 65, 300, 699, 700]), (42, [700, 2, 129, 511, 37, 640])], list(range(B)))


def test_noalloc_many_splits_ragged_matches_oracle():
    # 9 splits per sequence: the partial layout and the combine across splits; ragged
    # lengths leave some splits short or empty
    B, H, Hkv, cap = 8, 32, 8, 4608
    assert _splits(B, H, cap) == (9, 9)
    lens = [[1, 513, 1024, 2047, 3000, 4095, 4600, 4608], [4608, 4607, 17, 512, 2560, 3333, 1, 4100]]
    _check(B, H, Hkv, cap, [(43, lens[0]), (44, lens[1])], list(range(B)))


def test_noalloc_split_count_capped_by_its_scratch():
    # 64 x 32 heads x 8192 keys: 512-key units would make 16 splits, the fixed array
    # holds 15 (64 * 32 * 130 * 4 bytes each); the chunks grow instead
    B, H, Hkv, cap = 64, 32, 8, 8192
    assert _splits(B, H, cap) == (16, 15)
    lens = [cap - (37 * b) % 3000 for b in range(B)]
    _check(B, H, Hkv, cap, [(45, lens), (46, lens[::-1])], [0, 1, 31, 62, 63])


def test_noalloc_wait_running_out_gives_nan():
    # a 1 ns wait limit makes the kernel's waits on its first tiles run out: the
    # whole output must be NaN (never a mix of stale partials), and with the limit
    # restored the next call is right again. A call in which no wait happened to run
    # out must be entirely right; the short limit is tried up to three times.
    B, H, Hkv, cap = 64, 32, 8, 8192
    lens = [cap] * B
    q, k, v, kl = _inputs(47, B, H, Hkv, cap, lens)
    got = torch.empty(B, 1, H, D, dtype=torch.bfloat16, device="cuda")
    ref = _oracle(q, k, v, lens, [0, 63])
    poisoned = False
    set_wait_timeout_ns(1)
    try:
        for _ in range(3):
            got.zero_()
            attn_decode_noalloc(q, k, v, kl, got)
            torch.cuda.synchronize()
            if torch.isnan(got).all():
                poisoned = True
                break
            assert torch.isfinite(got).all()
            assert all(rel_err(got[b, 0], ref[j]) <= _stage_bound(ref[j]) for j, b in enumerate((0, 63)))
    finally:
        set_wait_timeout_ns(0)
    assert poisoned
    attn_decode_noalloc(q, k, v, kl, got)
    torch.cuda.synchronize()
    assert torch.isfinite(got).all()
    assert all(rel_err(got[b, 0], ref[j]) <= _stage_bound(ref[j]) for j, b in enumerate((0, 63)))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 2048 x 32 heads x (128 + 2) x 4 bytes > 16 MiB: refused on the host before any launch
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = lib().blk_attn_decode_noalloc(p, p, p, ctypes.c_void_p(lens.data_ptr()), 2048, 32, 8, 128, 16, p, None)
    assert st == 2  # BLK_ERR_UNSUPPORTED
    assert b"16 MiB" in lib().blk_last_error_message()
