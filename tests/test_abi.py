"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "blk.h")


@pytest.fixture(scope="module")
def L():
    from llama_family_decoder_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return binding.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(blk_[a-z_0-9]+)\s*\(", text)))


def test_header_symbols_exported(L):
    from llama_family_decoder_gb300 import binding
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n
    # the binding declares a signature for each of them
    assert set(names) == set(binding.SIGNATURES)


def test_error_strings_and_version(L):
    assert L.blk_error_string(0) == b"BLK_OK"
    assert L.blk_error_string(6) == b"BLK_ERR_TIMEOUT"
    assert b"sm_103a" in L.blk_version()


def test_xielu_effective_matches_oracle(L):
    from llama_family_decoder_gb300 import xielu_effective
    for raw in [(-3.0, 2.0), (0.0, 0.0), (5.0, -1.5)]:
        ap, an = xielu_effective(*raw)
        ref = oracle.xielu_effective(*raw)
        np.testing.assert_allclose([ap, an], ref, rtol=1e-6)


def _desc(**kw):
    from llama_family_decoder_gb300.binding import blk_desc
    base = dict(hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn=1024, rope_theta=1e4, eps=1e-5, act=1,
                xielu_alpha_p=0.8, xielu_alpha_n=0.8, xielu_beta=0.5, xielu_eps=-1e-6, qk_norm=0, dtype=0,
                max_batch=1, max_seq=64)
    base.update(kw)
    return blk_desc(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(n_kv_heads=3), 1),          # heads not a multiple of kv heads
    (dict(head_dim=63), 1),           # odd head_dim
    (dict(hidden=0), 1),
    (dict(eps=0.0), 1),
    (dict(act=7), 1),
    (dict(dtype=1, head_dim=64), 2),  # bf16 path wants head_dim 128
    (dict(dtype=1, head_dim=128, hidden=260), 2),
    (dict(sliding_window=-1), 1),     # "afmoe" options: a negative window
    (dict(attn_gate=2), 1),           # flags are 0 or 1
    (dict(no_rope=1, rope_type=1, rope_factor=2.0, rope_orig_max_pos=64, rope_low=1.0, rope_high=32.0), 1),
])
def test_create_rejects_bad_descriptors(L, kw, code):
    h = ctypes.c_void_p()
    d = _desc(**kw)
    assert L.blk_create(ctypes.byref(d), ctypes.byref(h)) == code
    assert h.value is None
    assert L.blk_last_error_message()


def test_stage_argument_checks_on_host(L):
    # null and misaligned pointers are rejected before any device work
    assert L.blk_rmsnorm(None, None, 4, 256, 1e-5, None, 1, None) == 1
    assert L.blk_rmsnorm(ctypes.c_void_p(0x1001), ctypes.c_void_p(0x2000), 4, 256, 1e-5,
                         ctypes.c_void_p(0x3000), 1, None) == 3
    assert L.blk_rmsnorm(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), 4, 260, 1e-5,
                         ctypes.c_void_p(0x3000), 1, None) == 2
    assert L.blk_forward(None, None, 1, 1, None, None, -1, None, None, 0, None, None) == 1
    assert L.blk_workspace_bytes(None, 1, 1, 0) == 0
    assert L.blk_destroy(None) == 0


def test_debug_gemm_argument_checks_on_host(L):
    # the bare GEMM's sizes, split and CTA-pair options are checked before any device work
    a, b, c = (ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000))
    gemm = L.blk_debug_gemm_bf16
    assert gemm(a, b, c, 256, 256, 64, 96, 1, 0, None) == 1    # a tile width not built
    assert gemm(a, b, c, 256, 256, 60, 256, 1, 0, None) == 1   # K not a multiple of 8
    assert gemm(a, b, c, 256, 256, 64, 256, 2, 0, None) == 1   # split-K needs 64-wide tiles
    assert gemm(a, b, c, 256, 256, 64, 64, 2, 1, None) == 1    # a CTA pair takes no K split
    assert gemm(a, b, c, 256, 256, 64, 128, 1, 1, None) == 1   # ... and tiles of 192 columns or more
    assert b"pair" in L.blk_last_error_message()
    assert gemm(ctypes.c_void_p(0x1008), b, c, 256, 256, 64, 256, 1, 1, None) == 3  # misaligned
