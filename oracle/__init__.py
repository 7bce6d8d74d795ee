"""fp64 CPU oracle for one Llama-style decoder block (test infrastructure).

This package is the checker, not the product. Only the test suite, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
it. It shares no code with the CUDA path under ``llama_family_decoder_gb300``.
"""
from .block import (  # noqa: F401
    BlockConfig,
    RopeScaling,
    rope_attention_factor,
    rms_norm,
    rope_inv_freq,
    rope,
    causal_gqa_attention,
    silu,
    sigmoid,
    relu2,
    xielu,
    xielu_effective,
    softplus,
    block_forward,
    padding_run,
    mlp,
    decode_step,
    prefill_with_cache,
    model_forward,
)
