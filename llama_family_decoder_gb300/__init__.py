"""GB300-native (sm_103a) forward pass of one Llama-style decoder block.

The compute lives in libblk.so (C ABI in include/blk.h, CUDA kernels under
csrc/); this package holds its ctypes binding and the seeded synthetic-input
generator.
"""
from .binding import (  # noqa: F401
    BlkError,
    DecoderBlock,
    lib,
    make_weights_struct,
    rmsnorm,
    set_wait_timeout_ns,
    xielu_effective,
)
