"""The bare tcgen05 GEMM core (TMA -> smem ring -> tcgen05.mma -> TMEM -> tcgen05.ld)
against an fp64 matmul of the same bf16 operands, over tile shapes, ragged
M/N/K tails, and the swap-AB split-K partial layout used by decode."""
import pytest
import torch

from llama_family_decoder_gb300.binding import debug_gemm_bf16

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    b = torch.randn(N, K, generator=g).to(torch.bfloat16)
    return a, b


@pytest.mark.parametrize("M,N,K,bn", [
    (128, 256, 64, 256),      # one tile, one k-block
    (256, 512, 1024, 256),    # several tiles and k-blocks
    (200, 1000, 1000, 256),   # ragged M, N and K
    (300, 384, 520, 128),
    (64, 192, 4096, 64),
    (1000, 136, 136, 128),
    (384, 4096, 1000, 224),   # 18 full 224-wide tiles plus a 64-column tail
    (300, 1000, 520, 192),
])
def test_gemm_matches_fp64(M, N, K, bn):
    a, b = _operands(M, N, K, seed=M + N + K)
    c = debug_gemm_bf16(a.cuda(), b.cuda(), bn=bn)
    torch.cuda.synchronize()
    ref = a.double() @ b.double().T
    # bf16 output rounding (<= 2^-9 relative) plus a small fp32-accumulation allowance
    bound = 2.0 ** -8 * ref.abs() + 1e-4 * ref.pow(2).mean().sqrt()
    bad = ((c.double().cpu() - ref).abs() > bound).sum()
    assert bad == 0, int(bad)


@pytest.mark.parametrize("M,N,K,bn", [
    (256, 256, 64, 256),      # one pair tile, one k-block
    (512, 768, 1024, 256),    # several pair tiles and k-blocks
    (300, 1000, 1000, 224),   # ragged M (the odd CTA's rows past M), N and K
    (100, 400, 520, 192),     # the odd CTA's rows all past M, its B half of the last tile too
    (2048, 4096, 4096, 256),  # more tiles than pairs: the persistent loop
])
def test_gemm_cta_pair_matches_fp64(M, N, K, bn):
    # tcgen05 cta_group::2: 256-row tiles over two CTAs, each holding half of B
    a, b = _operands(M, N, K, seed=3 * M + N + K)
    c = debug_gemm_bf16(a.cuda(), b.cuda(), bn=bn, pair=True)
    torch.cuda.synchronize()
    ref = a.double() @ b.double().T
    bound = 2.0 ** -8 * ref.abs() + 1e-4 * ref.pow(2).mean().sqrt()
    bad = ((c.double().cpu() - ref).abs() > bound).sum()
    assert bad == 0, int(bad)


@pytest.mark.parametrize("M,N,K,splits", [(64, 384, 4096, 4), (5, 1000, 1000, 3), (64, 6144, 512, 2)])
def test_gemm_split_partials(M, N, K, splits):
    a, b = _operands(M, N, K, seed=7 * M + N)
    parts = debug_gemm_bf16(a.cuda(), b.cuda(), bn=64, split_k=splits)
    torch.cuda.synchronize()
    ref = a.double() @ b.double().T
    got = parts.double().sum(0).cpu()
    err = (got - ref).abs().max() / ref.pow(2).mean().sqrt()
    assert err < 1e-5, float(err)  # fp32 partial sums, no output rounding
