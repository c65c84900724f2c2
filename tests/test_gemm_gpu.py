"""The tcgen05/TMA GEMM (the building block of the materialise-P path)
against a float64 CPU matrix product, for every operand major-ness."""

import pytest
import torch

from parity_util import relerr

pytestmark = pytest.mark.gpu


def _operands(batch, M, N, K, ak, bk, seed):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(batch, M, K, generator=g).to(torch.bfloat16)   # logical A (M x K)
    B = torch.randn(batch, K, N, generator=g).to(torch.bfloat16)   # logical B (K x N)
    a_st = A if ak else A.transpose(1, 2).contiguous()              # [M][K] or [K][M]
    b_st = B.transpose(1, 2).contiguous() if bk else B              # [N][K] or [K][N]
    ref = torch.matmul(A.double(), B.double())
    return a_st, b_st, ref


@pytest.mark.parametrize("ak,bk", [(1, 1), (1, 0), (0, 1), (0, 0)])
@pytest.mark.parametrize("batch,M,N,K", [(1, 128, 128, 64), (2, 256, 256, 192),
                                         (3, 200, 136, 72), (1, 128, 64, 128),
                                         (2, 384, 512, 320)])
@pytest.mark.parametrize("c_f32", [True, False])
def test_gemm(cuda_dev, ak, bk, batch, M, N, K, c_f32):
    from io_aware_exact_05_gb300 import attn

    a, b, ref = _operands(batch, M, N, K, ak, bk, seed=M * 7 + N + K + ak * 2 + bk)
    c = torch.full((batch, M, N), float("nan"), device=cuda_dev,
                   dtype=torch.float32 if c_f32 else torch.bfloat16)
    attn.attn_gemm_bf16(a.to(cuda_dev), b.to(cuda_dev), c, batch, M, N, K, ak, bk, alpha=0.5)
    assert attn.attn_status() == 0
    err = relerr(c, 0.5 * ref)
    assert err <= (1e-5 if c_f32 else 1e-2), err


def test_gemm_ragged_kmajor(cuda_dev):
    from io_aware_exact_05_gb300 import attn

    batch, M, N, K = 2, 130, 70, 40
    a, b, ref = _operands(batch, M, N, K, 1, 1, seed=5)
    c = torch.full((batch, M, N), float("nan"), device=cuda_dev)
    attn.attn_gemm_bf16(a.to(cuda_dev), b.to(cuda_dev), c, batch, M, N, K, 1, 1)
    assert attn.attn_status() == 0
    assert relerr(c, ref) <= 1e-5


@pytest.mark.parametrize("M,N,c_f32", [(130, 72, True), (130, 70, True), (200, 72, False),
                                       (200, 68, False), (257, 40, True)])
def test_gemm_ragged_epilogues(cuda_dev, M, N, c_f32):
    # C rows that are 16-byte multiples go out through TMA tile stores (rows
    # and columns past C's edge clipped by the tensor map), others through
    # direct stores: both, with ragged M and N
    from io_aware_exact_05_gb300 import attn

    batch, K = 2, 48
    a, b, ref = _operands(batch, M, N, K, 1, 1, seed=M + N)
    c = torch.full((batch, M, N), float("nan"), device=cuda_dev,
                   dtype=torch.float32 if c_f32 else torch.bfloat16)
    attn.attn_gemm_bf16(a.to(cuda_dev), b.to(cuda_dev), c, batch, M, N, K, 1, 1)
    assert attn.attn_status() == 0
    assert relerr(c, ref) <= (1e-5 if c_f32 else 1e-2)


@pytest.mark.parametrize("M,N,ak,bk", [(300, 260, 1, 1), (300, 264, 1, 1), (129, 256, 1, 1),
                                       (264, 264, 0, 0), (264, 264, 1, 0)])
def test_gemm_two_m_tiles(cuda_dev, M, N, ak, bk):
    # long contractions with bf16 outputs and N > 128 run two 128-row M tiles
    # per CTA against the same staged B block: a second tile that is partly
    # or wholly past M, C rows through TMA tile stores (N * 2 bytes a
    # multiple of 16) or direct stores, and MN-major operands
    from io_aware_exact_05_gb300 import attn

    batch, K = 2, 320
    a, b, ref = _operands(batch, M, N, K, ak, bk, seed=M * 3 + N + ak + 2 * bk)
    c = torch.full((batch, M, N), float("nan"), device=cuda_dev, dtype=torch.bfloat16)
    attn.attn_gemm_bf16(a.to(cuda_dev), b.to(cuda_dev), c, batch, M, N, K, ak, bk, alpha=0.25)
    assert attn.attn_status() == 0
    assert relerr(c, 0.25 * ref) <= 1e-2
