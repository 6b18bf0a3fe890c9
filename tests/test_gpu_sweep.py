"""A sweep of GEMM shapes around the tile edges, bit-exact.

Integer-valued bf16 operands in [-3, 3] make every fp32 partial sum an
exact integer, so C = bf16(A B^T) has one correct value whatever the
summation order.  The shapes put M, N and K on both sides of the 256-row /
256-column tile and 64-deep k-block edges (extents are multiples of 8, the
boundary's rule), give launches of fewer tiles than SM pairs and of more
(several rounds of the persistent grid, a last raster group narrower than
8 row tiles), and K of one partial k-block.  Every operand layout the path
uses, on SM pairs and on single SMs.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, section 尾声: the GEMM mainloop whose accumulator the
epilogue programs read).
"""
import pytest
import torch

from tests._parity import assert_device_ok
from tests.test_gpu_exact import ints

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")

# (M, N, K)
SHAPES = [
    (8, 8, 8),          # one tile, one partial k-block
    (8, 264, 72),       # one row, a column tile edge crossed by 8, K over one k-block by 8
    (264, 8, 136),      # the transpose case
    (248, 256, 64),     # just under a tile row, exactly one tile column and k-block
    (256, 248, 56),     # exactly one tile row, just under a column tile and a k-block
    (264, 264, 264),    # every extent one tile plus 8
    (520, 9992, 8),     # 3 x 40 tiles (more than one round), K = 8
    (1032, 4104, 200),  # 5 x 17 tiles, ragged in all three extents
    (2056, 2568, 72),   # 9 x 11 tiles: the last raster group is one row tile wide
    (4104, 136, 1032),  # 17 x 1 tiles, K = 16 k-blocks plus 8
]


def exact(A, Bt):
    """bf16 of the exact integer product A Bt^T (float64 BLAS: every partial
    sum is an integer below 2^53), rounded once."""
    v = A.to(torch.float64) @ Bt.to(torch.float64).T
    assert float(v.abs().max()) < 2 ** 24
    return v.to(torch.float32).to(torch.bfloat16)


@pytest.mark.parametrize("pair", [True, False], ids=["sm_pair", "single_sm"])
@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_shape_sweep_bit_exact(M, N, K, a_mn, b_mn, pair):
    A = ints((M, K), -3, 3, 41)
    Bt = ints((N, K), -3, 3, 42)
    Ad = (A.T.contiguous() if a_mn else A).to(torch.bfloat16).cuda()
    Bd = (Bt.T.contiguous() if b_mn else Bt).to(torch.bfloat16).cuda()
    Cd = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    C.coda_set_sm_pairing(pair)
    try:
        C.coda_gemm(Ad, a_mn, Bd, b_mn, Cd, M, N, K)
        torch.cuda.synchronize()
    finally:
        C.coda_set_sm_pairing(True)
    assert_device_ok()
    got = Cd.cpu()
    ref = exact(A, Bt)
    bad = (got != ref).nonzero()
    assert bad.numel() == 0, f"{bad.shape[0]} elements differ, first at {bad[0].tolist()}"
