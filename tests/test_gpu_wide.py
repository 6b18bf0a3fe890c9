"""GEMMs on 256 x 512 pair tiles (coda_set_wide_tiles): two 256-column
accumulator halves per A tile, the first J k-blocks feeding only the first
half and repeated at the end for the second, so that one half's epilogue
runs while the other accumulates; a last wave of at most half the SM pairs
runs as 256-column half tiles on a ring of 32 KB stages.  Only GEMMs with
K of at least 16384 take them (the RMSNorm-backward data gradient of the
block at the 7B and 70B widths).

Checked with wide tiles on, at sizes where the launcher takes them (asked
of the library's own rule through its test hook), in each schedule: all
wide tiles, wide tiles then half tiles, half tiles only:
  * known-answer integer GEMMs bit-exact in every operand layout (any fp32
    summation order gives the exact integer);
  * the block's dgrad2 with the RMSNorm-backward epilogue elementwise
    against the oracle fed the GPU's own stage inputs, with cuBLAS on the
    same inputs beside it, and close to the 256-column tiles' result; the
    other backward stages (on 256-column tiles at this K) beside it;
  * two runs bit-identical.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, section 尾声: the epilogue program sees a whole tile's
accumulator; here each 256-column half of a wide tile is such a tile).
"""
import pytest
import torch

import oracle as O
from coda_inputs import BlockShape, block_inputs
from tests._parity import assert_device_ok, assert_elem, assert_frob, edge_sample, f64
from tests.test_gpu_exact import ints

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402

LEAD = 8


def exact(A, Bt):
    """bf16 of the exact integer product A Bt^T (float64 BLAS: every partial
    sum is an integer below 2^53)."""
    v = A.to(torch.float64) @ Bt.to(torch.float64).T
    assert float(v.abs().max()) < 2 ** 24
    return v.to(torch.float32).to(torch.bfloat16)


@pytest.fixture
def wide_on():
    C.coda_set_sm_pairing(True)
    C.coda_set_wide_tiles(LEAD)
    yield
    torch.cuda.synchronize()
    C.coda_set_wide_tiles(0)


def test_wide_option_range():
    lib = C.load_library()
    h = C.handle()
    assert lib.coda_set_wide_tiles(h, -1) == 1  # CODA_ERR_INVALID_ARG
    assert lib.coda_set_wide_tiles(h, 65) == 1
    assert lib.coda_set_wide_tiles(h, 0) == 0
    assert C.coda_debug_wide_applies(8192, 4096, 28672) == 0
    C.coda_set_wide_tiles(8)
    try:
        assert C.coda_debug_wide_applies(8192, 4096, 28672) == 1   # 7B dgrad2
        assert C.coda_debug_wide_applies(28672, 4096, 8192) == 0   # 7B wgrad2: K too short
        assert C.coda_debug_wide_applies(8192, 3840, 28672) == 0   # an odd number of column tiles
    finally:
        C.coda_set_wide_tiles(0)


# (M, N, K), K at least 256 k-blocks: all wide tiles (64 on 76 pairs), wide
# tiles then half tiles (80: 76 + 4 split in 8 halves), half tiles only (32),
# ragged edges in M, N and K
SHAPES = [(2048, 4096, 16384), (2560, 4096, 16384), (1024, 4096, 16384), (1800, 3904, 16448)]


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_wide_gemm_bit_exact(a_mn, b_mn, M, N, K, wide_on):
    assert C.coda_debug_wide_applies(M, N, K) == 1
    A = ints((M, K), -3, 3, 31)
    Bt = ints((N, K), -3, 3, 32)
    Ad = (A.T.contiguous() if a_mn else A).to(torch.bfloat16).cuda()
    Bd = (Bt.T.contiguous() if b_mn else Bt).to(torch.bfloat16).cuda()
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm(Ad, a_mn, Bd, b_mn, Cd, M, N, K)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(Cd.cpu(), exact(A, Bt))


# dgrad2 (M x d x 2F = 2560 x 4096 x 16384): 80 wide tiles, wide then half
# tiles; wgrad2 (K = M = 2560) stays on 256-column tiles
WIDE_BLOCK = BlockShape("wide", 2560, 1024, 4096, 16384)


def test_wide_block_stages_against_oracle(wide_on):
    s = WIDE_BLOCK
    assert C.coda_debug_wide_applies(s.M, s.d, s.N2) == 1
    assert C.coda_debug_wide_applies(s.N2, s.d, s.M) == 0
    x = block_inputs(s, 0, "cuda")
    b = BlockBuffers(x)
    b.forward()
    b.backward_stages()
    assert_device_ok()
    W2t, g = f64(x["W2t"]), f64(x["g"])
    H = f64(b.H)
    dH_ref, dg_ref = O.stage_dgrad2_rmsbwd(f64(b.dP), W2t, g, H, f64(b.c))
    acc = torch.mm(b.dP, b.W2t, out_dtype=torch.float32)
    dH_cub = (b.g.float() * acc - b.c[:, None] * b.H.float()).to(torch.bfloat16)
    dg_cub = (acc * b.H.float()).sum(0)
    del acc
    assert_elem(b.dH, dH_ref, "dH", cublas=dH_cub)
    assert_elem(b.dg, dg_ref, "dg", cublas=dg_cub)
    # the weight gradient sums M = 2560 rows (rms ~ 45): at least 64 whole
    # rows and 64 whole columns (tile edges included), as at full size, with
    # cuBLAS on the same inputs
    cub = (torch.mm(b.dP.t(), b.H, out_dtype=torch.float32) * b.g.float()).to(torch.bfloat16)
    dP = f64(b.dP)
    ri, ci = edge_sample(s.N2, 64, 5), edge_sample(s.d, 64, 6)
    assert_elem(f64(b.dW2t)[ri], O.stage_wgrad2(H, dP[:, ri], g), "dW2t rows", cublas=f64(cub)[ri])
    assert_elem(f64(b.dW2t)[:, ci], O.stage_wgrad2(H[:, ci], dP, g[ci]), "dW2t columns", cublas=f64(cub)[:, ci])
    # the same stages on 256-column tiles: equal up to fp32 summation order,
    # so the bf16 outputs differ at most where a rounding flips, by one bf16
    # ulp (2^-8 relative) there
    got = {k: getattr(b, k).clone() for k in ("dH", "dg", "dW2t", "dX", "dW1t")}
    C.coda_set_wide_tiles(0)
    b.backward_stages()
    torch.cuda.synchronize()
    for k, v in got.items():
        assert_frob(v, getattr(b, k), f"{k} wide vs 256-column", tol=2.0 ** -8)
    C.coda_set_wide_tiles(LEAD)


def test_wide_is_deterministic(wide_on):
    x = block_inputs(WIDE_BLOCK, 1, "cuda")
    b = BlockBuffers(x)
    b.step()
    torch.cuda.synchronize()
    first = {k: getattr(b, k).clone() for k in ("out", "dH", "dg", "dW2t", "dX", "dW1t")}
    for _ in range(2):
        b.step()
        torch.cuda.synchronize()
        for k, v in first.items():
            assert torch.equal(getattr(b, k), v), k
    assert_device_ok()
