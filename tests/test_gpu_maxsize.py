"""Maximum sizes: outputs past 2^31 elements and 4 GiB, so that every byte
offset the epilogues and combine kernels form needs 64 bits.

* A plain GEMM whose output has more than 2^31 elements (integer operands:
  one exact result whatever the summation order), on SM pairs and single
  SMs, A read K-major and MN-major; sampled rows on both sides of the
  2^31-element and 2^32-byte boundaries and the last rows, prefilled with
  NaN so that an unwritten element shows.
* The 7B block forward and backward at 16x the 7B token count (M = 131072:
  z and dP hold 3.8e9 elements, 7.5 GB each): row-wise outputs on sampled
  rows, including the rows that straddle the 2^31-, 2^32- and 3*2^31-byte
  offsets of z and dP, against the oracle fed the GPU's own stage inputs;
  the reductions over all rows (dg, dW2t, dW1t) against cuBLAS in fp32 on
  the same inputs (relative Frobenius).

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, sections 尾声 and 实验结果: the block at the 7B hidden size).
"""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import BlockShape, block_inputs
from tests._parity import assert_device_ok, assert_elem, assert_frob, f64
from tests.test_gpu_exact import ints

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402


def boundary_rows(M, pitch_bytes, extra=()):
    """Rows holding the byte offsets k * 2^31 of a [M][pitch] tensor, their
    neighbours, the first and last rows."""
    rows = {0, 1, M - 2, M - 1, *extra}
    k = 1
    while k * 2 ** 31 < M * pitch_bytes:
        r = (k * 2 ** 31) // pitch_bytes
        rows |= {r - 1, r, r + 1}
        k += 1
    return sorted(r for r in rows if 0 <= r < M)


@pytest.mark.parametrize("pair,a_mn", [(True, False), (True, True), (False, False)],
                         ids=["sm_pair", "sm_pair_a_mn", "single_sm"])
def test_gemm_output_past_2_31_elements(pair, a_mn):
    M, N, K = 557056, 4096, 72          # 2.28e9 output elements, 4.6 GB
    assert M * N > 2 ** 31
    A = ints((M, K), -3, 3, 61)
    Bt = ints((N, K), -3, 3, 62)
    Ad = (A.T.contiguous() if a_mn else A).to(torch.bfloat16).cuda()
    # an MN-major A goes with an MN-major B (the layouts the path uses)
    Bd = (Bt.T.contiguous() if a_mn else Bt).to(torch.bfloat16).cuda()
    Cd = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    C.coda_set_sm_pairing(pair)
    try:
        C.coda_gemm(Ad, a_mn, Bd, a_mn, Cd, M, N, K)
        torch.cuda.synchronize()
    finally:
        C.coda_set_sm_pairing(True)
    assert_device_ok()
    rows = boundary_rows(M, N * 2, extra=(2 ** 31 // N - 1, 2 ** 31 // N, 2 ** 31 // N + 1))
    got = Cd[torch.as_tensor(rows, device="cuda")].cpu()
    ref = (A[rows].to(torch.float64) @ Bt.to(torch.float64).T).to(torch.float32).to(torch.bfloat16)
    assert torch.equal(got, ref)
    del Cd


def test_block_at_16x_the_7b_tokens():
    s = BlockShape("7b_m131072", 131072, 4096, 4096, 28672)
    M, d, F, K1 = s.M, s.d, s.F, s.K1
    x = block_inputs(s, 0, "cuda")
    b = BlockBuffers(x)
    b.forward()
    b.backward_stages()
    assert_device_ok()
    rows = boundary_rows(M, s.N2 * 2, extra=(M // 2,))
    ri = torch.as_tensor(rows, device="cuda")
    W1t, W2t, g = f64(b.W1t), f64(b.W2t), f64(b.g)

    def r(t):
        return f64(t[ri])

    H = r(b.H)
    assert_elem(H, O.gemm_residual(r(b.X), W1t, r(b.R)), "H")
    assert_elem(r(b.psum), O.partial_sumsq(H, C.PARTIAL_COLS), "psum", tol=1e-4)
    rstd = r(b.rstd)
    assert_elem(rstd, O.rstd_from_partials(r(b.psum), d, s.eps), "rstd", tol=1e-5)
    z_ref = O.rowscale_gemm(H, f64(b.W2gt), rstd)
    assert_elem(r(b.z), z_ref, "z")
    assert_elem(r(b.out), O.swiglu(z_ref), "out")
    dP_ref, c_ref = O.stage_swiglu_bwd(r(b.dY), r(b.z), rstd, d)
    assert_elem(r(b.dP), dP_ref, "dP")
    assert_elem(r(b.c), c_ref, "c")
    dH_ref, _ = O.stage_dgrad2_rmsbwd(r(b.dP), W2t, g, H, r(b.c))
    # cuBLAS's counterpart from the 1024-row block that holds each sampled
    # row: asked for a handful of rows alone, cuBLAS picks a kernel that
    # splits the 28672-long sum, whose rounding is not that of a launch over
    # all the rows (with 1024 or more rows its fp32 sums match this
    # library's to the last bit on a zero-sum probe)
    acc = torch.stack([torch.mm(b.dP[(i // 1024) * 1024:(i // 1024 + 1) * 1024], b.W2t,
                                out_dtype=torch.float32)[i % 1024] for i in rows])
    dH_cub = (b.g.float() * acc - b.c[ri, None] * b.H[ri].float()).to(torch.bfloat16)
    assert_elem(r(b.dH), dH_ref, "dH", cublas=dH_cub)
    assert_elem(r(b.dX), O.stage_dgrad1(r(b.dH), W1t), "dX")
    # reductions over all 131072 rows: against cuBLAS (fp32 result) on the
    # same inputs, in row blocks
    gf = b.g.float()
    dg = torch.zeros(d, device="cuda")
    for s0 in range(0, M, 16384):
        s1 = min(M, s0 + 16384)
        acc = torch.mm(b.dP[s0:s1], b.W2t, out_dtype=torch.float32)
        dg += (acc * b.H[s0:s1].float()).sum(0)
        del acc
    assert_frob(b.dg, f64(dg), "dg vs cuBLAS")
    dW2 = torch.mm(b.dP.t(), b.H, out_dtype=torch.float32) * gf
    assert_frob(b.dW2t, f64(dW2), "dW2t vs cuBLAS")
    del dW2
    dW1 = torch.mm(b.dH.t(), b.X, out_dtype=torch.float32)
    assert_frob(b.dW1t, f64(dW1), "dW1t vs cuBLAS")
    del dW1, b, x
    torch.cuda.empty_cache()
