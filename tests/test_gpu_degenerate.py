"""Degenerate inputs of the block, against the oracle:

  * rows whose residual stream is exactly zero (X and R rows zero): h = 0,
    rstd = 1 / sqrt(eps), z = 0, and the row's data gradients vanish exactly
    (every product in the row is zero);
  * SwiGLU saturation: |z| up to about 200 in GEMM2's epilogue and up to 120
    in the SwiGLU backward, where exp overflows in fp32 and the sigmoid must
    come out as exactly 0 or 1 rather than NaN.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, section 尾声: RMSNorm through the partial sums of squares
and the deferred row scale; SwiGLU in the second GEMM's epilogue).
"""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import BlockShape, block_inputs
from tests._parity import assert_device_ok, assert_elem, assert_frob, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402
from tests.test_gpu_parity import pairing  # noqa: E402,F401

EPS = 1e-5


def test_zero_rows(pairing):
    s = BlockShape("zero_rows", 300, 200, 328, 528)
    x = {k: v.cuda() for k, v in block_inputs(s, 0, "cpu").items()}
    rows = [0, 77, 299]
    x["X"][rows] = 0
    x["R"][rows] = 0
    b = BlockBuffers(x)
    b.forward()
    b.backward_stages()
    torch.cuda.synchronize()
    assert_device_ok()
    ri = torch.as_tensor(rows, device="cuda")
    assert torch.count_nonzero(b.H[ri]) == 0
    np.testing.assert_allclose(f64(b.rstd)[rows], 1.0 / np.sqrt(EPS), rtol=1e-6)
    for name in ("z", "out", "dP", "dH", "dX"):
        assert torch.count_nonzero(getattr(b, name)[ri]) == 0, name
    assert torch.count_nonzero(b.c[ri]) == 0
    assert torch.isfinite(b.dg).all() and torch.isfinite(b.dW2t.float()).all()
    ref = O.block_backward(*(f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t", "dY")), EPS, True)
    for k_gpu, k_ref in (("out", "out"), ("dH", "dR"), ("dX", "dX"), ("dW1t", "dW1t"), ("dW2t", "dW2t"),
                         ("dg", "dg")):
        assert_frob(getattr(b, k_gpu), ref[k_ref], f"{k_gpu} with zero rows")


def test_gemm2_epilogue_saturation(pairing):
    """z = rstd * (H W2g) with a large row scale: silu's sigmoid saturates at
    0 (exp overflowing) and 1; out is graded against the oracle's SwiGLU of
    the GPU's own z, and z against the oracle's row-scaled GEMM."""
    M, d, F = 264, 256, 264
    g = torch.Generator().manual_seed(31)
    H = torch.randn(M, d, generator=g).to(torch.bfloat16)
    W2g = (torch.randn(2 * F, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    rstd = torch.full((M,), 60.0)
    rstd[::3] = 120.0
    z = torch.empty(M, 2 * F, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm_rowscale_swiglu(H.cuda(), W2g.cuda(), rstd.cuda(), out, z, C.CODA_EPI_SWIGLU)
    torch.cuda.synchronize()
    assert_device_ok()
    zf = f64(z)
    assert np.abs(zf).max() > 100 and np.isfinite(zf).all()
    z_ref = O.rowscale_gemm(f64(H), f64(W2g), f64(rstd))
    assert_elem(z, z_ref, "z (saturating)")
    assert torch.isfinite(out.float()).all()
    # out is formed from the epilogue's fp32 z, not from the bf16 z it stores:
    # the oracle takes the exact z of the same stage inputs
    z32 = rstd.cuda()[:, None] * torch.mm(H.cuda(), W2g.cuda().t(), out_dtype=torch.float32)
    out_cub = (z32[:, :F] * torch.sigmoid(z32[:, :F]) * z32[:, F:]).to(torch.bfloat16)
    assert_elem(out, O.swiglu(z_ref), "out (saturating)", cublas=out_cub)


def test_swiglu_backward_saturation():
    M, F, d = 130, 264, 256
    g = torch.Generator().manual_seed(32)
    z = (torch.rand(M, 2 * F, generator=g) * 240 - 120).to(torch.bfloat16)
    z[:, :8] = torch.tensor([-120.0, -100.0, -88.0, -30.0, 30.0, 88.0, 100.0, 120.0]).to(torch.bfloat16)
    dY = torch.randn(M, F, generator=g).to(torch.bfloat16)
    rstd = 0.5 + torch.rand(M, generator=g)
    dP = torch.empty(M, 2 * F, dtype=torch.bfloat16, device="cuda")
    c = torch.empty(M, device="cuda")
    C.coda_swiglu_bwd(dY.cuda(), z.cuda(), rstd.cuda(), dP, c, d)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.isfinite(dP.float()).all() and torch.isfinite(c).all()
    dP_ref, c_ref = O.stage_swiglu_bwd(f64(dY), f64(z), f64(rstd), d)
    assert_elem(dP, dP_ref, "dP (saturating)")
    assert_elem(c, c_ref, "c (saturating)")
