"""Known-answer GEMMs.  Small-integer operands are exact in bf16 and in e4m3,
and every sum stays below 2^24, so each fp32 accumulation order gives the
exact integer.  The stored bf16 is then that integer rounded once, to nearest
even.  The library's output must match bit for bit, for:
  * every operand layout (A K-major or MN-major, B K-major or MN-major);
  * both kernel forms (SM pairs, one SM per tile);
  * power-of-two row / column scales (exact in fp32);
  * the grouped launch of the first layer's data and weight gradients;
  * e4m3 operands with unit scales;
  * the generic 8-bit GEMM for every layout and every pair of formats
    (e4m3 / e5m2), with power-of-two operand scales.
Ragged sizes span several tiles in every dimension.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, section 尾声: the mainloop is a tiled multiply-accumulate
and the epilogue sees the exact accumulator).
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests._parity import assert_device_ok

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from tests.test_gpu_parity import pairing  # noqa: E402,F401


def ints(shape, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int64)


def exact_bf16(A, Bt, row=None, col=None):
    """bf16 of the exact product A Bt^T (int64), optionally times power-of-two
    row / column scales, rounded once."""
    v = (A @ Bt.T).to(torch.float64)
    if row is not None:
        v = v * row.to(torch.float64)[:, None]
    if col is not None:
        v = v * col.to(torch.float64)[None, :]
    assert v.numel() == 0 or float(v.abs().max()) < 2 ** 24
    return v.to(torch.float32).to(torch.bfloat16)


def dev_bf16(t):
    return t.to(torch.bfloat16).cuda()


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K", [(520, 776, 1000), (256, 256, 64), (8, 8, 8)])
def test_gemm_layouts_bit_exact(a_mn, b_mn, M, N, K, pairing):
    A = ints((M, K), -3, 3, 1)
    Bt = ints((N, K), -3, 3, 2)
    Ad = dev_bf16(A.T.contiguous() if a_mn else A)
    Bd = dev_bf16(Bt.T.contiguous() if b_mn else Bt)
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm(Ad, a_mn, Bd, b_mn, Cd, M, N, K)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(Cd.cpu(), exact_bf16(A, Bt))


def test_power_of_two_scales_bit_exact(pairing):
    M, N, K = 300, 520, 200
    A = ints((M, K), -4, 4, 3)
    Bt = ints((N, K), -4, 4, 4)
    row = torch.pow(2.0, ints((M,), -3, 3, 5).to(torch.float32))
    col = torch.pow(2.0, ints((N,), -2, 2, 6).to(torch.float32)).to(torch.bfloat16)
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm(dev_bf16(A), False, dev_bf16(Bt), False, Cd, M, N, K, row_scale=row.cuda(), col_scale=col.cuda())
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(Cd.cpu(), exact_bf16(A, Bt, row, col.to(torch.float32)))


@pytest.mark.parametrize("M,K1,d", [(1000, 520, 328), (4096, 1024, 1024)])
def test_grouped_first_layer_backward_bit_exact(M, K1, d):
    dH = ints((M, d), -2, 2, 7)
    X = ints((M, K1), -2, 2, 8)
    W1t = ints((d, K1), -2, 2, 9)
    dX = torch.empty(M, K1, dtype=torch.bfloat16, device="cuda")
    dW1t = torch.empty(d, K1, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm_res_prms_bwd(dev_bf16(dH), dev_bf16(X), dev_bf16(W1t), dX, dW1t, None)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(dX.cpu(), exact_bf16(dH, W1t.T.contiguous()))      # dX = dH W1t
    assert torch.equal(dW1t.cpu(), exact_bf16(dH.T.contiguous(), X.T.contiguous()))  # dW1t = dH^T X


def test_fp8_operands_bit_exact(pairing):
    M, N2, K = 300, 776, 1024
    A = ints((M, K), -4, 4, 10)
    Bt = ints((N2, K), -4, 4, 11)
    Aq = torch.from_numpy(O.e4m3_encode(A.numpy().astype(np.float64))).cuda()
    Bq = torch.from_numpy(O.e4m3_encode(Bt.numpy().astype(np.float64))).cuda()
    one = torch.ones(1, device="cuda")
    rstd = torch.ones(M, device="cuda")
    out = torch.empty(M, N2, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm_rowscale_swiglu_fp8(Aq, one, Bq, one, rstd, out, None, C.CODA_EPI_PLAIN)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(out.cpu(), exact_bf16(A, Bt))


ENC = {0: O.e4m3_encode, 1: O.e5m2_encode}


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True)])
@pytest.mark.parametrize("a_fmt,b_fmt", [(0, 0), (1, 0), (0, 1), (1, 1)], ids=["e4e4", "e5e4", "e4e5", "e5e5"])
def test_fp8_gemm_layouts_and_formats_bit_exact(a_mn, b_mn, a_fmt, b_fmt, pairing):
    M, N, K = 528, 784, 1024       # ragged tiles in M and N, 8 k-blocks of 128
    A = ints((M, K), -4, 4, 12)
    Bt = ints((N, K), -4, 4, 13)
    Aq = ENC[a_fmt]((A.T if a_mn else A).numpy().astype(np.float64))
    Bq = ENC[b_fmt]((Bt.T if b_mn else Bt).numpy().astype(np.float64))
    sA = torch.tensor([0.5], device="cuda")
    sB = torch.tensor([4.0], device="cuda")
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm_fp8(torch.from_numpy(np.ascontiguousarray(Aq)).cuda(), a_mn, a_fmt, sA,
                    torch.from_numpy(np.ascontiguousarray(Bq)).cuda(), b_mn, b_fmt, sB, Cd, M, N, K)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(Cd.cpu(), exact_bf16(A, Bt, torch.full((M,), 2.0)))   # sA * sB = 2


@pytest.mark.parametrize("K", [300, 1, 0])
def test_fp8_gemm_ragged_token_k_bit_exact(K, pairing):
    """Both operands MN-major: K is their row count (a token count for a weight
    gradient), ragged against the 128-deep k-block; K = 0 is an empty sum."""
    M, N = 544, 336
    A = ints((M, K), -4, 4, 14)
    Bt = ints((N, K), -4, 4, 15)
    Aq = np.ascontiguousarray(O.e5m2_encode(A.T.numpy().astype(np.float64)))
    Bq = np.ascontiguousarray(O.e4m3_encode(Bt.T.numpy().astype(np.float64)))
    Cd = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm_fp8(torch.from_numpy(Aq).cuda(), True, 1, None, torch.from_numpy(Bq).cuda(), True, 0, None,
                    Cd, M, N, K)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(Cd.cpu(), exact_bf16(A, Bt))


@pytest.mark.parametrize("M,K1,d", [(1000, 528, 336), (300, 256, 512), (1, 256, 256), (0, 256, 256),
                                    (4096, 1024, 1024)])
def test_fp8_grouped_first_layer_backward_bit_exact(M, K1, d, pairing):
    """dX = sdH sW1 dH W1 and dW1t = sdH sX dH^T X from e5m2 dH and e4m3 W1 / X
    codes, one grouped launch with SM pairing (two launches without): the
    exact products times the power-of-two scales, rounded once (ragged tiles,
    ragged token count, one row, an empty batch)."""
    dH = ints((M, d), -4, 4, 16)
    X = ints((M, K1), -4, 4, 17)
    W1t = ints((d, K1), -4, 4, 18)
    dHq = torch.from_numpy(np.ascontiguousarray(O.e5m2_encode(dH.numpy().astype(np.float64)))).cuda()
    Xq = torch.from_numpy(np.ascontiguousarray(O.e4m3_encode(X.numpy().astype(np.float64)))).cuda()
    W1q = torch.from_numpy(np.ascontiguousarray(O.e4m3_encode(W1t.numpy().astype(np.float64)))).cuda()
    sdH, sX, sW1 = (torch.tensor([v], device="cuda") for v in (0.5, 2.0, 0.25))
    dX = torch.full((M, K1), 7.0, dtype=torch.bfloat16, device="cuda")
    dW1t = torch.full((d, K1), 7.0, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm_res_prms_bwd_fp8(dHq, C.E5M2, sdH, Xq, sX, W1q, sW1, C.E4M3, dX, dW1t)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(dX.cpu(), exact_bf16(dH, W1t.T.contiguous(), torch.full((M,), 0.125)))   # sdH * sW1
    assert torch.equal(dW1t.cpu(), exact_bf16(dH.T.contiguous(), X.T.contiguous(), torch.full((d,), 1.0)))  # sdH * sX
