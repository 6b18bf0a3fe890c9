"""FP8 (e4m3, per-tensor scale) operands for the same epilogue programs
(Synced write-up, section 背景: FP8 makes the matmul faster, raising the share
of the memory-bound operations the epilogues absorb).

* quantisation: codes and scales bit-exact against the oracle's e4m3
  rounding (the division by the scale in fp32 on both sides);
* GEMMs: against the oracle fed the dequantised codes (elementwise bar);
* end to end against the bf16-input oracle: relative Frobenius <= 8e-2,
  the bound two e4m3 roundings per product give (unit roundoff 2^-4 each,
  about 3.6 % rms per operand, combined over both GEMMs)."""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import BlockShape, block_inputs
from tests._parity import assert_device_ok, assert_elem, assert_frob, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")


@pytest.fixture(params=[True, False], ids=["sm_pair", "single_sm"])
def pairing(request):
    C.coda_set_sm_pairing(request.param)
    yield request.param
    C.coda_set_sm_pairing(True)


def quantize(x, g=None):
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty(2, device="cuda")
    C.coda_fp8_quantize(x, q, s, g)
    return q, s


def dequant(q, s):
    return O.e4m3_decode(q.cpu().numpy()) * float(s[1].item())


@pytest.mark.parametrize("shape,scale", [((300, 528), 1.0), ((64, 4096), 0.02), ((8, 16), 1e-3)])
def test_quantize_codes_bit_exact(shape, scale):
    g = torch.Generator().manual_seed(shape[0])
    x = (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)
    q, s = quantize(x.cuda())
    assert_device_ok()
    xf = x.float().numpy()
    amax = np.float32(np.max(np.abs(xf)))
    assert s[0].item() == amax
    sc = O.fp8_scale(xf)
    assert np.float32(s[1].item()) == sc
    assert np.array_equal(q.cpu().numpy(), O.fp8_quantize(xf, sc))


def test_quantize_with_folded_weight_bit_exact():
    g = torch.Generator().manual_seed(3)
    W = (torch.randn(528, 336, generator=g) * 0.02).to(torch.bfloat16)
    gw = (torch.rand(336, generator=g) + 0.5).to(torch.bfloat16)
    q, s = quantize(W.cuda(), gw.cuda())
    assert_device_ok()
    v = W.float().numpy() * gw.float().numpy()[None, :]      # exact in fp32
    sc = O.fp8_scale(v)
    assert np.float32(s[1].item()) == sc
    assert np.array_equal(q.cpu().numpy(), O.fp8_quantize(v, sc))


@pytest.mark.parametrize("shape,scale", [((300, 528), 1.0), ((64, 4096), 1e-4), ((8, 16), 30.0)])
def test_quantize_e5m2_codes_bit_exact(shape, scale):
    g = torch.Generator().manual_seed(shape[0] + 1)
    x = (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    s = torch.empty(2, device="cuda")
    C.coda_fp8_quantize_e5m2(x.cuda(), q, s)
    assert_device_ok()
    xf = x.float().numpy()
    sc = O.fp8_scale(xf, "e5m2")
    assert np.float32(s[1].item()) == sc
    assert np.array_equal(q.cpu().numpy(), O.fp8_quantize(xf, sc, "e5m2"))


def test_quantize_zero_tensor():
    q, s = quantize(torch.zeros(16, 32, dtype=torch.bfloat16, device="cuda"))
    assert_device_ok()
    assert s[1].item() == 1.0 and int(q.sum()) == 0


SHAPES = {"ragged": BlockShape("ragged", 300, 208, 336, 544), "whole": BlockShape("whole", 384, 256, 512, 1024)}


def _forward_fp8(s):
    x = {k: v.cuda() for k, v in block_inputs(s, 0, "cpu", with_dy=False).items()}
    Xq, sX = quantize(x["X"])
    W1q, sW1 = quantize(x["W1t"])
    W2q, sW2 = quantize(x["W2t"], x["g"])
    H = torch.empty(s.M, s.d, dtype=torch.bfloat16, device="cuda")
    psum = torch.empty(s.M, C.coda_prms_num_tiles(s.d), device="cuda")
    C.coda_gemm_res_prms_fp8(Xq, sX[1:], W1q, sW1[1:], x["R"], H, psum)
    rstd = torch.empty(s.M, device="cuda")
    C.coda_rstd_combine(psum, s.d, s.eps, rstd)
    Hq, sH = quantize(H)
    out = torch.empty(s.M, s.F, dtype=torch.bfloat16, device="cuda")
    z = torch.empty(s.M, s.N2, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm_rowscale_swiglu_fp8(Hq, sH[1:], W2q, sW2[1:], rstd, out, z)
    return dict(x=x, Xq=Xq, sX=sX, W1q=W1q, sW1=sW1, W2q=W2q, sW2=sW2, H=H, psum=psum, rstd=rstd, Hq=Hq, sH=sH,
                out=out, z=z)


@pytest.mark.parametrize("name", ["ragged", "whole"])
def test_fp8_forward_stages(name, pairing):
    s = SHAPES[name]
    r = _forward_fp8(s)
    assert_device_ok()
    Xd, W1d = dequant(r["Xq"], r["sX"]), dequant(r["W1q"], r["sW1"])
    assert_elem(r["H"], O.gemm_residual(Xd, W1d, f64(r["x"]["R"])), "H")
    H = f64(r["H"])
    assert_elem(r["psum"], O.partial_sumsq(H, C.PARTIAL_COLS), "psum", tol=1e-4)
    Hd, W2d = dequant(r["Hq"], r["sH"]), dequant(r["W2q"], r["sW2"])
    z_ref = O.rowscale_gemm(Hd, W2d, f64(r["rstd"]))
    assert_elem(r["z"], z_ref, "z")
    assert_elem(r["out"], O.swiglu(z_ref), "out")


def test_fp8_forward_end_to_end():
    s = SHAPES["whole"]
    r = _forward_fp8(s)
    assert_device_ok()
    x = r["x"]
    full = O.block_forward(*(f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t")), s.eps, True)
    assert_frob(r["H"], full["h"], "H e2e", tol=8e-2)
    assert_frob(r["out"], full["out"], "out e2e", tol=8e-2)
