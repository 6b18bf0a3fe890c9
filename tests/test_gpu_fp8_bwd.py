"""FP8 forward and backward of the block (the FP8 operand variant of every
epilogue program): e4m3 activations and weights, e5m2 gradients, each with
one fp32 scale per tensor.

Strict checks, stage by stage, against the oracle fed the GPU's own codes:
  * the e5m2 codes and scales of dP and dH are bit-exact (the quantiser's
    input is the bf16 tensor the GPU wrote);
  * dgrad2 with the RMSNorm backward (dH, dg), wgrad2 (dW2t), dgrad1 (dX) and
    wgrad1 (dW1t) meet the bf16 elementwise bar against the oracle fed the
    dequantised codes (the GEMMs accumulate exact products in fp32).

End to end against the fp64 oracle chained from the bf16 inputs, relative
Frobenius bounds derived from the quantisation error.  Round to nearest in a
format with p mantissa bits leaves an rms relative error of about
2^-(p+1)/sqrt(3) per element: 3.6 % for e4m3 (p = 3) and 7.2 % for e5m2
(p = 2).  Independent operand errors add in quadrature through a GEMM:
  * out: two e4m3 operands per GEMM, two GEMMs: <= 8e-2;
  * dP carries the forward's error (~5 %) and its e5m2 rounding (7.2 %),
    about 9 %; dH = g acc - c h, dW2t and dg add an e4m3 operand (3.6 %):
    about 10-11 %, bound 0.15;
  * dX and dW1t take dH (about 11 %) rounded again to e5m2 (7.2 %) times
    an e4m3 operand (3.6 %): about 14 %, bound 0.2.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, section 背景: FP8 makes the matmul faster and raises the
share of the memory-bound work the epilogues absorb).
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
SHAPES = {"ragged": BlockShape("ragged", 300, 208, 336, 544), "whole": BlockShape("whole", 384, 256, 512, 1024),
          "one_row": BlockShape("one_row", 1, 64, 64, 128)}


def deq(codes, scale_pair, fmt):
    return O.fp8_decode(codes.cpu().numpy(), fmt) * float(scale_pair[1].item())


def run_fp8(s, seed=0):
    x = {k: v.cuda() for k, v in block_inputs(s, seed, "cpu").items()}
    b = BlockBuffers(x)
    b.fp8_quantize_weights()
    b.forward_fp8()
    b.backward_fp8()
    torch.cuda.synchronize()
    assert_device_ok()
    return x, b


@pytest.mark.parametrize("name", ["ragged", "whole", "one_row"])
def test_fp8_backward_stages(name, pairing):
    s = SHAPES[name]
    x, b = run_fp8(s)
    check_fp8_backward_stages(s, x, b)


def check_fp8_forward_stages(s, x, b):
    """The FP8 forward of BlockBuffers stage by stage: the codes and scales
    of X and H bit-exact (the oracle's quantiser on the bf16 tensors), H,
    psum, rstd, z and out against the oracle fed the dequantised codes."""
    for src, q, sc in ((x["X"], b.Xq, b.s_a[0]), (b.H, b.Hq, b.s_a[1])):
        v = src.float().cpu().numpy()
        ref_scale = O.fp8_scale(v, "e4m3")
        assert np.float32(sc[1].item()) == ref_scale
        assert np.array_equal(q.cpu().numpy(), O.fp8_quantize(v, ref_scale, "e4m3"))
    Xd, W1d = deq(b.Xq, b.s_a[0], "e4m3"), deq(b.W1q, b.s_w[0], "e4m3")
    assert_elem(b.H, O.gemm_residual(Xd, W1d, f64(x["R"])), "H (fp8 gemm1)")
    H = f64(b.H)
    assert_elem(b.psum, O.partial_sumsq(H, C.PARTIAL_COLS), "psum (fp8 gemm1)", tol=1e-4)
    assert_elem(b.rstd, O.rstd_from_partials(f64(b.psum), s.d, EPS), "rstd", tol=1e-5)
    z_ref = O.rowscale_gemm(deq(b.Hq, b.s_a[1], "e4m3"), deq(b.W2gq, b.s_w[1], "e4m3"), f64(b.rstd))
    assert_elem(b.z, z_ref, "z (fp8 gemm2)")
    assert_elem(b.out, O.swiglu(z_ref), "out (fp8 gemm2)")


def check_fp8_backward_stages(s, x, b):
    g, H, c = f64(x["g"]), f64(b.H), f64(b.c)
    # dP's codes come straight from the SwiGLU backward: they must equal the
    # e5m2 codes of the bf16 dP that the unfused SwiGLU-backward kernel writes
    # from the same z and rstd, with the same c
    dP16 = torch.empty(s.M, s.N2, dtype=torch.bfloat16, device="cuda")
    c16 = torch.empty(s.M, dtype=torch.float32, device="cuda")
    C.coda_swiglu_bwd(b.dY, b.z, b.rstd, dP16, c16, s.d)
    torch.cuda.synchronize()
    assert torch.equal(b.c, c16)
    # gradient codes: bit-exact e5m2 of the bf16 tensors the GPU wrote
    for src, q, sc in ((dP16, b.dPq, b.s_a[2]), (b.dH, b.dHq, b.s_a[3])):
        v = src.float().cpu().numpy()
        ref_scale = O.fp8_scale(v, "e5m2")
        assert np.float32(sc[1].item()) == ref_scale
        assert np.array_equal(q.cpu().numpy(), O.fp8_quantize(v, ref_scale, "e5m2"))
    dP = deq(b.dPq, b.s_a[2], "e5m2")
    W2 = deq(b.W2q, b.s_w[2], "e4m3")
    Hq = deq(b.Hq, b.s_a[1], "e4m3")
    dH_ref, dg_ref = O.stage_dgrad2_rmsbwd(dP, W2, g, H, c)
    assert_elem(b.dH, dH_ref, "dH (fp8 dgrad2)")
    assert_elem(b.dg, dg_ref, "dg (fp8 dgrad2)")
    assert_elem(b.dW2t, O.stage_wgrad2(Hq, dP, g), "dW2t (fp8 wgrad2)")
    dHq = deq(b.dHq, b.s_a[3], "e5m2")
    W1 = deq(b.W1q, b.s_w[0], "e4m3")
    Xq = deq(b.Xq, b.s_a[0], "e4m3")
    assert_elem(b.dX, O.stage_dgrad1(dHq, W1), "dX (fp8 dgrad1)")
    assert_elem(b.dW1t, O.stage_wgrad1(dHq, Xq), "dW1t (fp8 wgrad1)")


@pytest.mark.parametrize("name", ["ragged", "whole"])
def test_fp8_forward_backward_end_to_end(name):
    s = SHAPES[name]
    x, b = run_fp8(s)
    ref = O.block_backward(*(f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t", "dY")), EPS, True)
    bounds = {"out": 8e-2, "dR": 0.15, "dW2t": 0.15, "dg": 0.15, "dX": 0.2, "dW1t": 0.2}
    for k_gpu, k_ref in (("out", "out"), ("dH", "dR"), ("dW2t", "dW2t"), ("dg", "dg"), ("dX", "dX"),
                         ("dW1t", "dW1t")):
        assert_frob(getattr(b, k_gpu), ref[k_ref], f"fp8 {k_gpu} e2e", tol=bounds[k_ref])


@pytest.mark.parametrize("fmt,name", [(C.E4M3, "e4m3"), (C.E5M2, "e5m2")])
@pytest.mark.parametrize("M,F", [(300, 272), (1, 8), (64, 1040)])
def test_swiglu_bwd_fp8_codes(fmt, name, M, F):
    """coda_swiglu_bwd_fp8 against its unfused definition: the codes, amax
    and scale of the bf16 dP that coda_swiglu_bwd writes, quantised by the
    oracle; c bit-equal to coda_swiglu_bwd's; and dP against the oracle's
    SwiGLU backward within the bf16 bar."""
    g = torch.Generator().manual_seed(M * 7 + F)
    dY = torch.randn(M, F, generator=g).to(torch.bfloat16).cuda()
    z = (2.0 * torch.randn(M, 2 * F, generator=g)).to(torch.bfloat16).cuda()
    rstd = (0.5 + torch.rand(M, generator=g)).cuda()
    d = 256
    dPq = torch.empty(M, 2 * F, dtype=torch.uint8, device="cuda")
    sc = torch.empty(2, device="cuda")
    c = torch.empty(M, device="cuda")
    C.coda_swiglu_bwd_fp8(dY, z, rstd, fmt, dPq, sc, c, d)
    dP16 = torch.empty(M, 2 * F, dtype=torch.bfloat16, device="cuda")
    c16 = torch.empty(M, device="cuda")
    C.coda_swiglu_bwd(dY, z, rstd, dP16, c16, d)
    torch.cuda.synchronize()
    assert_device_ok()
    v = dP16.float().cpu().numpy()
    ref_scale = O.fp8_scale(v, name)
    assert np.float32(sc[0].item()) == np.float32(np.abs(v).max())
    assert np.float32(sc[1].item()) == ref_scale
    assert np.array_equal(dPq.cpu().numpy(), O.fp8_quantize(v, ref_scale, name))
    assert torch.equal(c, c16)
    dP_ref, c_ref = O.stage_swiglu_bwd(f64(dY), f64(z), f64(rstd), d)
    assert_elem(dP16, dP_ref, "dP (bf16)")
    assert_elem(c, c_ref, "c")


def _swiglu_case(M, F, seed, dy_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    dY = (dy_scale * torch.randn(M, F, generator=g)).to(torch.bfloat16).cuda()
    z = (2.0 * torch.randn(M, 2 * F, generator=g)).to(torch.bfloat16).cuda()
    rstd = (0.5 + torch.rand(M, generator=g)).cuda()
    return dY, z, rstd


@pytest.mark.parametrize("fmt,name", [(C.E4M3, "e4m3"), (C.E5M2, "e5m2")])
@pytest.mark.parametrize("M,F", [(300, 272), (64, 1040)])
@pytest.mark.parametrize("dy_scale", [1.0, 3000.0], ids=["in_range", "saturating"])
def test_swiglu_bwd_fp8_delayed_codes(fmt, name, M, F, dy_scale):
    """Delayed scaling: step A (exact, two passes) leaves its amax in the
    state; step B's single pass quantises its bf16 dP with the scale the
    oracle derives from A's amax (saturating where B exceeds A's range, the
    second case), reports B's own amax for the next step, and writes the c
    of coda_swiglu_bwd bit for bit."""
    d = 256
    dPq = torch.empty(M, 2 * F, dtype=torch.uint8, device="cuda")
    sc = torch.empty(2, device="cuda")
    c = torch.empty(M, device="cuda")
    dP16 = torch.empty(M, 2 * F, dtype=torch.bfloat16, device="cuda")
    c16 = torch.empty(M, device="cuda")
    dYa, za, ra = _swiglu_case(M, F, 11)
    C.coda_swiglu_bwd_fp8(dYa, za, ra, fmt, dPq, sc, c, d)
    C.coda_swiglu_bwd(dYa, za, ra, dP16, c16, d)
    torch.cuda.synchronize()
    prev_scale = O.fp8_scale(dP16.float().cpu().numpy(), name)
    dYb, zb, rb = _swiglu_case(M, F, 12, dy_scale)
    C.coda_swiglu_bwd_fp8_delayed(dYb, zb, rb, fmt, dPq, sc, c, d)
    C.coda_swiglu_bwd(dYb, zb, rb, dP16, c16, d)
    torch.cuda.synchronize()
    assert_device_ok()
    v = dP16.float().cpu().numpy()
    assert np.float32(sc[1].item()) == prev_scale
    assert np.float32(sc[0].item()) == np.float32(np.abs(v).max())
    codes = dPq.cpu().numpy()
    assert np.array_equal(codes, O.fp8_quantize(v, prev_scale, name))
    fmax = 448.0 if name == "e4m3" else 57344.0
    if dy_scale > 1.0:   # B far outside A's range: the codes saturate (and still match)
        assert (np.abs(v) / prev_scale > fmax).any()
    assert torch.equal(c, c16)


def test_fp8_delayed_scaling_end_to_end_and_graph():
    """Steps with delayed dP scaling: after an exact first step, a delayed
    step on new inputs meets the FP8 end-to-end bounds against the oracle;
    a CUDA graph of the delayed step replays bit-identically to the same
    eager sequence."""
    s = SHAPES["ragged"]
    xa = {k: v.cuda() for k, v in block_inputs(s, 0, "cpu").items()}
    xb = {k: v.cuda() for k, v in block_inputs(s, 1, "cpu").items()}
    ins = ("X", "R", "dY")
    b = BlockBuffers({k: v.clone() for k, v in xa.items()})
    b.fp8_quantize_weights()
    b.step_fp8(delayed=True)             # the first step takes the exact form
    eager = []
    for x in (xb, xa, xb):
        for k in ins:
            getattr(b, k).copy_(x[k])
        b.step_fp8(delayed=True)
        torch.cuda.synchronize()
        eager.append({k: getattr(b, k).clone() for k in ("out", "dH", "dX", "dW1t", "dW2t", "dg")})
    assert_device_ok()
    ref = O.block_backward(*(f64(xa[k]) if k in ("W1t", "g", "W2t") else f64(xb[k])
                             for k in ("X", "W1t", "R", "g", "W2t", "dY")), EPS, True)
    bounds = {"out": 8e-2, "dR": 0.15, "dW2t": 0.15, "dg": 0.15, "dX": 0.2, "dW1t": 0.2}
    for k_gpu, k_ref in (("out", "out"), ("dH", "dR"), ("dW2t", "dW2t"), ("dg", "dg"), ("dX", "dX"),
                         ("dW1t", "dW1t")):
        assert_frob(eager[2][k_gpu], ref[k_ref], f"fp8 delayed {k_gpu} e2e", tol=bounds[k_ref])

    g = BlockBuffers({k: v.clone() for k, v in xa.items()})
    g.fp8_quantize_weights()
    g.capture_step(fp8=True, delayed=True)   # its eager step is the exact first step
    for x, want in zip((xb, xa, xb), eager):
        for k in ins:
            getattr(g, k).copy_(x[k])
        g.replay()
        torch.cuda.synchronize()
        for k, v in want.items():
            assert torch.equal(getattr(g, k), v), k
    assert_device_ok()


def test_swiglu_bwd_fp8_empty():
    z0 = torch.empty(0, 16, dtype=torch.bfloat16, device="cuda")
    sc = torch.full((2,), 9.0, device="cuda")
    C.coda_swiglu_bwd_fp8(torch.empty(0, 8, dtype=torch.bfloat16, device="cuda"), z0,
                          torch.empty(0, device="cuda"), C.E5M2, torch.empty(0, 16, dtype=torch.uint8, device="cuda"),
                          sc, torch.empty(0, device="cuda"), 64)
    torch.cuda.synchronize()
    assert sc.tolist() == [0.0, 1.0]


def test_fp8_empty_batch():
    """M = 0 through the whole FP8 step: the weight gradients are empty sums
    (zero), dg is zero, and the activation / gradient scales are {0, 1}."""
    s = BlockShape("empty", 0, 64, 64, 128)
    b = BlockBuffers({k: v.cuda() for k, v in block_inputs(s, 0, "cpu").items()})
    b.fp8_quantize_weights()
    for t in (b.dW2t, b.dW1t, b.dg):
        t.fill_(1.0)
    b.s_a.fill_(7.0)
    b.step_fp8()
    torch.cuda.synchronize()
    assert_device_ok()
    for t in (b.dW2t, b.dW1t, b.dg):
        assert torch.count_nonzero(t) == 0
    assert b.s_a.tolist() == [[0.0, 1.0]] * 4


def test_fp8_argument_errors():
    """The 8-bit entry points reject what their header excludes, without
    launching anything."""
    lib = C.load_library()
    h = C.handle()
    st = torch.cuda.current_stream().cuda_stream
    u = torch.empty(4096, dtype=torch.uint8, device="cuda")
    bfb = torch.empty(4096, dtype=torch.bfloat16, device="cuda")
    f = torch.empty(64, device="cuda")
    p = u.data_ptr()
    # coda_gemm_fp8: a format outside {0, 1}
    assert lib.coda_gemm_fp8(h, p, 0, 2, None, p, 0, 0, None, bfb.data_ptr(), 32, 32, 32, None, None, st) == 1
    # MN-major A with K-major B is not a supported combination
    assert lib.coda_gemm_fp8(h, p, 1, 0, None, p, 0, 0, None, bfb.data_ptr(), 32, 32, 32, None, None, st) == 3
    # K-major K not a multiple of 16 (8-bit rows are 16-byte multiples)
    assert lib.coda_gemm_fp8(h, p, 0, 0, None, p, 0, 0, None, bfb.data_ptr(), 32, 32, 24, None, None, st) == 2
    # MN-major M not a multiple of 16
    assert lib.coda_gemm_fp8(h, p, 1, 0, None, p, 1, 0, None, bfb.data_ptr(), 24, 32, 32, None, None, st) == 2
    # coda_swiglu_bwd_fp8: a format outside {0, 1}
    assert lib.coda_swiglu_bwd_fp8(h, bfb.data_ptr(), bfb.data_ptr(), f.data_ptr(), 3, p, f.data_ptr(),
                                   f.data_ptr(), 8, 16, 64, st) == 1
    # coda_gemm_dgrad_rmsbwd_fp8: N2 not a multiple of 16
    assert lib.coda_gemm_dgrad_rmsbwd_fp8(h, p, 1, f.data_ptr(), p, 0, f.data_ptr(), bfb.data_ptr(), bfb.data_ptr(),
                                          f.data_ptr(), bfb.data_ptr(), f.data_ptr(), 8, 24, 64, st) == 2
    assert_device_ok()
