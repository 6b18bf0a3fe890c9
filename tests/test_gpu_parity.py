"""CUDA path vs the fp64 oracle at sizes the oracle finishes in seconds that
still span several tiles and ragged tails (128-row, 256-column tiles, K
blocks of 64).  Every call goes through the C ABI.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, sections 尾声 and 五种积木).
"""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import BlockShape, TINY, block_inputs
from tests._parity import assert_device_ok, assert_elem, assert_frob, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402

EPS = 1e-5

SHAPES = {
    # ragged in every dimension: 3 M tiles (last 44 rows), K1 = 200 (ragged
    # K block), d = 328 (2 column tiles), F = 264 (3 gate tiles of 128)
    "ragged": BlockShape("ragged", 300, 200, 328, 528),
    # whole tiles, 3 x 2 tiles, two TMEM buffers per CTA in use
    "whole": BlockShape("whole", 384, 256, 512, 1024),
    # a single row, a single K block
    "one_row": BlockShape("one_row", 1, 64, 64, 128),
}


@pytest.fixture(params=[True, False], ids=["sm_pair", "single_sm"])
def pairing(request):
    """Run the test with the 2-SM pair GEMM kernel and with the 1-SM one."""
    C.coda_set_sm_pairing(request.param)
    yield request.param
    C.coda_set_sm_pairing(True)


def dev_inputs(s, seed=0):
    return {k: v.cuda() for k, v in block_inputs(s, seed, "cpu", with_dy=s.swiglu).items()}


# --------------------------------------------------------------------------
# the mainloop with a plain epilogue, every operand major
# --------------------------------------------------------------------------

@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K", [(200, 328, 136), (128, 256, 64), (8, 8, 8), (520, 776, 1000)])
def test_gemm_layouts(a_mn, b_mn, M, N, K, pairing):
    # fan-in scaled operands (as in the block workloads) so outputs are O(1)
    # and the elementwise bar's 1e-3 floor is on the data's own scale
    g = torch.Generator().manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    Ad = (A.t().contiguous() if a_mn else A).cuda()
    Bd = (B.t().contiguous() if b_mn else B).cuda()
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm(Ad, a_mn, Bd, b_mn, Cd, M, N, K)
    assert_device_ok()
    assert_elem(Cd, O.matmul_nt(f64(A), f64(B)), "C")


def test_gemm_row_and_col_scale(pairing):
    M, N, K = 264, 264, 192
    g = torch.Generator().manual_seed(5)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    rs = torch.rand(M, generator=g) + 0.5
    cs = (torch.rand(N, generator=g) + 0.5).to(torch.bfloat16)
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm(A.cuda(), False, B.cuda(), False, Cd, M, N, K, rs.cuda(), cs.cuda())
    ref = O.matmul_nt(f64(A), f64(B)) * f64(rs)[:, None] * f64(cs)[None, :]
    assert_elem(Cd, ref, "scaled C")


# --------------------------------------------------------------------------
# forward: each stage against the oracle on the GPU's own stage inputs (O2),
# the output against the chained oracle (O1)
# --------------------------------------------------------------------------

def check_forward(s: BlockShape, b: BlockBuffers, x: dict):
    X, W1t, R, g, W2t = (f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t"))
    H = f64(b.H)
    assert_elem(b.W2gt, O.fold_weight(W2t, g), "W2gt")
    assert_elem(b.H, O.gemm_residual(X, W1t, R), "H")
    bn = C.PARTIAL_COLS
    assert_elem(b.psum, O.partial_sumsq(H, bn), "psum", tol=1e-4)
    assert_elem(b.rstd, O.rstd_from_partials(f64(b.psum), s.d, EPS), "rstd", tol=1e-5)
    z_ref = O.rowscale_gemm(H, f64(b.W2gt), f64(b.rstd))
    if s.swiglu:
        assert_elem(b.z, z_ref, "z")
        assert_elem(b.out, O.swiglu(z_ref), "out")
    else:
        assert_elem(b.z, z_ref, "out (plain)")
    full = O.block_forward(X, W1t, R, g, W2t, EPS, s.swiglu)
    assert_frob(b.H, full["h"], "H e2e")
    assert_frob(b.rstd, full["rstd"], "rstd e2e")
    assert_frob(b.out, full["out"], "out e2e")


@pytest.mark.parametrize("name", ["ragged", "whole", "one_row"])
def test_forward_parity(name, pairing):
    s = SHAPES[name]
    x = dev_inputs(s)
    b = BlockBuffers(x, swiglu=True, backward=False)
    b.forward()
    assert_device_ok()
    check_forward(s, b, x)


def test_tiny_config_plain(pairing):
    """The tiny forward workload: X[256,512], W1, W2 [512,512], PLAIN
    epilogue (row scale only), outputs h, rstd, out[256,512]."""
    x = dev_inputs(TINY)
    b = BlockBuffers(x, swiglu=False, backward=False)
    b.forward()
    assert_device_ok()
    check_forward(TINY, b, x)


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------

def check_backward_stages(s, b, x):
    X, W1t, g, W2t, dY = (f64(x[k]) for k in ("X", "W1t", "g", "W2t", "dY"))
    H, z, rstd = f64(b.H), f64(b.z), f64(b.rstd)
    dP_ref, c_ref = O.stage_swiglu_bwd(dY, z, rstd, s.d)
    assert_elem(b.dP, dP_ref, "dP")
    assert_elem(b.c, c_ref, "c")
    dH_ref, dg_ref = O.stage_dgrad2_rmsbwd(f64(b.dP), W2t, g, H, f64(b.c))
    assert_elem(b.dH, dH_ref, "dH")
    assert_elem(b.dg, dg_ref, "dg")
    assert_elem(b.dW2t, O.stage_wgrad2(H, f64(b.dP), g), "dW2t")
    assert_elem(b.dX, O.stage_dgrad1(f64(b.dH), W1t), "dX")
    assert_elem(b.dW1t, O.stage_wgrad1(f64(b.dH), X), "dW1t")


@pytest.mark.parametrize("name", ["ragged", "whole", "one_row"])
def test_backward_stage_parity(name, pairing):
    s = SHAPES[name]
    x = dev_inputs(s)
    b = BlockBuffers(x)
    b.forward()
    b.backward_stages()
    assert_device_ok()
    check_backward_stages(s, b, x)


@pytest.mark.parametrize("name", ["ragged", "whole"])
def test_fwd_bwd_end_to_end(name):
    s = SHAPES[name]
    x = dev_inputs(s)
    b = BlockBuffers(x)
    b.step()
    assert_device_ok()
    ref = O.block_backward(*(f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t", "dY")), EPS, True)
    for k_gpu, k_ref in (("out", "out"), ("dH", "dR"), ("dX", "dX"), ("dW1t", "dW1t"), ("dW2t", "dW2t"),
                         ("dg", "dg")):
        assert_frob(getattr(b, k_gpu), ref[k_ref], f"{k_gpu} e2e")


def test_composite_backward_equals_stages_and_is_deterministic():
    s = SHAPES["ragged"]
    x = dev_inputs(s)
    a = BlockBuffers(x)
    a.forward()
    a.backward_stages()
    got = {k: getattr(a, k).clone() for k in ("dH", "dX", "dW1t", "dW2t", "dg")}
    for _ in range(2):
        a.backward()
        torch.cuda.synchronize()
        for k, v in got.items():
            assert torch.equal(getattr(a, k), v), k


def test_unfused_ablation_matches_oracle(pairing):
    s = SHAPES["ragged"]
    x = dev_inputs(s)
    b = BlockBuffers(x, unfused=True)
    b.step()
    assert_device_ok()
    ref = O.block_backward(*(f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t", "dY")), EPS, True)
    for k_gpu, k_ref in (("out", "out"), ("dH", "dR"), ("dX", "dX"), ("dW1t", "dW1t"), ("dW2t", "dW2t"),
                         ("dg", "dg")):
        assert_frob(getattr(b, k_gpu), ref[k_ref], f"unfused {k_gpu}")


# --------------------------------------------------------------------------
# edge cases and argument errors
# --------------------------------------------------------------------------

def test_empty_batch_is_a_no_op():
    s = BlockShape("empty", 0, 64, 64, 128)
    x = dev_inputs(s)
    b = BlockBuffers(x)
    b.dW2t.fill_(1.0)
    b.dg.fill_(1.0)
    b.step()
    assert_device_ok()
    assert torch.count_nonzero(b.dW2t) == 0 and torch.count_nonzero(b.dg) == 0
    # the same through the stage calls (dgpart has no rows; the combine writes dg = 0)
    b.dW2t.fill_(1.0)
    b.dg.fill_(1.0)
    b.forward()
    b.backward_stages()
    assert_device_ok()
    assert torch.count_nonzero(b.dW2t) == 0 and torch.count_nonzero(b.dg) == 0


def test_argument_errors():
    d = torch.empty(64, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(64, 64, dtype=torch.bfloat16, device="cuda")
    lib = C.load_library()
    h = C.handle()
    s = torch.cuda.current_stream().cuda_stream
    # misaligned pointer
    assert lib.coda_gemm(h, d.data_ptr() + 2, 0, d.data_ptr(), 0, out.data_ptr(), 64, 64, 64, None, None, s) == 2
    # null pointer
    assert lib.coda_gemm(h, None, 0, d.data_ptr(), 0, out.data_ptr(), 64, 64, 64, None, None, s) == 1
    # extent not a multiple of 8
    assert lib.coda_gemm(h, d.data_ptr(), 0, d.data_ptr(), 0, out.data_ptr(), 64, 60, 64, None, None, s) == 2
    # unsupported major combination
    assert lib.coda_gemm(h, d.data_ptr(), 1, d.data_ptr(), 0, out.data_ptr(), 64, 64, 64, None, None, s) == 3
    # bad epilogue flag
    assert lib.coda_gemm_rowscale_swiglu(h, d.data_ptr(), d.data_ptr(), d.data_ptr(), out.data_ptr(), None,
                                         64, 64, 64, 7, s) == 3
    # workspace too small
    assert lib.coda_gemm_rowscale_swiglu_bwd(h, *([d.data_ptr()] * 10), 16, 64, 64, 128, s) == 4
    with pytest.raises(TypeError):
        C.coda_gemm(d, False, d, False, out, 64, 64, 64, row_scale=torch.empty(64, device="cuda"),
                    col_scale=torch.empty(64, device="cuda", dtype=torch.float32))
    assert_device_ok()


# --------------------------------------------------------------------------
# the light combine folded into GEMM2's epilogue (row scale from the partial
# sums, no separate combine launch)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["ragged", "whole", "one_row"])
def test_forward_fused_rstd_parity(name, pairing):
    s = SHAPES[name]
    x = dev_inputs(s)
    b = BlockBuffers(x, swiglu=True, backward=False, fuse_rstd=True)
    b.forward()
    assert_device_ok()
    check_forward(s, b, x)


def test_tiny_config_plain_fused_rstd():
    x = dev_inputs(TINY)
    b = BlockBuffers(x, swiglu=False, backward=False, fuse_rstd=True)
    b.forward()
    assert_device_ok()
    check_forward(TINY, b, x)


def test_fwd_bwd_end_to_end_fused_rstd():
    s = SHAPES["ragged"]
    x = dev_inputs(s)
    b = BlockBuffers(x, fuse_rstd=True)
    b.step()
    assert_device_ok()
    ref = O.block_backward(*(f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t", "dY")), EPS, True)
    for k_gpu, k_ref in (("out", "out"), ("rstd", "rstd"), ("dH", "dR"), ("dX", "dX"), ("dW1t", "dW1t"),
                         ("dW2t", "dW2t"), ("dg", "dg")):
        assert_frob(getattr(b, k_gpu), ref[k_ref], f"{k_gpu} e2e")


# --------------------------------------------------------------------------
# RMSNorm weight applied on the activation side (Hg written by GEMM1's
# epilogue, GEMM2 on the unfolded W2): no per-step fold pass over W2
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["ragged", "whole", "one_row"])
@pytest.mark.parametrize("fuse_rstd", [False, True])
def test_forward_g_on_activation(name, fuse_rstd, pairing):
    s = SHAPES[name]
    x = dev_inputs(s)
    b = BlockBuffers(x, swiglu=True, backward=False, g_on_activation=True, fuse_rstd=fuse_rstd)
    b.forward()
    assert_device_ok()
    X, W1t, R, g, W2t = (f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t"))
    H = f64(b.H)
    assert_elem(b.H, O.gemm_residual(X, W1t, R), "H")
    assert_elem(b.Hg, H * g[None, :], "Hg")
    assert_elem(b.psum, O.partial_sumsq(H, C.PARTIAL_COLS), "psum", tol=1e-4)
    assert_elem(b.rstd, O.rstd_from_partials(f64(b.psum), s.d, EPS), "rstd", tol=1e-5)
    z_ref = O.rowscale_gemm(f64(b.Hg), W2t, f64(b.rstd))
    assert_elem(b.z, z_ref, "z")
    assert_elem(b.out, O.swiglu(z_ref), "out")
    full = O.block_forward(X, W1t, R, g, W2t, EPS, True)
    assert_frob(b.out, full["out"], "out e2e")


def test_fwd_bwd_end_to_end_g_on_activation():
    s = SHAPES["ragged"]
    x = dev_inputs(s)
    b = BlockBuffers(x, g_on_activation=True, fuse_rstd=True)
    b.step()
    assert_device_ok()
    ref = O.block_backward(*(f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t", "dY")), EPS, True)
    for k_gpu, k_ref in (("out", "out"), ("dH", "dR"), ("dX", "dX"), ("dW1t", "dW1t"), ("dW2t", "dW2t"),
                         ("dg", "dg")):
        assert_frob(getattr(b, k_gpu), ref[k_ref], f"{k_gpu} e2e")
