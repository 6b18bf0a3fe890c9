"""Further epilogue programs on the block's path, against the fp64 oracle:

* the SwiGLU backward in the epilogue of the down projection's data-gradient
  GEMM (dY stays on chip; c is formed from per-tile partial sums inside the
  RMSNorm-backward epilogue of dgrad2);

graded per stage on the GPU's own stage inputs (elementwise) and end to end
against the chain rule (Frobenius).  Synced write-up, section 尾声 (the
re-parameterisation holds for SwiGLU and for the backward) and 实验结果
(SwiGLU backward)."""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import BlockShape, block_inputs, down_proj_inputs
from tests._parity import assert_device_ok, assert_elem, assert_frob, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402

SHAPES = {
    "ragged": BlockShape("ragged", 300, 200, 328, 528),
    "whole": BlockShape("whole", 384, 256, 512, 1024),
}


@pytest.fixture(params=[True, False], ids=["sm_pair", "single_sm"])
def pairing(request):
    C.coda_set_sm_pairing(request.param)
    yield request.param
    C.coda_set_sm_pairing(True)


def _setup(s):
    x = {k: v.cuda() for k, v in block_inputs(s, 0, "cpu", with_dy=False).items()}
    dp = {k: v.cuda() for k, v in down_proj_inputs(s, 0, "cpu").items()}
    b = BlockBuffers(dict(x, dY=torch.empty(s.M, s.F, dtype=torch.bfloat16, device="cuda")))
    b.forward()
    return x, dp, b


@pytest.mark.parametrize("name", ["ragged", "whole"])
def test_down_proj_dgrad_swiglu_bwd_stage(name, pairing):
    s = SHAPES[name]
    x, dp, b = _setup(s)
    cpart = torch.empty(s.M, C.coda_prms_num_tiles(s.F), device="cuda")
    C.coda_gemm_dgrad_swiglu_bwd(dp["dYb"], dp["W3t"], b.z, b.rstd, b.dP, cpart)
    assert_device_ok()
    dY = O.down_proj_dgrad(f64(dp["dYb"]), f64(dp["W3t"]))
    z, rstd = f64(b.z), f64(b.rstd)
    dP_ref, c_ref = O.stage_swiglu_bwd(dY, z, rstd, s.d)
    assert_elem(b.dP, dP_ref, "dP")
    cp_ref = O.swiglu_c_partials(dY, z, C.PARTIAL_COLS)
    assert_elem(cpart, cp_ref, "cpart")
    assert_elem(f64(cpart).sum(axis=1) * rstd ** 2 / s.d, c_ref, "c from cpart")


@pytest.mark.parametrize("name", ["ragged", "whole"])
def test_dgrad_rmsbwd_with_cpart_stage(name, pairing):
    s = SHAPES[name]
    x, dp, b = _setup(s)
    cpart = torch.empty(s.M, C.coda_prms_num_tiles(s.F), device="cuda")
    C.coda_gemm_dgrad_swiglu_bwd(dp["dYb"], dp["W3t"], b.z, b.rstd, b.dP, cpart)
    C.coda_gemm_dgrad_rmsbwd_cpart(b.dP, b.W2t, b.H, b.g, b.rstd, cpart, b.dH, b.dgpart)
    C.coda_dg_combine(b.dgpart, b.dg)
    assert_device_ok()
    c = f64(cpart).sum(axis=1) * f64(b.rstd) ** 2 / s.d
    dH_ref, dg_ref = O.stage_dgrad2_rmsbwd(f64(b.dP), f64(x["W2t"]), f64(x["g"]), f64(b.H), c)
    assert_elem(b.dH, dH_ref, "dH")
    assert_elem(b.dg, dg_ref, "dg")


def test_backward_from_down_proj_end_to_end():
    s = SHAPES["ragged"]
    x, dp, b = _setup(s)
    b.backward_from_down_proj(dp["dYb"], dp["W3t"])
    assert_device_ok()
    dY = O.down_proj_dgrad(f64(dp["dYb"]), f64(dp["W3t"]))
    ref = O.block_backward(*(f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t")), dY, s.eps, True)
    for k_gpu, k_ref in (("dH", "dR"), ("dX", "dX"), ("dW1t", "dW1t"), ("dW2t", "dW2t"), ("dg", "dg")):
        assert_frob(getattr(b, k_gpu), ref[k_ref], f"{k_gpu} e2e")


def test_fused_matches_unfused_route():
    """dY through HBM (plain GEMM to bf16 + the streaming SwiGLU backward) vs
    on chip: same dP up to the bf16 rounding of dY."""
    s = SHAPES["whole"]
    x, dp, b = _setup(s)
    cpart = torch.empty(s.M, C.coda_prms_num_tiles(s.F), device="cuda")
    C.coda_gemm_dgrad_swiglu_bwd(dp["dYb"], dp["W3t"], b.z, b.rstd, b.dP, cpart)
    dP_fused = b.dP.clone()
    dY = torch.empty(s.M, s.F, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm(dp["dYb"], False, dp["W3t"], True, dY, s.M, s.F, s.d)
    C.coda_swiglu_bwd(dY, b.z, b.rstd, b.dP, b.c, s.d)
    assert_device_ok()
    assert_frob(dP_fused, f64(b.dP), "dP fused vs unfused", tol=1e-2)
    # c is a sum with cancellation: the bf16 rounding of dY on the HBM route
    # moves rows near zero by ~1e-5 absolute, so compare on c's own scale
    assert_frob(f64(cpart).sum(axis=1) * f64(b.rstd) ** 2 / s.d, f64(b.c), "c fused vs unfused", tol=2e-2)


# --------------------------------------------------------------------------
# RoPE in the QKV projection's epilogue (rotate-half, head_dim 128)
# --------------------------------------------------------------------------

def _rope_inputs(M, d, n_heads, seed):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(M, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(n_heads * 128, d, generator=g) * 0.02).to(torch.bfloat16)
    return X.cuda(), W.cuda()


def _tables(S, base=10000.0):
    cos_t = torch.empty(S, 64, device="cuda")
    sin_t = torch.empty(S, 64, device="cuda")
    C.coda_rope_table(cos_t, sin_t, base)
    return cos_t, sin_t


def test_rope_table():
    cos_t, sin_t = _tables(2048)
    assert_device_ok()
    th = O.rope_angles(np.arange(2048), 128)
    assert_elem(cos_t, np.cos(th), "cos", tol=1e-5)
    assert_elem(sin_t, np.sin(th), "sin", tol=1e-5)


@pytest.mark.parametrize("M,d,Hq,Hkv,S", [(300, 328, 4, 2, 128), (512, 512, 2, 1, 512), (264, 136, 3, 0, 100),
                                          (256, 256, 2, 2, 64)])
def test_gemm_qkv_rope_parity(M, d, Hq, Hkv, S, pairing):
    X, W = _rope_inputs(M, d, Hq + 2 * Hkv, M + d)
    cos_t, sin_t = _tables(S)
    qkv = torch.empty(M, (Hq + 2 * Hkv) * 128, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm_qkv_rope(X, W, cos_t, sin_t, qkv, Hq, Hkv)
    assert_device_ok()
    ref = O.qkv_rope(f64(X), f64(W), Hq, Hkv, 128, S)
    assert_elem(qkv, ref, "qkv")
    assert_frob(qkv, ref, "qkv")


def test_rope_apply_standalone_and_fused_agree():
    M, d, Hq, Hkv, S = 512, 512, 4, 2, 128
    X, W = _rope_inputs(M, d, Hq + 2 * Hkv, 7)
    cos_t, sin_t = _tables(S)
    N = (Hq + 2 * Hkv) * 128
    plain = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm(X, False, W, False, plain, M, N, d)
    ref = O.rope_rotate_half(f64(plain)[:, :(Hq + Hkv) * 128], np.arange(M) % S, 128)
    C.coda_rope_apply(plain, cos_t, sin_t, Hq, Hkv)
    fused = torch.empty_like(plain)
    C.coda_gemm_qkv_rope(X, W, cos_t, sin_t, fused, Hq, Hkv)
    assert_device_ok()
    assert_elem(plain[:, :(Hq + Hkv) * 128], ref, "standalone RoPE")
    assert_frob(fused, f64(plain), "fused vs unfused", tol=1e-2)


def test_rope_rejects_other_head_dims():
    lib = C.load_library()
    p = torch.empty(16, device="cuda").data_ptr()
    st = lib.coda_gemm_qkv_rope(C.handle(), p, p, p, p, p, 128, 128, 2, 1, 64, 16,
                                torch.cuda.current_stream().cuda_stream)
    assert st == 3
