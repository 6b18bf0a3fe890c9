"""FP8 forward and backward at the full workload sizes (7B and 70B blocks),
in the launch configuration the bench times, on sampled outputs.

  * scales: the GPU's scale of every quantised tensor equals the oracle's
    fp8_scale of the whole tensor (its amax taken on the host);
  * codes: sampled rows of every code tensor are bit-exact against the
    oracle's quantisation with that scale;
  * GEMM stages: sampled rows / columns of H, z, out, dH, dg, dW2t, dX and
    dW1t meet the bf16 elementwise bar against the oracle fed the GPU's own
    codes, dequantised (the products are exact and accumulate in fp32);
  * end to end on the sampled rows against the oracle chained from the bf16
    inputs: the forward output within the e4m3 bound (Frobenius 8e-2), the
    row-local data gradients dR and dX within 0.15 and 0.2 (the bounds of
    the small-shape FP8 backward test, from the e4m3 / e5m2 rounding).

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, section 背景: FP8 makes the matmul faster and raises the
share of the memory-bound work the epilogues absorb; sections 尾声 / 实验结果
for the block and its 7B / 70B hidden sizes).
"""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import B7, B70, block_inputs
from tests._parity import assert_device_ok, assert_elem, assert_frob, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402


def sample(n, k, seed):
    r = np.random.default_rng(seed)
    idx = set(r.choice(n, size=min(k, n), replace=False).tolist()) | {0, n - 1}
    return np.array(sorted(idx))


def idx(a):
    return torch.as_tensor(a, device="cuda")


def scale_of(pair):
    return np.float32(pair[1].item())


def deq(codes, pair, fmt):
    """Values of a code tensor (any slice, on the GPU) times its scale."""
    return O.fp8_decode(codes.cpu().numpy(), fmt) * float(scale_of(pair))


def check_codes(src_f32, codes, pair, fmt, rows, name):
    """The scale from the whole tensor, the codes of the sampled rows."""
    v = src_f32.cpu().numpy()
    s = O.fp8_scale(v, fmt)
    assert scale_of(pair) == s, f"{name}: scale {scale_of(pair)} != {s}"
    got = codes[idx(rows)].cpu().numpy()
    assert np.array_equal(got, O.fp8_quantize(v[rows], s, fmt)), f"{name}: codes"


def check_fp8_block(shape):
    x = block_inputs(shape, 0, "cuda")
    b = BlockBuffers(x)
    b.fp8_quantize_weights()
    b.forward_fp8()
    b.backward_fp8()
    torch.cuda.synchronize()
    assert_device_ok()
    M, d, F, K1 = shape.M, shape.d, shape.F, shape.K1
    rows = sample(M, 10, 11)
    jcols = sample(F, 16, 12)
    kcols = sample(d, 16, 13)
    icols = sample(K1, 16, 14)
    ncols = np.concatenate([jcols, F + jcols])
    g = f64(b.g)

    # codes and scales (the folded weight quantises fp32(W2t * g))
    check_codes(b.X.float(), b.Xq, b.s_a[0], "e4m3", rows, "Xq")
    check_codes(b.H.float(), b.Hq, b.s_a[1], "e4m3", rows, "Hq")
    check_codes(b.W1t.float(), b.W1q, b.s_w[0], "e4m3", sample(d, 10, 15), "W1q")
    check_codes(x["W2t"].cpu().float() * x["g"].cpu().float(), b.W2gq, b.s_w[1], "e4m3", ncols, "W2gq")
    check_codes(b.W2t.float(), b.W2q, b.s_w[2], "e4m3", ncols, "W2q")
    check_codes(b.dH.float(), b.dHq, b.s_a[3], "e5m2", rows, "dHq")
    # dP's codes against the bf16 dP the unfused SwiGLU backward writes
    C.coda_swiglu_bwd(b.dY, b.z, b.rstd, b.dP, torch.empty_like(b.c), b.d)
    torch.cuda.synchronize()
    check_codes(b.dP.float(), b.dPq, b.s_a[2], "e5m2", rows, "dPq")

    # forward GEMMs on the codes
    W1 = deq(b.W1q, b.s_w[0], "e4m3")
    H = f64(b.H[idx(rows)])
    assert_elem(H, O.gemm_residual(deq(b.Xq[idx(rows)], b.s_a[0], "e4m3"), W1, f64(b.R[idx(rows)])), "H (fp8)")
    rstd = f64(b.rstd)[rows]
    assert_elem(rstd, O.rstd_from_partials(f64(b.psum[idx(rows)]), d, shape.eps), "rstd", tol=1e-5)
    z_ref = O.rowscale_gemm(deq(b.Hq[idx(rows)], b.s_a[1], "e4m3"), deq(b.W2gq[idx(ncols)], b.s_w[1], "e4m3"), rstd)
    assert_elem(f64(b.z[idx(rows)])[:, ncols], z_ref, "z (fp8)")
    assert_elem(f64(b.out[idx(rows)])[:, jcols], O.swiglu(z_ref), "out (fp8)")
    # the forward output end to end, from the bf16 inputs
    full = O.block_forward(f64(b.X[idx(rows)]), f64(b.W1t), f64(b.R[idx(rows)]), g, f64(b.W2t[idx(ncols)]),
                           shape.eps, True)
    assert_frob(f64(b.out[idx(rows)])[:, jcols], full["out"], "out fp8 e2e", tol=8e-2)

    # backward GEMMs on the codes
    W2k = deq(b.W2q[:, idx(kcols)], b.s_w[2], "e4m3")
    dg = np.zeros(len(kcols))
    for s0 in range(0, M, 1024):
        e = min(M, s0 + 1024)
        _, part = O.stage_dgrad2_rmsbwd(deq(b.dPq[s0:e], b.s_a[2], "e5m2"), W2k, g[kcols],
                                        f64(b.H[s0:e])[:, kcols], f64(b.c[s0:e]))
        dg += part
    dh_ref, _ = O.stage_dgrad2_rmsbwd(deq(b.dPq[idx(rows)], b.s_a[2], "e5m2"), W2k, g[kcols],
                                      f64(b.H[idx(rows)])[:, kcols], f64(b.c)[rows])
    assert_elem(f64(b.dH[idx(rows)])[:, kcols], dh_ref, "dH (fp8)")
    assert_elem(f64(b.dg)[kcols], dg, "dg (fp8)")
    dW2_ref = O.stage_wgrad2(deq(b.Hq[:, idx(kcols)], b.s_a[1], "e4m3"), deq(b.dPq[:, idx(ncols)], b.s_a[2], "e5m2"),
                             g[kcols])
    assert_elem(f64(b.dW2t[idx(ncols)])[:, kcols], dW2_ref, "dW2t (fp8)")
    assert_elem(f64(b.dX[idx(rows)]), O.stage_dgrad1(deq(b.dHq[idx(rows)], b.s_a[3], "e5m2"), W1), "dX (fp8)")
    dW1_ref = O.stage_wgrad1(deq(b.dHq[:, idx(kcols)], b.s_a[3], "e5m2"), deq(b.Xq[:, idx(icols)], b.s_a[0], "e4m3"))
    assert_elem(f64(b.dW1t[idx(kcols)])[:, icols], dW1_ref, "dW1t (fp8)")
    # the data gradients end to end: a row's dR and dX depend on that row alone
    ref = O.block_backward(f64(b.X[idx(rows)]), f64(b.W1t), f64(b.R[idx(rows)]), g, f64(b.W2t),
                           f64(b.dY[idx(rows)]), shape.eps, True)
    assert_frob(f64(b.dH[idx(rows)]), ref["dR"], "dR fp8 e2e", tol=0.15)
    assert_frob(f64(b.dX[idx(rows)]), ref["dX"], "dX fp8 e2e", tol=0.2)


def test_7b_fp8_forward_backward_full_size():
    check_fp8_block(B7)


def test_70b_fp8_forward_backward_full_size():
    check_fp8_block(B70)
