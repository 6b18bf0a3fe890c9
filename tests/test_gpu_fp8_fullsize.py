"""FP8 forward and backward at the full workload sizes (7B and 70B blocks),
in the launch configuration the bench times, on whole rows and columns.

  * scales: the GPU's scale of every quantised tensor equals the oracle's
    fp8_scale of the whole tensor (its amax taken on the host);
  * codes: at least 256 whole rows of every activation code tensor (first
    and last row tiles, both sides of the tile edges, random others) and
    whole rows of the weight codes are bit-exact against the oracle's
    quantisation with that scale;
  * GEMM stages against the oracle fed the GPU's own codes, dequantised (the
    products are exact and accumulate in fp32), at the bf16 elementwise bar:
    whole rows of H, z, out and dX; every row of dH and all of dg; at least
    64 whole rows and 64 whole columns of dW2t and dW1t.  Each GEMM output is
    also computed by cuBLASLt on the same codes and scales (torch._scaled_mm,
    fp32 result, the epilogue's arithmetic in fp32): the long-K sums named in
    tests/_parity.py pass when no worse than 1.25x cuBLASLt;
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
from tests._parity import assert_device_ok, assert_elem, assert_elem_chunks, assert_frob, edge_sample, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402

CHUNK = 1024
E4M3, E5M2 = torch.float8_e4m3fn, torch.float8_e5m2


def idx(a):
    return torch.as_tensor(a, device="cuda")


def scale_of(pair):
    return np.float32(pair[1].item())


def deq(codes, pair, fmt):
    """Values of a code tensor (any slice, on the GPU) times its scale."""
    return O.fp8_decode(codes.cpu().numpy(), fmt) * float(scale_of(pair))


def check_codes(src_f32, codes, pair, fmt, rows, name):
    """The scale from the whole tensor, the codes of whole rows."""
    v = src_f32.cpu().numpy()
    s = O.fp8_scale(v, fmt)
    assert scale_of(pair) == s, f"{name}: scale {scale_of(pair)} != {s}"
    got = codes[idx(rows)].cpu().numpy()
    assert np.array_equal(got, O.fp8_quantize(v[rows], s, fmt)), f"{name}: codes"


def pad16(ix):
    """Indices padded (with their first) to a multiple of 16, as cuBLASLt's
    8-bit GEMM wants; the comparator's extra columns are sliced off."""
    ix = np.asarray(ix)
    return np.concatenate([ix, np.full((-len(ix)) % 16, ix[0])])


def lt(a_codes, a_fmt, a_pair, b_codes_kn, b_fmt, b_pair):
    """cuBLASLt: sa * sb * A B in fp32, A [m][k] row-major codes, B given as
    [k][n] (made column-major here)."""
    a = a_codes.contiguous().view(a_fmt)
    b = b_codes_kn.t().contiguous().t().view(b_fmt)
    return torch._scaled_mm(a, b, a_pair[1], b_pair[1], out_dtype=torch.float32)


def check_fp8_block(shape):
    x = block_inputs(shape, 0, "cuda")
    b = BlockBuffers(x)
    b.fp8_quantize_weights()
    b.forward_fp8()
    b.backward_fp8()
    torch.cuda.synchronize()
    assert_device_ok()
    M, d, F, K1 = shape.M, shape.d, shape.F, shape.K1
    rows = pad16(edge_sample(M, 256, 11))
    jcols = edge_sample(F, 32, 12)
    kcols = pad16(edge_sample(d, 64, 13))
    icols = pad16(edge_sample(K1, 64, 14))
    ncols = pad16(np.concatenate([jcols, F + jcols]))
    ri, ki, ii, ni = idx(rows), idx(kcols), idx(icols), idx(ncols)
    bf = torch.bfloat16
    g = f64(b.g)
    gf = b.g.float()
    sX, sH, sdP, sdH = b.s_a
    sW1, sW2g, sW2 = b.s_w

    # codes and scales (the folded weight quantises fp32(W2t * g))
    check_codes(b.X.float(), b.Xq, sX, "e4m3", rows, "Xq")
    check_codes(b.H.float(), b.Hq, sH, "e4m3", rows, "Hq")
    check_codes(b.W1t.float(), b.W1q, sW1, "e4m3", kcols, "W1q")
    check_codes(x["W2t"].cpu().float() * x["g"].cpu().float(), b.W2gq, sW2g, "e4m3", ncols, "W2gq")
    check_codes(b.W2t.float(), b.W2q, sW2, "e4m3", ncols, "W2q")
    check_codes(b.dH.float(), b.dHq, sdH, "e5m2", rows, "dHq")
    # dP's codes against the bf16 dP the unfused SwiGLU backward writes
    C.coda_swiglu_bwd(b.dY, b.z, b.rstd, b.dP, torch.empty_like(b.c), b.d)
    torch.cuda.synchronize()
    check_codes(b.dP.float(), b.dPq, sdP, "e5m2", rows, "dPq")

    # forward GEMMs on the codes: whole rows
    W1 = deq(b.W1q, sW1, "e4m3")
    H = f64(b.H[ri])
    cub = (lt(b.Xq[ri], E4M3, sX, b.W1q.t(), E4M3, sW1) + b.R[ri].float()).to(bf)
    assert_elem(H, O.gemm_residual(deq(b.Xq[ri], sX, "e4m3"), W1, f64(b.R[ri])), "H (fp8)", cublas=cub)
    assert_elem(b.rstd, O.rstd_from_partials(f64(b.psum), d, shape.eps), "rstd", tol=1e-5)
    rstd = f64(b.rstd)[rows]
    z_ref = O.rowscale_gemm(deq(b.Hq[ri], sH, "e4m3"), deq(b.W2gq, sW2g, "e4m3"), rstd)
    z32 = b.rstd[ri, None] * lt(b.Hq[ri], E4M3, sH, b.W2gq.t(), E4M3, sW2g)
    assert_elem(f64(b.z[ri]), z_ref, "z (fp8)", cublas=z32.to(bf))
    zg, zu = z32[:, :F], z32[:, F:]
    assert_elem(f64(b.out[ri]), O.swiglu(z_ref), "out (fp8)", cublas=(zg * torch.sigmoid(zg) * zu).to(bf))
    del z_ref, z32, zg, zu
    # the forward output end to end, from the bf16 inputs
    full = O.block_forward(f64(b.X[ri]), f64(b.W1t), f64(b.R[ri]), g, f64(b.W2t), shape.eps, True)
    assert_frob(f64(b.out[ri]), full["out"], "out fp8 e2e", tol=8e-2)
    del full

    # dgrad2 + RMSNorm backward: every row of dH, all of dg
    W2 = deq(b.W2q, sW2, "e4m3")
    Hall = f64(b.H)
    c_all = f64(b.c)
    dg = np.zeros(d)
    dg_cub = np.zeros(d)
    parts = []
    for s0 in range(0, M, CHUNK):
        e = min(M, s0 + CHUNK)
        dh, part = O.stage_dgrad2_rmsbwd(deq(b.dPq[s0:e], sdP, "e5m2"), W2, g, Hall[s0:e], c_all[s0:e])
        dg += part
        acc = lt(b.dPq[s0:e], E5M2, sdP, b.W2q, E4M3, sW2)
        dg_cub += f64((acc * b.H[s0:e].float()).sum(0))
        parts.append((b.dH[s0:e], dh, (gf * acc - b.c[s0:e, None] * b.H[s0:e].float()).to(bf)))
        del acc
    assert_elem_chunks(parts, "dH (fp8)")
    del parts, W2
    assert_elem(b.dg, dg, "dg (fp8)", cublas=dg_cub)
    # wgrad2: whole columns (fixed k) and whole rows (fixed n) of dW2t
    dP_all = deq(b.dPq, sdP, "e5m2")
    Hq_all = deq(b.Hq, sH, "e4m3")
    dPqT = b.dPq.t().contiguous()
    cub = (lt(dPqT, E5M2, sdP, b.Hq[:, ki], E4M3, sH) * gf[ki]).to(bf)
    assert_elem(f64(b.dW2t[:, ki]), O.stage_wgrad2(Hq_all[:, kcols], dP_all, g[kcols]), "dW2t columns (fp8)",
                cublas=cub)
    cub = (lt(dPqT[ni], E5M2, sdP, b.Hq, E4M3, sH) * gf).to(bf)
    assert_elem(f64(b.dW2t[ni]), O.stage_wgrad2(Hq_all, dP_all[:, ncols], g), "dW2t rows (fp8)", cublas=cub)
    del dP_all, dPqT, cub
    # dgrad1 (whole rows) and wgrad1 (whole rows and columns of dW1t)
    dHq_rows = deq(b.dHq[ri], sdH, "e5m2")
    assert_elem(f64(b.dX[ri]), O.stage_dgrad1(dHq_rows, W1), "dX (fp8)",
                cublas=lt(b.dHq[ri], E5M2, sdH, b.W1q, E4M3, sW1).to(bf))
    dH_all = deq(b.dHq, sdH, "e5m2")
    X_all = deq(b.Xq, sX, "e4m3")
    dHqT = b.dHq.t().contiguous()
    assert_elem(f64(b.dW1t[ki]), O.stage_wgrad1(dH_all[:, kcols], X_all), "dW1t rows (fp8)",
                cublas=lt(dHqT[ki], E5M2, sdH, b.Xq, E4M3, sX).to(bf))
    assert_elem(f64(b.dW1t[:, ii]), O.stage_wgrad1(dH_all, X_all[:, icols]), "dW1t columns (fp8)",
                cublas=lt(dHqT, E5M2, sdH, b.Xq[:, ii], E4M3, sX).to(bf))
    del dH_all, X_all, dHqT, Hq_all
    # the data gradients end to end: a row's dR and dX depend on that row alone
    ref = O.block_backward(f64(b.X[ri]), f64(b.W1t), f64(b.R[ri]), g, f64(b.W2t), f64(b.dY[ri]), shape.eps, True)
    assert_frob(f64(b.dH[ri]), ref["dR"], "dR fp8 e2e", tol=0.15)
    assert_frob(f64(b.dX[ri]), ref["dX"], "dX fp8 e2e", tol=0.2)


def test_7b_fp8_forward_backward_full_size():
    check_fp8_block(B7)


def test_70b_fp8_forward_backward_full_size():
    check_fp8_block(B70)
