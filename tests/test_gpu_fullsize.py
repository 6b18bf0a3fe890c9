"""Parity at the full workload sizes, in the launch configuration the bench
times (same entry points, persistent grids), on sampled outputs the fp64
oracle can compute row by row or column by column.

Each stage is graded elementwise against the oracle fed the GPU's own stage
inputs; the forward output is also graded end to end (Frobenius) against the
oracle chained from the seeded inputs on the sampled rows.  Workloads: the 1B
forward, the 7B and 70B forward+backward, and the LM-head cross-entropy
(Synced write-up, sections 尾声 / 五种积木 / 实验结果: GEMM-RMSNorm-GEMM at
the 1B, 7B and 70B hidden sizes).
"""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import B1, B7, B70, LMHEAD, block_inputs, ce_inputs
from tests._parity import assert_device_ok, assert_elem, assert_frob, elem_err, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402


def sample(n, k, seed):
    r = np.random.default_rng(seed)
    idx = set(r.choice(n, size=min(k, n), replace=False).tolist()) | {0, n - 1}
    return np.array(sorted(idx))


def rows_of(t, idx):
    return f64(t[torch.as_tensor(idx, device=t.device)])


def cols_of(t, idx):
    return f64(t[:, torch.as_tensor(idx, device=t.device)])


def dgrad2_sampled(b, kcols, rows, chunk=1024):
    """Oracle dH[rows][:, kcols] and dg[kcols] from the GPU's stage inputs
    (dP, c, H), summing the oracle's dg over row chunks."""
    W2k = cols_of(b.W2t, kcols)
    gk = f64(b.g)[kcols]
    dg = np.zeros(len(kcols))
    for s in range(0, b.M, chunk):
        e = min(b.M, s + chunk)
        _, part = O.stage_dgrad2_rmsbwd(f64(b.dP[s:e]), W2k, gk, cols_of(b.H[s:e], kcols), f64(b.c[s:e]))
        dg += part
    dh, _ = O.stage_dgrad2_rmsbwd(rows_of(b.dP, rows), W2k, gk, rows_of(b.H, rows)[:, kcols], f64(b.c)[rows])
    return dh, dg


def check_block(shape, backward: bool):
    x = block_inputs(shape, 0, "cuda")
    b = BlockBuffers(x, backward=backward)
    b.forward()
    if backward:
        b.backward_stages()
    assert_device_ok()
    M, d, F = shape.M, shape.d, shape.F
    rows = sample(M, 12, 1)
    jcols = sample(F, 16, 2)
    kcols = sample(d, 16, 3)
    ncols = np.concatenate([jcols, F + jcols])
    W1t = f64(b.W1t)
    g = f64(b.g)
    # a1 fold
    assert_elem(rows_of(b.W2gt, ncols), O.fold_weight(rows_of(b.W2t, ncols), g), "W2gt")
    # a2 GEMM1 + residual, partial RMS
    H = rows_of(b.H, rows)
    assert_elem(H, O.gemm_residual(rows_of(b.X, rows), W1t, rows_of(b.R, rows)), "H")
    assert_elem(rows_of(b.psum, rows), O.partial_sumsq(H, C.PARTIAL_COLS), "psum", tol=1e-4)
    # a3 combine
    rstd = f64(b.rstd)[rows]
    assert_elem(rstd, O.rstd_from_partials(rows_of(b.psum, rows), d, shape.eps), "rstd", tol=1e-5)
    # a4 GEMM2 + row scale + SwiGLU on sampled gate/up columns
    z_ref = O.rowscale_gemm(H, rows_of(b.W2gt, ncols), rstd)
    assert_elem(rows_of(b.z, rows)[:, ncols], z_ref, "z")
    out_ref = O.swiglu(z_ref)
    assert_elem(rows_of(b.out, rows)[:, jcols], out_ref, "out")
    # end to end on the sampled rows and columns
    full = O.block_forward(rows_of(b.X, rows), W1t, rows_of(b.R, rows), g, rows_of(b.W2t, ncols), shape.eps, True)
    assert_frob(rows_of(b.out, rows)[:, jcols], full["out"], "out e2e")
    assert_frob(H, full["h"], "H e2e")
    if not backward:
        return
    # a5 SwiGLU backward
    dP_ref, c_ref = O.stage_swiglu_bwd(rows_of(b.dY, rows), rows_of(b.z, rows), rstd, d)
    assert_elem(rows_of(b.dP, rows), dP_ref, "dP")
    assert_elem(f64(b.c)[rows], c_ref, "c")
    # a6 + a7 dgrad2 with the RMSNorm backward, dg
    dh_ref, dg_ref = dgrad2_sampled(b, kcols, rows)
    assert_elem(rows_of(b.dH, rows)[:, kcols], dh_ref, "dH")
    assert_elem(f64(b.dg)[kcols], dg_ref, "dg")
    # a8 wgrad2
    dW2_ref = O.stage_wgrad2(cols_of(b.H, kcols), cols_of(b.dP, ncols), g[kcols])
    e_ours = assert_elem(rows_of(b.dW2t, ncols)[:, kcols], dW2_ref, "dW2t")
    ni, ki = torch.as_tensor(ncols, device="cuda"), torch.as_tensor(kcols, device="cuda")
    cub = torch.matmul(b.dP[:, ni].t(), b.H[:, ki]).float() * b.g[ki].float()
    assert e_ours <= 1.25 * elem_err(cub, dW2_ref) + 1e-3
    # a9 dgrad1, a10 wgrad1; dgrad1 also against cuBLAS (bf16 in, fp32
    # accumulate, bf16 out) on the same inputs: no worse than it
    dX_ref = O.stage_dgrad1(rows_of(b.dH, rows), W1t)
    e_ours = assert_elem(rows_of(b.dX, rows), dX_ref, "dX")
    ri = torch.as_tensor(rows, device="cuda")
    e_cublas = elem_err(torch.matmul(b.dH[ri], b.W1t), dX_ref)
    assert e_ours <= 1.25 * e_cublas + 1e-3, (e_ours, e_cublas)
    icols = sample(shape.K1, 16, 4)
    assert_elem(rows_of(b.dW1t, kcols)[:, icols], O.stage_wgrad1(cols_of(b.dH, kcols), cols_of(b.X, icols)),
                "dW1t")
    # the composite backward reproduces the stage calls exactly
    ref = {k: getattr(b, k).clone() for k in ("dH", "dW2t", "dg", "dX", "dW1t")}
    b.backward()
    torch.cuda.synchronize()
    for k, v in ref.items():
        assert torch.equal(getattr(b, k), v), k


def test_1b_forward_full_size():
    check_block(B1, backward=False)


def test_7b_forward_backward_full_size():
    check_block(B7, backward=True)


def test_70b_forward_backward_full_size():
    check_block(B70, backward=True)


def test_lmhead_ce_full_size():
    s = LMHEAD
    x = ce_inputs(s, 0, "cuda")
    M, d, V = s.M, s.d, s.V
    ws = torch.empty(C.coda_lmhead_ce_workspace_bytes(M, d, V, True), dtype=torch.uint8, device="cuda")
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(M, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    dH = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(V, d, dtype=torch.bfloat16, device="cuda")
    C.coda_lmhead_ce(x["H"], x["Wt"], x["labels"], loss, lse, am, dH, dW, ws)
    assert_device_ok()
    rows = sample(M, 12, 5)
    y = x["labels"].cpu().numpy().astype(np.int64)
    Hs = rows_of(x["H"], rows)
    Wt = f64(x["Wt"])
    Hall = f64(x["H"])
    fw = O.ce_forward(Hs, Wt, y[rows])
    assert_elem(f64(lse)[rows], fw["lse"], "lse", tol=1e-4)
    # argmax on the sampled rows (ties within the fp32 error may go either way)
    L = O.logits_rows(Hs, Wt)
    srt = np.sort(L, axis=1)
    decided = srt[:, -1] - srt[:, -2] > 1e-3
    got = am.cpu().numpy()[rows]
    assert np.array_equal(got[decided], O.argmax_lowest(L)[decided])
    # mean loss = mean(lse - L[y]); the label logits for every row from the oracle
    zy = np.einsum("md,md->m", Hall, Wt[y])
    assert abs(loss.item() - float(np.mean(f64(lse) - zy))) <= 1e-4 * abs(loss.item())
    # dH on sampled rows: the oracle's per-row gradient rescaled from 1/len(rows) to 1/M
    bw = O.ce_backward(Hs, Wt, y[rows])
    assert_frob(rows_of(dH, rows), bw["dH"] * (len(rows) / M), "dH")
    # dW on sampled vocabulary rows (including some labels) given the GPU's lse
    vcols = np.unique(np.concatenate([sample(V, 24, 6), y[rows[:6]]]))
    dW_ref = O.ce_weight_grad_given_lse(Hall, Wt[vcols], vcols, y, f64(lse), M)
    assert_frob(rows_of(dW, vcols), dW_ref, "dW")


def test_7b_block_executor_full_size():
    """The block executor on host buffers at the 7B size, as the bench's
    end-to-end figure drives it: two pipelined steps with different inputs,
    each bit-identical to the separate calls on the same inputs (whose parity
    with the oracle the tests above establish)."""
    from gemm_epilogue_transformer_tma_gb300.path import HostBlockStepper
    w = {k: v for k, v in block_inputs(B7, 0, "cuda").items() if k in ("W1t", "g", "W2t")}
    steps = [block_inputs(B7, seed, "cuda") for seed in (1, 2)]
    st = HostBlockStepper(w["W1t"], w["g"], w["W2t"], B7.M, B7.eps)
    host_in = [{k: x[k].cpu().pin_memory() for k in ("X", "R", "dY")} for x in steps]
    outs = [st.host_buffers(out=True, dX=True, dR=True) for _ in steps]
    for hi, o in zip(host_in, outs):
        st.submit(hi["X"], hi["R"], hi["dY"], **o)
    st.sync()
    del host_in
    for i, (x, o) in enumerate(zip(steps, outs)):
        b = BlockBuffers(dict(w, **{k: x[k] for k in ("X", "R", "dY")}))
        b.step()
        torch.cuda.synchronize()
        assert_device_ok()
        for k_host, k_ref in (("out", "out"), ("dX", "dX"), ("dR", "dH")):
            assert torch.equal(o[k_host], getattr(b, k_ref).cpu()), (i, k_host)
        if i == len(steps) - 1:
            for k in ("dW1t", "dW2t", "dg"):
                assert torch.equal(getattr(st, k), getattr(b, k)), k
        del b
        torch.cuda.empty_cache()
    st.close()
