"""Parity at the full workload sizes, in the launch configuration the bench
times (same entry points, persistent grids), on whole rows and whole columns
the fp64 oracle computes in seconds.

Each stage is graded elementwise against the oracle fed the GPU's own stage
inputs: whole rows (every column) of H, z, out, dP and dX on at least 256
rows, taken from the first and last row tiles, both sides of the 128- and
256-row tile edges and at random; every row of psum, rstd, c and dH (dH and
dg from a full row-blocked oracle pass of the second GEMM's data gradient);
all of dg; at least 64 whole columns and 64 whole rows of dW2t and dW1t,
including the first and last column tiles and the gate/up boundary.  The
forward output is also graded end to end (Frobenius) against the oracle
chained from the seeded inputs on the sampled rows.  Workloads: the 1B
forward, the 7B and 70B forward+backward (each on the default 256 x 256 pair
tiles and on the opt-in 256 x 512 tiles), and the LM-head cross-entropy
(Synced write-up, sections 尾声 / 五种积木 / 实验结果: GEMM-RMSNorm-GEMM at
the 1B, 7B and 70B hidden sizes).
"""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import B1, B7, B70, LMHEAD, block_inputs, ce_inputs
from tests._ce import check_argmax, check_label_rows, edge_labels, known_answer_ce
from tests._parity import assert_device_ok, assert_elem, assert_elem_chunks, assert_frob, edge_sample, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402

CHUNK = 1024  # rows per oracle block for the whole-tensor passes


def rows_of(t, idx):
    return f64(t[torch.as_tensor(idx, device=t.device)])


def cols_of(t, idx):
    return f64(t[:, torch.as_tensor(idx, device=t.device)])


def row_blocks(M):
    return [(s, min(M, s + CHUNK)) for s in range(0, M, CHUNK)]


def mm_f32(A, B):
    """cuBLAS bf16 GEMM A B with its fp32 result (fp32 accumulation, no
    rounding of the product to bf16): the library's counterpart where an
    epilogue consumes the fp32 accumulator."""
    return torch.mm(A, B, out_dtype=torch.float32)


def check_block(shape, backward: bool):
    x = block_inputs(shape, 0, "cuda")
    b = BlockBuffers(x, backward=backward)
    b.forward()
    if backward:
        b.backward_stages()
    assert_device_ok()
    M, d, F, K1 = shape.M, shape.d, shape.F, shape.K1
    rows = edge_sample(M, 256, 1)
    jcols = edge_sample(F, 32, 2)
    ncols = np.concatenate([jcols, F + jcols])          # gate and matching up rows of W2t
    kcols = edge_sample(d, 64, 3)
    icols = edge_sample(K1, 64, 4)
    ri, ni, ki, ii = (torch.as_tensor(v, device="cuda") for v in (rows, ncols, kcols, icols))
    bf = torch.bfloat16
    W1t = f64(b.W1t)
    W2t = f64(b.W2t)
    g = f64(b.g)
    # a1 fold: whole rows of W2gt (gate and up)
    assert_elem(rows_of(b.W2gt, ncols), O.fold_weight(W2t[ncols], g), "W2gt")
    # a2 GEMM1 + residual (whole rows), partial RMS (every row)
    H = rows_of(b.H, rows)
    cub = (mm_f32(b.X[ri], b.W1t.t()) + b.R[ri].float()).to(bf)
    assert_elem(H, O.gemm_residual(rows_of(b.X, rows), W1t, rows_of(b.R, rows)), "H", cublas=cub)
    Hall = f64(b.H)
    psum_all = f64(b.psum)
    assert_elem(psum_all, O.partial_sumsq(Hall, C.PARTIAL_COLS), "psum", tol=1e-4)
    # a3 combine, every row
    assert_elem(b.rstd, O.rstd_from_partials(psum_all, d, shape.eps), "rstd", tol=1e-5)
    rstd = f64(b.rstd)[rows]
    # a4 GEMM2 + row scale + SwiGLU, whole rows
    z_ref = O.rowscale_gemm(H, f64(b.W2gt), rstd)
    z32 = b.rstd[ri, None] * mm_f32(b.H[ri], b.W2gt.t())
    assert_elem(rows_of(b.z, rows), z_ref, "z", cublas=z32.to(bf))
    out_ref = O.swiglu(z_ref)
    zg, zu = z32[:, :F], z32[:, F:]
    assert_elem(rows_of(b.out, rows), out_ref, "out", cublas=(zg * torch.sigmoid(zg) * zu).to(bf))
    del z32, zg, zu
    # end to end on the sampled rows
    full = O.block_forward(rows_of(b.X, rows), W1t, rows_of(b.R, rows), g, W2t, shape.eps, True)
    assert_frob(rows_of(b.out, rows), full["out"], "out e2e")
    assert_frob(H, full["h"], "H e2e")
    del full, z_ref, out_ref
    if not backward:
        return
    # a5 SwiGLU backward: dP on whole rows, c on every row
    dP_ref, _ = O.stage_swiglu_bwd(rows_of(b.dY, rows), rows_of(b.z, rows), rstd, d)
    assert_elem(rows_of(b.dP, rows), dP_ref, "dP")
    rstd_all = f64(b.rstd)
    c_ref = np.concatenate([O.stage_swiglu_bwd(f64(b.dY[s:e]), f64(b.z[s:e]), rstd_all[s:e], d)[1]
                            for s, e in row_blocks(M)])
    assert_elem(b.c, c_ref, "c")
    # a6 + a7 dgrad2 with the RMSNorm backward: dH on every row, all of dg
    c_all = f64(b.c)
    dg_ref = np.zeros(d)
    gf = b.g.float()
    dg_cub = np.zeros(d)
    parts = []
    for s, e in row_blocks(M):
        dh, part = O.stage_dgrad2_rmsbwd(f64(b.dP[s:e]), W2t, g, Hall[s:e], c_all[s:e])
        dg_ref += part
        acc = mm_f32(b.dP[s:e], b.W2t)
        cub = (gf * acc - b.c[s:e, None] * b.H[s:e].float()).to(bf)
        dg_cub += f64((acc * b.H[s:e].float()).sum(0))
        parts.append((b.dH[s:e], dh, cub))
        del acc
    assert_elem_chunks(parts, "dH")
    del parts
    assert_elem(b.dg, dg_ref, "dg", cublas=dg_cub)
    # a8 wgrad2: whole columns (fixed k) and whole rows (fixed n) of dW2t
    dP_all = f64(b.dP)
    cub = (mm_f32(b.dP.t(), b.H[:, ki]) * gf[ki]).to(bf)
    assert_elem(cols_of(b.dW2t, kcols), O.stage_wgrad2(Hall[:, kcols], dP_all, g[kcols]), "dW2t columns",
                cublas=cub)
    cub = (mm_f32(b.dP[:, ni].t(), b.H) * gf).to(bf)
    assert_elem(rows_of(b.dW2t, ncols), O.stage_wgrad2(Hall, dP_all[:, ncols], g), "dW2t rows", cublas=cub)
    del dP_all, cub
    # a9 dgrad1 (whole rows)
    dX_ref = O.stage_dgrad1(rows_of(b.dH, rows), W1t)
    assert_elem(rows_of(b.dX, rows), dX_ref, "dX", cublas=torch.matmul(b.dH[ri], b.W1t))
    # a10 wgrad1: whole rows (fixed k) and whole columns (fixed i) of dW1t
    dH_all = f64(b.dH)
    X_all = f64(b.X)
    assert_elem(rows_of(b.dW1t, kcols), O.stage_wgrad1(dH_all[:, kcols], X_all), "dW1t rows",
                cublas=torch.matmul(b.dH[:, ki].t(), b.X))
    assert_elem(cols_of(b.dW1t, icols), O.stage_wgrad1(dH_all, X_all[:, icols]), "dW1t columns",
                cublas=torch.matmul(b.dH.t(), b.X[:, ii]))
    del dH_all, X_all
    # the composite backward reproduces the stage calls exactly
    ref = {k: getattr(b, k).clone() for k in ("dH", "dW2t", "dg", "dX", "dW1t")}
    b.backward()
    torch.cuda.synchronize()
    for k, v in ref.items():
        assert torch.equal(getattr(b, k), v), k


def test_1b_forward_full_size():
    check_block(B1, backward=False)


@pytest.fixture(params=[0, 8], ids=["tiles_256", "wide_tiles"])
def wide_lead(request):
    """The default 256 x 256 pair tiles, and the opt-in 256 x 512 pair tiles
    (coda_set_wide_tiles, lead 8), which the data gradient of the second GEMM
    (K = 2F) takes at both block sizes."""
    C.coda_set_wide_tiles(request.param)
    yield request.param
    torch.cuda.synchronize()
    C.coda_set_wide_tiles(0)


def test_7b_forward_backward_full_size(wide_lead):
    if wide_lead:
        assert C.coda_debug_wide_applies(B7.M, B7.d, B7.N2) == 1
    check_block(B7, backward=True)


def test_70b_forward_backward_full_size(wide_lead):
    if wide_lead:
        assert C.coda_debug_wide_applies(B70.M, B70.d, B70.N2) == 1
    check_block(B70, backward=True)


def test_lmhead_ce_full_size():
    """Every row's label logit; lse, argmax, row loss and the label's column
    on at least 256 whole rows (all 128256 logits each), with labels placed
    on the 128- and 256-column tile edges, the backward chunk edges and the
    last vocabulary columns; dH and dW by Frobenius."""
    s = LMHEAD
    x = ce_inputs(s, 0, "cuda")
    M, d, V = s.M, s.d, s.V
    rows = edge_sample(M, 256, 5)
    edges = edge_labels(V)
    assert len(edges) <= len(rows)
    labels = x["labels"].clone()
    labels[torch.as_tensor(rows[:len(edges)], device="cuda")] = torch.tensor(edges, dtype=labels.dtype,
                                                                             device="cuda")
    ws = torch.empty(C.coda_lmhead_ce_workspace_bytes(M, d, V, True), dtype=torch.uint8, device="cuda")
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(M, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    dH = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(V, d, dtype=torch.bfloat16, device="cuda")
    C.coda_lmhead_ce(x["H"], x["Wt"], labels, loss, lse, am, dH, dW, ws)
    assert_device_ok()
    zy_gpu, row_loss_gpu = C.coda_lmhead_ce_row_results(ws, M, d, V, True)
    y = labels.cpu().numpy().astype(np.int64)
    Hall = f64(x["H"])
    Wt = f64(x["Wt"])
    # the label logit of every row: L[m, y_m] = H[m] . W[y_m]
    zy_ref = np.einsum("md,md->m", Hall, Wt[y])
    assert_elem(zy_gpu, zy_ref, "label logit (all rows)")
    # whole rows of logits on the sample: lse, argmax, row loss, label column
    Hs = Hall[rows]
    L = O.logits_rows(Hs, Wt)
    lse_ref = O.lse_rows(L)
    assert_elem(f64(lse)[rows], lse_ref, "lse", tol=1e-4)
    assert check_argmax(am.cpu()[rows], Hs, Wt, L=L) >= len(rows) - 4
    check_label_rows(zy_gpu, row_loss_gpu, L, y[rows], lse_ref, rows=rows)
    # mean loss = mean(lse - L[y]) over every row
    assert abs(loss.item() - float(np.mean(f64(lse) - zy_ref))) <= 1e-4 * abs(loss.item())
    # dH on sampled rows: the oracle's per-row gradient rescaled from 1/len(rows) to 1/M
    bw = O.ce_backward(Hs, Wt, y[rows])
    assert_frob(rows_of(dH, rows), bw["dH"] * (len(rows) / M), "dH")
    # dW on sampled vocabulary rows (the edge labels among them) given the GPU's lse
    vcols = np.unique(np.concatenate([edge_sample(V, 48, 6), np.asarray(edges)]))
    dW_ref = O.ce_weight_grad_given_lse(Hall, Wt[vcols], vcols, y, f64(lse), M)
    assert_frob(rows_of(dW, vcols), dW_ref, "dW")


def test_lmhead_ce_known_answer_full_size():
    """Label logit and argmax bit-exact on all 8192 rows at the full
    vocabulary (integer logits +-pi(v), see tests/_ce.py), labels on every
    tile and chunk edge."""
    s = LMHEAD
    H, Wt, lab, zy_ref, am_ref = known_answer_ce(s.M, s.d, s.V, seed=7)
    Hd, Wd, ld = H.cuda(), Wt.cuda(), lab.cuda()
    del H, Wt
    ws = torch.empty(C.coda_lmhead_ce_workspace_bytes(s.M, s.d, s.V, False), dtype=torch.uint8, device="cuda")
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(s.M, device="cuda")
    am = torch.empty(s.M, dtype=torch.int32, device="cuda")
    C.coda_lmhead_ce(Hd, Wd, ld, loss, lse, am, None, None, ws)
    assert_device_ok()
    zy_gpu, _ = C.coda_lmhead_ce_row_results(ws, s.M, s.d, s.V, False)
    assert np.array_equal(f64(zy_gpu), zy_ref)
    assert np.array_equal(am.cpu().numpy().astype(np.int64), am_ref)


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
