"""LM-head cross-entropy on FP8 operands (the FP8 variant of the blocked
log-sum-exp and softmax-gradient epilogue programs): e4m3 codes of H and W,
the recomputed dL of each vocabulary chunk kept as e5m2 codes with the
power-of-two scale fixed by |dL| <= 1/M.

  * against the oracle fed the GPU's own H / W codes: lse (elementwise),
    loss, argmax; dH and dW against the oracle's dL (fp64, from the
    dequantised logits) quantised to e5m2 with the same scale, then the two
    contractions (Frobenius: a code that rounds the other way at a tie of
    the fp32 and fp64 dL is invisible there);
  * end to end against the oracle on the bf16 inputs, within bounds from the
    formats' rounding error (e4m3 3.6 %, e5m2 7.2 % rms per element).

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, sections 五种积木: block log-sum-exp; 背景: FP8).
"""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import CEShape, ce_inputs
from tests._ce import check_label_rows, check_row_loss, known_answer_ce, known_answer_logits, with_edge_labels
from tests._parity import assert_device_ok, assert_elem, assert_frob, f64
from tests.test_gpu_ce import check_argmax, pairing  # noqa: F401

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")


def quantize(x):
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty(2, device="cuda")
    C.coda_fp8_quantize(x, q, s)
    return q, s


def deq(q, s, fmt="e4m3"):
    return O.fp8_decode(q.cpu().numpy(), fmt) * float(s[1].item())


def run_fp8_ce(Hq, sH, Wq, sW, labels, grads=True):
    M, d = Hq.shape
    V = Wq.shape[0]
    ws = torch.empty(C.coda_lmhead_ce_workspace_bytes(M, d, V, grads), dtype=torch.uint8, device="cuda")
    o = dict(loss=torch.empty(1, device="cuda"), lse=torch.empty(M, device="cuda"),
             argmax=torch.empty(M, dtype=torch.int32, device="cuda"))
    o["dH"] = torch.empty(M, d, dtype=torch.bfloat16, device="cuda") if grads else None
    o["dW"] = torch.empty(V, d, dtype=torch.bfloat16, device="cuda") if grads else None
    C.coda_lmhead_ce_fp8(Hq, sH[1:], Wq, sW[1:], labels, o["loss"], o["lse"], o["argmax"], o["dH"], o["dW"], ws)
    o["zy"], o["row_loss"] = C.coda_lmhead_ce_row_results(ws, M, d, V, grads)
    return o


@pytest.mark.parametrize("M,d,V", [(200, 144, 1008), (37, 256, 40000)])
def test_fp8_ce_parity(M, d, V, pairing):
    s = CEShape("t", M, d, V)
    x = {k: v.cuda() for k, v in ce_inputs(s, 0).items()}
    x["labels"] = with_edge_labels(x["labels"], V)
    Hq, sH = quantize(x["H"])
    Wq, sW = quantize(x["Wt"])
    o = run_fp8_ce(Hq, sH, Wq, sW, x["labels"])
    torch.cuda.synchronize()
    assert_device_ok()
    Hd, Wd, y = deq(Hq, sH), deq(Wq, sW), x["labels"].cpu().numpy()
    fw = O.ce_forward(Hd, Wd, y)
    assert_elem(o["lse"], fw["lse"], "lse (fp8)", tol=1e-4)
    assert abs(o["loss"].item() - fw["loss"]) <= 1e-4 * abs(fw["loss"])
    L = O.logits_rows(Hd, Wd)
    check_argmax(o["argmax"], Hd, Wd, L=L)
    check_label_rows(o["zy"], o["row_loss"], L, y, fw["lse"])
    # the backward's dL as the GPU keeps it: e5m2 codes with the scale fixed
    # by |dL| <= 1/M
    P = np.exp(L - fw["lse"][:, None])
    P[np.arange(M), y] -= 1.0
    dL = P / M
    s_dL = O.fp8_scale(np.array([1.0 / M], np.float32), "e5m2")
    assert np.max(np.abs(dL)) <= 1.0 / M
    dLd = O.fp8_decode(O.fp8_quantize(dL, s_dL, "e5m2"), "e5m2") * float(s_dL)
    assert_frob(o["dH"], dLd @ Wd, "dH (fp8, e5m2 dL)")
    assert_frob(o["dW"], dLd.T @ Hd, "dW (fp8, e5m2 dL)")
    # end to end against the bf16 inputs
    Hb, Wb = f64(x["H"]), f64(x["Wt"])
    fb = O.ce_forward(Hb, Wb, y)
    bb = O.ce_backward(Hb, Wb, y)
    assert abs(o["loss"].item() - fb["loss"]) <= 1e-2 * abs(fb["loss"])
    assert_frob(o["dH"], bb["dH"], "dH fp8 e2e", tol=0.15)
    assert_frob(o["dW"], bb["dWt"], "dW fp8 e2e", tol=0.15)


def test_fp8_ce_narrower_backward_chunks():
    """The 8-bit backward in 4096-column chunks (ten at V = 40000, each one
    grouped dH / dW launch): dW bit-equal to the default chunks' (its tiles do
    not change), dH within its fp32 summation order, and both against the
    oracle fed the same codes."""
    M, d, V = 37, 256, 40000
    s = CEShape("t", M, d, V)
    x = {k: v.cuda() for k, v in ce_inputs(s, 4).items()}
    x["labels"] = with_edge_labels(x["labels"], V, 4096)
    Hq, sH = quantize(x["H"])
    Wq, sW = quantize(x["Wt"])
    base = run_fp8_ce(Hq, sH, Wq, sW, x["labels"])
    C.coda_set_lmhead_chunk(4096)
    try:
        o = run_fp8_ce(Hq, sH, Wq, sW, x["labels"])
        torch.cuda.synchronize()
    finally:
        C.coda_set_lmhead_chunk(0)
    assert_device_ok()
    assert torch.equal(o["dW"], base["dW"])
    assert_frob(o["dH"], f64(base["dH"]), "dH vs default chunks (fp8)", tol=2 ** -8)
    Hd, Wd, y = deq(Hq, sH), deq(Wq, sW), x["labels"].cpu().numpy()
    L = O.logits_rows(Hd, Wd)
    lse = O.ce_forward(Hd, Wd, y)["lse"]
    P = np.exp(L - lse[:, None])
    P[np.arange(M), y] -= 1.0
    s_dL = O.fp8_scale(np.array([1.0 / M], np.float32), "e5m2")
    dLd = O.fp8_decode(O.fp8_quantize(P / M, s_dL, "e5m2"), "e5m2") * float(s_dL)
    assert_frob(o["dH"], dLd @ Wd, "dH (fp8, 4096-column chunks)")
    assert_frob(o["dW"], dLd.T @ Hd, "dW (fp8, 4096-column chunks)")


def test_fp8_ce_forward_only_and_argument_errors():
    s = CEShape("t", 64, 64, 512)
    x = {k: v.cuda() for k, v in ce_inputs(s, 1).items()}
    Hq, sH = quantize(x["H"])
    Wq, sW = quantize(x["Wt"])
    o = run_fp8_ce(Hq, sH, Wq, sW, x["labels"], grads=False)
    torch.cuda.synchronize()
    assert_device_ok()
    fw = O.ce_forward(deq(Hq, sH), deq(Wq, sW), x["labels"].cpu().numpy())
    assert_elem(o["lse"], fw["lse"], "lse (fp8, forward only)", tol=1e-4)
    lib = C.load_library()
    h = C.handle()
    st = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(C.coda_lmhead_ce_workspace_bytes(64, 64, 512, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty(64, device="cuda")
    args = [Hq.data_ptr(), sH[1:].data_ptr(), Wq.data_ptr(), sW[1:].data_ptr(), x["labels"].data_ptr(),
            out.data_ptr(), out.data_ptr(), None, None, None, ws.data_ptr(), ws.numel()]
    # d = 56: not a multiple of 16 (the 8-bit rows need 16-byte multiples)
    assert lib.coda_lmhead_ce_fp8(h, *args, 64, 56, 512, st) == 2
    # an empty batch has no mean
    assert lib.coda_lmhead_ce_fp8(h, *args, 0, 64, 512, st) == 1


@pytest.mark.parametrize("M,d,V", [(200, 64, 1008), (37, 256, 40000)])
def test_fp8_ce_label_logit_and_argmax_known_answer(M, d, V, pairing):
    """Label indexing and argmax bit-exact on every row with 8-bit operands:
    integer logits +-pi(v) written in base 8 (digits and powers of two exact
    in e4m3 under the power-of-two scales), labels on the tile and chunk
    edges."""
    H, Wt, lab, zy_ref, am_ref = known_answer_ce(M, d, V, seed=M + V, base=8)
    Hq, sH = quantize(H.cuda())
    Wq, sW = quantize(Wt.cuda())
    assert np.array_equal(deq(Hq, sH), f64(H)) and np.array_equal(deq(Wq, sW), f64(Wt))
    o = run_fp8_ce(Hq, sH, Wq, sW, lab.cuda(), grads=False)
    torch.cuda.synchronize()
    assert_device_ok()
    assert np.array_equal(f64(o["zy"]), zy_ref)
    assert np.array_equal(o["argmax"].cpu().numpy().astype(np.int64), am_ref)
    lse_ref = O.lse_rows(known_answer_logits(Wt, M, base=8))
    assert_elem(o["lse"], lse_ref, "lse (fp8, integer logits)", tol=1e-5)
    check_row_loss(o["row_loss"], lse_ref, zy_ref)
