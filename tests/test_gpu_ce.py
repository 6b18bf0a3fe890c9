"""LM-head cross-entropy with the blocked log-sum-exp epilogue vs the fp64
oracle (Synced write-up, section 五种积木: block reduction "block
log-sum-exp" and the stateful max / sum-exp statistics; the label logit is
gathered by the epilogue of the vocabulary tile that holds the label).

Small vocabularies that still span several 256-column tiles with a ragged
last tile, plus two 32768-column backward chunks (and ten of 4096 columns
with the chunk width set narrower).  Every row's label
logit and row loss is read back from the workspace and graded, with labels
placed on the 128- and 256-column tile edges, the backward chunk edges and
the last (ragged) tile."""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import CEShape, ce_inputs
from tests._ce import (check_argmax, check_label_rows, check_row_loss, known_answer_ce, known_answer_logits,
                      with_edge_labels)
from tests._parity import assert_device_ok, assert_elem, assert_frob, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")


@pytest.fixture(params=[True, False], ids=["sm_pair", "single_sm"])
def pairing(request):
    C.coda_set_sm_pairing(request.param)
    yield request.param
    C.coda_set_sm_pairing(True)


def run_ce(H, Wt, labels, grads=True):
    M, d = H.shape
    V = Wt.shape[0]
    ws = torch.empty(C.coda_lmhead_ce_workspace_bytes(M, d, V, grads), dtype=torch.uint8, device="cuda")
    out = dict(loss=torch.empty(1, device="cuda"), lse=torch.empty(M, device="cuda"),
               argmax=torch.empty(M, dtype=torch.int32, device="cuda"))
    dH = torch.empty(M, d, dtype=torch.bfloat16, device="cuda") if grads else None
    dW = torch.empty(V, d, dtype=torch.bfloat16, device="cuda") if grads else None
    C.coda_lmhead_ce(H, Wt, labels, out["loss"], out["lse"], out["argmax"], dH, dW, ws)
    out["dH"], out["dW"] = dH, dW
    out["zy"], out["row_loss"] = C.coda_lmhead_ce_row_results(ws, M, d, V, grads)
    return out


@pytest.mark.parametrize("M,d,V", [(200, 136, 1000), (128, 64, 256), (37, 256, 40000)])
def test_ce_parity(M, d, V, pairing):
    s = CEShape("t", M, d, V)
    x = {k: v.cuda() for k, v in ce_inputs(s, 0).items()}
    x["labels"] = with_edge_labels(x["labels"], V)
    o = run_ce(x["H"], x["Wt"], x["labels"])
    assert_device_ok()
    H, Wt, y = f64(x["H"]), f64(x["Wt"]), x["labels"].cpu().numpy()
    fw = O.ce_forward(H, Wt, y)
    bw = O.ce_backward(H, Wt, y)
    assert_elem(o["lse"], fw["lse"], "lse", tol=1e-4)
    assert abs(o["loss"].item() - fw["loss"]) <= 1e-4 * abs(fw["loss"])
    L = O.logits_rows(H, Wt)
    check_argmax(o["argmax"], H, Wt, L=L)
    check_label_rows(o["zy"], o["row_loss"], L, y, fw["lse"])
    assert_frob(o["dH"], bw["dH"], "dH")
    assert_frob(o["dW"], bw["dWt"], "dW")


@pytest.mark.parametrize("chunk,V", [(4096, 40000), (256, 5000)])
def test_ce_narrower_backward_chunks(chunk, V):
    """coda_set_lmhead_chunk: the backward in narrower vocabulary chunks (ten
    of 4096 columns; twenty of 256, one tile each) against the oracle, with
    labels on the chunk edges; dW equal to the default chunks' bit for bit
    (its tiles do not change), dH within its fp32 summation order."""
    lib = C.load_library()
    h = C.handle()
    for bad in (-256, 100, 255, 32768 + 256):
        assert lib.coda_set_lmhead_chunk(h, bad) == 1  # CODA_ERR_INVALID_ARG
    s = CEShape("t", 200, 136, V)
    x = {k: v.cuda() for k, v in ce_inputs(s, 3).items()}
    x["labels"] = with_edge_labels(x["labels"], V, chunk)
    base = run_ce(x["H"], x["Wt"], x["labels"])
    C.coda_set_lmhead_chunk(chunk)
    try:
        o = run_ce(x["H"], x["Wt"], x["labels"])
        assert_device_ok()
    finally:
        C.coda_set_lmhead_chunk(0)
    H, Wt, y = f64(x["H"]), f64(x["Wt"]), x["labels"].cpu().numpy()
    bw = O.ce_backward(H, Wt, y)
    assert torch.equal(o["lse"], base["lse"]) and torch.equal(o["loss"], base["loss"])
    assert torch.equal(o["dW"], base["dW"])
    assert_frob(o["dH"], bw["dH"], "dH")
    assert_frob(o["dW"], bw["dWt"], "dW")
    assert_frob(o["dH"], f64(base["dH"]), "dH vs default chunks", tol=2 ** -8)


def test_ce_forward_only_and_label_range():
    s = CEShape("t", 64, 64, 512)
    x = {k: v.cuda() for k, v in ce_inputs(s, 1).items()}
    lab = x["labels"].clone()
    lab[3] = 512          # out of range
    lab[5] = -1
    o = run_ce(x["H"], x["Wt"], lab, grads=False)
    st, bits = C.coda_sync_status()
    assert st == 7 and (bits & 0x100)
    H, Wt = f64(x["H"]), f64(x["Wt"])
    lse = O.lse_rows(O.logits_rows(H, Wt))
    assert_elem(o["lse"], lse, "lse", tol=1e-4)
    ok = np.ones(64, bool)
    ok[[3, 5]] = False
    L = O.logits_rows(H, Wt)
    yy = lab.cpu().numpy()
    per_row = np.where(ok, lse - L[np.arange(64), np.clip(yy, 0, 511)], 0.0)
    assert abs(o["loss"].item() - per_row.mean()) <= 1e-4 * abs(per_row.mean())
    # rows with a label outside [0, V) gather nothing and contribute 0
    zy, rl = f64(o["zy"]), f64(o["row_loss"])
    assert zy[3] == 0.0 and zy[5] == 0.0 and rl[3] == 0.0 and rl[5] == 0.0
    check_label_rows(zy[ok], rl[ok], L[ok], yy[ok], lse[ok])
    assert_device_ok()


def test_ce_argmax_ties_pick_lowest_column():
    M, d, V = 16, 64, 1024
    g = torch.Generator().manual_seed(3)
    H = torch.randn(M, d, generator=g).to(torch.bfloat16)
    Wt = (torch.randn(V, d, generator=g) * 0.02).to(torch.bfloat16)
    # exact duplicates of the winning column, in a later tile and in the same tile
    L = f64(H) @ f64(Wt).T
    win = O.argmax_lowest(L)
    for m in range(M):
        Wt[(win[m] + 300 + m) % V] = Wt[win[m]]
    L = f64(H) @ f64(Wt).T
    lab = torch.zeros(M, dtype=torch.int32)
    o = run_ce(H.cuda(), Wt.cuda(), lab.cuda(), grads=False)
    assert_device_ok()
    assert np.array_equal(o["argmax"].cpu().numpy(), O.argmax_lowest(L))


def test_ce_large_logits_and_edge_labels(pairing):
    """Logits of several hundred (exp overflows fp32 past about 88 unless the
    running maximum is subtracted): the blocked statistics and the backward's
    exp(L - lse) must stay finite and match the oracle; labels on the first
    and last vocabulary columns (the last one in the ragged last tile)."""
    s = CEShape("t", 96, 136, 1000)
    x = ce_inputs(s, 3)
    H = (x["H"].float() * 400).to(torch.bfloat16)
    lab = x["labels"].clone()
    lab[0], lab[1], lab[2] = 0, s.V - 1, s.V - 1
    o = run_ce(H.cuda(), x["Wt"].cuda(), lab.cuda())
    assert_device_ok()
    Hf, Wt, y = f64(H), f64(x["Wt"]), lab.numpy()
    L = O.logits_rows(Hf, Wt)
    assert np.abs(L).max() > 200
    fw = O.ce_forward(Hf, Wt, y)
    bw = O.ce_backward(Hf, Wt, y)
    for k in ("lse", "dH", "dW"):
        assert torch.isfinite(o[k].float()).all(), k
    assert_elem(o["lse"], fw["lse"], "lse (large logits)", tol=1e-4)
    assert abs(o["loss"].item() - fw["loss"]) <= 1e-4 * abs(fw["loss"])
    check_argmax(o["argmax"], Hf, Wt, L=L)
    # logits of several hundred: the fp32 accumulation error is ~1e-5 of them
    check_label_rows(o["zy"], o["row_loss"], L, y, fw["lse"], tol_gap=0.05)
    assert_frob(o["dH"], bw["dH"], "dH (large logits)")
    assert_frob(o["dW"], bw["dWt"], "dW (large logits)")


@pytest.mark.parametrize("M,d,V", [(200, 64, 1000), (37, 256, 40000), (256, 16, 128256)])
def test_ce_label_logit_and_argmax_known_answer(M, d, V, pairing):
    """Label indexing and argmax bit-exact on every row: integer logits
    L[m, v] = +-pi(v) for a fixed permutation pi (exact in any fp32
    summation order), labels on the tile and chunk edges."""
    H, Wt, lab, zy_ref, am_ref = known_answer_ce(M, d, V, seed=M + V)
    o = run_ce(H.cuda(), Wt.cuda(), lab.cuda(), grads=False)
    assert_device_ok()
    assert np.array_equal(f64(o["zy"]), zy_ref)
    assert np.array_equal(o["argmax"].cpu().numpy().astype(np.int64), am_ref)
    # lse = max + log sum exp(L - max) of the integer logits; the row loss
    lse_ref = O.lse_rows(known_answer_logits(Wt, M))
    assert_elem(o["lse"], lse_ref, "lse (integer logits)", tol=1e-5)
    check_row_loss(o["row_loss"], lse_ref, zy_ref)
