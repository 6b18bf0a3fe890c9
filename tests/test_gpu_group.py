"""Grouped launches of independent GEMM pairs: the first layer's data
gradient and weight gradient (dX, dW1) in one persistent SM-pair launch with
a balanced tile schedule (the LM-head's dH / dW chunk pairs use the same
kernel and are checked against the oracle in test_gpu_ce.py).  Each output
tile is computed by the same MMA sequence as in a separate launch, so the
grouped results must be bit-identical to two separate launches; they are
also checked against the oracle.  Sizes cover the schedule's cases: fewer
tiles than SM pairs, more than one wave, the heavy problem first or second,
ragged tails.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, sections 尾声 and 五种积木: the backward's GEMMs with their
epilogues).
"""
import pytest
import torch

import oracle as O
from tests._parity import assert_device_ok, assert_elem, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")


@pytest.mark.parametrize("M,K1,d", [
    (1280, 512, 256),    # wgrad heavier (K = M); fewer tiles than SM pairs
    (256, 512, 1024),    # dgrad heavier (K = d)
    (4096, 1024, 1024),  # 80 tiles: more than one wave, catch-up covers every light tile
    (8192, 2048, 2048),  # 320 tiles, heavy tiles fewer than SM pairs, round-robin tail
    (1000, 520, 328),    # ragged in every dimension
])
def test_dgrad_wgrad1_grouped_equals_separate(M, K1, d):
    g = torch.Generator(device="cuda").manual_seed(M + K1 + d)
    dH = torch.randn(M, d, device="cuda", generator=g).to(torch.bfloat16)
    X = torch.randn(M, K1, device="cuda", generator=g).to(torch.bfloat16)
    W1t = (torch.randn(d, K1, device="cuda", generator=g) / d ** 0.5).to(torch.bfloat16)
    dX = torch.empty(M, K1, device="cuda", dtype=torch.bfloat16)
    dW1t = torch.empty(d, K1, device="cuda", dtype=torch.bfloat16)
    C.coda_gemm_res_prms_bwd(dH, X, W1t, dX, dW1t, None)
    rX = torch.empty_like(dX)
    rW = torch.empty_like(dW1t)
    C.coda_gemm(dH, False, W1t, True, rX, M, K1, d)
    C.coda_gemm(dH, True, X, True, rW, d, K1, M)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(dX, rX)
    assert torch.equal(dW1t, rW)
    if M * K1 * d <= 1 << 28:
        assert_elem(dX, O.stage_dgrad1(f64(dH), f64(W1t)), "dX")
        assert_elem(dW1t, O.stage_wgrad1(f64(dH), f64(X)), "dW1t")
