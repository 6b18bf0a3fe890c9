"""Write guards: no kernel writes outside the buffers it is given.

compute-sanitizer is not available, so every output buffer of the path is
handed to the library as a view into a larger allocation whose bytes before
and after the view carry a sentinel pattern; after the calls the guard bytes
must be untouched.  An out-of-range row or column in an epilogue's plain
stores (the partial sums, c, the dg partials, the per-row label logits), a
tensor map with a wrong extent or pitch, or a combine kernel running past
its row count would change them.  Ragged shapes (tails in every extent), on
SM pairs and on single SMs, through the bf16 block forward and backward, the
unfused ablation, the FP8 block, the LM-head cross-entropy and the QKV RoPE
projection; the opt-in wide and split schedules on the GEMM they change.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, sections 尾声 and 五种积木: each epilogue writes only its
own tile of the output and its own partials).
"""
import pytest
import torch

from coda_inputs import BlockShape, CEShape, block_inputs, ce_inputs
from tests._guard import Guards
from tests._parity import assert_device_ok

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402

def guard_outputs(b, names, g):
    for k in names:
        t = getattr(b, k, None)
        if t is not None:
            setattr(b, k, g.like(t))


SHAPES = [BlockShape("ragged", 300, 200, 328, 528), BlockShape("one_row", 1, 64, 64, 128),
          BlockShape("tails", 777, 136, 392, 784)]
FWD = ("W2gt", "H", "psum", "rstd", "z", "out")
BWD = ("dP", "c", "dgpart", "dH", "dX", "dW1t", "dW2t", "dg", "ws")


@pytest.mark.parametrize("pair", [True, False], ids=["sm_pair", "single_sm"])
@pytest.mark.parametrize("s", SHAPES, ids=[s.name for s in SHAPES])
def test_block_writes_stay_in_bounds(s, pair):
    C.coda_set_sm_pairing(pair)
    try:
        g = Guards()
        b = BlockBuffers(block_inputs(s, 0, "cuda"))
        guard_outputs(b, FWD + BWD, g)
        b.forward()
        b.backward_stages()
        g.check("stages")
        b.step()              # the fused backward entry point (its workspace guarded too)
        g.check("fused step")
        assert_device_ok()
    finally:
        C.coda_set_sm_pairing(True)


def test_unfused_and_fp8_block_writes_stay_in_bounds():
    s = BlockShape("tails16", 777, 208, 400, 800)  # FP8 extents: multiples of 16
    g = Guards()
    b = BlockBuffers(block_inputs(s, 1, "cuda"), unfused=True)
    guard_outputs(b, FWD + BWD + ("Nrm", "ws_unfused"), g)
    b.forward_unfused()
    b.backward_unfused()
    g.check("unfused")
    b._fp8_buffers()
    guard_outputs(b, ("Xq", "Hq", "W1q", "W2gq", "W2q", "s_w", "s_a", "dPq", "dHq"), g)
    b.fp8_quantize_weights()
    b.forward_fp8()
    b.backward_fp8()
    b.backward_fp8(delayed=True)
    g.check("fp8")
    assert_device_ok()


@pytest.mark.parametrize("M,d,V", [(37, 256, 40000), (200, 136, 1000), (1, 64, 264)])
def test_lmhead_writes_stay_in_bounds(M, d, V):
    s = CEShape("t", M, d, V)
    x = {k: v.cuda() for k, v in ce_inputs(s, 2).items()}
    g = Guards()
    nws = C.coda_lmhead_ce_workspace_bytes(M, d, V, True)
    ws = g.new((nws,), torch.uint8)
    loss, lse = g.new((1,), torch.float32), g.new((M,), torch.float32)
    am = g.new((M,), torch.int32)
    dH, dW = g.new((M, d), torch.bfloat16), g.new((V, d), torch.bfloat16)
    C.coda_lmhead_ce(x["H"], x["Wt"], x["labels"], loss, lse, am, dH, dW, ws)
    C.coda_set_lmhead_chunk(256)
    try:
        C.coda_lmhead_ce(x["H"], x["Wt"], x["labels"], loss, lse, am, dH, dW, ws)
    finally:
        C.coda_set_lmhead_chunk(0)
    g.check("bf16 cross-entropy")
    if d % 16 == 0 and V % 16 == 0:
        Hq, Wq = g.new((M, d), torch.uint8), g.new((V, d), torch.uint8)
        sc = g.new((2, 2), torch.float32)
        C.coda_fp8_quantize(x["H"], Hq, sc[0])
        C.coda_fp8_quantize(x["Wt"], Wq, sc[1])
        C.coda_lmhead_ce_fp8(Hq, sc[0, 1:], Wq, sc[1, 1:], x["labels"], loss, lse, am, dH, dW, ws)
        g.check("FP8 cross-entropy")
    assert_device_ok()


def test_qkv_rope_writes_stay_in_bounds():
    M, d, hq, hkv, S = 300, 328, 3, 1, 100
    gen = torch.Generator().manual_seed(9)
    X = torch.randn(M, d, generator=gen).to(torch.bfloat16).cuda()
    W = (torch.randn((hq + 2 * hkv) * 128, d, generator=gen) * 0.02).to(torch.bfloat16).cuda()
    g = Guards()
    cos_t, sin_t = g.new((S, 64), torch.float32), g.new((S, 64), torch.float32)
    qkv = g.new((M, (hq + 2 * hkv) * 128), torch.bfloat16)
    C.coda_rope_table(cos_t, sin_t, 10000.0)
    C.coda_gemm_qkv_rope(X, W, cos_t, sin_t, qkv, hq, hkv)
    C.coda_rope_apply(qkv, cos_t, sin_t, hq, hkv)
    g.check("rope")
    assert_device_ok()


@pytest.mark.parametrize("sched", ["wide", "split"])
def test_opt_in_schedules_write_stay_in_bounds(sched):
    M, N, K = (1800, 3904, 16448) if sched == "wide" else (1800, 3904, 13000)
    gen = torch.Generator().manual_seed(10)
    A = torch.randn(M, K, generator=gen).to(torch.bfloat16).cuda()
    B = (torch.randn(N, K, generator=gen) / K ** 0.5).to(torch.bfloat16).cuda()
    g = Guards()
    out = g.new((M, N), torch.bfloat16)
    ws = None
    if sched == "wide":
        C.coda_set_wide_tiles(8)
        assert C.coda_debug_wide_applies(M, N, K) == 1
    else:
        ws = g.new((C.coda_split_workspace_bytes(),), torch.uint8)
        C.coda_set_split_workspace(ws)
    try:
        C.coda_gemm(A, False, B, False, out, M, N, K)
        torch.cuda.synchronize()
    finally:
        C.coda_set_wide_tiles(0)
        C.coda_set_split_workspace(None)
    g.check(sched)
    assert_device_ok()
