"""GEMMs whose last, partial wave is split along K across all SM pairs
(coda_set_split_workspace): the remainder tiles after the full waves are
each cut into equal k-ranges, dealt range-major to all pairs, and the pair
that runs a tile's last range adds the earlier ranges' fp32 partials before
its epilogue.

Checked with splitting on, at sizes where the launcher splits (asked of the
library's own rule through its test hook):
  * known-answer integer GEMMs bit-exact, every operand layout, bf16 and
    8-bit operands (any fp32 summation order gives the exact integer);
  * the block forward and backward stages (every epilogue program of the
    path) elementwise against the oracle fed the GPU's own stage inputs, and
    close to the unsplit run;
  * the LM-head cross-entropy statistics and gradient programs (at a hidden
    width long enough to split);
  * two runs bit-identical (the split is a fixed schedule).

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, section 尾声: the epilogue sees the whole tile's
accumulator, here summed from the split pieces before it runs).
"""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import BlockShape, CEShape, block_inputs, ce_inputs
from tests._parity import assert_device_ok, assert_elem, assert_frob, f64
from tests.test_gpu_exact import ints

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402

def splits(M, N, K, kb=64):
    """True when the SM-pair launcher splits an M x N x K launch (256 x 256
    tiles, kb-deep k-blocks) on this GPU's SM pairs."""
    tiles = -(-M // 256) * -(-N // 256)
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    return C.coda_debug_split_ranges(tiles, -(-K // kb), pairs) > 1


def exact(A, Bt, scale=1.0):
    """bf16 of the exact integer product A Bt^T (float64 BLAS: every partial
    sum is an integer below 2^53), times an exact power of two."""
    v = (A.to(torch.float64) @ Bt.to(torch.float64).T) * scale
    assert float(v.abs().max()) < 2 ** 24
    return v.to(torch.float32).to(torch.bfloat16)


@pytest.fixture
def split_on():
    ws = torch.empty(C.coda_split_workspace_bytes(), dtype=torch.uint8, device="cuda")
    C.coda_set_sm_pairing(True)
    C.coda_set_split_workspace(ws)
    yield ws
    torch.cuda.synchronize()
    C.coda_set_split_workspace(None)


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K", [(2048, 4096, 16384), (1800, 3904, 13000)])
def test_split_gemm_bit_exact(a_mn, b_mn, M, N, K, split_on):
    assert splits(M, N, K)
    A = ints((M, K), -3, 3, 21)
    Bt = ints((N, K), -3, 3, 22)
    Ad = (A.T.contiguous() if a_mn else A).to(torch.bfloat16).cuda()
    Bd = (Bt.T.contiguous() if b_mn else Bt).to(torch.bfloat16).cuda()
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm(Ad, a_mn, Bd, b_mn, Cd, M, N, K)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(Cd.cpu(), exact(A, Bt))


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (True, True)])
def test_split_fp8_gemm_bit_exact(a_mn, b_mn, split_on):
    M, N, K = 2048, 4096, 24576        # 8 x 16 tiles, 192 k-blocks of 128 codes
    assert splits(M, N, K, kb=128)
    A = ints((M, K), -4, 4, 23)
    Bt = ints((N, K), -4, 4, 24)
    Aq = O.e5m2_encode((A.T if a_mn else A).numpy().astype(np.float64))
    Bq = O.e4m3_encode((Bt.T if b_mn else Bt).numpy().astype(np.float64))
    sA = torch.tensor([0.5], device="cuda")
    sB = torch.tensor([4.0], device="cuda")
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm_fp8(torch.from_numpy(np.ascontiguousarray(Aq)).cuda(), a_mn, 1, sA,
                    torch.from_numpy(np.ascontiguousarray(Bq)).cuda(), b_mn, 0, sB, Cd, M, N, K)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(Cd.cpu(), exact(A, Bt, 2.0))   # sA * sB = 2


# dgrad2 (M x d x 2F = 2048 x 4096 x 16384, 256 k-blocks) splits; the
# step's shorter-K GEMMs do not
SPLIT_BLOCK = BlockShape("split", 2048, 2048, 4096, 16384)


def test_split_block_stages_against_oracle(split_on):
    """The block at a size whose dgrad2 (the RMSNorm-backward epilogue)
    splits; every stage against the oracle on the GPU's own inputs."""
    s = SPLIT_BLOCK
    assert splits(s.M, s.d, s.N2)
    x = block_inputs(s, 0, "cuda")
    b = BlockBuffers(x)
    b.forward()
    b.backward_stages()
    assert_device_ok()
    X, W1t, R, g, W2t, dY = (f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t", "dY"))
    H = f64(b.H)
    assert_elem(b.H, O.gemm_residual(X, W1t, R), "H")
    assert_elem(b.psum, O.partial_sumsq(H, C.PARTIAL_COLS), "psum", tol=1e-4)
    z_ref = O.rowscale_gemm(H, f64(b.W2gt), f64(b.rstd))
    assert_elem(b.z, z_ref, "z")
    assert_elem(b.out, O.swiglu(z_ref), "out")
    # dgrad2 sums K = 16384 terms: dH and dg are compared with cuBLAS on the
    # same inputs as at full size
    dH_ref, dg_ref = O.stage_dgrad2_rmsbwd(f64(b.dP), W2t, g, H, f64(b.c))
    acc = torch.mm(b.dP, b.W2t, out_dtype=torch.float32)
    dH_cub = (b.g.float() * acc - b.c[:, None] * b.H.float()).to(torch.bfloat16)
    dg_cub = (acc * b.H.float()).sum(0)
    del acc
    assert_elem(b.dH, dH_ref, "dH", cublas=dH_cub)
    assert_elem(b.dg, dg_ref, "dg", cublas=dg_cub)
    # the weight gradients sum M = 2048 rows (rms ~ 26): compared with cuBLAS
    # on the same inputs as at full size
    cub = (torch.mm(b.dP.t(), b.H, out_dtype=torch.float32) * b.g.float()).to(torch.bfloat16)
    assert_elem(b.dW2t, O.stage_wgrad2(H, f64(b.dP), g), "dW2t", cublas=cub)
    assert_elem(b.dX, O.stage_dgrad1(f64(b.dH), W1t), "dX", cublas=torch.matmul(b.dH, b.W1t))
    assert_elem(b.dW1t, O.stage_wgrad1(f64(b.dH), X), "dW1t", cublas=torch.matmul(b.dH.t(), b.X))
    full = O.block_forward(X, W1t, R, g, W2t, s.eps, True)
    assert_frob(b.out, full["out"], "out e2e")
    # the same step unsplit: equal up to fp32 summation order, so the bf16
    # outputs differ at most where a rounding flips, by one bf16 ulp
    # (2^-8 relative) there
    got = {k: getattr(b, k).clone() for k in ("H", "z", "out", "dH", "dg", "dW2t", "dX", "dW1t")}
    C.coda_set_split_workspace(None)
    b.forward()
    b.backward_stages()
    torch.cuda.synchronize()
    for k, v in got.items():
        assert_frob(v, getattr(b, k), f"{k} split vs unsplit", tol=2.0 ** -8)
    C.coda_set_split_workspace(split_on)


def test_split_is_deterministic(split_on):
    x = block_inputs(SPLIT_BLOCK, 1, "cuda")
    b = BlockBuffers(x)
    b.step()
    torch.cuda.synchronize()
    first = {k: getattr(b, k).clone() for k in ("out", "dH", "dg", "dW2t", "dX", "dW1t")}
    for _ in range(2):
        b.step()
        torch.cuda.synchronize()
        for k, v in first.items():
            assert torch.equal(getattr(b, k), v), k
    assert_device_ok()


def test_split_lmhead_ce(split_on):
    """At a hidden width of 12288 (192 k-blocks) the statistics GEMM (314
    tiles) and each vocabulary chunk's gradient recompute (128 tiles) split;
    lse, loss, label logits and argmax against the oracle, dH and dW by
    Frobenius."""
    s = CEShape("split_ce", 512, 12288, 40000)
    assert splits(s.M, s.V, s.d) and splits(s.M, 16384, s.d)
    x = {k: v.cuda() for k, v in ce_inputs(s, 0).items()}
    M, d, V = s.M, s.d, s.V
    ws = torch.empty(C.coda_lmhead_ce_workspace_bytes(M, d, V, True), dtype=torch.uint8, device="cuda")
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(M, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    dH = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(V, d, dtype=torch.bfloat16, device="cuda")
    C.coda_lmhead_ce(x["H"], x["Wt"], x["labels"], loss, lse, am, dH, dW, ws)
    assert_device_ok()
    H, Wt, y = f64(x["H"]), f64(x["Wt"]), x["labels"].cpu().numpy()
    fw = O.ce_forward(H, Wt, y)
    assert_elem(lse, fw["lse"], "lse", tol=1e-4)
    assert abs(loss.item() - fw["loss"]) <= 1e-4 * abs(fw["loss"])
    L = O.logits_rows(H, Wt)
    srt = np.sort(L, axis=1)
    decided = srt[:, -1] - srt[:, -2] > 1e-3
    assert np.array_equal(am.cpu().numpy()[decided], O.argmax_lowest(L)[decided])
    zy, _ = C.coda_lmhead_ce_row_results(ws, M, d, V, True)
    assert_elem(zy, L[np.arange(M), y], "label logit")
    bw = O.ce_backward(H, Wt, y)
    assert_frob(dH, bw["dH"], "dH")
    assert_frob(dW, bw["dWt"], "dW")
