"""Seeded random shapes through the whole block and the LM-head cross-entropy,
against the fp64 oracle fed the GPU's own stage inputs.

The hand-picked shapes of the other parity tests sit on chosen tile edges;
these draw M, K1, d, F and V from a fixed seed (extents multiples of 8, the
boundary's rule; M any positive size), so that tails of every width
against the 128-row / 256-column tiles, the 64-deep k-blocks, the 128-column
partial sums and the 16384-column vocabulary chunks come up without being
chosen.  Every stage is graded as in the hand-picked tests (and the block's
outputs are bit-identical over two runs), the block also on
8-bit operands (extents multiples of 16 there), and the further epilogue
programs (the SwiGLU backward in the down projection's data gradient, RoPE
in the QKV projection) on shapes of their own; each shape runs on SM pairs
or on single SMs, alternately.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, sections 尾声 and 五种积木).
"""
import numpy as np
import pytest
import torch

import oracle as O
from coda_inputs import BlockShape, CEShape, block_inputs, ce_inputs, down_proj_inputs
from tests._ce import check_argmax, check_label_rows, with_edge_labels
from tests._parity import assert_device_ok, assert_elem, assert_frob, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402
from tests.test_gpu_ce import run_ce  # noqa: E402
from tests.test_gpu_fp8_bwd import check_fp8_backward_stages, check_fp8_forward_stages, run_fp8  # noqa: E402
from tests.test_gpu_parity import check_backward_stages, check_forward  # noqa: E402


def block_shapes(n=32, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.integers(1, 1100))
        K1 = 8 * int(rng.integers(1, 80))
        d = 8 * int(rng.integers(1, 96))
        F = 8 * int(rng.integers(1, 72))
        out.append(BlockShape(f"fuzz{i}", M, K1, d, 2 * F))
    return out


def fp8_block_shapes(n=8, seed=2026):
    """8-bit operands: extents multiples of 16 (TMA rows of 16 bytes)."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.integers(1, 900))
        K1 = 16 * int(rng.integers(1, 40))
        d = 16 * int(rng.integers(1, 48))
        F = 16 * int(rng.integers(1, 36))
        out.append(BlockShape(f"fuzz_fp8_{i}", M, K1, d, 2 * F))
    return out


def ce_shapes(n=12, seed=2025):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.integers(1, 400))
        d = 8 * int(rng.integers(1, 48))
        V = 8 * int(rng.integers(1, 5000))
        out.append(CEShape(f"fuzz{i}", M, d, V))
    return out


BLOCKS = block_shapes()
OUTPUTS = ("H", "psum", "rstd", "z", "out", "dP", "c", "dgpart", "dH", "dg", "dW2t", "dX", "dW1t")
FP8_BLOCKS = fp8_block_shapes()
CES = ce_shapes()


@pytest.mark.parametrize("i", range(len(BLOCKS)), ids=[f"M{s.M}_K{s.K1}_d{s.d}_N{s.N2}" for s in BLOCKS])
def test_block_random_shape(i):
    s = BLOCKS[i]
    C.coda_set_sm_pairing(i % 2 == 0)
    try:
        x = {k: v.cuda() for k, v in block_inputs(s, i, "cpu").items()}
        b = BlockBuffers(x)
        b.forward()
        b.backward_stages()
        assert_device_ok()
        first = {k: getattr(b, k).clone() for k in OUTPUTS}
        # a second run: every reduction is a fixed-order combine, so the
        # results must be bit-identical
        b.forward()
        b.backward_stages()
        assert_device_ok()
    finally:
        C.coda_set_sm_pairing(True)
    for k in OUTPUTS:
        assert torch.equal(getattr(b, k), first[k]), f"{k} differs between two runs"
    check_forward(s, b, x)
    check_backward_stages(s, b, x)


@pytest.mark.parametrize("i", range(len(FP8_BLOCKS)),
                         ids=[f"M{s.M}_K{s.K1}_d{s.d}_N{s.N2}" for s in FP8_BLOCKS])
def test_fp8_block_random_shape(i):
    """The block on e4m3 activations and weights and e5m2 gradients."""
    s = FP8_BLOCKS[i]
    C.coda_set_sm_pairing(i % 2 == 0)
    try:
        x, b = run_fp8(s, seed=100 + i)
    finally:
        C.coda_set_sm_pairing(True)
    check_fp8_forward_stages(s, x, b)
    check_fp8_backward_stages(s, x, b)


@pytest.mark.parametrize("i", range(len(CES)), ids=[f"M{s.M}_d{s.d}_V{s.V}" for s in CES])
def test_ce_random_shape(i):
    s = CES[i]
    C.coda_set_sm_pairing(i % 2 == 0)
    try:
        x = {k: v.cuda() for k, v in ce_inputs(s, i).items()}
        x["labels"] = with_edge_labels(x["labels"], s.V)
        o = run_ce(x["H"], x["Wt"], x["labels"])
        assert_device_ok()
    finally:
        C.coda_set_sm_pairing(True)
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


# the next epilogue programs on the same kind of random shapes: the SwiGLU
# backward inside the down projection's data-gradient GEMM with dgrad2 on its
# c partials, and RoPE in the QKV projection's epilogue
NEXT_BLOCKS = block_shapes(n=8, seed=2027)


@pytest.mark.parametrize("i", range(len(NEXT_BLOCKS)),
                         ids=[f"M{s.M}_K{s.K1}_d{s.d}_N{s.N2}" for s in NEXT_BLOCKS])
def test_down_proj_swiglu_bwd_random_shape(i):
    s = NEXT_BLOCKS[i]
    C.coda_set_sm_pairing(i % 2 == 0)
    try:
        x = {k: v.cuda() for k, v in block_inputs(s, i, "cpu", with_dy=False).items()}
        dp = {k: v.cuda() for k, v in down_proj_inputs(s, i, "cpu").items()}
        b = BlockBuffers(dict(x, dY=torch.empty(s.M, s.F, dtype=torch.bfloat16, device="cuda")))
        b.forward()
        cpart = torch.empty(s.M, C.coda_prms_num_tiles(s.F), device="cuda")
        C.coda_gemm_dgrad_swiglu_bwd(dp["dYb"], dp["W3t"], b.z, b.rstd, b.dP, cpart)
        C.coda_gemm_dgrad_rmsbwd_cpart(b.dP, b.W2t, b.H, b.g, b.rstd, cpart, b.dH, b.dgpart)
        C.coda_dg_combine(b.dgpart, b.dg)
        assert_device_ok()
    finally:
        C.coda_set_sm_pairing(True)
    dY = O.down_proj_dgrad(f64(dp["dYb"]), f64(dp["W3t"]))
    z, rstd = f64(b.z), f64(b.rstd)
    dP_ref, c_ref = O.stage_swiglu_bwd(dY, z, rstd, s.d)
    assert_elem(b.dP, dP_ref, "dP")
    assert_elem(cpart, O.swiglu_c_partials(dY, z, C.PARTIAL_COLS), "cpart")
    c = f64(cpart).sum(axis=1) * rstd ** 2 / s.d
    dH_ref, dg_ref = O.stage_dgrad2_rmsbwd(f64(b.dP), f64(x["W2t"]), f64(x["g"]), f64(b.H), c)
    assert_elem(b.dH, dH_ref, "dH")
    assert_elem(b.dg, dg_ref, "dg")


def rope_shapes(n=8, seed=2028):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.integers(1, 1100))
        d = 8 * int(rng.integers(1, 80))
        hq = int(rng.integers(1, 6))
        hkv = int(rng.integers(0, hq + 1))
        S = int(rng.integers(1, 700))
        out.append((M, d, hq, hkv, S))
    return out


ROPES = rope_shapes()


@pytest.mark.parametrize("i", range(len(ROPES)), ids=[f"M{m}_d{d}_q{q}_kv{k}_S{s}" for m, d, q, k, s in ROPES])
def test_qkv_rope_random_shape(i):
    M, d, hq, hkv, S = ROPES[i]
    g = torch.Generator().manual_seed(500 + i)
    X = torch.randn(M, d, generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn((hq + 2 * hkv) * 128, d, generator=g) * 0.02).to(torch.bfloat16).cuda()
    cos_t = torch.empty(S, 64, device="cuda")
    sin_t = torch.empty(S, 64, device="cuda")
    qkv = torch.empty(M, (hq + 2 * hkv) * 128, dtype=torch.bfloat16, device="cuda")
    C.coda_set_sm_pairing(i % 2 == 0)
    try:
        C.coda_rope_table(cos_t, sin_t, 10000.0)
        C.coda_gemm_qkv_rope(X, W, cos_t, sin_t, qkv, hq, hkv)
        assert_device_ok()
    finally:
        C.coda_set_sm_pairing(True)
    ref = O.qkv_rope(f64(X), f64(W), hq, hkv, 128, S)
    assert_elem(qkv, ref, "qkv")


# the opt-in schedules on random shapes, with integer operands (one exact
# result whatever the summation order): 256 x 512 pair tiles (K of at least
# 16384 and an even number of 256-column tiles) and split last waves
def exact_product(A, Bt):
    v = A.to(torch.float64) @ Bt.to(torch.float64).T
    assert float(v.abs().max()) < 2 ** 24
    return v.to(torch.float32).to(torch.bfloat16)


def wide_shapes(n=5, seed=2029):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.integers(1, 2600))
        if i % 3 == 2:
            M = 8 * max(1, M // 8)  # A read MN-major: its rows of M elements obey the 8-element rule
        N = 512 * int(rng.integers(1, 9)) - 8 * int(rng.integers(0, 32))
        K = 16384 + 8 * int(rng.integers(0, 512))
        out.append((M, N, K))
    return out


def split_shapes(n=5, seed=2030, pairs=76):
    """Random shapes that the launcher splits on a GPU of `pairs` SM pairs
    (asked of the library's own rule, which runs on the host)."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        M = int(rng.integers(300, 2600))
        if len(out) % 3 == 2:
            M = 8 * (M // 8)  # A read MN-major (see wide_shapes)
        N = 8 * int(rng.integers(40, 560))
        K = 8 * int(rng.integers(400, 2000))
        tiles = -(-M // 256) * -(-N // 256)
        if C.coda_debug_split_ranges(tiles, -(-K // 64), pairs) > 1:
            out.append((M, N, K))
    return out


WIDES = wide_shapes()
try:
    SPLITS = split_shapes()
except ImportError:  # the library is not built: nothing to collect here (GPU tests only)
    SPLITS = []


def _int_gemm(M, N, K, a_mn, b_mn, seed):
    from tests.test_gpu_exact import ints
    A, Bt = ints((M, K), -3, 3, seed), ints((N, K), -3, 3, seed + 1)
    Ad = (A.T.contiguous() if a_mn else A).to(torch.bfloat16).cuda()
    Bd = (Bt.T.contiguous() if b_mn else Bt).to(torch.bfloat16).cuda()
    Cd = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    C.coda_gemm(Ad, a_mn, Bd, b_mn, Cd, M, N, K)
    torch.cuda.synchronize()
    assert_device_ok()
    return Cd.cpu(), exact_product(A, Bt)


@pytest.mark.parametrize("i", range(len(WIDES)), ids=[f"M{m}_N{n}_K{k}" for m, n, k in WIDES])
def test_wide_tiles_random_shape(i):
    M, N, K = WIDES[i]
    C.coda_set_sm_pairing(True)
    C.coda_set_wide_tiles(8)
    try:
        assert C.coda_debug_wide_applies(M, N, K) == 1
        got, ref = _int_gemm(M, N, K, i % 3 == 2, i % 3 != 0, 700 + 2 * i)
    finally:
        C.coda_set_wide_tiles(0)
    assert torch.equal(got, ref)


@pytest.mark.parametrize("i", range(len(SPLITS)), ids=[f"M{m}_N{n}_K{k}" for m, n, k in SPLITS])
def test_split_tiles_random_shape(i):
    M, N, K = SPLITS[i]
    ws = torch.empty(C.coda_split_workspace_bytes(), dtype=torch.uint8, device="cuda")
    C.coda_set_sm_pairing(True)
    C.coda_set_split_workspace(ws)
    try:
        tiles = -(-M // 256) * -(-N // 256)
        pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
        assert C.coda_debug_split_ranges(tiles, -(-K // 64), pairs) > 1
        got, ref = _int_gemm(M, N, K, i % 3 == 2, i % 3 != 0, 800 + 2 * i)
    finally:
        C.coda_set_split_workspace(None)
    assert torch.equal(got, ref)
