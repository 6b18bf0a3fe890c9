"""The boundary's error behaviour as include/coda.h states it: every
argument error is returned synchronously, before anything is launched, with
the documented status; an empty problem returns CODA_OK and launches
nothing; and the context works normally afterwards.

Called through the raw C ABI (ctypes), so that null, misaligned and
ill-sized arguments reach the library unfiltered by the Python binding.
Every case below is rejected by the entry point's argument checks, which run
before any tensor map is encoded or kernel launched.
"""
import ctypes

import pytest
import torch

from tests._parity import assert_device_ok

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")

OK, INVALID, ALIGN, UNSUPPORTED, WS_SMALL = 0, 1, 2, 3, 4


@pytest.fixture
def env():
    lib, h = C.load_library(), C.handle()
    st = torch.cuda.current_stream().cuda_stream
    bf = dict(dtype=torch.bfloat16, device="cuda")
    bufs = {"A": torch.zeros(256 * 256 + 64, **bf), "B": torch.zeros(256 * 256 + 64, **bf),
            "C": torch.zeros(256 * 256 + 64, **bf), "f": torch.zeros(4096, device="cuda")}
    yield lib, h, st, bufs
    torch.cuda.synchronize()
    assert_device_ok()


def p(t, byte_offset=0):
    return ctypes.c_void_p(t.data_ptr() + byte_offset)


def test_gemm_argument_errors(env):
    lib, h, st, b = env
    A, B, Cc = p(b["A"]), p(b["B"]), p(b["C"])

    def gemm(a=A, amn=0, bb=B, bmn=0, c=Cc, M=128, N=128, K=64):
        return lib.coda_gemm(h, a, amn, bb, bmn, c, M, N, K, None, None, st)

    assert gemm(a=None) == INVALID                 # null A with rows to compute
    assert gemm(c=None) == INVALID
    assert gemm(bb=None) == INVALID
    assert gemm(a=p(b["A"], 2)) == ALIGN           # not 16-byte aligned
    assert gemm(c=p(b["C"], 8)) == ALIGN
    assert gemm(N=100) == ALIGN                    # contiguous extent not a multiple of 8
    assert gemm(K=36) == ALIGN
    assert gemm(K=0) == INVALID
    assert gemm(N=-8) == INVALID
    assert gemm(M=-1) == INVALID
    assert gemm(M=2 ** 31) == INVALID              # beyond the extent limit
    assert gemm(amn=1, bmn=0) == UNSUPPORTED       # MN-major A needs MN-major B
    assert gemm(amn=1, bmn=1, M=100) == ALIGN      # MN-major A: M is its contiguous extent
    assert lib.coda_gemm(None, A, 0, B, 0, Cc, 128, 128, 64, None, None, st) == INVALID
    assert gemm(a=None, c=None, M=0) == OK         # an empty problem: nothing to launch


def test_block_entry_point_errors(env):
    lib, h, st, b = env
    A, B, Cc, f = p(b["A"]), p(b["B"]), p(b["C"]), p(b["f"])
    # the fold writes a new tensor: in place is refused
    assert lib.coda_fold_rmsnorm_weight(h, A, B, A, 64, 64, st) == INVALID
    assert lib.coda_fold_rmsnorm_weight(h, A, B, Cc, 64, 12, st) == ALIGN
    # GEMM1: the residual and H must be distinct buffers
    assert lib.coda_gemm_res_prms(h, A, B, Cc, Cc, f, 64, 64, 64, st) == INVALID
    assert lib.coda_gemm_res_prms(h, A, B, Cc, A, p(b["f"], 4), 64, 64, 64, st) == ALIGN
    # the combine: eps must be a number >= 0, T and d positive
    assert lib.coda_rstd_combine(h, f, 64, 1, 64, ctypes.c_float(-1e-5), f, st) == INVALID
    assert lib.coda_rstd_combine(h, f, 64, 1, 64, ctypes.c_float(float("nan")), f, st) == INVALID
    assert lib.coda_rstd_combine(h, f, 64, 0, 64, ctypes.c_float(1e-5), f, st) == INVALID
    # GEMM2: unknown flags, z with the PLAIN program, a SwiGLU half not a multiple of 8
    assert lib.coda_gemm_rowscale_swiglu(h, A, B, f, Cc, None, 64, 64, 128, 7, st) == UNSUPPORTED
    assert lib.coda_gemm_rowscale_swiglu(h, A, B, f, Cc, A, 64, 64, 128, C.CODA_EPI_PLAIN, st) == INVALID
    assert lib.coda_gemm_rowscale_swiglu(h, A, B, f, Cc, None, 64, 64, 24, C.CODA_EPI_SWIGLU, st) == ALIGN
    # the SwiGLU backward: every pointer checked
    assert lib.coda_swiglu_bwd(h, None, B, f, Cc, f, 64, 64, 64, st) == INVALID
    assert lib.coda_swiglu_bwd(h, A, B, f, p(b["C"], 2), f, 64, 64, 64, st) == ALIGN
    # empty batches are valid and launch nothing
    assert lib.coda_swiglu_bwd(h, None, None, None, None, None, 0, 64, 64, st) == OK
    assert lib.coda_gemm_res_prms(h, None, B, None, None, None, 0, 64, 64, st) == OK


def test_lmhead_errors(env):
    lib, h, st, b = env
    M, d, V = 64, 64, 512
    H, W = p(b["A"]), p(b["B"])
    labels = torch.zeros(M, dtype=torch.int32, device="cuda")
    loss, lse = torch.zeros(1, device="cuda"), torch.zeros(M, device="cuda")
    dH = torch.zeros(M, d, dtype=torch.bfloat16, device="cuda")
    dW = torch.zeros(V, d, dtype=torch.bfloat16, device="cuda")
    need = lib.coda_lmhead_ce_workspace_bytes(M, d, V, 1)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")

    def ce(M=M, ws_bytes=need, dh=p(dH), dw=p(dW), lab=p(labels)):
        return lib.coda_lmhead_ce(h, H, W, lab, p(loss), p(lse), None, dh, dw, p(ws), ws_bytes, M, d, V, st)

    assert ce(ws_bytes=need - 1) == WS_SMALL
    assert ce(M=0) == INVALID                     # the mean over no rows is undefined
    assert ce(dw=None) == INVALID                 # gradients come in pairs
    assert ce(lab=None) == INVALID
    assert lib.coda_lmhead_ce_workspace_bytes(0, d, V, 1) == 0


def test_handle_errors():
    lib = C.load_library()
    out = ctypes.c_void_p()
    assert lib.coda_create(ctypes.byref(out), -1) == INVALID
    assert lib.coda_create(ctypes.byref(out), 4096) == INVALID
    assert lib.coda_set_wait_timeout_ns(None, 1000) == INVALID
    assert lib.coda_set_sm_pairing(None, 1) == INVALID


def test_context_works_after_rejected_calls(env):
    lib, h, st, b = env
    M = N = K = 64
    A = torch.randint(-3, 4, (M, K), device="cuda").to(torch.bfloat16)
    B = torch.randint(-3, 4, (N, K), device="cuda").to(torch.bfloat16)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    assert lib.coda_gemm(h, p(A), 0, p(B), 0, p(out), M, N, K, None, None, st) == OK
    torch.cuda.synchronize()
    assert torch.equal(out, (A.double() @ B.double().T).to(torch.bfloat16))
