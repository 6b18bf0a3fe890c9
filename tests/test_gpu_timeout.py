"""Failure detection without a GPU fault: every wait inside the GEMM kernels
is time-bounded.  The test hook leaves a shared-memory stage unfilled, or
stops one CTA of an SM pair before its first copy, so the MMA warp's wait
can never complete; the wait must expire after the short limit, the kernel
must record CODA_ERR_TIMEOUT in the device status word, observe every copy
it issued land and return, and the context must stay usable (a normal GEMM
right after is checked against the oracle)."""
import pytest
import torch

import oracle as O
from tests._parity import assert_device_ok, assert_elem, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")

TIMEOUT_BITS = 0x1 | 0x2 | 0x4   # producer / MMA / epilogue wait expired
DRAIN_BIT = 0x8                   # a drain on the way out expired (must not happen)


def _gemm(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C.coda_gemm(A.cuda(), False, B.cuda(), False, Cd, M, N, K)
    return A, B, Cd


@pytest.mark.parametrize("pair,mode", [(True, 1), (True, 2), (False, 1)],
                         ids=["sm_pair_leader_skips", "sm_pair_peer_stops", "single_sm"])
def test_expired_wait_is_reported_and_the_context_survives(pair, mode):
    """mode 1: the first CTA never arms its first stage (the second CTA's
    copies for it land unobserved by any MMA); mode 2: the first pair's second
    CTA issues no copy (the first CTA's stages expect bytes that never come).
    Both leave copies that only the end-of-producer hand-off observes."""
    assert_device_ok()
    C.coda_set_sm_pairing(pair)
    C.coda_set_wait_timeout_ns(50_000_000)  # 50 ms
    C.coda_debug_skip_first_stage(mode)
    try:
        _gemm(256, 256, 512, 1)
        st, bits = C.coda_sync_status()
    finally:
        C.coda_debug_skip_first_stage(0)
        C.coda_set_wait_timeout_ns(0)
        C.coda_set_sm_pairing(True)
    assert st == 6, f"expected CODA_ERR_TIMEOUT, got {C.STATUS_NAMES.get(st)} bits={bits:#x}"
    # the MMA warp waits on the unfilled stage, and the producer waits for the
    # MMA to release it: whichever limit is noticed first raises the abort
    assert bits & TIMEOUT_BITS, f"a bounded wait should have expired (bits={bits:#x})"
    assert not bits & DRAIN_BIT, f"in-flight copies did not drain (bits={bits:#x})"
    # the status word was cleared by the read, and the context still works
    C.coda_set_sm_pairing(pair)
    A, B, Cd = _gemm(264, 520, 200, 2)
    C.coda_set_sm_pairing(True)
    assert_device_ok()
    assert_elem(Cd, O.matmul_nt(f64(A), f64(B)), "C after timeout")


@pytest.mark.parametrize("mode", [1, 2], ids=["leader_stops", "peer_stops"])
def test_wide_tiles_expired_wait(mode):
    """The 256 x 512 pair-tile kernel, whose producers fill two rings (wide
    stages of one or two B halves, then half-tile stages): one CTA of the
    first pair issues no copy (1: the first CTA, so every fill of the second
    lands on a stage only the end-of-producer hand-off arms; 2: the second
    CTA, so the first CTA's stages wait for bytes that never come).  The
    wait must expire, no drain may, and a wide GEMM right after is exact."""
    from tests.test_gpu_exact import ints
    assert_device_ok()
    C.coda_set_sm_pairing(True)
    C.coda_set_wide_tiles(8)
    try:
        assert C.coda_debug_wide_applies(256, 512, 16384) == 1
        C.coda_set_wait_timeout_ns(50_000_000)  # 50 ms
        C.coda_debug_skip_first_stage(mode)
        try:
            _gemm(256, 512, 16384, 3)
            st, bits = C.coda_sync_status()
        finally:
            C.coda_debug_skip_first_stage(0)
            C.coda_set_wait_timeout_ns(0)
        assert st == 6, f"expected CODA_ERR_TIMEOUT, got {C.STATUS_NAMES.get(st)} bits={bits:#x}"
        assert bits & TIMEOUT_BITS, f"a bounded wait should have expired (bits={bits:#x})"
        assert not bits & DRAIN_BIT, f"in-flight copies did not drain (bits={bits:#x})"
        # integer operands: one exact result whatever the summation order
        M, N, K = 1024, 4096, 16384
        assert C.coda_debug_wide_applies(M, N, K) == 1
        A, Bt = ints((M, K), -3, 3, 51), ints((N, K), -3, 3, 52)
        Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        C.coda_gemm(A.to(torch.bfloat16).cuda(), False, Bt.to(torch.bfloat16).cuda(), False, Cd, M, N, K)
        torch.cuda.synchronize()
    finally:
        C.coda_set_wide_tiles(0)
    assert_device_ok()
    ref = (A.to(torch.float64) @ Bt.to(torch.float64).T).to(torch.float32).to(torch.bfloat16)
    assert torch.equal(Cd.cpu(), ref)


@pytest.mark.parametrize("mode", [1, 2], ids=["leader_skips", "peer_stops"])
def test_grouped_launch_expired_wait(mode):
    """The grouped SM-pair launch (dX and dW1 of the first layer in one
    persistent kernel) under both hook modes: the wait must expire, no drain
    may, and the grouped launch right after must equal two separate GEMMs."""
    assert_device_ok()
    M, K1, d = 1280, 512, 256
    g = torch.Generator(device="cuda").manual_seed(7)
    dH = torch.randn(M, d, device="cuda", generator=g).to(torch.bfloat16)
    X = torch.randn(M, K1, device="cuda", generator=g).to(torch.bfloat16)
    W1t = (torch.randn(d, K1, device="cuda", generator=g) / d ** 0.5).to(torch.bfloat16)
    dX = torch.empty(M, K1, device="cuda", dtype=torch.bfloat16)
    dW1t = torch.empty(d, K1, device="cuda", dtype=torch.bfloat16)
    C.coda_set_sm_pairing(True)
    C.coda_set_wait_timeout_ns(50_000_000)  # 50 ms
    C.coda_debug_skip_first_stage(mode)
    try:
        C.coda_gemm_res_prms_bwd(dH, X, W1t, dX, dW1t, None)
        st, bits = C.coda_sync_status()
    finally:
        C.coda_debug_skip_first_stage(0)
        C.coda_set_wait_timeout_ns(0)
    assert st == 6, f"expected CODA_ERR_TIMEOUT, got {C.STATUS_NAMES.get(st)} bits={bits:#x}"
    assert bits & TIMEOUT_BITS, f"a bounded wait should have expired (bits={bits:#x})"
    assert not bits & DRAIN_BIT, f"in-flight copies did not drain (bits={bits:#x})"
    C.coda_gemm_res_prms_bwd(dH, X, W1t, dX, dW1t, None)
    rX, rW = torch.empty_like(dX), torch.empty_like(dW1t)
    C.coda_gemm(dH, False, W1t, True, rX, M, K1, d)
    C.coda_gemm(dH, True, X, True, rW, d, K1, M)
    torch.cuda.synchronize()
    assert_device_ok()
    assert torch.equal(dX, rX)
    assert torch.equal(dW1t, rW)
