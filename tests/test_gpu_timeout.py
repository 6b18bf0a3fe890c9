"""Failure detection without a GPU fault: every wait inside the GEMM kernels
is time-bounded.  The test hook leaves one shared-memory stage unfilled, so
the MMA warp's wait can never complete; the wait must expire after the short
limit, the kernel must record CODA_ERR_TIMEOUT in the device status word,
drain its own in-flight copies and return, and the context must stay usable
(a normal GEMM right after is checked against the oracle)."""
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


@pytest.mark.parametrize("pair", [True, False], ids=["sm_pair", "single_sm"])
def test_expired_wait_is_reported_and_the_context_survives(pair):
    assert_device_ok()
    C.coda_set_sm_pairing(pair)
    C.coda_set_wait_timeout_ns(50_000_000)  # 50 ms
    C.coda_debug_skip_first_stage(True)
    try:
        _gemm(256, 256, 512, 1)
        st, bits = C.coda_sync_status()
    finally:
        C.coda_debug_skip_first_stage(False)
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
