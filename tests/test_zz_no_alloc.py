"""The allocation-free entry point, coda_gemm_dgrad_rmsbwd_noalloc.

It is for callers that cannot allocate device memory at all (a host
framework that hands over only input and output tensors while its own pool
owns the rest of the device, or a latency-critical caller that must not pay
for an allocation): its dg partial sums live in a fixed array inside the
library.  Here its dH and dg are checked against the allocating pair
coda_gemm_dgrad_rmsbwd + coda_dg_combine on two calls in a row with
different inputs (so anything the first call left in the shared array would
show), and an over-size problem must be refused before any launch.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import pytest
import torch

from tests._parity import ELEM_TOL, assert_device_ok, assert_elem

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")


def _inputs(M, N2, d, seed):
    g = torch.Generator().manual_seed(seed)
    bf = torch.bfloat16
    x = {
        "dP": (torch.randn(M, N2, generator=g) * 0.5).to(bf),
        "W2t": (torch.randn(N2, d, generator=g) * 0.02).to(bf),
        "H": torch.randn(M, d, generator=g).to(bf),
        "g": (torch.rand(d, generator=g) + 0.5).to(bf),
        "c": torch.randn(M, generator=g) * 1e-3,
    }
    return {k: v.cuda() for k, v in x.items()}


def _allocating(x, M, d):
    dH = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    dg = torch.empty(d, dtype=torch.float32, device="cuda")
    dgpart = torch.empty(C.coda_dgpart_rows(M), d, dtype=torch.float32, device="cuda")
    C.coda_gemm_dgrad_rmsbwd(x["dP"], x["W2t"], x["H"], x["g"], x["c"], dH, dgpart)
    C.coda_dg_combine(dgpart, dg)
    return dH, dg


def _no_alloc(x, M, d):
    dH = torch.full((M, d), 7.0, dtype=torch.bfloat16, device="cuda")
    dg = torch.full((d,), 7.0, dtype=torch.float32, device="cuda")
    C.coda_gemm_dgrad_rmsbwd_noalloc(x["dP"], x["W2t"], x["H"], x["g"], x["c"], dH, dg)
    return dH, dg


@pytest.mark.parametrize("M,N2,d", [(300, 528, 328), (1024, 2048, 512)])
def test_noalloc_matches_allocating_entry_point_twice(M, N2, d):
    for call, seed in enumerate((11, 12)):
        x = _inputs(M, N2, d, seed)
        ref_dH, ref_dg = _allocating(x, M, d)
        got_dH, got_dg = _no_alloc(x, M, d)
        assert_device_ok()
        assert_elem(got_dH, ref_dH, f"dH (call {call})", tol=ELEM_TOL)
        assert_elem(got_dg, ref_dg, f"dg (call {call})", tol=ELEM_TOL)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # coda_dgpart_rows(M) * d * 4 bytes > 8 MiB: 4*ceil(16512/128) rows * 4096
    lib = C.load_library()
    M, N2, d = 16512, 64, 4096
    assert C.coda_dgpart_rows(M) * d * 4 > (8 << 20)
    dummy = torch.empty(16, dtype=torch.float32, device="cuda").data_ptr()
    st = lib.coda_gemm_dgrad_rmsbwd_noalloc(C.handle(), dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                            M, N2, d, torch.cuda.current_stream().cuda_stream)
    assert st == 4  # CODA_ERR_WORKSPACE_TOO_SMALL, nothing launched
    assert_device_ok()
