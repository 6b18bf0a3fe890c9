"""The allocation-free entry point, coda_gemm_dgrad_rmsbwd_noalloc.

It is for callers that cannot allocate device memory at all (a host
framework that hands over only input and output tensors while its own pool
owns the rest of the device, or a latency-critical caller that must not pay
for an allocation): its dg partial sums live in a fixed 8 MiB array inside
the library.  It runs the same kernels in the same order as the allocating
pair coda_gemm_dgrad_rmsbwd + coda_dg_combine, so its dH and dg must be
bit-identical to theirs; that is checked on two calls in a row with
different inputs (anything the first call left in the shared array would
show), at problem sizes that fill the array exactly, and for an empty batch.
A problem one row block beyond the array must be refused before any launch.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import pytest
import torch

from tests._parity import assert_device_ok

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")

SCRATCH_BYTES = 8 << 20


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


@pytest.mark.parametrize("M,N2,d", [
    (300, 528, 328),     # ragged in every dimension
    (1024, 2048, 512),
    (8192, 64, 8192),    # coda_dgpart_rows(M) * d * 4 == 8 MiB exactly
    (16384, 64, 4096),   # the same edge at d = 4096
])
def test_noalloc_matches_allocating_entry_point_twice(M, N2, d):
    assert C.coda_dgpart_rows(M) * d * 4 <= SCRATCH_BYTES
    for call, seed in enumerate((11, 12)):
        x = _inputs(M, N2, d, seed + M)
        ref_dH, ref_dg = _allocating(x, M, d)
        got_dH, got_dg = _no_alloc(x, M, d)
        assert_device_ok()
        assert torch.equal(got_dH, ref_dH), f"dH differs on call {call}"
        assert torch.equal(got_dg, ref_dg), f"dg differs on call {call}"
        del x, ref_dH, ref_dg, got_dH, got_dg


def test_noalloc_empty_batch_writes_zero_dg():
    d, N2 = 328, 528
    x = _inputs(0, N2, d, 5)
    got_dH, got_dg = _no_alloc(x, 0, d)
    assert_device_ok()
    assert got_dH.numel() == 0
    assert torch.equal(got_dg, torch.zeros(d, device="cuda"))


def test_noalloc_rejects_problems_beyond_its_scratch():
    # one 128-row block past the edge: coda_dgpart_rows(16512) * 4096 * 4 > 8 MiB
    lib = C.load_library()
    M, N2, d = 16512, 64, 4096
    assert C.coda_dgpart_rows(M) * d * 4 > SCRATCH_BYTES
    assert C.coda_dgpart_rows(M - 128) * d * 4 == SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.float32, device="cuda").data_ptr()
    st = lib.coda_gemm_dgrad_rmsbwd_noalloc(C.handle(), dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                            M, N2, d, torch.cuda.current_stream().cuda_stream)
    assert st == 4  # CODA_ERR_WORKSPACE_TOO_SMALL, nothing launched
    assert_device_ok()
