"""Host-only checks of the C ABI: the library loads, exports every entry
point include/coda.h declares with the binding's signature table matching,
and the pure host queries (tile counts, workspace sizes, status strings)
answer without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", n) for n in ("coda.h", "coda_testing.h")]


@pytest.fixture(scope="module")
def lib():
    from gemm_epilogue_transformer_tma_gb300 import build
    build.build()
    import gemm_epilogue_transformer_tma_gb300 as C
    return C.load_library()


def declared():
    src = "".join(open(h).read() for h in HEADERS)
    return set(re.findall(r"^\s*(?:coda_status_t|const char\*|int64_t|size_t|int)\s+(coda_\w+)\s*\(", src, re.M))


def test_header_declares_the_named_entry_points():
    names = declared()
    for n in ("coda_gemm_res_prms", "coda_rstd_combine", "coda_gemm_rowscale_swiglu",
              "coda_gemm_rowscale_swiglu_bwd", "coda_gemm_res_prms_bwd", "coda_lmhead_ce"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import gemm_epilogue_transformer_tma_gb300 as C
    names = declared()
    assert names == set(C.SIGNATURES), (names ^ set(C.SIGNATURES))
    out = subprocess.run(["nm", "-D", "--defined-only", C.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (coda_\w+)", out))
    assert names <= exported, names - exported
    for n in names:
        assert hasattr(lib, n)


def test_host_queries(lib):
    assert lib.coda_prms_num_tiles(4096) == 32   # 128-column partials
    assert lib.coda_prms_num_tiles(328) == 3
    assert lib.coda_dgpart_rows(300) == 12
    assert lib.coda_bwd_workspace_bytes(0, 64, 128) == 0
    M, d, N2 = 8192, 4096, 28672
    assert lib.coda_bwd_workspace_bytes(M, d, N2) >= M * N2 * 2 + M * 4 + 4 * (M // 128) * d * 4
    assert lib.coda_lmhead_ce_workspace_bytes(8192, 2048, 128256, 0) >= 3 * 8192 * 1002 * 4
    assert lib.coda_lmhead_ce_workspace_bytes(8192, 2048, 128256, 1) > lib.coda_lmhead_ce_workspace_bytes(
        8192, 2048, 128256, 0)
    # the executor's arena: W2g alone for an empty batch, 0 for an invalid shape
    assert lib.coda_block_arena_bytes(0, 64, 64, 128, 1) == 128 * 64 * 2
    assert lib.coda_block_arena_bytes(8, 64, 64, 0, 1) == 0
    assert lib.coda_block_arena_bytes(M, 4096, d, N2, 1) > lib.coda_block_arena_bytes(M, 4096, d, N2, 0) > \
        2 * M * (4096 + d + N2 // 2) * 2
    # FP8: codes instead of W2g and the bf16 workspace, so a smaller arena
    assert 0 < lib.coda_block_arena_bytes(M, 4096, d, N2, 3) < lib.coda_block_arena_bytes(M, 4096, d, N2, 1)
    # per-row CE results: label logits then row losses, after the three
    # [M][ceil(V/128)] partial arrays, inside the workspace
    M, d, V = 8192, 2048, 128256
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    for grads in (0, 1):
        assert lib.coda_lmhead_ce_row_offsets(M, d, V, grads, ctypes.byref(a), ctypes.byref(b)) == 0
        part = -(-(M * (V // 128) * 4) // 256) * 256
        assert a.value == 3 * part and b.value == a.value + M * 4
        assert b.value + M * 4 <= lib.coda_lmhead_ce_workspace_bytes(M, d, V, grads)
    assert lib.coda_lmhead_ce_row_offsets(0, d, V, 0, None, None) == 1
    assert lib.coda_status_string(0) == b"ok"
    assert b"time limit" in lib.coda_status_string(6)


def test_null_handle_is_rejected_without_a_gpu(lib):
    # validation runs before any CUDA call
    assert lib.coda_set_wait_timeout_ns(None, 1) == 1
    assert lib.coda_gemm(None, None, 0, None, 0, None, 8, 8, 8, None, None, None) == 1
    assert lib.coda_destroy(None) == 0
    out = ctypes.c_void_p()
    assert lib.coda_block_create(None, 8, 64, 64, 128, 1e-5, 1, *([None] * 7), 0, ctypes.byref(out)) == 1
    assert lib.coda_block_quantize_weights(None) == 1
    assert lib.coda_block_step_host(None, None, None, None, None, None, None, None) == 1
    assert lib.coda_block_sync(None, None) == 1
    assert lib.coda_block_destroy(None) == 0
