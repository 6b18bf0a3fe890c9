"""Host-only check of the wide-tile (256 x 512) schedule of the SM-pair GEMM,
run with the kernel's own iterators through the library's test hook, no GPU
needed: every 256 x 256 output tile is computed by exactly one unit, wide
units come before half-tile units on every cluster, and each accumulator
half sees every k-block exactly once, from the block that starts its sum to
the block where the kernel commits it."""
import pytest


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tma_gb300 import build
    build.build()
    import gemm_epilogue_transformer_tma_gb300 as C
    return C


def test_every_tile_and_kblock_once(C):
    checked = 0
    for P in (1, 2, 3, 7, 38, 74, 76):
        for M in (256, 1800, 2048, 4096, 8192, 28672):
            for N in (512, 1000, 3904, 4096, 8192):
                for K in (64, 100, 1024, 4096, 8192, 28672):
                    for lead in (0, 1, 8, 16, 64):
                        assert C.coda_debug_wide_schedule_violations(M, N, K, P, lead) == 0, (M, N, K, P, lead)
                        checked += 1
    assert checked > 5000


def test_odd_column_tiles_are_refused(C):
    # 3 column tiles of 256: no wide tiling (the launcher keeps 256-column tiles)
    assert C.coda_debug_wide_schedule_violations(4096, 768, 4096, 76, 16) == -1
    assert C.coda_debug_wide_schedule_violations(4096, 4096, 4096, 0, 16) == -1

