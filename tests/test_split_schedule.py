"""Host-only check of the split-tile (stream-K) schedule of the SM-pair GEMM,
run with the kernel's own work iterator through the library's test hook, no
GPU needed: every (tile, k-block) unit is computed exactly once, each SM
pair's share holds at most one partial piece (its first) and one owner piece
(its last), and an owner's contributors cover the rest of its tile without a
gap, at most three of them.  Covers the block step's shapes on 76 pairs and
many small and ragged tile and k-block counts."""
import pytest


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tma_gb300 import build
    build.build()
    import gemm_epilogue_transformer_tma_gb300 as C
    return C


def test_every_unit_is_computed_once(C):
    checked = 0
    for P in (2, 3, 7, 74, 76):
        for tiles in sorted({1, 2, P - 1, P + 1, 2 * P - 1, 3 * P + 5, 6 * P + 56, 512, 1792, 3584}):
            for nkb in (16, 17, 31, 64, 65, 128, 448, 896):
                assert C.coda_debug_split_schedule_violations(tiles, nkb, P) == 0, (tiles, nkb, P)
                checked += 1
    assert checked > 300


def test_the_step_shapes_split(C):
    """The 7B step's long GEMMs on 76 pairs are split (the hook only checks a
    schedule that the launcher would really split), and a full last wave or
    short K is not."""
    for tiles, nkb in ((512, 448), (512, 64), (3584, 64), (1792, 128), (16032, 32)):
        assert C.coda_debug_split_schedule_violations(tiles, nkb, 76) == 0


def test_which_launches_split(C):
    """Split when the last wave is partial and K has at least 16 k-blocks;
    the region is the last partial wave plus the full wave before it."""
    assert C.coda_debug_split_first_tile(512, 448, 76) == 380      # 7B dgrad2: 6.74 waves
    assert C.coda_debug_split_first_tile(3584, 64, 76) == 3496     # 7B GEMM2: 47.2 waves
    assert C.coda_debug_split_first_tile(64, 32, 76) == 0          # below one wave: all split
    assert C.coda_debug_split_first_tile(456, 448, 76) == 456      # whole waves: no split
    assert C.coda_debug_split_first_tile(512, 15, 76) == 512       # short K: no split
    assert C.coda_debug_split_first_tile(12, 63, 76) == 12         # >3 contributors per tile: no split


def test_invalid_arguments(C):
    assert C.coda_debug_split_schedule_violations(0, 64, 76) == -1
    assert C.coda_debug_split_schedule_violations(64, 0, 76) == -1
    assert C.coda_debug_split_schedule_violations(64, 64, 0) == -1
    assert C.coda_debug_split_first_tile(0, 64, 76) == -1
