"""Host-only check of the split-tile schedule of the SM-pair GEMM, run with
the kernel's own work iterator through the library's test hooks, no GPU
needed.  The remainder tiles after the full waves are each cut into equal
k-ranges dealt range-major and round-robin; the hook checks that every
(tile, k-block) unit is computed exactly once, that every split piece is a
partial (an earlier range, in a slot of its own) or the owner (the last
range), that each cluster meets its partial pieces before its owner pieces,
and that each owner's slots hold its tile's earlier ranges in order without
a gap."""
import pytest


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tma_gb300 import build
    build.build()
    import gemm_epilogue_transformer_tma_gb300 as C
    return C


def test_every_unit_is_computed_once(C):
    checked = split = 0
    for P in (2, 3, 7, 74, 76):
        for tiles in sorted({1, 2, P - 1, P + 1, 2 * P - 1, 3 * P + 5, 6 * P + 56, 128, 512, 1792}):
            for nkb in (96, 97, 128, 200, 255, 448, 896):
                assert C.coda_debug_split_schedule_violations(tiles, nkb, P) == 0, (tiles, nkb, P)
                checked += 1
                split += C.coda_debug_split_ranges(tiles, nkb, P) > 1
    assert checked > 300 and split > 100


def test_which_launches_split(C):
    """The remainder after the full waves is split when its k-ranges finish
    in fewer rounds than one whole round, each range has at least 48
    k-blocks, and the ranges number at most 6."""
    # 7B and 70B dgrad2: 6 full waves, 56 tiles left, 4 ranges take 3 quarter-rounds
    assert C.coda_debug_split_first_tile(512, 448, 76) == 456
    assert C.coda_debug_split_ranges(512, 448, 76) == 4
    assert C.coda_debug_split_ranges(512, 896, 76) == 4
    # below one wave: all tiles are the remainder
    assert C.coda_debug_split_first_tile(128, 256, 76) == 76 and C.coda_debug_split_ranges(128, 256, 76) == 4
    # no split: whole waves, ranges under 48 k-blocks, or no count that beats one round
    assert C.coda_debug_split_first_tile(456, 448, 76) == 456
    assert C.coda_debug_split_ranges(512, 64, 76) == 1        # GEMM1 / GEMM2 shapes, K = 4096
    assert C.coda_debug_split_ranges(1792, 128, 76) == 1      # wgrad2 shape, K = 8192
    assert C.coda_debug_split_ranges(64, 256, 76) == 1        # 64 of 76 pairs: no count of ranges gains


def test_invalid_arguments(C):
    assert C.coda_debug_split_schedule_violations(0, 64, 76) == -1
    assert C.coda_debug_split_schedule_violations(64, 0, 76) == -1
    assert C.coda_debug_split_schedule_violations(64, 64, 0) == -1
    assert C.coda_debug_split_first_tile(0, 64, 76) == -1
    assert C.coda_debug_split_ranges(64, 64, 0) == -1
