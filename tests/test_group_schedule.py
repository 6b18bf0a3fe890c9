"""Host-only check of the tile schedule of the grouped GEMM launches (two
independent GEMMs, e.g. a layer's data and weight gradients, in one
persistent SM-pair launch).  Every role of the kernel computes its tile
sequence with the same arithmetic; the library's host build of that
function is checked here, without a GPU: every tile of both problems must be
visited by exactly one cluster, for any cluster count, tile counts and
catch-up size, including empty problems and problems smaller than a wave."""
import pytest


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tma_gb300 import build
    build.build()
    import gemm_epilogue_transformer_tma_gb300 as C
    return C


def test_every_tile_is_visited_exactly_once(C):
    checked = 0
    for P in (1, 2, 3, 5, 8, 76):
        for nH in sorted({0, 1, P - 1, P, P + 1, 3 * P + 2, 10 * P + 7}):
            for nL in sorted({0, 1, 5, P, 4 * P + 3, 23 * P + 40}):
                for q in (0, 1, 2, 4, 9):
                    for heavy in (0, 1):
                        assert C.coda_debug_group_schedule_violations(P, heavy, nH, nL, q) == 0, \
                            (P, heavy, nH, nL, q)
                        checked += 1
    assert checked > 1000


@pytest.mark.parametrize("P,heavy,nH,nL,q", [
    (76, 0, 512, 1792, 4),   # dgrad2 + wgrad2 of the 7B block
    (76, 1, 256, 512, 2),    # dgrad1 + wgrad1 of the 7B block (wgrad heavier)
    (76, 0, 256, 512, 2),    # LM-head dH + dW of one vocabulary chunk
    (76, 1, 64, 256, 4),     # fewer heavy tiles than clusters
])
def test_step_shapes(C, P, heavy, nH, nL, q):
    assert C.coda_debug_group_schedule_violations(P, heavy, nH, nL, q) == 0


def test_invalid_arguments_are_rejected(C):
    assert C.coda_debug_group_schedule_violations(0, 0, 1, 1, 1) == -1
    assert C.coda_debug_group_schedule_violations(4, 2, 1, 1, 1) == -1
    assert C.coda_debug_group_schedule_violations(4, 0, -1, 1, 1) == -1
