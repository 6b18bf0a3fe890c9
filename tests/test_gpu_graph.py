"""The whole step recorded as one CUDA graph (the launch path a training loop
would replay): replays give results bit-identical to eager steps on the same
inputs, also after the inputs are overwritten in place between replays, for
the bf16 step and the FP8 step.  Every kernel is deterministic (fixed
reduction orders), so equality is exact.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, section 尾声: the block as a short fixed sequence of
GEMM-epilogue launches).
"""
import pytest
import torch

from coda_inputs import BlockShape, block_inputs
from tests._parity import assert_device_ok

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers  # noqa: E402

SHAPE = BlockShape("graph", 520, 256, 384, 1056)   # F = 528: ragged against 128-column halves
OUTS = ("H", "rstd", "z", "out", "dH", "dg", "dW2t", "dX", "dW1t")
INS = ("X", "R", "dY")


def snapshot(b):
    return {k: getattr(b, k).clone() for k in OUTS}


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_graph_replay_matches_eager(fp8):
    x = block_inputs(SHAPE, 0, "cuda")
    x2 = block_inputs(SHAPE, 1, "cuda")
    b = BlockBuffers({k: v.clone() for k, v in x.items()})
    if fp8:
        b.fp8_quantize_weights()
    run = b.step_fp8 if fp8 else b.step
    run()
    torch.cuda.synchronize()
    eager1 = snapshot(b)
    for k in INS:
        getattr(b, k).copy_(x2[k])
    run()
    torch.cuda.synchronize()
    eager2 = snapshot(b)
    for k in INS:
        getattr(b, k).copy_(x[k])
    b.capture_step(fp8=fp8)
    for inputs, want in ((x2, eager2), (x, eager1), (x2, eager2)):
        for k in INS:
            getattr(b, k).copy_(inputs[k])
        b.replay()
        torch.cuda.synchronize()
        assert_device_ok()
        for k in OUTS:
            assert torch.equal(getattr(b, k), want[k]), k
