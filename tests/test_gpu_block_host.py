"""The block step executor (coda_block_*): the whole fused step issued from
native code on page-locked host inputs, with the copies of one step
overlapping the kernels of its neighbours.

  * over several steps with different inputs, every result read back (out,
    dX, dR) is bit-identical to the separate calls (BlockBuffers.step) on the
    same inputs, and the weight gradients left on the device are those of
    the last step: slot reuse and the overlap never mix steps up;
  * a step's results are complete once coda_block_wait_step for it returns;
  * end to end against the oracle on one small case;
  * forward only, the empty batch, and argument errors (pageable host
    memory, a short arena, a gradient buffer without backward) refused
    before anything is enqueued.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
(Synced write-up, section 尾声: the block as GEMM1 + residual + partial RMS,
a light combine, GEMM2 + row scale + SwiGLU, and a block-local backward).
"""
import ctypes

import pytest
import torch

import oracle as O
from coda_inputs import BlockShape, block_inputs
from tests._parity import assert_device_ok, assert_frob, f64

pytestmark = pytest.mark.gpu

C = pytest.importorskip("gemm_epilogue_transformer_tma_gb300")
from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers, HostBlockStepper  # noqa: E402

SHAPES = {
    "ragged": BlockShape("ragged", 300, 200, 328, 528),
    "whole": BlockShape("whole", 384, 256, 512, 1024),
}
WEIGHTS = ("W1t", "g", "W2t")


def pinned(t):
    return t.cpu().contiguous().pin_memory()


def reference(s, w, x):
    b = BlockBuffers(dict(w, **{k: x[k] for k in x if k not in WEIGHTS}), backward=s.backward)
    b.step()
    torch.cuda.synchronize()
    return b


@pytest.mark.parametrize("name", ["ragged", "whole"])
def test_steps_match_separate_calls(name):
    s = SHAPES[name]
    w = {k: v for k, v in block_inputs(s, 0, "cuda").items() if k in WEIGHTS}
    steps = [block_inputs(s, seed, "cuda") for seed in (1, 2, 3, 4, 5)]
    st = HostBlockStepper(w["W1t"], w["g"], w["W2t"], s.M, s.eps)
    host_in = [{k: pinned(x[k]) for k in ("X", "R", "dY")} for x in steps]
    host_out = [st.host_buffers(out=True, dX=True, dR=True) for _ in steps]
    ids = [st.submit(hi["X"], hi["R"], hi["dY"], **ho) for hi, ho in zip(host_in, host_out)]
    assert ids == list(range(len(steps)))
    # step 1's results are complete once its wait returns, while later steps may still run
    st.wait(1)
    ref1 = reference(s, w, steps[1])
    assert torch.equal(host_out[1]["dX"], ref1.dX.cpu())
    st.sync()
    assert_device_ok()
    for i, x in enumerate(steps):
        ref = ref1 if i == 1 else reference(s, w, x)
        for k_host, k_ref in (("out", "out"), ("dX", "dX"), ("dR", "dH")):
            assert torch.equal(host_out[i][k_host], getattr(ref, k_ref).cpu()), (i, k_host)
    for k in ("dW1t", "dW2t", "dg"):
        assert torch.equal(getattr(st, k), getattr(ref, k)), k
    st.close()


def test_end_to_end_against_the_oracle():
    s = SHAPES["ragged"]
    x = block_inputs(s, 0, "cuda")
    st = HostBlockStepper(x["W1t"], x["g"], x["W2t"], s.M, s.eps)
    hi = {k: pinned(x[k]) for k in ("X", "R", "dY")}
    ho = st.host_buffers(out=True, dX=True, dR=True)
    st.submit(hi["X"], hi["R"], hi["dY"], **ho)
    st.sync()
    ref = O.block_backward(*(f64(x[k]) for k in ("X", "W1t", "R", "g", "W2t", "dY")), s.eps, True)
    for got, k_ref in ((ho["out"], "out"), (ho["dX"], "dX"), (ho["dR"], "dR"), (st.dW1t, "dW1t"),
                       (st.dW2t, "dW2t"), (st.dg, "dg")):
        assert_frob(got, ref[k_ref], f"executor {k_ref}")
    st.close()


def test_forward_only():
    s = BlockShape("fwd", 300, 200, 328, 528, backward=False)
    w = {k: v for k, v in block_inputs(s, 0, "cuda").items() if k in WEIGHTS}
    steps = [block_inputs(s, seed, "cuda") for seed in (1, 2, 3)]
    st = HostBlockStepper(w["W1t"], w["g"], w["W2t"], s.M, s.eps, backward=False)
    outs = [st.host_buffers(out=True) for _ in steps]
    for x, o in zip(steps, outs):
        st.submit(pinned(x["X"]), pinned(x["R"]), **o)
    st.sync()
    for x, o in zip(steps, outs):
        assert torch.equal(o["out"], reference(s, w, x).out.cpu())
    st.close()


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_empty_batch_zeroes_the_weight_gradients(fp8):
    s = BlockShape("empty", 0, 64, 64, 128)
    x = block_inputs(s, 0, "cuda")
    st = HostBlockStepper(x["W1t"], x["g"], x["W2t"], 0, s.eps, fp8=fp8)
    for t in (st.dW1t, st.dW2t, st.dg):
        t.fill_(1.0)
    st.submit(None, None, None)
    st.sync()
    for t in (st.dW1t, st.dW2t, st.dg):
        assert not t.any()
    st.close()


def test_argument_errors():
    s = SHAPES["ragged"]
    x = block_inputs(s, 0, "cuda")
    lib = C.load_library()
    st = HostBlockStepper(x["W1t"], x["g"], x["W2t"], s.M, s.eps)
    hi = {k: pinned(x[k]) for k in ("X", "R", "dY")}
    pageable = x["X"].cpu().contiguous()
    sid = ctypes.c_int64(-1)
    # pageable host memory is refused by the library itself (the binding refuses it first)
    assert lib.coda_block_step_host(st.blk, pageable.data_ptr(), hi["R"].data_ptr(), hi["dY"].data_ptr(),
                                    None, None, None, ctypes.byref(sid)) == 1
    with pytest.raises(ValueError):
        st.submit(pageable, hi["R"], hi["dY"])
    # a backward step without its upstream gradient
    assert lib.coda_block_step_host(st.blk, hi["X"].data_ptr(), hi["R"].data_ptr(), None, None, None, None,
                                    None) == 1
    # nothing was enqueued: the next step is still step 0
    assert st.submit(hi["X"], hi["R"], hi["dY"]) == 0
    st.sync()
    # waiting on a step that was never submitted
    assert lib.coda_block_wait_step(st.blk, 5) == 1
    st.close()

    # a forward-only executor takes no gradient buffers
    fw = HostBlockStepper(x["W1t"], x["g"], x["W2t"], s.M, s.eps, backward=False)
    assert lib.coda_block_step_host(fw.blk, hi["X"].data_ptr(), hi["R"].data_ptr(), hi["dY"].data_ptr(), None,
                                    None, None, None) == 1
    fw.close()

    # an arena one byte short, and a non-SwiGLU-sized N2
    need = C.coda_block_arena_bytes(s.M, s.K1, s.d, s.N2, C.CODA_BLOCK_BACKWARD)
    arena = torch.empty(need, dtype=torch.uint8, device="cuda")
    dW1t = torch.empty(s.d, s.K1, dtype=torch.bfloat16, device="cuda")
    dW2t = torch.empty(s.N2, s.d, dtype=torch.bfloat16, device="cuda")
    dg = torch.empty(s.d, dtype=torch.float32, device="cuda")
    out = ctypes.c_void_p()
    h = C.handle()
    args = [x["W1t"].data_ptr(), x["g"].data_ptr(), x["W2t"].data_ptr(), dW1t.data_ptr(), dW2t.data_ptr(),
            dg.data_ptr(), arena.data_ptr()]
    assert lib.coda_block_create(h, s.M, s.K1, s.d, s.N2, s.eps, 1, *args, need - 1, ctypes.byref(out)) == 4
    assert out.value is None
    assert lib.coda_block_create(h, s.M, s.K1, s.d, 520, s.eps, 1, *args, need, ctypes.byref(out)) == 2
    assert lib.coda_block_create(h, s.M, s.K1, s.d, s.N2, 0.0, 1, *args, need, ctypes.byref(out)) == 1
    assert lib.coda_block_create(h, s.M, s.K1, s.d, s.N2, s.eps, 8, *args, need, ctypes.byref(out)) == 1
    assert lib.coda_block_create(h, s.M, s.K1, s.d, s.N2, s.eps, 1 | 4, *args, need, ctypes.byref(out)) == 1
    assert lib.coda_block_create(h, s.M, s.K1, s.d, s.N2, s.eps, 1, *args, need, ctypes.byref(out)) == 0
    assert lib.coda_block_destroy(out) == 0


def test_work_on_the_executor_stream_is_ordered_between_steps():
    # a weight update enqueued on the executor's compute stream after step 0
    # is seen by step 1 and not by step 0
    s = SHAPES["ragged"]
    w = {k: v.clone() for k, v in block_inputs(s, 0, "cuda").items() if k in WEIGHTS}
    x = block_inputs(s, 1, "cuda")
    st = HostBlockStepper(w["W1t"], w["g"], w["W2t"], s.M, s.eps)
    hi = {k: pinned(x[k]) for k in ("X", "R", "dY")}
    outs = [st.host_buffers(out=True, dX=True) for _ in range(2)]
    st.submit(hi["X"], hi["R"], hi["dY"], **outs[0])
    with torch.cuda.stream(st.stream()):
        w["W1t"].mul_(2.0)
        w["g"].mul_(0.5)
    st.submit(hi["X"], hi["R"], hi["dY"], **outs[1])
    st.sync()
    w0 = {k: v for k, v in block_inputs(s, 0, "cuda").items() if k in WEIGHTS}
    for o, weights in ((outs[0], w0), (outs[1], w)):
        ref = reference(s, weights, x)
        assert torch.equal(o["out"], ref.out.cpu())
        assert torch.equal(o["dX"], ref.dX.cpu())
    st.close()


FP8_SHAPE = BlockShape("ragged_fp8", 300, 208, 336, 544)


@pytest.mark.parametrize("delayed", [False, True], ids=["exact", "delayed"])
def test_fp8_steps_match_separate_calls(delayed):
    """FP8 executor steps on host buffers bit-identical to BlockBuffers'
    FP8 steps on the same inputs in the same order (with delayed scaling
    the dP state carries from step to step on both sides)."""
    s = FP8_SHAPE
    w = {k: v for k, v in block_inputs(s, 0, "cuda").items() if k in WEIGHTS}
    steps = [block_inputs(s, seed, "cuda") for seed in (1, 2, 3, 4)]
    st = HostBlockStepper(w["W1t"], w["g"], w["W2t"], s.M, s.eps, fp8=True, delayed=delayed)
    host_in = [{k: pinned(x[k]) for k in ("X", "R", "dY")} for x in steps]
    outs = [st.host_buffers(out=True, dX=True, dR=True) for _ in steps]
    for hi, o in zip(host_in, outs):
        st.submit(hi["X"], hi["R"], hi["dY"], **o)
    st.sync()
    ref = BlockBuffers(dict(w, **{k: steps[0][k].clone() for k in ("X", "R", "dY")}))
    ref.fp8_quantize_weights()
    for i, x in enumerate(steps):
        for k in ("X", "R", "dY"):
            getattr(ref, k).copy_(x[k])
        ref.step_fp8(delayed=delayed)
        torch.cuda.synchronize()
        for k_host, k_ref in (("out", "out"), ("dX", "dX"), ("dR", "dH")):
            assert torch.equal(outs[i][k_host], getattr(ref, k_ref).cpu()), (i, k_host)
    assert_device_ok()
    for k in ("dW1t", "dW2t", "dg"):
        assert torch.equal(getattr(st, k), getattr(ref, k)), k
    st.close()


def test_fp8_step_needs_quantised_weights():
    s = FP8_SHAPE
    x = block_inputs(s, 0, "cuda")
    lib = C.load_library()
    flags = C.CODA_BLOCK_BACKWARD | C.CODA_BLOCK_FP8
    need = C.coda_block_arena_bytes(s.M, s.K1, s.d, s.N2, flags)
    arena = torch.empty(need, dtype=torch.uint8, device="cuda")
    grads = [torch.empty(s.d, s.K1, dtype=torch.bfloat16, device="cuda"),
             torch.empty(s.N2, s.d, dtype=torch.bfloat16, device="cuda"),
             torch.empty(s.d, dtype=torch.float32, device="cuda")]
    out = ctypes.c_void_p()
    assert lib.coda_block_create(C.handle(), s.M, s.K1, s.d, s.N2, s.eps, flags, x["W1t"].data_ptr(),
                                 x["g"].data_ptr(), x["W2t"].data_ptr(), *(t.data_ptr() for t in grads),
                                 arena.data_ptr(), need, ctypes.byref(out)) == 0
    hi = {k: pinned(x[k]) for k in ("X", "R", "dY")}
    assert lib.coda_block_step_host(out, hi["X"].data_ptr(), hi["R"].data_ptr(), hi["dY"].data_ptr(), None, None,
                                    None, None) == 1
    assert lib.coda_block_quantize_weights(out) == 0
    assert lib.coda_block_step_host(out, hi["X"].data_ptr(), hi["R"].data_ptr(), hi["dY"].data_ptr(), None, None,
                                    None, None) == 0
    assert lib.coda_block_sync(out, None) == 0
    assert lib.coda_block_destroy(out) == 0
