"""One pass of the hot path through the C ABI: device buffers for a
GEMM-Residual-PartialRMS-GEMM(+SwiGLU) block and the call sequence of its
forward and backward, fused or unfused (ablation).

Orchestration only: buffer allocation (torch, on the device) and the order of
library calls.  No arithmetic happens here.
"""
from __future__ import annotations

import torch

from . import (CODA_EPI_PLAIN, CODA_EPI_SWIGLU, E4M3, E5M2, coda_bwd_workspace_bytes, coda_dg_combine,
               coda_fp8_quantize, coda_fp8_quantize_e5m2, coda_gemm_dgrad_rmsbwd_fp8, coda_gemm_fp8,
               coda_swiglu_bwd_fp8_delayed, coda_gemm_res_prms_bwd_fp8,
               coda_gemm_res_prms_fp8, coda_gemm_rowscale_swiglu_fp8,
               coda_dgpart_rows, coda_fold_rmsnorm_weight, coda_gemm_dgrad_rmsbwd, coda_gemm_prms_rowscale_swiglu,
               coda_gemm_dgrad_rmsbwd_cpart, coda_gemm_dgrad_swiglu_bwd, coda_gemm_res_prms, coda_gemm_res_prms_g,
               coda_gemm_res_prms_bwd, coda_gemm_rowscale_swiglu, coda_gemm_rowscale_swiglu_bwd,
               coda_gemm_wgrad_gscale, coda_prms_num_tiles, coda_rstd_combine, coda_swiglu_bwd, coda_swiglu_bwd_fp8,
               coda_unfused_bwd, coda_unfused_fwd, coda_unfused_workspace_bytes)
from . import (CODA_BLOCK_BACKWARD, CODA_BLOCK_FP8, CODA_BLOCK_FP8_DELAYED, coda_block_arena_bytes,
               coda_block_create, coda_block_destroy, coda_block_quantize_weights, coda_block_step_host,
               coda_block_stream, coda_block_sync, coda_block_wait_step, STATUS_NAMES)

BF = torch.bfloat16
F32 = torch.float32


class BlockBuffers:
    """All tensors of one block problem on one device.

    inputs: X[M,K1], W1t[d,K1], R[M,d], g[d], W2t[N2,d], dY[M,F] (backward)
    forward: W2gt, H, psum, rstd, z (saved), out
    backward: dP, c, dgpart (stages), dH (= dR), dX, dW1t, dW2t, dg
    """

    def __init__(self, inputs: dict, swiglu: bool = True, backward: bool = True, eps: float = 1e-5,
                 unfused: bool = False, fuse_rstd: bool = False, g_on_activation: bool = False):
        dev = inputs["X"].device
        self.swiglu = swiglu
        self.eps = eps
        self.with_backward = backward
        self.unfused = unfused
        self.fuse_rstd = fuse_rstd
        self.g_on_activation = g_on_activation
        for k, v in inputs.items():
            setattr(self, k, v.contiguous())
        self.M, self.K1 = self.X.shape
        self.d = self.W1t.shape[0]
        self.N2 = self.W2t.shape[0]
        self.F = self.N2 // 2 if swiglu else self.N2
        M, d, N2 = self.M, self.d, self.N2
        e = dict(device=dev)
        self.W2gt = torch.empty(N2, d, dtype=BF, **e)
        self.H = torch.empty(M, d, dtype=BF, **e)
        self.Hg = torch.empty(M, d, dtype=BF, **e) if g_on_activation else None
        self.psum = torch.empty(M, coda_prms_num_tiles(d), dtype=F32, **e)
        self.rstd = torch.empty(M, dtype=F32, **e)
        self.z = torch.empty(M, N2, dtype=BF, **e)
        self.out = torch.empty(M, self.F, dtype=BF, **e) if swiglu else self.z
        if unfused:
            self.Nrm = torch.empty(M, d, dtype=BF, **e)
            self.ws_unfused = torch.empty(max(1, coda_unfused_workspace_bytes(M, d, N2)), dtype=torch.uint8, **e)
        if backward:
            self.dP = torch.empty(M, N2, dtype=BF, **e)
            self.c = torch.empty(M, dtype=F32, **e)
            # no rows for an empty batch: the dg combine then writes dg = 0
            self.dgpart = torch.empty(coda_dgpart_rows(M), d, dtype=F32, **e)
            self.dH = torch.empty(M, d, dtype=BF, **e)
            self.dX = torch.empty(M, self.K1, dtype=BF, **e)
            self.dW1t = torch.empty(d, self.K1, dtype=BF, **e)
            self.dW2t = torch.empty(N2, d, dtype=BF, **e)
            self.dg = torch.empty(d, dtype=F32, **e)
            self.ws = torch.empty(max(1, coda_bwd_workspace_bytes(M, d, N2)), dtype=torch.uint8, **e)

    # -- fused path ----------------------------------------------------------
    def forward(self, save_z: bool = True):
        """fold g -> GEMM1 + residual + partial RMS -> rstd combine ->
        GEMM2 + row scale + SwiGLU (z saved for the backward)."""
        if self.unfused:
            return self.forward_unfused()
        if self.g_on_activation:
            # g broadcast in GEMM1's epilogue: GEMM2 takes Hg and the unfolded W2
            coda_gemm_res_prms_g(self.X, self.W1t, self.R, self.g, self.H, self.Hg, self.psum)
            A2, B2 = self.Hg, self.W2t
        else:
            self.gemm1_and_fold()
            A2, B2 = self.H, self.W2gt
        if self.fuse_rstd:
            # the combine runs inside GEMM2's epilogue, which also stores rstd
            flags = CODA_EPI_SWIGLU if self.swiglu else CODA_EPI_PLAIN
            coda_gemm_prms_rowscale_swiglu(A2, B2, self.psum, self.eps, self.rstd,
                                           self.out if self.swiglu else self.z,
                                           (self.z if save_z else None) if self.swiglu else None, flags)
            return
        coda_rstd_combine(self.psum, self.d, self.eps, self.rstd)
        if self.swiglu:
            coda_gemm_rowscale_swiglu(A2, B2, self.rstd, self.out, self.z if save_z else None, CODA_EPI_SWIGLU)
        else:
            coda_gemm_rowscale_swiglu(A2, B2, self.rstd, self.z, None, CODA_EPI_PLAIN)

    def gemm1_and_fold(self):
        """GEMM1 + residual + partial RMS on the current stream, and the fold
        W2g = g * W2 beside it on a second stream; returns with the current
        stream ordered after both.  The fold reads only the weights and is
        HBM-bound.  GEMM1 is tensor-bound and leaves shared memory, threads
        and registers free on every SM, so the two share the SMs.  GEMM1 is
        launched first: its persistent CTAs take their SMs before the fold's
        CTAs fill them."""
        self._beside(lambda: coda_gemm_res_prms(self.X, self.W1t, self.R, self.H, self.psum),
                     lambda side: coda_fold_rmsnorm_weight(self.W2t, self.g, self.W2gt, stream=side))

    def _beside(self, main_call, side_call):
        """main_call on the current stream and side_call(side_stream) on a
        second stream, both ordered after everything before on the current
        stream; returns with the current stream ordered after both.  For a
        tensor-bound persistent GEMM (launched first, its CTAs take their
        SMs) with an independent HBM-bound kernel that fills the SMs'
        remaining threads and registers."""
        main = torch.cuda.current_stream(self.X.device)
        if getattr(self, "_side", None) is None:
            self._side = torch.cuda.Stream(device=self.X.device)
            self._ev_in = torch.cuda.Event()
            self._ev_side = torch.cuda.Event()
        self._ev_in.record(main)
        main_call()
        self._side.wait_event(self._ev_in)
        side_call(self._side)
        self._ev_side.record(self._side)
        main.wait_event(self._ev_side)

    def backward_stages(self):
        """The backward as separate stage calls (dP, c, dgpart stay visible)."""
        coda_swiglu_bwd(self.dY, self.z, self.rstd, self.dP, self.c, self.d)
        coda_gemm_dgrad_rmsbwd(self.dP, self.W2t, self.H, self.g, self.c, self.dH, self.dgpart)
        coda_dg_combine(self.dgpart, self.dg)
        coda_gemm_wgrad_gscale(self.H, self.dP, self.g, self.dW2t)
        coda_gemm_res_prms_bwd(self.dH, self.X, self.W1t, self.dX, self.dW1t, self.dH)

    def backward(self):
        """SwiGLU bwd -> dgrad2 + RMSNorm bwd -> dg combine -> wgrad2 ->
        dgrad1 -> wgrad1 (composite calls)."""
        if self.unfused:
            return self.backward_unfused()
        coda_gemm_rowscale_swiglu_bwd(self.dY, self.z, self.rstd, self.H, self.W2t, self.g, self.dH,
                                      self.dW2t, self.dg, self.ws)
        coda_gemm_res_prms_bwd(self.dH, self.X, self.W1t, self.dX, self.dW1t, self.dH)

    def step(self):
        """One pass of the whole path: forward, then backward if requested."""
        self.forward()
        if self.with_backward:
            self.backward()

    def step_fp8(self, delayed: bool = False):
        """One pass with FP8 operands (weights quantised beforehand by
        fp8_quantize_weights); delayed: dP's codes scaled by the previous
        step's amax (one pass instead of two)."""
        self.forward_fp8()
        if self.with_backward:
            self.backward_fp8(delayed)

    # -- CUDA graphs ----------------------------------------------------------
    def capture_step(self, fp8: bool = False, delayed: bool = False):
        """Record one step (step or step_fp8) into a CUDA graph and return
        it; replay() then reruns it on whatever the input buffers hold.  One
        eager step runs first, so that the library handle, tensor maps and
        the fold's side stream exist before the capture (none of them may be
        created inside it).  The fold's fork to the side stream and its join
        back are recorded as graph edges."""
        run = (lambda: self.step_fp8(delayed)) if fp8 else self.step
        run()
        torch.cuda.synchronize(self.X.device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run()
        self._graph = graph
        return graph

    def replay(self):
        self._graph.replay()

    # -- backward from the down projection's upstream gradient ---------------
    def backward_from_down_proj(self, dYb, W3t):
        """The backward when the block's output feeds a down projection
        y = out W3 (W3t[d, F]) with upstream gradient dYb[M, d]: dY stays on
        chip -- the down projection's data-gradient GEMM runs the SwiGLU
        backward in its epilogue, and dgrad2's epilogue forms c from its
        partial sums."""
        if not hasattr(self, "cpart"):
            self.cpart = torch.empty(self.M, coda_prms_num_tiles(self.F), dtype=F32, device=self.X.device)
        coda_gemm_dgrad_swiglu_bwd(dYb, W3t, self.z, self.rstd, self.dP, self.cpart)
        coda_gemm_dgrad_rmsbwd_cpart(self.dP, self.W2t, self.H, self.g, self.rstd, self.cpart, self.dH, self.dgpart)
        coda_dg_combine(self.dgpart, self.dg)
        coda_gemm_wgrad_gscale(self.H, self.dP, self.g, self.dW2t)
        coda_gemm_res_prms_bwd(self.dH, self.X, self.W1t, self.dX, self.dW1t, self.dH)

    # -- FP8 operands: e4m3 activations and weights, e5m2 gradients -----------
    def _fp8_buffers(self):
        if getattr(self, "Xq", None) is not None:
            return
        M, K1, d, N2 = self.M, self.K1, self.d, self.N2
        u8 = dict(dtype=torch.uint8, device=self.X.device)
        self.Xq = torch.empty(M, K1, **u8)
        self.Hq = torch.empty(M, d, **u8)
        self.W1q = torch.empty(d, K1, **u8)
        self.W2gq = torch.empty(N2, d, **u8)
        self.W2q = torch.empty(N2, d, **u8)
        # {amax, scale} per tensor: weights W1, W2*g, W2; activations X, H,
        # gradients dP, dH
        self.s_w = torch.empty(3, 2, dtype=F32, device=self.X.device)
        self.s_a = torch.empty(4, 2, dtype=F32, device=self.X.device)
        self._dp_amax_ready = False  # s_a[2] holds an amax of dP (delayed scaling)
        if self.with_backward:
            self.dPq = torch.empty(M, N2, **u8)
            self.dHq = torch.empty(M, d, **u8)

    def fp8_quantize_weights(self):
        """Per-tensor e4m3 codes of W1t, of W2t with g folded in (forward) and
        of W2t alone (dgrad2); needed once per weight update."""
        self._fp8_buffers()
        coda_fp8_quantize(self.W1t, self.W1q, self.s_w[0])
        coda_fp8_quantize(self.W2t, self.W2gq, self.s_w[1], self.g)
        if self.with_backward:
            coda_fp8_quantize(self.W2t, self.W2q, self.s_w[2])

    def fp8_forward_calls(self):
        """The forward on e4m3 operands as named calls (X and H quantised in
        the step, the weights by fp8_quantize_weights): the same epilogue
        programs as the bf16 forward."""
        self._fp8_buffers()
        return [
            ("quantize_X", lambda: coda_fp8_quantize(self.X, self.Xq, self.s_a[0])),
            ("gemm1_res_prms_fp8", lambda: coda_gemm_res_prms_fp8(self.Xq, self.s_a[0, 1:], self.W1q,
                                                                  self.s_w[0, 1:], self.R, self.H, self.psum)),
            ("rstd_combine", lambda: coda_rstd_combine(self.psum, self.d, self.eps, self.rstd)),
            ("quantize_H", lambda: coda_fp8_quantize(self.H, self.Hq, self.s_a[1])),
            ("gemm2_rowscale_swiglu_fp8", lambda: coda_gemm_rowscale_swiglu_fp8(
                self.Hq, self.s_a[1, 1:], self.W2gq, self.s_w[1, 1:], self.rstd, self.out, self.z)),
        ]

    def _swiglu_bwd_codes(self, delayed: bool):
        """dP's e5m2 codes and c.  Delayed: scaled by the previous step's
        amax of dP, one pass (the first step of a run, with no previous amax,
        takes the exact two-pass form)."""
        if delayed and self._dp_amax_ready:
            coda_swiglu_bwd_fp8_delayed(self.dY, self.z, self.rstd, E5M2, self.dPq, self.s_a[2], self.c, self.d)
        else:
            coda_swiglu_bwd_fp8(self.dY, self.z, self.rstd, E5M2, self.dPq, self.s_a[2], self.c, self.d)
        self._dp_amax_ready = True

    def fp8_backward_calls(self, delayed: bool = False):
        """The backward as named calls, with e5m2 gradients (dP, dH) against
        the e4m3 codes of the forward's activations and weights: the SwiGLU
        backward writes dP's codes directly (with delayed, scaled by the
        previous step's amax of dP, in one pass); dgrad2 runs the RMSNorm
        backward in its epilogue; the weight gradients and the first layer's
        data gradient are 8-bit GEMMs on the same codes read MN-major."""
        self._fp8_buffers()
        M, K1, d, N2 = self.M, self.K1, self.d, self.N2
        return [
            ("swiglu_bwd_e5m2", lambda: self._swiglu_bwd_codes(delayed)),
            ("dgrad2_rmsbwd_fp8", lambda: coda_gemm_dgrad_rmsbwd_fp8(
                self.dPq, E5M2, self.s_a[2, 1:], self.W2q, E4M3, self.s_w[2, 1:], self.H, self.g, self.c, self.dH,
                self.dgpart)),
            ("dg_combine", lambda: coda_dg_combine(self.dgpart, self.dg)),
            # dW2t[n][k] = g[k] sum_m dP[m][n] H[m][k]; dH's codes (needed
            # only by the first layer's gradients) beside it
            ("wgrad2_gscale_fp8+quantize_dH", lambda: self._beside(
                lambda: coda_gemm_fp8(self.dPq, True, E5M2, self.s_a[2, 1:], self.Hq, True, E4M3, self.s_a[1, 1:],
                                      self.dW2t, N2, d, M, col_scale=self.g),
                lambda side: coda_fp8_quantize_e5m2(self.dH, self.dHq, self.s_a[3], stream=side))),
            # dX = dH W1 (W1t codes [d][K1] read MN-major) and dW1t = dH^T X,
            # one grouped launch
            ("dgrad1_wgrad1_fp8", lambda: coda_gemm_res_prms_bwd_fp8(
                self.dHq, E5M2, self.s_a[3, 1:], self.Xq, self.s_a[0, 1:], self.W1q, self.s_w[0, 1:], E4M3, self.dX,
                self.dW1t)),
        ]

    def forward_fp8(self):
        for _, f in self.fp8_forward_calls():
            f()

    def backward_fp8(self, delayed: bool = False):
        for _, f in self.fp8_backward_calls(delayed):
            f()

    # -- unfused ablation -----------------------------------------------------
    def forward_unfused(self):
        coda_unfused_fwd(self.X, self.W1t, self.R, self.g, self.W2t, self.H, self.rstd, self.Nrm, self.z,
                         self.out, self.ws_unfused, self.eps, CODA_EPI_SWIGLU if self.swiglu else CODA_EPI_PLAIN)

    def backward_unfused(self):
        coda_unfused_bwd(self.dY, self.X, self.W1t, self.g, self.W2t, self.H, self.rstd, self.Nrm, self.z,
                         self.dH, self.dX, self.dW1t, self.dW2t, self.dg, self.ws_unfused)


class HostBlockStepper:
    """The fused step through the library's block executor (coda_block_*):
    each step's X, R (and dY) come from page-locked host tensors and its
    results go back to page-locked host tensors, with the copies of one step
    overlapping the kernels of its neighbours.  The executor issues the
    whole step natively; this class owns its device arena and the weight
    gradients, nothing more.

    W1t[d,K1], g[d], W2t[N2,d]: device bf16 weights, read by every step.
    With backward, every step overwrites dW1t, dW2t and dg (device).  With
    fp8, the steps run on 8-bit operands (delayed: dP's codes scaled by the
    previous step's amax); quantize_weights() must follow every weight
    update (the constructor calls it once)."""

    def __init__(self, W1t, g, W2t, M: int, eps: float = 1e-5, backward: bool = True, fp8: bool = False,
                 delayed: bool = False):
        dev = W1t.device
        self.d, self.K1 = W1t.shape
        self.N2 = W2t.shape[0]
        self.F = self.N2 // 2
        self.M = M
        self.backward = backward
        self.W1t, self.g, self.W2t = W1t, g, W2t
        e = dict(device=dev)
        self.dW1t = torch.empty(self.d, self.K1, dtype=BF, **e) if backward else None
        self.dW2t = torch.empty(self.N2, self.d, dtype=BF, **e) if backward else None
        self.dg = torch.empty(self.d, dtype=F32, **e) if backward else None
        flags = (CODA_BLOCK_BACKWARD if backward else 0) | (CODA_BLOCK_FP8 if fp8 else 0) | \
            (CODA_BLOCK_FP8_DELAYED if delayed else 0)
        nbytes = coda_block_arena_bytes(M, self.K1, self.d, self.N2, flags)
        self.arena = torch.empty(max(1, nbytes), dtype=torch.uint8, **e)
        self.blk = coda_block_create(M, self.K1, self.d, self.N2, eps, flags, W1t, g, W2t,
                                     self.dW1t, self.dW2t, self.dg, self.arena)
        self.fp8 = fp8
        if fp8:
            self.quantize_weights()

    def quantize_weights(self):
        """FP8: enqueue the weights' e4m3 quantisation on the executor's
        stream (after every weight update)."""
        coda_block_quantize_weights(self.blk)

    def host_buffers(self, out: bool = False, dX: bool = True, dR: bool = False) -> dict:
        """Page-locked host tensors for the results a step should read back."""
        M, K1, d, F = self.M, self.K1, self.d, self.F
        want = {"out": (out, (M, F)), "dX": (dX and self.backward, (M, K1)), "dR": (dR and self.backward, (M, d))}
        return {k: torch.empty(shape, dtype=BF).pin_memory() for k, (on, shape) in want.items() if on}

    def submit(self, X, R, dY=None, out=None, dX=None, dR=None) -> int:
        """Enqueue one step; returns its index.  The host inputs stay in use,
        and the results are not ready, until wait(index) or sync()."""
        return coda_block_step_host(self.blk, self.M, self.K1, self.d, self.F, X, R, dY, out, dX, dR)

    def wait(self, step: int):
        coda_block_wait_step(self.blk, step)

    def sync(self):
        """Wait for every submitted step; raises on a device-side error."""
        st, bits = coda_block_sync(self.blk)
        if st != 0:
            raise RuntimeError(f"block executor: {STATUS_NAMES.get(st, st)} (device bits {bits:#x})")

    def stream(self) -> torch.cuda.ExternalStream:
        """The executor's compute stream, for work ordered between steps."""
        return torch.cuda.ExternalStream(coda_block_stream(self.blk), device=self.W1t.device)

    def close(self):
        if getattr(self, "blk", None):
            coda_block_destroy(self.blk)
            self.blk = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
