"""Python binding of libcoda (include/coda.h): Transformer-block memory-bound
operations run as GEMM epilogues on sm_103a.

Argument marshalling only: every function here takes torch tensors already
on the GPU, checks dtype/shape/contiguity, and calls the C entry point of the
same name with raw pointers and extents on the current torch stream.  All
arithmetic runs in the library's CUDA kernels.  There is no fallback: if
libcoda.so is missing or cannot be loaded, importing the binding's entry
points raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcoda.so")

CODA_EPI_SWIGLU = 0
CODA_EPI_PLAIN = 1
# columns covered by one block-reduction partial (psum, CE statistics, c
# partials): partial j of a row covers columns [128 j, 128 j + 128)
PARTIAL_COLS = 128

STATUS_NAMES = {
    0: "CODA_OK", 1: "CODA_ERR_INVALID_ARG", 2: "CODA_ERR_ALIGNMENT", 3: "CODA_ERR_UNSUPPORTED",
    4: "CODA_ERR_WORKSPACE_TOO_SMALL", 5: "CODA_ERR_CUDA", 6: "CODA_ERR_TIMEOUT", 7: "CODA_ERR_LABEL_RANGE",
}


class CodaError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({msg})")
        self.code = code


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_U32 = ctypes.c_uint32
_INT = ctypes.c_int
_F32 = ctypes.c_float
_SZ = ctypes.c_size_t

# name -> (restype, argtypes), mirroring include/coda.h
SIGNATURES = {
    "coda_create": (_INT, [ctypes.POINTER(_P), _INT]),
    "coda_destroy": (_INT, [_P]),
    "coda_status_string": (ctypes.c_char_p, [_INT]),
    "coda_sync_status": (_INT, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "coda_set_wait_timeout_ns": (_INT, [_P, _U64]),
    "coda_debug_skip_first_stage": (_INT, [_P, _INT]),
    "coda_debug_group_schedule_violations": (_INT, [_INT, _INT, _INT, _INT, _INT]),
    "coda_debug_split_schedule_violations": (_INT, [_INT, _INT, _INT]),
    "coda_debug_split_first_tile": (_INT, [_INT, _INT, _INT]),
    "coda_debug_split_ranges": (_INT, [_INT, _INT, _INT]),
    "coda_debug_wide_schedule_violations": (_INT, [_INT, _INT, _INT, _INT, _INT]),
    "coda_debug_wide_applies": (_INT, [_P, _INT, _INT, _INT]),
    "coda_set_sm_pairing": (_INT, [_P, _INT]),
    "coda_set_wide_tiles": (_INT, [_P, _INT]),
    "coda_set_lmhead_chunk": (_INT, [_P, _I64]),
    "coda_split_workspace_bytes": (_SZ, [_P]),
    "coda_set_split_workspace": (_INT, [_P, _P, _SZ, _P]),
    "coda_prms_num_tiles": (_I64, [_I64]),
    "coda_dgpart_rows": (_I64, [_I64]),
    "coda_gemm": (_INT, [_P, _P, _INT, _P, _INT, _P, _I64, _I64, _I64, _P, _P, _P]),
    "coda_fold_rmsnorm_weight": (_INT, [_P, _P, _P, _P, _I64, _I64, _P]),
    "coda_gemm_res_prms": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_gemm_res_prms_g": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_rstd_combine": (_INT, [_P, _P, _I64, _I64, _I64, _F32, _P, _P]),
    "coda_gemm_rowscale_swiglu": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _U32, _P]),
    "coda_gemm_prms_rowscale_swiglu": (_INT, [_P, _P, _P, _P, _I64, _F32, _P, _P, _P, _I64, _I64, _I64, _U32, _P]),
    "coda_swiglu_bwd": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_gemm_dgrad_rmsbwd": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_gemm_dgrad_rmsbwd_noalloc": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_gemm_dgrad_swiglu_bwd": (_INT, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_gemm_dgrad_rmsbwd_cpart": (_INT, [_P, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _I64, _I64, _I64, _P]),
    "coda_dg_combine": (_INT, [_P, _P, _I64, _I64, _P, _P]),
    "coda_gemm_wgrad_gscale": (_INT, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_bwd_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "coda_gemm_rowscale_swiglu_bwd": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                             _I64, _I64, _I64, _P]),
    "coda_gemm_res_prms_bwd": (_INT, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_block_arena_bytes": (_SZ, [_I64, _I64, _I64, _I64, _U32]),
    "coda_block_create": (_INT, [_P, _I64, _I64, _I64, _I64, _F32, _U32, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                 ctypes.POINTER(_P)]),
    "coda_block_quantize_weights": (_INT, [_P]),
    "coda_block_step_host": (_INT, [_P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(_I64)]),
    "coda_block_wait_step": (_INT, [_P, _I64]),
    "coda_block_sync": (_INT, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "coda_block_stream": (_INT, [_P, ctypes.POINTER(_P)]),
    "coda_block_destroy": (_INT, [_P]),
    "coda_rope_table": (_INT, [_P, _P, _P, _I64, _I64, _F32, _P]),
    "coda_gemm_qkv_rope": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _P]),
    "coda_rope_apply": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _P]),
    "coda_fp8_quantize": (_INT, [_P, _P, _P, _P, _P, _I64, _I64, _P]),
    "coda_fp8_quantize_e5m2": (_INT, [_P, _P, _P, _P, _P, _I64, _I64, _P]),
    "coda_swiglu_bwd_fp8": (_INT, [_P, _P, _P, _P, _INT, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_swiglu_bwd_fp8_delayed": (_INT, [_P, _P, _P, _P, _INT, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_gemm_fp8": (_INT, [_P, _P, _INT, _INT, _P, _P, _INT, _INT, _P, _P, _I64, _I64, _I64, _P, _P, _P]),
    "coda_gemm_res_prms_bwd_fp8": (_INT, [_P, _P, _INT, _P, _P, _P, _P, _P, _INT, _P, _P, _I64, _I64, _I64, _P]),
    "coda_gemm_dgrad_rmsbwd_fp8": (_INT, [_P, _P, _INT, _P, _P, _INT, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_gemm_res_prms_fp8": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "coda_gemm_rowscale_swiglu_fp8": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _U32, _P]),
    "coda_lmhead_ce_workspace_bytes": (_SZ, [_I64, _I64, _I64, _INT]),
    "coda_lmhead_ce_row_offsets": (_INT, [_I64, _I64, _I64, _INT, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "coda_lmhead_ce": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I64, _I64, _P]),
    "coda_lmhead_ce_fp8": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I64, _I64, _P]),
    "coda_unfused_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "coda_unfused_fwd": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                _I64, _I64, _I64, _I64, _F32, _U32, _P]),
    "coda_unfused_bwd": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                _I64, _I64, _I64, _I64, _P]),
}

_lib = None
_lib_lock = threading.Lock()
_handles: dict[int, int] = {}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libcoda.so (built by gemm_epilogue_transformer_tma_gb300.build) and
    declare every entry point's signature.  Raises if it is missing."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with "
                              "`python -m gemm_epilogue_transformer_tma_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(code: int, where: str):
    if code != 0:
        msg = load_library().coda_status_string(code).decode()
        raise CodaError(code, where, msg)


def handle(device: int | None = None) -> int:
    """The library handle of a CUDA device (created once per device)."""
    lib = load_library()
    dev = torch.cuda.current_device() if device is None else int(device)
    h = _handles.get(dev)
    if h is None:
        hp = _P()
        _check(lib.coda_create(ctypes.byref(hp), dev), "coda_create")
        h = hp.value
        _handles[dev] = h
    return h


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _shape(t, shape, name):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


BF = torch.bfloat16
F32 = torch.float32
I32 = torch.int32


def _h(t: torch.Tensor) -> int:
    return handle(t.device.index)


# ---------------------------------------------------------------------------
def coda_sync_status(device: int | None = None, stream=None) -> tuple[int, int]:
    """Synchronise the stream, read and clear the device status word.
    Returns (status, raw_bits); does not raise."""
    lib = load_library()
    bits = ctypes.c_int32(0)
    st = lib.coda_sync_status(handle(device), _stream(stream), ctypes.byref(bits))
    return st, bits.value


def coda_set_wait_timeout_ns(ns: int, device: int | None = None):
    _check(load_library().coda_set_wait_timeout_ns(handle(device), ns), "coda_set_wait_timeout_ns")


def coda_set_sm_pairing(enable: bool, device: int | None = None):
    """GEMMs on SM pairs (2-SM MMA, default) or one SM per tile."""
    _check(load_library().coda_set_sm_pairing(handle(device), int(enable)), "coda_set_sm_pairing")


def coda_set_wide_tiles(lead_kblocks: int, device: int | None = None):
    """256 x 512 pair tiles for the long-K backward GEMMs with lead J =
    lead_kblocks k-blocks; 0 turns them off (see include/coda.h)."""
    _check(load_library().coda_set_wide_tiles(handle(device), int(lead_kblocks)), "coda_set_wide_tiles")


def coda_set_lmhead_chunk(cols: int, device: int | None = None):
    """Vocabulary columns per LM-head backward chunk (a multiple of 256 up to
    32768; 0 = the default, 32768); see include/coda.h."""
    _check(load_library().coda_set_lmhead_chunk(handle(device), int(cols)), "coda_set_lmhead_chunk")


def coda_split_workspace_bytes(device: int | None = None) -> int:
    """Bytes of the split-tile scratch coda_set_split_workspace takes."""
    return load_library().coda_split_workspace_bytes(handle(device))


def coda_set_split_workspace(ws, device: int | None = None, stream=None):
    """Give the device's handle a split-tile scratch (a uint8 CUDA tensor of at
    least coda_split_workspace_bytes()), or None to stop splitting tiles.
    The caller keeps ws alive while it is set (see include/coda.h)."""
    if ws is None:
        _check(load_library().coda_set_split_workspace(handle(device), None, 0, _stream(stream)),
               "coda_set_split_workspace")
        return
    _check(load_library().coda_set_split_workspace(handle(device), _ptr(ws, torch.uint8, "ws"),
                                                   ws.numel() * ws.element_size(), _stream(stream)),
           "coda_set_split_workspace")


def coda_debug_skip_first_stage(enable: int, device: int | None = None):
    """Failure-detection test hook (see include/coda_testing.h)."""
    _check(load_library().coda_debug_skip_first_stage(handle(device), int(enable)), "coda_debug_skip_first_stage")


def coda_prms_num_tiles(d: int) -> int:
    return load_library().coda_prms_num_tiles(d)


def coda_dgpart_rows(M: int) -> int:
    return load_library().coda_dgpart_rows(M)


def coda_gemm(A, a_mn_major: bool, B, b_mn_major: bool, C, M: int, N: int, K: int,
              row_scale=None, col_scale=None, stream=None):
    """C[M,N] = row_scale * col_scale * A B (see include/coda.h)."""
    _shape(A, (K, M) if a_mn_major else (M, K), "A")
    _shape(B, (K, N) if b_mn_major else (N, K), "B")
    _shape(C, (M, N), "C")
    if row_scale is not None:
        _shape(row_scale, (M,), "row_scale")
    if col_scale is not None:
        _shape(col_scale, (N,), "col_scale")
    _check(load_library().coda_gemm(_h(C), _ptr(A, BF, "A"), int(a_mn_major), _ptr(B, BF, "B"), int(b_mn_major),
                                    _ptr(C, BF, "C"), M, N, K, _ptr(row_scale, F32, "row_scale"),
                                    _ptr(col_scale, BF, "col_scale"), _stream(stream)), "coda_gemm")


def coda_fold_rmsnorm_weight(W2t, g, W2gt, stream=None):
    N2, d = W2t.shape
    _shape(g, (d,), "g")
    _shape(W2gt, (N2, d), "W2gt")
    _check(load_library().coda_fold_rmsnorm_weight(_h(W2t), _ptr(W2t, BF, "W2t"), _ptr(g, BF, "g"),
                                                   _ptr(W2gt, BF, "W2gt"), N2, d, _stream(stream)),
           "coda_fold_rmsnorm_weight")


def coda_gemm_res_prms(X, W1t, R, H, psum, stream=None):
    M, K1 = X.shape
    d = W1t.shape[0]
    _shape(W1t, (d, K1), "W1t")
    _shape(R, (M, d), "R")
    _shape(H, (M, d), "H")
    _shape(psum, (M, coda_prms_num_tiles(d)), "psum")
    _check(load_library().coda_gemm_res_prms(_h(X), _ptr(X, BF, "X"), _ptr(W1t, BF, "W1t"), _ptr(R, BF, "R"),
                                             _ptr(H, BF, "H"), _ptr(psum, F32, "psum"), M, K1, d, _stream(stream)),
           "coda_gemm_res_prms")


def coda_gemm_res_prms_g(X, W1t, R, g, H, Hg, psum, stream=None):
    """coda_gemm_res_prms that also writes Hg = bf16(H * g) (the RMSNorm
    weight applied on the activation side)."""
    M, K1 = X.shape
    d = W1t.shape[0]
    _shape(W1t, (d, K1), "W1t")
    _shape(R, (M, d), "R")
    _shape(g, (d,), "g")
    _shape(H, (M, d), "H")
    _shape(Hg, (M, d), "Hg")
    _shape(psum, (M, coda_prms_num_tiles(d)), "psum")
    _check(load_library().coda_gemm_res_prms_g(_h(X), _ptr(X, BF, "X"), _ptr(W1t, BF, "W1t"), _ptr(R, BF, "R"),
                                               _ptr(g, BF, "g"), _ptr(H, BF, "H"), _ptr(Hg, BF, "Hg"),
                                               _ptr(psum, F32, "psum"), M, K1, d, _stream(stream)),
           "coda_gemm_res_prms_g")


def coda_rstd_combine(psum, d: int, eps: float, rstd, stream=None):
    M, T = psum.shape
    _shape(rstd, (M,), "rstd")
    _check(load_library().coda_rstd_combine(_h(psum), _ptr(psum, F32, "psum"), M, T, d, eps,
                                            _ptr(rstd, F32, "rstd"), _stream(stream)), "coda_rstd_combine")


def coda_gemm_rowscale_swiglu(H, W2gt, rstd, out, z_save=None, flags=CODA_EPI_SWIGLU, stream=None):
    M, d = H.shape
    N2 = W2gt.shape[0]
    _shape(W2gt, (N2, d), "W2gt")
    _shape(rstd, (M,), "rstd")
    _shape(out, (M, N2 // 2 if flags == CODA_EPI_SWIGLU else N2), "out")
    if z_save is not None:
        _shape(z_save, (M, N2), "z_save")
    _check(load_library().coda_gemm_rowscale_swiglu(_h(H), _ptr(H, BF, "H"), _ptr(W2gt, BF, "W2gt"),
                                                    _ptr(rstd, F32, "rstd"), _ptr(out, BF, "out"),
                                                    _ptr(z_save, BF, "z_save"), M, d, N2, flags, _stream(stream)),
           "coda_gemm_rowscale_swiglu")


def coda_gemm_prms_rowscale_swiglu(H, W2gt, psum, eps, rstd, out, z_save=None, flags=CODA_EPI_SWIGLU,
                                   stream=None):
    """GEMM2 with the row scale derived from GEMM1's partial sums in its
    epilogue (no separate combine launch); rstd may be None."""
    M, d = H.shape
    N2 = W2gt.shape[0]
    T = psum.shape[1]
    _shape(W2gt, (N2, d), "W2gt")
    _shape(psum, (M, T), "psum")
    if rstd is not None:
        _shape(rstd, (M,), "rstd")
    _shape(out, (M, N2 // 2 if flags == CODA_EPI_SWIGLU else N2), "out")
    if z_save is not None:
        _shape(z_save, (M, N2), "z_save")
    _check(load_library().coda_gemm_prms_rowscale_swiglu(_h(H), _ptr(H, BF, "H"), _ptr(W2gt, BF, "W2gt"),
                                                         _ptr(psum, F32, "psum"), T, eps, _ptr(rstd, F32, "rstd"),
                                                         _ptr(out, BF, "out"), _ptr(z_save, BF, "z_save"),
                                                         M, d, N2, flags, _stream(stream)),
           "coda_gemm_prms_rowscale_swiglu")


def coda_swiglu_bwd(dY, z, rstd, dP, c, d: int, stream=None):
    M, F = dY.shape
    _shape(z, (M, 2 * F), "z")
    _shape(rstd, (M,), "rstd")
    _shape(dP, (M, 2 * F), "dP")
    _shape(c, (M,), "c")
    _check(load_library().coda_swiglu_bwd(_h(dY), _ptr(dY, BF, "dY"), _ptr(z, BF, "z"), _ptr(rstd, F32, "rstd"),
                                          _ptr(dP, BF, "dP"), _ptr(c, F32, "c"), M, F, d, _stream(stream)),
           "coda_swiglu_bwd")


def coda_gemm_dgrad_rmsbwd(dP, W2t, H, g, c, dH, dgpart, stream=None):
    M, N2 = dP.shape
    d = W2t.shape[1]
    _shape(W2t, (N2, d), "W2t")
    _shape(H, (M, d), "H")
    _shape(g, (d,), "g")
    _shape(c, (M,), "c")
    _shape(dH, (M, d), "dH")
    _shape(dgpart, (coda_dgpart_rows(M), d), "dgpart")
    _check(load_library().coda_gemm_dgrad_rmsbwd(_h(dP), _ptr(dP, BF, "dP"), _ptr(W2t, BF, "W2t"), _ptr(H, BF, "H"),
                                                 _ptr(g, BF, "g"), _ptr(c, F32, "c"), _ptr(dH, BF, "dH"),
                                                 _ptr(dgpart, F32, "dgpart"), M, N2, d, _stream(stream)),
           "coda_gemm_dgrad_rmsbwd")


def coda_gemm_dgrad_rmsbwd_noalloc(dP, W2t, H, g, c, dH, dg, stream=None):
    """coda_gemm_dgrad_rmsbwd + coda_dg_combine without any device allocation:
    the dg partial sums live in the library's own fixed 8 MiB array."""
    M, N2 = dP.shape
    d = W2t.shape[1]
    _shape(W2t, (N2, d), "W2t")
    _shape(H, (M, d), "H")
    _shape(g, (d,), "g")
    _shape(c, (M,), "c")
    _shape(dH, (M, d), "dH")
    _shape(dg, (d,), "dg")
    _check(load_library().coda_gemm_dgrad_rmsbwd_noalloc(_h(dP), _ptr(dP, BF, "dP"), _ptr(W2t, BF, "W2t"),
                                                         _ptr(H, BF, "H"), _ptr(g, BF, "g"), _ptr(c, F32, "c"),
                                                         _ptr(dH, BF, "dH"), _ptr(dg, F32, "dg"), M, N2, d,
                                                         _stream(stream)), "coda_gemm_dgrad_rmsbwd_noalloc")


def coda_gemm_dgrad_swiglu_bwd(dYb, W3t, z, rstd, dP, cpart, stream=None):
    """dY = dYb W3 on chip, SwiGLU backward in the epilogue: dP and the c
    partial sums (see include/coda.h)."""
    M, d = dYb.shape
    F = W3t.shape[1]
    _shape(W3t, (d, F), "W3t")
    _shape(z, (M, 2 * F), "z")
    _shape(rstd, (M,), "rstd")
    _shape(dP, (M, 2 * F), "dP")
    _shape(cpart, (M, coda_prms_num_tiles(F)), "cpart")
    _check(load_library().coda_gemm_dgrad_swiglu_bwd(_h(dYb), _ptr(dYb, BF, "dYb"), _ptr(W3t, BF, "W3t"),
                                                     _ptr(z, BF, "z"), _ptr(rstd, F32, "rstd"), _ptr(dP, BF, "dP"),
                                                     _ptr(cpart, F32, "cpart"), M, d, F, _stream(stream)),
           "coda_gemm_dgrad_swiglu_bwd")


def coda_gemm_dgrad_rmsbwd_cpart(dP, W2t, H, g, rstd, cpart, dH, dgpart, stream=None):
    M, N2 = dP.shape
    d = W2t.shape[1]
    Tc = cpart.shape[1]
    _shape(W2t, (N2, d), "W2t")
    _shape(H, (M, d), "H")
    _shape(g, (d,), "g")
    _shape(rstd, (M,), "rstd")
    _shape(cpart, (M, Tc), "cpart")
    _shape(dH, (M, d), "dH")
    _shape(dgpart, (coda_dgpart_rows(M), d), "dgpart")
    _check(load_library().coda_gemm_dgrad_rmsbwd_cpart(
        _h(dP), _ptr(dP, BF, "dP"), _ptr(W2t, BF, "W2t"), _ptr(H, BF, "H"), _ptr(g, BF, "g"),
        _ptr(rstd, F32, "rstd"), _ptr(cpart, F32, "cpart"), Tc, _ptr(dH, BF, "dH"), _ptr(dgpart, F32, "dgpart"),
        M, N2, d, _stream(stream)), "coda_gemm_dgrad_rmsbwd_cpart")


def coda_dg_combine(dgpart, dg, stream=None):
    rows, d = dgpart.shape
    _shape(dg, (d,), "dg")
    _check(load_library().coda_dg_combine(_h(dg), _ptr(dgpart, F32, "dgpart"), rows, d, _ptr(dg, F32, "dg"),
                                          _stream(stream)), "coda_dg_combine")


def coda_gemm_wgrad_gscale(H, dP, g, dW2t, stream=None):
    M, d = H.shape
    N2 = dP.shape[1]
    _shape(dP, (M, N2), "dP")
    _shape(g, (d,), "g")
    _shape(dW2t, (N2, d), "dW2t")
    _check(load_library().coda_gemm_wgrad_gscale(_h(H), _ptr(H, BF, "H"), _ptr(dP, BF, "dP"), _ptr(g, BF, "g"),
                                                 _ptr(dW2t, BF, "dW2t"), M, N2, d, _stream(stream)),
           "coda_gemm_wgrad_gscale")


def coda_debug_group_schedule_violations(P: int, heavy: int, nH: int, nL: int, q: int) -> int:
    """Host check of the grouped launches' tile schedule (see include/coda_testing.h)."""
    return load_library().coda_debug_group_schedule_violations(P, heavy, nH, nL, q)


def coda_debug_split_schedule_violations(tiles: int, num_kb: int, clusters: int) -> int:
    """Host check of the split-tile schedule (see include/coda_testing.h)."""
    return load_library().coda_debug_split_schedule_violations(tiles, num_kb, clusters)


def coda_debug_split_first_tile(tiles: int, num_kb: int, clusters: int) -> int:
    """First split tile the launcher would choose, tiles if none (see include/coda_testing.h)."""
    return load_library().coda_debug_split_first_tile(tiles, num_kb, clusters)


def coda_debug_split_ranges(tiles: int, num_kb: int, clusters: int) -> int:
    """k-ranges per split tile the launcher would choose, 1 if none (see include/coda_testing.h)."""
    return load_library().coda_debug_split_ranges(tiles, num_kb, clusters)


def coda_debug_wide_schedule_violations(M: int, N: int, K: int, clusters: int, lead: int) -> int:
    """Host-side check of the wide-tile schedule (see include/coda_testing.h)."""
    return load_library().coda_debug_wide_schedule_violations(M, N, K, clusters, lead)


def coda_debug_wide_applies(M: int, N: int, K: int, device: int | None = None) -> int:
    """1 if a long-K backward GEMM of this size would take wide tiles on the
    device's handle now (see include/coda_testing.h)."""
    return load_library().coda_debug_wide_applies(handle(device), M, N, K)


def coda_bwd_workspace_bytes(M: int, d: int, N2: int) -> int:
    return load_library().coda_bwd_workspace_bytes(M, d, N2)


def coda_gemm_rowscale_swiglu_bwd(dY, z, rstd, H, W2t, g, dH, dW2t, dg, ws, stream=None):
    M, d = H.shape
    N2 = W2t.shape[0]
    _shape(dY, (M, N2 // 2), "dY")
    _shape(z, (M, N2), "z")
    _shape(rstd, (M,), "rstd")
    _shape(W2t, (N2, d), "W2t")
    _shape(g, (d,), "g")
    _shape(dH, (M, d), "dH")
    _shape(dW2t, (N2, d), "dW2t")
    _shape(dg, (d,), "dg")
    _check(load_library().coda_gemm_rowscale_swiglu_bwd(
        _h(H), _ptr(dY, BF, "dY"), _ptr(z, BF, "z"), _ptr(rstd, F32, "rstd"), _ptr(H, BF, "H"),
        _ptr(W2t, BF, "W2t"), _ptr(g, BF, "g"), _ptr(dH, BF, "dH"), _ptr(dW2t, BF, "dW2t"), _ptr(dg, F32, "dg"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), M, d, N2, _stream(stream)),
        "coda_gemm_rowscale_swiglu_bwd")


def coda_gemm_res_prms_bwd(dH, X, W1t, dX, dW1t, dR=None, stream=None):
    M, K1 = X.shape
    d = W1t.shape[0]
    _shape(dH, (M, d), "dH")
    _shape(W1t, (d, K1), "W1t")
    _shape(dX, (M, K1), "dX")
    _shape(dW1t, (d, K1), "dW1t")
    if dR is not None:
        _shape(dR, (M, d), "dR")
    _check(load_library().coda_gemm_res_prms_bwd(_h(X), _ptr(dH, BF, "dH"), _ptr(X, BF, "X"), _ptr(W1t, BF, "W1t"),
                                                 _ptr(dX, BF, "dX"), _ptr(dW1t, BF, "dW1t"), _ptr(dR, BF, "dR"),
                                                 M, K1, d, _stream(stream)), "coda_gemm_res_prms_bwd")


def _host_ptr(t: torch.Tensor | None, dtype, shape, name) -> int | None:
    """A page-locked host tensor's address (the block executor's copy
    engines read and write it asynchronously)."""
    if t is None:
        return None
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    _shape(t, shape, name)
    if not t.is_pinned():
        raise ValueError(f"{name} must be in page-locked memory (pin_memory())")
    return t.data_ptr()


CODA_BLOCK_BACKWARD = 1
CODA_BLOCK_FP8 = 2
CODA_BLOCK_FP8_DELAYED = 4


def coda_block_arena_bytes(M: int, K1: int, d: int, N2: int, flags: int) -> int:
    return load_library().coda_block_arena_bytes(M, K1, d, N2, int(flags))


def coda_block_create(M: int, K1: int, d: int, N2: int, eps: float, flags: int, W1t, g, W2t,
                      dW1t, dW2t, dg, arena) -> int:
    """Create a block step executor (include/coda.h) on the weights' device;
    returns its handle.  flags: CODA_BLOCK_* bits.  arena: a uint8 device
    tensor of at least coda_block_arena_bytes bytes, kept alive by the
    caller."""
    backward = bool(flags & CODA_BLOCK_BACKWARD)
    _shape(W1t, (d, K1), "W1t")
    _shape(g, (d,), "g")
    _shape(W2t, (N2, d), "W2t")
    if backward:
        _shape(dW1t, (d, K1), "dW1t")
        _shape(dW2t, (N2, d), "dW2t")
        _shape(dg, (d,), "dg")
    out = _P()
    with torch.cuda.device(W1t.device):
        _check(load_library().coda_block_create(
            _h(W1t), M, K1, d, N2, eps, int(flags), _ptr(W1t, BF, "W1t"), _ptr(g, BF, "g"), _ptr(W2t, BF, "W2t"),
            _ptr(dW1t, BF, "dW1t"), _ptr(dW2t, BF, "dW2t"), _ptr(dg, F32, "dg"), _ptr(arena, torch.uint8, "arena"),
            arena.numel(), ctypes.byref(out)), "coda_block_create")
    return out.value


def coda_block_step_host(blk: int, M: int, K1: int, d: int, F: int, X, R, dY=None, out=None, dX=None,
                         dR=None) -> int:
    """Enqueue one step on page-locked host tensors; returns the step index."""
    sid = _I64(0)
    _check(load_library().coda_block_step_host(
        blk, _host_ptr(X, BF, (M, K1), "X"), _host_ptr(R, BF, (M, d), "R"), _host_ptr(dY, BF, (M, F), "dY"),
        _host_ptr(out, BF, (M, F), "out"), _host_ptr(dX, BF, (M, K1), "dX"), _host_ptr(dR, BF, (M, d), "dR"),
        ctypes.byref(sid)), "coda_block_step_host")
    return sid.value


def coda_block_quantize_weights(blk: int):
    """FP8 executors: enqueue the e4m3 quantisation of the weights."""
    _check(load_library().coda_block_quantize_weights(blk), "coda_block_quantize_weights")


def coda_block_wait_step(blk: int, step: int):
    _check(load_library().coda_block_wait_step(blk, step), "coda_block_wait_step")


def coda_block_sync(blk: int) -> tuple[int, int]:
    """Wait for every submitted step; returns (status, raw_bits) like
    coda_sync_status, without raising."""
    bits = ctypes.c_int32(0)
    st = load_library().coda_block_sync(blk, ctypes.byref(bits))
    return st, bits.value


def coda_block_stream(blk: int) -> int:
    """The executor's compute stream, as a cudaStream_t value."""
    s = _P()
    _check(load_library().coda_block_stream(blk, ctypes.byref(s)), "coda_block_stream")
    return s.value or 0


def coda_block_destroy(blk: int):
    _check(load_library().coda_block_destroy(blk), "coda_block_destroy")


def coda_rope_table(cos_t, sin_t, base=10000.0, stream=None):
    """cos / sin tables [S, head_dim / 2] of the rotary embedding."""
    S, half = cos_t.shape
    _shape(sin_t, (S, half), "sin_t")
    _check(load_library().coda_rope_table(_h(cos_t), _ptr(cos_t, F32, "cos_t"), _ptr(sin_t, F32, "sin_t"), S,
                                          2 * half, base, _stream(stream)), "coda_rope_table")


def coda_gemm_qkv_rope(X, Wqkv_t, cos_t, sin_t, qkv, n_q_heads, n_kv_heads, head_dim=128, stream=None):
    """qkv = X Wqkv with RoPE on the q and k heads in the GEMM epilogue."""
    M, d = X.shape
    N = (n_q_heads + 2 * n_kv_heads) * head_dim
    S = cos_t.shape[0]
    _shape(Wqkv_t, (N, d), "Wqkv_t")
    _shape(qkv, (M, N), "qkv")
    _shape(cos_t, (S, head_dim // 2), "cos_t")
    _check(load_library().coda_gemm_qkv_rope(_h(X), _ptr(X, BF, "X"), _ptr(Wqkv_t, BF, "Wqkv_t"),
                                             _ptr(cos_t, F32, "cos_t"), _ptr(sin_t, F32, "sin_t"),
                                             _ptr(qkv, BF, "qkv"), M, d, n_q_heads, n_kv_heads, head_dim, S,
                                             _stream(stream)), "coda_gemm_qkv_rope")


def coda_rope_apply(qkv, cos_t, sin_t, n_q_heads, n_kv_heads, head_dim=128, stream=None):
    """Standalone in-place RoPE on an existing qkv (the unfused baseline)."""
    M, N = qkv.shape
    S = cos_t.shape[0]
    if N != (n_q_heads + 2 * n_kv_heads) * head_dim:
        raise ValueError("qkv width does not match the head counts")
    _check(load_library().coda_rope_apply(_h(qkv), _ptr(qkv, BF, "qkv"), _ptr(cos_t, F32, "cos_t"),
                                          _ptr(sin_t, F32, "sin_t"), M, n_q_heads, n_kv_heads, head_dim, S,
                                          _stream(stream)), "coda_rope_apply")


U8 = torch.uint8


def coda_fp8_quantize(src, dst, amax_scale, g=None, stream=None):
    """Per-tensor e4m3 quantisation of src (times g per column if given);
    dst: uint8 codes of src's shape; amax_scale: fp32 [2] <- {amax, scale}."""
    rows, cols = src.shape
    _shape(dst, (rows, cols), "dst")
    _shape(amax_scale, (2,), "amax_scale")
    if g is not None:
        _shape(g, (cols,), "g")
    _check(load_library().coda_fp8_quantize(_h(src), _ptr(src, BF, "src"), _ptr(g, BF, "g"),
                                            _ptr(amax_scale, F32, "amax_scale"), _ptr(dst, U8, "dst"), rows, cols,
                                            _stream(stream)), "coda_fp8_quantize")


def coda_fp8_quantize_e5m2(src, dst, amax_scale, g=None, stream=None):
    """Per-tensor e5m2 quantisation (scale: the smallest power of two with
    amax / scale <= 57344), like coda_fp8_quantize."""
    rows, cols = src.shape
    _shape(dst, (rows, cols), "dst")
    _shape(amax_scale, (2,), "amax_scale")
    if g is not None:
        _shape(g, (cols,), "g")
    _check(load_library().coda_fp8_quantize_e5m2(_h(src), _ptr(src, BF, "src"), _ptr(g, BF, "g"),
                                                 _ptr(amax_scale, F32, "amax_scale"), _ptr(dst, U8, "dst"), rows,
                                                 cols, _stream(stream)), "coda_fp8_quantize_e5m2")


E4M3, E5M2 = 0, 1


def coda_swiglu_bwd_fp8(dY, z, rstd, fmt: int, dPq, amax_scale, c, d: int, stream=None):
    """coda_swiglu_bwd with dP delivered as 8-bit codes (fmt E4M3 / E5M2) and
    {amax, scale}; dP itself is never written (see include/coda.h)."""
    M, F = dY.shape
    _shape(z, (M, 2 * F), "z")
    _shape(rstd, (M,), "rstd")
    _shape(dPq, (M, 2 * F), "dPq")
    _shape(amax_scale, (2,), "amax_scale")
    _shape(c, (M,), "c")
    _check(load_library().coda_swiglu_bwd_fp8(_h(dY), _ptr(dY, BF, "dY"), _ptr(z, BF, "z"), _ptr(rstd, F32, "rstd"),
                                              int(fmt), _ptr(dPq, U8, "dPq"), _ptr(amax_scale, F32, "amax_scale"),
                                              _ptr(c, F32, "c"), M, F, d, _stream(stream)), "coda_swiglu_bwd_fp8")


def coda_swiglu_bwd_fp8_delayed(dY, z, rstd, fmt: int, dPq, amax_scale, c, d: int, stream=None):
    """coda_swiglu_bwd_fp8 with delayed scaling: amax_scale[0] holds the
    previous dP's amax on entry; on exit {this dP's amax, the scale used}
    (see include/coda.h)."""
    M, F = dY.shape
    _shape(z, (M, 2 * F), "z")
    _shape(rstd, (M,), "rstd")
    _shape(dPq, (M, 2 * F), "dPq")
    _shape(amax_scale, (2,), "amax_scale")
    _shape(c, (M,), "c")
    _check(load_library().coda_swiglu_bwd_fp8_delayed(
        _h(dY), _ptr(dY, BF, "dY"), _ptr(z, BF, "z"), _ptr(rstd, F32, "rstd"), int(fmt), _ptr(dPq, U8, "dPq"),
        _ptr(amax_scale, F32, "amax_scale"), _ptr(c, F32, "c"), M, F, d, _stream(stream)),
        "coda_swiglu_bwd_fp8_delayed")


def coda_gemm_fp8(A, a_mn_major: bool, a_format: int, sA, B, b_mn_major: bool, b_format: int, sB, C,
                  M: int, N: int, K: int, row_scale=None, col_scale=None, stream=None):
    """C[M,N] = row_scale * col_scale * sA * sB * A B on 8-bit codes (see include/coda.h)."""
    _shape(A, (K, M) if a_mn_major else (M, K), "A")
    _shape(B, (K, N) if b_mn_major else (N, K), "B")
    _shape(C, (M, N), "C")
    _check(load_library().coda_gemm_fp8(_h(C), _ptr(A, U8, "A"), int(a_mn_major), int(a_format),
                                        _ptr(sA, F32, "sA"), _ptr(B, U8, "B"), int(b_mn_major), int(b_format),
                                        _ptr(sB, F32, "sB"), _ptr(C, BF, "C"), M, N, K,
                                        _ptr(row_scale, F32, "row_scale"), _ptr(col_scale, BF, "col_scale"),
                                        _stream(stream)), "coda_gemm_fp8")


def coda_gemm_res_prms_bwd_fp8(dHq, dh_format: int, sdH, Xq, sX, W1q, sW1, w_format: int, dX, dW1t,
                               stream=None):
    """dX = sdH sW1 dHq W1q and dW1t = sdH sX dHq^T Xq on 8-bit codes, one
    grouped launch (see include/coda.h)."""
    M, d = dHq.shape
    K1 = W1q.shape[1]
    _shape(W1q, (d, K1), "W1q")
    _shape(Xq, (M, K1), "Xq")
    _shape(dX, (M, K1), "dX")
    _shape(dW1t, (d, K1), "dW1t")
    _check(load_library().coda_gemm_res_prms_bwd_fp8(
        _h(dW1t), _ptr(dHq, U8, "dHq"), int(dh_format), _ptr(sdH, F32, "sdH"), _ptr(Xq, U8, "Xq"),
        _ptr(sX, F32, "sX"), _ptr(W1q, U8, "W1q"), _ptr(sW1, F32, "sW1"), int(w_format), _ptr(dX, BF, "dX"),
        _ptr(dW1t, BF, "dW1t"), M, K1, d, _stream(stream)), "coda_gemm_res_prms_bwd_fp8")


def coda_gemm_dgrad_rmsbwd_fp8(dPq, dp_format: int, sdP, W2q, w_format: int, sW2, H, g, c, dH, dgpart,
                               stream=None):
    """dgrad2 with the RMSNorm-backward epilogue on 8-bit operands (see include/coda.h)."""
    M, N2 = dPq.shape
    d = W2q.shape[1]
    _shape(W2q, (N2, d), "W2q")
    _shape(H, (M, d), "H")
    _shape(g, (d,), "g")
    _shape(c, (M,), "c")
    _shape(dH, (M, d), "dH")
    _shape(dgpart, (coda_dgpart_rows(M), d), "dgpart")
    _check(load_library().coda_gemm_dgrad_rmsbwd_fp8(
        _h(dPq), _ptr(dPq, U8, "dPq"), int(dp_format), _ptr(sdP, F32, "sdP"), _ptr(W2q, U8, "W2q"), int(w_format),
        _ptr(sW2, F32, "sW2"), _ptr(H, BF, "H"), _ptr(g, BF, "g"), _ptr(c, F32, "c"), _ptr(dH, BF, "dH"),
        _ptr(dgpart, F32, "dgpart"), M, N2, d, _stream(stream)), "coda_gemm_dgrad_rmsbwd_fp8")


def coda_gemm_res_prms_fp8(Xq, sX, W1q, sW1, R, H, psum, stream=None):
    """GEMM1 + residual + partial RMS on e4m3 operands (scales: 1-element
    fp32 device tensors, e.g. amax_scale[1:])."""
    M, K1 = Xq.shape
    d = W1q.shape[0]
    _shape(W1q, (d, K1), "W1q")
    _shape(R, (M, d), "R")
    _shape(H, (M, d), "H")
    _shape(psum, (M, coda_prms_num_tiles(d)), "psum")
    _check(load_library().coda_gemm_res_prms_fp8(_h(Xq), _ptr(Xq, U8, "Xq"), _ptr(sX, F32, "sX"),
                                                 _ptr(W1q, U8, "W1q"), _ptr(sW1, F32, "sW1"), _ptr(R, BF, "R"),
                                                 _ptr(H, BF, "H"), _ptr(psum, F32, "psum"), M, K1, d,
                                                 _stream(stream)), "coda_gemm_res_prms_fp8")


def coda_gemm_rowscale_swiglu_fp8(Hq, sH, W2gq, sW2, rstd, out, z_save=None, flags=CODA_EPI_SWIGLU, stream=None):
    M, d = Hq.shape
    N2 = W2gq.shape[0]
    _shape(W2gq, (N2, d), "W2gq")
    _shape(rstd, (M,), "rstd")
    _shape(out, (M, N2 // 2 if flags == CODA_EPI_SWIGLU else N2), "out")
    if z_save is not None:
        _shape(z_save, (M, N2), "z_save")
    _check(load_library().coda_gemm_rowscale_swiglu_fp8(_h(Hq), _ptr(Hq, U8, "Hq"), _ptr(sH, F32, "sH"),
                                                        _ptr(W2gq, U8, "W2gq"), _ptr(sW2, F32, "sW2"),
                                                        _ptr(rstd, F32, "rstd"), _ptr(out, BF, "out"),
                                                        _ptr(z_save, BF, "z_save"), M, d, N2, flags,
                                                        _stream(stream)), "coda_gemm_rowscale_swiglu_fp8")


def coda_lmhead_ce_workspace_bytes(M: int, d: int, V: int, with_grads: bool) -> int:
    return load_library().coda_lmhead_ce_workspace_bytes(M, d, V, int(with_grads))


def coda_lmhead_ce_row_offsets(M: int, d: int, V: int, with_grads: bool):
    """Byte offsets (label logits, row losses) of the per-row fp32 results
    that coda_lmhead_ce / coda_lmhead_ce_fp8 leave in their workspace."""
    a, b = _SZ(0), _SZ(0)
    _check(load_library().coda_lmhead_ce_row_offsets(M, d, V, int(with_grads), ctypes.byref(a), ctypes.byref(b)),
           "coda_lmhead_ce_row_offsets")
    return a.value, b.value


def coda_lmhead_ce_row_results(ws, M: int, d: int, V: int, with_grads: bool):
    """Views (label logits [M], row losses [M], fp32) into a workspace that a
    completed coda_lmhead_ce call with these sizes has filled."""
    a, b = coda_lmhead_ce_row_offsets(M, d, V, with_grads)
    flat = ws.view(torch.uint8).reshape(-1)
    return (flat[a:a + 4 * M].view(torch.float32), flat[b:b + 4 * M].view(torch.float32))


def coda_lmhead_ce(Hs, Wt, labels, loss, lse, argmax, dHs, dWt, ws, stream=None):
    M, d = Hs.shape
    V = Wt.shape[0]
    _shape(Wt, (V, d), "Wt")
    _shape(labels, (M,), "labels")
    _shape(loss, (1,), "loss")
    _shape(lse, (M,), "lse")
    if argmax is not None:
        _shape(argmax, (M,), "argmax")
    if dHs is not None:
        _shape(dHs, (M, d), "dHs")
        _shape(dWt, (V, d), "dWt")
    _check(load_library().coda_lmhead_ce(
        _h(Hs), _ptr(Hs, BF, "Hs"), _ptr(Wt, BF, "Wt"), _ptr(labels, I32, "labels"), _ptr(loss, F32, "loss"),
        _ptr(lse, F32, "lse"), _ptr(argmax, I32, "argmax"), _ptr(dHs, BF, "dHs"), _ptr(dWt, BF, "dWt"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), M, d, V, _stream(stream)), "coda_lmhead_ce")


def coda_lmhead_ce_fp8(Hq, sH, Wq, sW, labels, loss, lse, argmax, dHs, dWt, ws, stream=None):
    """coda_lmhead_ce on e4m3 codes of H and W (scales sH, sW: the scale
    element of coda_fp8_quantize's {amax, scale}); dL kept as e5m2 codes in
    the backward (see include/coda.h)."""
    M, d = Hq.shape
    V = Wq.shape[0]
    _shape(Wq, (V, d), "Wq")
    _shape(labels, (M,), "labels")
    _shape(loss, (1,), "loss")
    _shape(lse, (M,), "lse")
    if argmax is not None:
        _shape(argmax, (M,), "argmax")
    if dHs is not None:
        _shape(dHs, (M, d), "dHs")
        _shape(dWt, (V, d), "dWt")
    _check(load_library().coda_lmhead_ce_fp8(
        _h(Hq), _ptr(Hq, U8, "Hq"), _ptr(sH, F32, "sH"), _ptr(Wq, U8, "Wq"), _ptr(sW, F32, "sW"),
        _ptr(labels, I32, "labels"), _ptr(loss, F32, "loss"), _ptr(lse, F32, "lse"), _ptr(argmax, I32, "argmax"),
        _ptr(dHs, BF, "dHs"), _ptr(dWt, BF, "dWt"), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), M, d, V,
        _stream(stream)), "coda_lmhead_ce_fp8")


def coda_unfused_workspace_bytes(M: int, d: int, N2: int) -> int:
    return load_library().coda_unfused_workspace_bytes(M, d, N2)


def coda_unfused_fwd(X, W1t, R, g, W2t, H, rstd, Nrm, z, out, ws, eps=1e-5, flags=CODA_EPI_SWIGLU, stream=None):
    M, K1 = X.shape
    d = W1t.shape[0]
    N2 = W2t.shape[0]
    _check(load_library().coda_unfused_fwd(
        _h(X), _ptr(X, BF, "X"), _ptr(W1t, BF, "W1t"), _ptr(R, BF, "R"), _ptr(g, BF, "g"), _ptr(W2t, BF, "W2t"),
        _ptr(H, BF, "H"), _ptr(rstd, F32, "rstd"), _ptr(Nrm, BF, "Nrm"), _ptr(z, BF, "z"), _ptr(out, BF, "out"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), M, K1, d, N2, eps, flags, _stream(stream)),
        "coda_unfused_fwd")


def coda_unfused_bwd(dY, X, W1t, g, W2t, H, rstd, Nrm, z, dH, dX, dW1t, dW2t, dg, ws, stream=None):
    M, K1 = X.shape
    d = W1t.shape[0]
    N2 = W2t.shape[0]
    _check(load_library().coda_unfused_bwd(
        _h(X), _ptr(dY, BF, "dY"), _ptr(X, BF, "X"), _ptr(W1t, BF, "W1t"), _ptr(g, BF, "g"), _ptr(W2t, BF, "W2t"),
        _ptr(H, BF, "H"), _ptr(rstd, F32, "rstd"), _ptr(Nrm, BF, "Nrm"), _ptr(z, BF, "z"), _ptr(dH, BF, "dH"),
        _ptr(dX, BF, "dX"), _ptr(dW1t, BF, "dW1t"), _ptr(dW2t, BF, "dW2t"), _ptr(dg, F32, "dg"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), M, K1, d, N2, _stream(stream)),
        "coda_unfused_bwd")
