"""Plain fp64 definitions of every quantity on the CODA hot path.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing in the product
imports this file.

Notation follows the write-up: h is the residual-stream activation after the
first GEMM, r the RMSNorm row scale, g the RMSNorm weight, z the second GEMM's
output split into gate/up halves.  Shapes:
    X[M,K1]  W1t[d,K1]  R[M,d]  g[d]  W2t[N2,d]  (N2 = 2F, rows [0,F) gate,
    rows [F,2F) up)   dY[M,F]   H[M,d]  Wt[V,d]  labels[M]
Weights are in nn.Linear layout (row = output feature), so the mathematical
weight is the transpose: h = X @ W1t.T + R.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "matmul_nt", "gemm_residual", "rms_rstd", "partial_sumsq",
    "rstd_from_partials", "rmsnorm", "fold_weight", "rowscale_gemm", "silu",
    "silu_grad", "swiglu", "block_forward", "swiglu_backward",
    "block_backward", "stage_swiglu_bwd", "stage_dgrad2_rmsbwd",
    "stage_wgrad2", "stage_dgrad1", "stage_wgrad1", "logits_rows",
    "lse_rows", "lse_tile_partials", "lse_combine", "ce_forward",
    "ce_backward", "argmax_lowest", "ce_weight_grad_given_lse", "down_proj_dgrad",
    "swiglu_c_partials", "rope_angles", "rope_rotate_half", "qkv_rope", "e4m3_round", "e4m3_encode",
    "e4m3_decode", "e5m2_round", "e5m2_encode", "e5m2_decode", "fp8_scale", "fp8_quantize", "fp8_decode",
]


# ----------------------------------------------------------------------------
# GEMM and the first epilogue (residual add, partial RMS)
# ----------------------------------------------------------------------------

def matmul_nt(A: np.ndarray, Bt: np.ndarray) -> np.ndarray:
    """C[m,n] = sum_k A[m,k] * Bt[n,k]: the mainloop's contraction (尾声 section:
    "the mainloop does the tiled multiply-accumulate")."""
    return np.asarray(A, np.float64) @ np.asarray(Bt, np.float64).T


def gemm_residual(X, W1t, R):
    """h = X W1 + R: GEMM followed by the residual add (尾声 section, the
    GEMM-RMSNorm-GEMM pattern "matmul, residual add, RMS normalisation")."""
    return matmul_nt(X, W1t) + np.asarray(R, np.float64)


def rms_rstd(h, eps: float = 1e-5):
    """r[m] = 1 / sqrt(mean_k h[m,k]^2 + eps): the RMSNorm row scale r
    (尾声 section, "the row scale factor r is a scalar shared by the row").
    eps inside the square root, added to the mean square."""
    h = np.asarray(h, np.float64)
    return 1.0 / np.sqrt(np.mean(h * h, axis=1) + eps)


def partial_sumsq(h, bn: int):
    """psum[m,j] = sum over the j-th block of bn columns of h[m,:]^2: the
    block-local "partial RMS" that GEMM1's epilogue emits per output tile
    (尾声 section; 五种积木 section, block reduction "local RMS").  The last
    block may be ragged."""
    h = np.asarray(h, np.float64)
    M, d = h.shape
    T = -(-d // bn)
    out = np.zeros((M, T), np.float64)
    for j in range(T):
        blk = h[:, j * bn:(j + 1) * bn]
        out[:, j] = np.sum(blk * blk, axis=1)
    return out


def rstd_from_partials(psum, d: int, eps: float = 1e-5):
    """The "very light auxiliary reduction kernel" of the 尾声 section:
    merge per-tile partial sums of squares into r[m]."""
    psum = np.asarray(psum, np.float64)
    return 1.0 / np.sqrt(np.sum(psum, axis=1) / d + eps)


def rmsnorm(h, g, eps: float = 1e-5):
    """Standard RMSNorm: n[m,k] = r[m] * h[m,k] * g[k]."""
    r = rms_rstd(h, eps)
    return np.asarray(h, np.float64) * r[:, None] * np.asarray(g, np.float64)[None, :]


# ----------------------------------------------------------------------------
# second GEMM: folded RMSNorm weight, deferred row scale, SwiGLU
# ----------------------------------------------------------------------------

def fold_weight(W2t, g):
    """W2g = diag(g) W2, i.e. W2gt[n,k] = W2t[n,k] * g[k]: the RMSNorm weight
    broadcast (五种积木 section, vector load of the RMSNorm weight) folded into
    the second GEMM's B operand."""
    return np.asarray(W2t, np.float64) * np.asarray(g, np.float64)[None, :]


def rowscale_gemm(h, W2gt, rstd):
    """z[m,:] = r[m] * (h W2g)[m,:]: the row scale applied after the
    contraction, which is legal because r is one scalar per row (尾声 section,
    r "commutes with the following matmul")."""
    return np.asarray(rstd, np.float64)[:, None] * matmul_nt(h, W2gt)


def silu(x):
    """silu(x) = x * sigmoid(x) = x / (1 + exp(-x))."""
    x = np.asarray(x, np.float64)
    return x / (1.0 + np.exp(-x))


def silu_grad(x):
    """d silu / dx = s (1 + x (1 - s)) with s = sigmoid(x)."""
    x = np.asarray(x, np.float64)
    s = 1.0 / (1.0 + np.exp(-x))
    return s * (1.0 + x * (1.0 - s))


def swiglu(z):
    """out = silu(z_gate) * z_up, with z = [z_gate | z_up] split in two halves
    along the columns (SwiGLU activation, listed among the elementwise
    epilogue transforms of the 五种积木 section)."""
    z = np.asarray(z, np.float64)
    F = z.shape[1] // 2
    return silu(z[:, :F]) * z[:, F:]


def block_forward(X, W1t, R, g, W2t, eps: float = 1e-5, swiglu_act: bool = True):
    """Unfused forward of the GEMM-Residual-RMSNorm-GEMM(-SwiGLU) block:
    h = X W1 + R ; n = RMSNorm(h; g) ; z = n W2 ; out = SwiGLU(z) (or z).

    This is the textbook sequence of the 尾声 section ("three separate
    operators"), with no re-parameterisation: the RMSNorm is applied in full
    before the second GEMM.  Returns a dict with h, rstd, n, z, out.
    """
    h = gemm_residual(X, W1t, R)
    r = rms_rstd(h, eps)
    n = h * r[:, None] * np.asarray(g, np.float64)[None, :]
    z = matmul_nt(n, W2t)
    out = swiglu(z) if swiglu_act else z
    return {"h": h, "rstd": r, "n": n, "z": z, "out": out}


# ----------------------------------------------------------------------------
# backward: textbook chain rule (unfused) ...
# ----------------------------------------------------------------------------

def swiglu_backward(dY, z):
    """dZ = [dZ_gate | dZ_up] for out = silu(z_gate) * z_up."""
    z = np.asarray(z, np.float64)
    dY = np.asarray(dY, np.float64)
    F = z.shape[1] // 2
    zg, zu = z[:, :F], z[:, F:]
    return np.concatenate([dY * zu * silu_grad(zg), dY * silu(zg)], axis=1)


def block_backward(X, W1t, R, g, W2t, dY, eps: float = 1e-5, swiglu_act: bool = True):
    """Gradients of sum(out * dY) through the unfused block, by the plain
    chain rule in the order the forward was written (no fused identities):

        dZ from the SwiGLU derivative      dW2 = n^T dZ      dN = dZ W2^T
        dg = sum_m dN * (r h)              dn = dN * g
        dh = r dn - (r^3 / d) h sum_k(dn h)
        dR = dh          dX = dh W1^T      dW1 = X^T dh

    Returned in storage layout: dW1t[d,K1], dW2t[N2,d].  The write-up states
    (尾声 section) that the backward inherits the forward's block-local
    structure; the fused stage definitions below are checked against this.
    """
    X = np.asarray(X, np.float64)
    g = np.asarray(g, np.float64)
    W2t = np.asarray(W2t, np.float64)
    W1t = np.asarray(W1t, np.float64)
    fw = block_forward(X, W1t, R, g, W2t, eps, swiglu_act)
    h, r, n, z = fw["h"], fw["rstd"], fw["n"], fw["z"]
    d = h.shape[1]
    dZ = swiglu_backward(dY, z) if swiglu_act else np.asarray(dY, np.float64)
    dW2t = dZ.T @ n                      # dW2[k,n] = sum_m n[m,k] dZ[m,n]
    dN = dZ @ W2t                        # dN[m,k] = sum_n dZ[m,n] W2[k,n]
    xhat = h * r[:, None]
    dg = np.sum(dN * xhat, axis=0)
    dn = dN * g[None, :]
    proj = np.sum(dn * h, axis=1)
    dh = r[:, None] * dn - (r ** 3 / d)[:, None] * h * proj[:, None]
    dX = dh @ W1t                        # dX[m,i] = sum_k dh[m,k] W1[i,k]
    dW1t = dh.T @ X                      # dW1[i,k] = sum_m X[m,i] dh[m,k]
    return {"dZ": dZ, "dW2t": dW2t, "dg": dg, "dh": dh, "dR": dh,
            "dX": dX, "dW1t": dW1t, **fw}


# ----------------------------------------------------------------------------
# ... and the fused stage definitions, each fed by the previous stage's
# (possibly bf16-rounded) outputs.  These are what each GPU stage is meant to
# compute; tests pin their composition to block_backward above.
# ----------------------------------------------------------------------------

def stage_swiglu_bwd(dY, z, rstd, d: int):
    """SwiGLU backward stage: dP = r * dZ and c[m] = (r[m]^2 / d) *
    sum_n dZ[m,n] z[m,n], where d is the hidden width (the RMSNorm length).
    dP is the row-scaled gradient fed to the second GEMM's data and weight
    gradients; c is the scalar of the RMSNorm backward."""
    dZ = swiglu_backward(dY, z)
    r = np.asarray(rstd, np.float64)
    zz = np.asarray(z, np.float64)
    return r[:, None] * dZ, (r * r / d) * np.sum(dZ * zz, axis=1)


def down_proj_dgrad(dYb, W3t):
    """Gradient reaching the SwiGLU output through a down projection
    y = out W3 (nn.Linear layout W3t[d, F]): dY[m, j] = sum_k dYb[m, k]
    W3t[k, j]."""
    return np.asarray(dYb, np.float64) @ np.asarray(W3t, np.float64)


def swiglu_c_partials(dY, z, bn: int):
    """Per (row, tile of bn gate columns) partial sums of dZ * z over the gate
    columns of the tile and the matching up columns: the block reduction a
    SwiGLU-backward epilogue emits; sum_j of them times r^2 / d is c of
    stage_swiglu_bwd."""
    z = np.asarray(z, np.float64)
    F = z.shape[1] // 2
    dZ = swiglu_backward(dY, z)
    prod = dZ[:, :F] * z[:, :F] + dZ[:, F:] * z[:, F:]
    T = -(-F // bn)
    return np.stack([prod[:, j * bn:(j + 1) * bn].sum(axis=1) for j in range(T)], axis=1)


def stage_dgrad2_rmsbwd(dP, W2t, g, h, c):
    """RMSNorm backward in the epilogue of the second GEMM's data gradient:
    acc = dP W2^T ; dh = g * acc - c[m] h ; dg = sum_m acc * h."""
    acc = np.asarray(dP, np.float64) @ np.asarray(W2t, np.float64)
    h = np.asarray(h, np.float64)
    dh = acc * np.asarray(g, np.float64)[None, :] - np.asarray(c, np.float64)[:, None] * h
    dg = np.sum(acc * h, axis=0)
    return dh, dg


def stage_wgrad2(h, dP, g):
    """dW2t[n,k] = g[k] * sum_m h[m,k] dP[m,n] (storage layout [N2,d])."""
    return (np.asarray(dP, np.float64).T @ np.asarray(h, np.float64)) * np.asarray(g, np.float64)[None, :]


def stage_dgrad1(dh, W1t):
    """dX = dh W1^T, i.e. dX[m,i] = sum_k dh[m,k] W1t[k,i]."""
    return np.asarray(dh, np.float64) @ np.asarray(W1t, np.float64)


def stage_wgrad1(dh, X):
    """dW1t[k,i] = sum_m dh[m,k] X[m,i] (storage layout [d,K1])."""
    return np.asarray(dh, np.float64).T @ np.asarray(X, np.float64)


# ----------------------------------------------------------------------------
# LM-head cross-entropy with a blocked log-sum-exp
# ----------------------------------------------------------------------------

def logits_rows(H, Wt):
    """L[m,v] = sum_k H[m,k] Wt[v,k]."""
    return matmul_nt(H, Wt)


def lse_rows(L):
    """log sum_v exp(L[m,v]) computed with the max shift."""
    L = np.asarray(L, np.float64)
    mx = np.max(L, axis=1)
    return mx + np.log(np.sum(np.exp(L - mx[:, None]), axis=1))


def argmax_lowest(L):
    """Per-row argmax; on ties the lowest column index wins."""
    return np.argmax(np.asarray(L, np.float64), axis=1).astype(np.int64)


def lse_tile_partials(L, bn: int):
    """Block log-sum-exp statistics per (row, column tile): running max and
    sum of exp(L - max) (五种积木 section: block reduction "block log-sum-exp"
    and the stateful max / sum-exp statistics of online normalisation)."""
    L = np.asarray(L, np.float64)
    M, V = L.shape
    T = -(-V // bn)
    mx = np.zeros((M, T))
    se = np.zeros((M, T))
    for j in range(T):
        blk = L[:, j * bn:(j + 1) * bn]
        mx[:, j] = np.max(blk, axis=1)
        se[:, j] = np.sum(np.exp(blk - mx[:, j:j + 1]), axis=1)
    return mx, se


def lse_combine(mx, se):
    """Merge per-tile (max, sum-exp) pairs: lse = m* + log sum_j se_j
    exp(mx_j - m*), m* = max_j mx_j."""
    mx = np.asarray(mx, np.float64)
    se = np.asarray(se, np.float64)
    ms = np.max(mx, axis=1)
    return ms + np.log(np.sum(se * np.exp(mx - ms[:, None]), axis=1))


def ce_forward(H, Wt, labels, row_chunk: int = 256):
    """Mean softmax cross-entropy of logits H W against integer labels.

    Rows are processed in chunks so that no [M,V] array is ever held.
    Returns dict(loss, lse[M], zy[M], argmax[M]).
    """
    H = np.asarray(H, np.float64)
    Wt = np.asarray(Wt, np.float64)
    labels = np.asarray(labels, np.int64)
    M = H.shape[0]
    lse = np.zeros(M)
    zy = np.zeros(M)
    am = np.zeros(M, np.int64)
    for s in range(0, M, row_chunk):
        L = logits_rows(H[s:s + row_chunk], Wt)
        lse[s:s + row_chunk] = lse_rows(L)
        idx = labels[s:s + row_chunk]
        zy[s:s + row_chunk] = L[np.arange(L.shape[0]), idx]
        am[s:s + row_chunk] = argmax_lowest(L)
    return {"loss": float(np.mean(lse - zy)), "lse": lse, "zy": zy, "argmax": am}


def ce_backward(H, Wt, labels, row_chunk: int = 256):
    """dL = (softmax(L) - onehot(y)) / M ; dH = dL W^T ; dWt = dL^T H."""
    H = np.asarray(H, np.float64)
    Wt = np.asarray(Wt, np.float64)
    labels = np.asarray(labels, np.int64)
    M = H.shape[0]
    dH = np.zeros_like(H)
    dWt = np.zeros_like(Wt)
    for s in range(0, M, row_chunk):
        L = logits_rows(H[s:s + row_chunk], Wt)
        P = np.exp(L - lse_rows(L)[:, None])
        P[np.arange(L.shape[0]), labels[s:s + row_chunk]] -= 1.0
        P /= M
        dH[s:s + row_chunk] = P @ Wt
        dWt += P.T @ H[s:s + row_chunk]
    return {"dH": dH, "dWt": dWt}


def ce_weight_grad_given_lse(H, Wt_cols, cols, labels, lse, M: int):
    """Rows `cols` of dWt given each row's log-sum-exp:
    dWt[v] = sum_m ((exp(L[m,v] - lse[m]) - [y_m == v]) / M) H[m], with
    L[m,v] = H[m] . Wt[v].  Wt_cols holds the rows `cols` of Wt; M is the
    batch size of the mean (the rows of H may be all of them)."""
    H = np.asarray(H, np.float64)
    L = H @ np.asarray(Wt_cols, np.float64).T
    P = np.exp(L - np.asarray(lse, np.float64)[:, None])
    P -= (np.asarray(labels, np.int64)[:, None] == np.asarray(cols, np.int64)[None, :])
    return (P / M).T @ H


# ----------------------------------------------------------------------------
# rotary position embedding on the QKV projection (an elementwise epilogue
# transform in the write-up's 五种积木 section)
# ----------------------------------------------------------------------------

def rope_angles(positions, head_dim: int, base: float = 10000.0):
    """theta[p, i] = position_p * base^(-2 i / head_dim), i < head_dim / 2."""
    pos = np.asarray(positions, np.float64)
    i = np.arange(head_dim // 2, dtype=np.float64)
    return pos[:, None] * base ** (-2.0 * i / head_dim)[None, :]


def rope_rotate_half(x, positions, head_dim: int, base: float = 10000.0):
    """Rotate each head of x[M, heads * head_dim] (rotate-half pairing: element
    i pairs with i + head_dim/2): out_i = x_i cos - x_{i+D/2} sin,
    out_{i+D/2} = x_{i+D/2} cos + x_i sin, angles from row m's position."""
    x = np.asarray(x, np.float64)
    M, n = x.shape
    h = head_dim // 2
    th = rope_angles(positions, head_dim, base)
    cos, sin = np.cos(th), np.sin(th)
    out = np.empty_like(x)
    for s0 in range(0, n, head_dim):
        a = x[:, s0:s0 + h]
        b = x[:, s0 + h:s0 + head_dim]
        out[:, s0:s0 + h] = a * cos - b * sin
        out[:, s0 + h:s0 + head_dim] = b * cos + a * sin
    return out


def qkv_rope(X, Wqkv_t, n_q_heads: int, n_kv_heads: int, head_dim: int, seq_len: int, base: float = 10000.0):
    """qkv = X Wqkv (nn.Linear layout Wqkv_t[(Hq + 2 Hkv) D, d], columns q | k |
    v), then RoPE on the q and k heads at position m mod seq_len; v as is."""
    qkv = matmul_nt(X, Wqkv_t)
    M = qkv.shape[0]
    pos = np.arange(M) % seq_len
    rot = (n_q_heads + n_kv_heads) * head_dim
    out = qkv.copy()
    out[:, :rot] = rope_rotate_half(qkv[:, :rot], pos, head_dim, base)
    return out


# ----------------------------------------------------------------------------
# FP8 (e4m3) operands with per-tensor scaling (the write-up's 背景 section:
# FP8 makes the matmul faster, raising the relative cost of the memory-bound
# operations the epilogues absorb)
# ----------------------------------------------------------------------------
# e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; normal numbers
# 2^-6 .. 448, subnormals k * 2^-9; no infinities (saturating conversion).

E4M3_MAX = 448.0


def e4m3_round(x):
    """Round to the nearest e4m3 value, ties to even, saturating at +-448.
    Input: float64 array (the value to convert, already in the precision
    the conversion sees)."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)                       # below 2^-6: subnormal quantum 2^-9
    quantum = np.exp2(e - 3)
    q = np.round(a / quantum) * quantum         # np.round: half to even
    q = np.minimum(q, E4M3_MAX)
    return np.where(a > 0, np.sign(x) * q, 0.0 * x)


def e4m3_encode(v):
    """Byte encoding of e4m3 values (exactly representable, |v| <= 448)."""
    v = np.asarray(v, np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    out = np.zeros(a.shape, np.uint8)
    sub = (a > 0) & (a < 2.0 ** -6)
    out[sub] = (a[sub] / 2.0 ** -9).astype(np.uint8)
    nrm = a >= 2.0 ** -6
    e = np.floor(np.log2(a[nrm]))
    man = a[nrm] / np.exp2(e) - 1.0
    out[nrm] = ((e + 7).astype(np.uint8) << 3) | np.round(man * 8).astype(np.uint8)
    return out | sign


def e4m3_decode(b):
    """Value of e4m3 byte codes (the NaN codes 0x7f / 0xff are not produced
    by a saturating conversion)."""
    b = np.asarray(b, np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    return sign * val


E5M2_MAX = 57344.0


def e5m2_round(x):
    """Round to the nearest e5m2 value (sign, 5 exponent bits with bias 15, 2
    mantissa bits), ties to even, saturating at +-57344.  Normal exponents
    -14..15; below 2^-14 the subnormal quantum is 2^-16."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -14, 15)
    quantum = np.exp2(e - 2)
    q = np.round(a / quantum) * quantum         # np.round: half to even
    q = np.minimum(q, E5M2_MAX)
    return np.where(a > 0, np.sign(x) * q, 0.0 * x)


def e5m2_encode(v):
    """Byte encoding of e5m2 values (exactly representable, |v| <= 57344)."""
    v = np.asarray(v, np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    out = np.zeros(a.shape, np.uint8)
    sub = (a > 0) & (a < 2.0 ** -14)
    out[sub] = (a[sub] / 2.0 ** -16).astype(np.uint8)
    nrm = a >= 2.0 ** -14
    e = np.floor(np.log2(a[nrm]))
    man = a[nrm] / np.exp2(e) - 1.0
    out[nrm] = ((e + 15).astype(np.uint8) << 2) | np.round(man * 4).astype(np.uint8)
    return out | sign


def e5m2_decode(b):
    """Value of e5m2 byte codes with a finite value (exponent field < 31; the
    inf / NaN codes are not produced by a saturating conversion)."""
    b = np.asarray(b, np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 2) & 0x1F
    m = b & 0x3
    val = np.where(e == 0, m * 2.0 ** -16, (1.0 + m / 4.0) * np.exp2(e - 15.0))
    return sign * val


FP8_FORMATS = {"e4m3": (E4M3_MAX, e4m3_round, e4m3_encode, e4m3_decode),
               "e5m2": (E5M2_MAX, e5m2_round, e5m2_encode, e5m2_decode)}


def fp8_scale(x, fmt="e4m3"):
    """Per-tensor scale: the smallest power of two s with amax / s <= fmax
    (448 for e4m3, 57344 for e5m2), amax the largest magnitude of x in fp32,
    so the largest element lands in (fmax / 2, fmax]; 1 for an all-zero
    tensor; s >= 2^-126.  With a power of two, x / s and code * s are exact:
    every element is rounded once, by the format.  (The method's pages name
    FP8 only as a faster matmul and fix no scaling rule; this is the reading
    taken.)"""
    amax = float(np.max(np.abs(np.asarray(x, np.float32)))) if np.size(x) else 0.0
    if amax == 0.0:
        return np.float32(1.0)
    ma, ea = np.frexp(amax)                     # amax = ma * 2^ea, ma in [0.5, 1)
    mf, ef = np.frexp(FP8_FORMATS[fmt][0])      # fmax = 0.875 * 2^ef
    k = int(ea) - int(ef) + (1 if ma > mf else 0)
    return np.float32(2.0 ** max(k, -126))


def fp8_quantize(x, scale, fmt="e4m3"):
    """Codes of x / scale rounded to the format (x taken in fp32, as the
    quantiser reads it; the division by a power-of-two scale is exact)."""
    _, rnd, enc, _ = FP8_FORMATS[fmt]
    q = np.asarray(x, np.float32).astype(np.float64) / float(scale)
    return enc(rnd(q))


def fp8_decode(b, fmt="e4m3"):
    """Values of fp8 byte codes in the given format."""
    return FP8_FORMATS[fmt][3](b)
