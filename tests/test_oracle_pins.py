"""Pins for the fp64 oracle: every check here is independent of the oracle's
own formulas (brute force, closed forms, finite differences, an independent
autograd library, hand-worked fixtures), so a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them.

Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs" as
summarised by the Synced article (sections 尾声 and 五种积木).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# GEMM
# --------------------------------------------------------------------------

def brute_nt(A, Bt):
    M, K = A.shape
    N = Bt.shape[0]
    C = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += A[m, k] * Bt[n, k]
            C[m, n] = s
    return C


def test_matmul_bruteforce():
    r = rng(1)
    A = r.standard_normal((3, 5))
    Bt = r.standard_normal((4, 5))
    np.testing.assert_allclose(O.matmul_nt(A, Bt), brute_nt(A, Bt), rtol=1e-13, atol=1e-13)


def test_gemm_integer_known_answer():
    # integer-valued operands: the exact result is an integer matrix
    A = np.array([[1, 2, 3], [0, -1, 4]], float)
    Bt = np.array([[1, 0, 0], [0, 1, 0], [1, 1, 1], [2, -1, 0]], float)
    expect = np.array([[1, 2, 6, 0], [0, -1, 3, 1]], float)
    assert np.array_equal(O.matmul_nt(A, Bt), expect)
    R = np.ones((2, 4))
    assert np.array_equal(O.gemm_residual(A, Bt, R), expect + 1)


# --------------------------------------------------------------------------
# RMSNorm, partial RMS and the combine
# --------------------------------------------------------------------------

@pytest.mark.parametrize("c", [0.0, 0.5, 3.0, -2.0])
def test_rstd_constant_row(c):
    eps = 1e-5
    h = np.full((2, 37), c)
    np.testing.assert_allclose(O.rms_rstd(h, eps), 1.0 / math.sqrt(c * c + eps), rtol=1e-15)


def test_rstd_bruteforce_mean_not_sum():
    h = np.array([[3.0, 4.0, 0.0, 0.0]])
    # mean of squares = 25/4
    assert O.rms_rstd(h, 0.0)[0] == pytest.approx(1.0 / 2.5, rel=1e-15)


@pytest.mark.parametrize("bn", [1, 16, 100, 128, 300])
def test_partial_sumsq_tiling_invariance(bn):
    h = rng(2).standard_normal((5, 300))
    ps = O.partial_sumsq(h, bn)
    assert ps.shape == (5, -(-300 // bn))
    np.testing.assert_allclose(ps.sum(axis=1), (h * h).sum(axis=1), rtol=1e-13)
    # brute force of each block
    for j in range(ps.shape[1]):
        for m in range(5):
            s = 0.0
            for k in range(j * bn, min(300, (j + 1) * bn)):
                s += h[m, k] ** 2
            assert ps[m, j] == pytest.approx(s, rel=1e-13)


def test_rstd_from_partials_matches_rstd():
    h = rng(3).standard_normal((7, 96)) * 2
    for bn in (8, 32, 96):
        np.testing.assert_allclose(O.rstd_from_partials(O.partial_sumsq(h, bn), 96, 1e-5),
                                   O.rms_rstd(h, 1e-5), rtol=1e-14)


def test_rmsnorm_unit_rms():
    h = rng(4).standard_normal((6, 64)) * 7
    n = O.rmsnorm(h, np.ones(64), eps=0.0)
    np.testing.assert_allclose(np.mean(n * n, axis=1), 1.0, rtol=1e-13)


# --------------------------------------------------------------------------
# the re-parameterisation: fold g, defer r past the second GEMM
# --------------------------------------------------------------------------

def test_fold_and_rowscale_commute():
    r = rng(5)
    M, d, N2 = 6, 10, 14          # d != N2 so a transposed g would not broadcast
    h = r.standard_normal((M, d))
    g = r.uniform(0.5, 1.5, d)
    W2t = r.standard_normal((N2, d))
    rstd = O.rms_rstd(h, 1e-5)
    z_fused = O.rowscale_gemm(h, O.fold_weight(W2t, g), rstd)
    # unfused: explicit normalised activation, then a brute-force GEMM
    n = np.array([[h[m, k] * rstd[m] * g[k] for k in range(d)] for m in range(M)])
    np.testing.assert_allclose(z_fused, brute_nt(n, W2t), rtol=1e-12, atol=1e-13)


def test_fold_weight_bruteforce():
    W2t = np.arange(12, dtype=float).reshape(3, 4)
    g = np.array([1.0, 2.0, 0.5, -1.0])
    expect = np.array([[W2t[i, k] * g[k] for k in range(4)] for i in range(3)])
    assert np.array_equal(O.fold_weight(W2t, g), expect)


# --------------------------------------------------------------------------
# SwiGLU
# --------------------------------------------------------------------------

def test_silu_special_values():
    assert O.silu(0.0) == 0.0
    assert O.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert O.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(O.silu(-40.0)) < 1e-15
    assert O.silu_grad(0.0) == pytest.approx(0.5, rel=1e-15)


def test_silu_grad_finite_difference():
    x = np.linspace(-6, 6, 41)
    e = 1e-6
    fd = (O.silu(x + e) - O.silu(x - e)) / (2 * e)
    np.testing.assert_allclose(O.silu_grad(x), fd, rtol=1e-8, atol=1e-9)


def test_swiglu_halves():
    z = np.array([[0.0, 2.0, 5.0, 7.0],      # gate=[0,2], up=[5,7]
                  [30.0, -30.0, 3.0, 4.0]])
    out = O.swiglu(z)
    assert out.shape == (2, 2)
    assert out[0, 0] == 0.0                   # silu(0) * 5
    assert out[0, 1] == pytest.approx(2.0 / (1 + math.exp(-2.0)) * 7.0, rel=1e-15)
    assert out[1, 0] == pytest.approx(30.0 * 3.0, rel=1e-12)
    assert out[1, 1] == pytest.approx(-30.0 / (1 + math.exp(30.0)) * 4.0, rel=1e-12)


# --------------------------------------------------------------------------
# backward: finite differences and an independent autograd
# --------------------------------------------------------------------------

def _tiny_block(seed, swiglu_act=True, M=3, K1=4, d=5, F=3):
    r = rng(seed)
    N2 = 2 * F if swiglu_act else F
    return dict(X=r.standard_normal((M, K1)), W1t=r.standard_normal((d, K1)) * 0.5,
                R=r.standard_normal((M, d)), g=r.uniform(0.5, 1.5, d),
                W2t=r.standard_normal((N2, d)) * 0.5, dY=r.standard_normal((M, F)))


def _loss(p, swiglu_act):
    fw = O.block_forward(p["X"], p["W1t"], p["R"], p["g"], p["W2t"], 1e-5, swiglu_act)
    return float(np.sum(fw["out"] * p["dY"]))


@pytest.mark.parametrize("swiglu_act", [True, False])
def test_block_backward_finite_difference(swiglu_act):
    p = _tiny_block(7, swiglu_act)
    gr = O.block_backward(p["X"], p["W1t"], p["R"], p["g"], p["W2t"], p["dY"], 1e-5, swiglu_act)
    names = {"X": "dX", "W1t": "dW1t", "R": "dR", "g": "dg", "W2t": "dW2t"}
    e = 1e-6
    for k, gk in names.items():
        a = p[k]
        fd = np.zeros_like(a)
        for idx in np.ndindex(a.shape):
            old = a[idx]
            a[idx] = old + e
            lp = _loss(p, swiglu_act)
            a[idx] = old - e
            lm = _loss(p, swiglu_act)
            a[idx] = old
            fd[idx] = (lp - lm) / (2 * e)
        np.testing.assert_allclose(gr[gk], fd, rtol=1e-6, atol=1e-7, err_msg=k)


def test_block_backward_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    p = _tiny_block(11, True, M=4, K1=6, d=8, F=5)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    h = t["X"] @ t["W1t"].T + t["R"]
    n = torch.nn.functional.rms_norm(h, (8,), weight=t["g"], eps=1e-5)
    z = n @ t["W2t"].T
    out = torch.nn.functional.silu(z[:, :5]) * z[:, 5:]
    (out * t["dY"]).sum().backward()
    gr = O.block_backward(p["X"], p["W1t"], p["R"], p["g"], p["W2t"], p["dY"], 1e-5, True)
    for k, gk in {"X": "dX", "W1t": "dW1t", "R": "dR", "g": "dg", "W2t": "dW2t"}.items():
        np.testing.assert_allclose(gr[gk], t[k].grad.numpy(), rtol=1e-11, atol=1e-12, err_msg=k)
    np.testing.assert_allclose(O.block_forward(p["X"], p["W1t"], p["R"], p["g"], p["W2t"])["out"],
                               out.detach().numpy(), rtol=1e-12, atol=1e-13)


def test_fused_stages_compose_to_textbook_backward():
    """The fused stage definitions (dP, c, dh = g*acc - c*h, dg = sum acc*h,
    dW2 = g * h^T dP) reproduce the chain-rule backward exactly in fp64."""
    p = _tiny_block(13, True, M=6, K1=7, d=9, F=4)
    ref = O.block_backward(p["X"], p["W1t"], p["R"], p["g"], p["W2t"], p["dY"])
    h = O.gemm_residual(p["X"], p["W1t"], p["R"])
    rstd = O.rstd_from_partials(O.partial_sumsq(h, 4), 9, 1e-5)
    z = O.rowscale_gemm(h, O.fold_weight(p["W2t"], p["g"]), rstd)
    np.testing.assert_allclose(O.swiglu(z), ref["out"], rtol=1e-12, atol=1e-13)
    dP, c = O.stage_swiglu_bwd(p["dY"], z, rstd, 9)
    dh, dg = O.stage_dgrad2_rmsbwd(dP, p["W2t"], p["g"], h, c)
    np.testing.assert_allclose(dh, ref["dh"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dg, ref["dg"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(O.stage_wgrad2(h, dP, p["g"]), ref["dW2t"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(O.stage_dgrad1(dh, p["W1t"]), ref["dX"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(O.stage_wgrad1(dh, p["X"]), ref["dW1t"], rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------------------
# blocked log-sum-exp and cross-entropy
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bn", [1, 7, 64, 200])
def test_lse_combine_identity(bn):
    L = rng(17).standard_normal((4, 200)) * 5
    mx, se = O.lse_tile_partials(L, bn)
    direct = np.log(np.sum(np.exp(L), axis=1))
    np.testing.assert_allclose(O.lse_combine(mx, se), direct, rtol=1e-13)
    np.testing.assert_allclose(O.lse_rows(L), direct, rtol=1e-13)


def test_lse_large_values_and_constant_row():
    L = np.full((1, 10), 1000.0)
    assert O.lse_rows(L)[0] == pytest.approx(1000.0 + math.log(10.0), rel=1e-15)
    mx, se = O.lse_tile_partials(L, 3)
    assert O.lse_combine(mx, se)[0] == pytest.approx(1000.0 + math.log(10.0), rel=1e-15)


def test_ce_uniform_logits_is_log_v():
    V, d, M = 37, 8, 5
    out = O.ce_forward(rng(1).standard_normal((M, d)), np.zeros((V, d)), np.arange(M) % V)
    assert out["loss"] == pytest.approx(math.log(V), rel=1e-15)


def test_ce_argmax_tie_lowest_index():
    H = np.array([[1.0, 2.0]])
    Wt = np.array([[0.0, 0.0], [1.0, 1.0], [-1.0, 0.0], [1.0, 1.0]])  # columns 1 and 3 tie
    out = O.ce_forward(H, Wt, np.array([2]))
    assert out["argmax"][0] == 1


def test_ce_backward_finite_difference_and_row_sum():
    r = rng(19)
    M, d, V = 3, 4, 6
    H = r.standard_normal((M, d))
    Wt = r.standard_normal((V, d))
    y = np.array([0, 5, 2])
    gr = O.ce_backward(H, Wt, y, row_chunk=2)
    e = 1e-6
    for a, ga in ((H, gr["dH"]), (Wt, gr["dWt"])):
        fd = np.zeros_like(a)
        for idx in np.ndindex(a.shape):
            old = a[idx]
            a[idx] = old + e
            lp = O.ce_forward(H, Wt, y, row_chunk=2)["loss"]
            a[idx] = old - e
            lm = O.ce_forward(H, Wt, y, row_chunk=2)["loss"]
            a[idx] = old
            fd[idx] = (lp - lm) / (2 * e)
        np.testing.assert_allclose(ga, fd, rtol=1e-6, atol=1e-9)
    # softmax minus one-hot sums to zero per row: with Wt = I columns, dH rows sum to 0
    Wi = np.eye(V)
    g2 = O.ce_backward(r.standard_normal((M, V)), Wi, y)
    np.testing.assert_allclose(g2["dH"].sum(axis=1), 0.0, atol=1e-15)


def test_ce_expected_loss_statistics():
    """L = H W with H ~ N(0,1), W ~ N(0, 0.02), d = 2048: logits are
    N(0, s^2), s^2 = d * 0.02^2 = 0.8192, so E[lse] ~= ln V + s^2/2 for large V
    and E[loss] ~= ln V + s^2 / 2."""
    r = rng(23)
    M, d, V = 64, 2048, 8192
    H = r.standard_normal((M, d))
    Wt = r.standard_normal((V, d)) * 0.02
    y = r.integers(0, V, M)
    loss = O.ce_forward(H, Wt, y, row_chunk=64)["loss"]
    assert loss == pytest.approx(math.log(V) + 0.8192 / 2, abs=0.25)


# --------------------------------------------------------------------------
# hand-worked fixtures
# --------------------------------------------------------------------------

def test_golden_block_forward_worked_example():
    f = json.load(open(os.path.join(GOLD, "block_fwd_worked.json")))
    arr = {k: np.array(f[k], float) for k in ("X", "W1t", "R", "g", "W2t")}
    fw = O.block_forward(arr["X"], arr["W1t"], arr["R"], arr["g"], arr["W2t"], f["eps"], True)
    for k, v in f["expect"].items():
        np.testing.assert_allclose(fw[k], np.array(v), rtol=1e-14, atol=1e-15, err_msg=k)
    # the fused route reaches the same numbers
    h = O.gemm_residual(arr["X"], arr["W1t"], arr["R"])
    rstd = O.rstd_from_partials(O.partial_sumsq(h, 1), 2, f["eps"])
    z = O.rowscale_gemm(h, O.fold_weight(arr["W2t"], arr["g"]), rstd)
    np.testing.assert_allclose(O.swiglu(z), np.array(f["expect"]["out"]), rtol=1e-14)


def test_golden_ce_worked_example():
    f = json.load(open(os.path.join(GOLD, "ce_worked.json")))
    H, Wt, y = np.array(f["H"], float), np.array(f["Wt"], float), np.array(f["labels"])
    fw = O.ce_forward(H, Wt, y)
    ex = f["expect"]
    assert fw["loss"] == pytest.approx(ex["loss"], rel=1e-14)
    np.testing.assert_allclose(fw["lse"], ex["lse"], rtol=1e-14)
    assert list(fw["argmax"]) == ex["argmax"]
    bw = O.ce_backward(H, Wt, y)
    np.testing.assert_allclose(bw["dH"], ex["dH"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(bw["dWt"], ex["dWt"], rtol=1e-13, atol=1e-15)


def test_ce_weight_grad_given_lse_matches_full_backward():
    r = rng(29)
    M, d, V = 6, 5, 40
    H = r.standard_normal((M, d))
    Wt = r.standard_normal((V, d))
    y = np.array([0, 3, 3, 39, 7, 12])
    full = O.ce_backward(H, Wt, y)["dWt"]
    cols = np.array([3, 12, 0, 25])
    lse = O.lse_rows(O.logits_rows(H, Wt))
    np.testing.assert_allclose(O.ce_weight_grad_given_lse(H, Wt[cols], cols, y, lse, M), full[cols],
                               rtol=1e-12, atol=1e-14)


def test_down_proj_dgrad_bruteforce():
    r = rng(31)
    dYb = r.standard_normal((3, 4))
    W3t = r.standard_normal((4, 5))
    ref = np.array([[sum(dYb[m, k] * W3t[k, j] for k in range(4)) for j in range(5)] for m in range(3)])
    np.testing.assert_allclose(O.down_proj_dgrad(dYb, W3t), ref, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("bn", [1, 3, 8, 11])
def test_swiglu_c_partials_sum_to_c(bn):
    """the partials, brute-forced per tile, reproduce stage_swiglu_bwd's c"""
    r = rng(37)
    M, F, d = 4, 11, 7
    z = r.standard_normal((M, 2 * F))
    dY = r.standard_normal((M, F))
    rstd = r.uniform(0.5, 2.0, M)
    cp = O.swiglu_c_partials(dY, z, bn)
    assert cp.shape == (M, -(-F // bn))
    _, c = O.stage_swiglu_bwd(dY, z, rstd, d)
    np.testing.assert_allclose(cp.sum(axis=1) * rstd ** 2 / d, c, rtol=1e-12)
    # brute force of one tile from the SwiGLU derivative's closed form
    m, j = 2, 0
    tot = 0.0
    for n in range(0, min(bn, F)):
        zg, zu, dy = z[m, n], z[m, F + n], dY[m, n]
        s = 1 / (1 + math.exp(-zg))
        tot += dy * zu * s * (1 + zg * (1 - s)) * zg + dy * zg * s * zu
    assert cp[m, j] == pytest.approx(tot, rel=1e-12)


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------

def test_rope_position_zero_is_identity_and_norm_preserved():
    r = rng(41)
    x = r.standard_normal((5, 3 * 8))
    np.testing.assert_array_equal(O.rope_rotate_half(x, np.zeros(5), 8), x)
    y = O.rope_rotate_half(x, np.arange(5) * 37, 8)
    for s0 in range(0, 24, 8):
        for i in range(4):
            n_in = x[:, s0 + i] ** 2 + x[:, s0 + i + 4] ** 2
            n_out = y[:, s0 + i] ** 2 + y[:, s0 + i + 4] ** 2
            np.testing.assert_allclose(n_out, n_in, rtol=1e-13)


def test_rope_two_dim_closed_form():
    # head_dim 2: one pair, angle = position (base^0 = 1)
    x = np.array([[1.0, 2.0]])
    p = 0.7
    y = O.rope_rotate_half(x, np.array([p]), 2)
    np.testing.assert_allclose(y, [[math.cos(p) - 2 * math.sin(p), 2 * math.cos(p) + math.sin(p)]], rtol=1e-15)
    # head_dim 4, base 100: angles p and p / 10, pairs (0, 2) and (1, 3)
    th = O.rope_angles([3.0], 4, 100.0)
    np.testing.assert_allclose(th, [[3.0, 0.3]], rtol=1e-15)
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    a, b = 3.0, 0.3
    expect = [1 * math.cos(a) - 3 * math.sin(a), 2 * math.cos(b) - 4 * math.sin(b),
              3 * math.cos(a) + 1 * math.sin(a), 4 * math.cos(b) + 2 * math.sin(b)]
    np.testing.assert_allclose(O.rope_rotate_half(x, [3.0], 4, 100.0), [expect], rtol=1e-14)


def test_rope_scores_depend_only_on_relative_position():
    r = rng(43)
    q = r.standard_normal((1, 16))
    k = r.standard_normal((1, 16))
    def score(m, n):
        return float((O.rope_rotate_half(q, [m], 16) @ O.rope_rotate_half(k, [n], 16).T).item())
    for m, n, t in ((5, 2, 11), (100, 7, 1000), (0, 9, 3)):
        assert score(m, n) == pytest.approx(score(m + t, n + t), rel=1e-10, abs=1e-12)


def test_qkv_rope_rotates_q_and_k_only():
    r = rng(47)
    M, d, D, Hq, Hkv, S = 6, 8, 4, 2, 1, 3
    X = r.standard_normal((M, d))
    W = r.standard_normal(((Hq + 2 * Hkv) * D, d))
    out = O.qkv_rope(X, W, Hq, Hkv, D, S)
    plain = X @ W.T
    rot = (Hq + Hkv) * D
    np.testing.assert_allclose(out[:, rot:], plain[:, rot:], rtol=1e-14)
    pos = np.arange(M) % S
    np.testing.assert_allclose(out[:, :rot], O.rope_rotate_half(plain[:, :rot], pos, D), rtol=1e-13)
    # rows at position 0 (m = 0, 3) are not rotated
    np.testing.assert_allclose(out[[0, 3]], plain[[0, 3]], rtol=1e-14)


# --------------------------------------------------------------------------
# e4m3 (FP8) rounding and encoding, from the format's definition
# --------------------------------------------------------------------------

@pytest.mark.parametrize("v,code", [(1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (2.0 ** -6, 0x08),
                                    (2.0 ** -9, 0x01), (0.875 * 2.0 ** -6, 0x07), (1.125, 0x39), (0.0, 0x00),
                                    (240.0, 0x77), (3.5, 0x46)])
def test_e4m3_known_encodings(v, code):
    assert int(O.e4m3_encode(np.array([v]))[0]) == code
    assert O.e4m3_decode(np.array([code], np.uint8))[0] == v


def test_e4m3_every_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)   # skip the NaN codes
    vals = O.e4m3_decode(codes)
    assert np.array_equal(O.e4m3_round(vals), vals)
    back = O.e4m3_encode(vals)
    # +0 and -0 both decode to zero; everything else is exact
    nz = codes != 0x80
    assert np.array_equal(back[nz], codes[nz])


def test_e4m3_rounding_rules():
    # ties to even: 1 + 1/16 lies halfway between 1 and 1.125 -> 1 (even mantissa)
    assert O.e4m3_round(1.0625) == 1.0
    assert O.e4m3_round(1.1875) == 1.25          # halfway 1.125 / 1.25 -> even mantissa 2
    # half the smallest subnormal rounds to 0, a hair above rounds up
    assert O.e4m3_round(2.0 ** -10) == 0.0
    assert O.e4m3_round(2.0 ** -10 * 1.001) == 2.0 ** -9
    # saturation
    assert O.e4m3_round(1000.0) == 448.0 and O.e4m3_round(-465.0) == -448.0
    # relative error of normal numbers <= 2^-4
    x = np.random.default_rng(5).uniform(2.0 ** -6, 448, 10000)
    assert np.max(np.abs(O.e4m3_round(x) - x) / x) <= 2.0 ** -4 + 1e-15
    # nearest: no representable value is closer
    grid = np.unique(np.abs(O.e4m3_decode(np.arange(0, 127, dtype=np.uint8))))
    for v in np.random.default_rng(6).uniform(0, 448, 500):
        best = grid[np.argmin(np.abs(grid - v))]
        assert abs(O.e4m3_round(v) - v) <= abs(best - v) + 1e-15


# --------------------------------------------------------------------------
# e5m2 (FP8 for gradients) rounding and encoding, from the format's definition
# --------------------------------------------------------------------------

@pytest.mark.parametrize("v,code", [(1.0, 0x3C), (-1.0, 0xBC), (57344.0, 0x7B), (2.0 ** -14, 0x04),
                                    (2.0 ** -16, 0x01), (3 * 2.0 ** -16, 0x03), (1.25, 0x3D), (3.0, 0x42),
                                    (0.0, 0x00), (1536.0, 0x66)])
def test_e5m2_known_encodings(v, code):
    assert int(O.e5m2_encode(np.array([v]))[0]) == code
    assert O.e5m2_decode(np.array([code], np.uint8))[0] == v


def test_e5m2_every_code_round_trips():
    codes = np.array([c for c in range(256) if ((c >> 2) & 0x1F) != 31], np.uint8)   # skip inf / NaN
    vals = O.e5m2_decode(codes)
    assert np.array_equal(O.e5m2_round(vals), vals)
    back = O.e5m2_encode(vals)
    nz = codes != 0x80
    assert np.array_equal(back[nz], codes[nz])


def test_e5m2_rounding_rules():
    assert O.e5m2_round(1.125) == 1.0              # halfway 1 / 1.25 -> even mantissa 0
    assert O.e5m2_round(1.375) == 1.5              # halfway 1.25 / 1.5 -> even mantissa 2
    assert O.e5m2_round(2.0 ** -17) == 0.0          # half the smallest subnormal
    assert O.e5m2_round(2.0 ** -17 * 1.001) == 2.0 ** -16
    assert O.e5m2_round(60000.0) == 57344.0 and O.e5m2_round(-1e6) == -57344.0
    x = np.random.default_rng(7).uniform(2.0 ** -14, 57344, 10000)
    assert np.max(np.abs(O.e5m2_round(x) - x) / x) <= 2.0 ** -3 + 1e-15
    grid = np.unique(np.abs(O.e5m2_decode(np.array([c for c in range(124)], np.uint8))))
    for v in np.random.default_rng(8).uniform(0, 57344, 500):
        best = grid[np.argmin(np.abs(grid - v))]
        assert abs(O.e5m2_round(v) - v) <= abs(best - v) + 1e-12


def test_fp8_scale_and_quantize_per_format():
    x = np.array([[0.5, -3.0], [2.0, 0.25]], np.float32)
    # 3 / 448 lies in (2^-8, 2^-7]: 3 / 2^-7 = 384 <= 448 < 768
    assert O.fp8_scale(x, "e4m3") == np.float32(2.0 ** -7)
    # 3 / 57344 lies in (2^-15, 2^-14]: 3 / 2^-14 = 49152 <= 57344
    assert O.fp8_scale(x, "e5m2") == np.float32(2.0 ** -14)
    for fmt, top in (("e4m3", 448.0), ("e5m2", 57344.0)):
        s = O.fp8_scale(x, fmt)
        codes = O.fp8_quantize(x, s, fmt)
        vals = O.fp8_decode(codes, fmt)
        # the largest magnitude lands in the top binade, unsaturated
        assert top / 2 < np.max(np.abs(vals)) <= top
        # 0.5, 3, 2 and 0.25 are exact in both formats, and so is x / s
        assert np.array_equal(vals * s, x.astype(np.float64))
        assert O.fp8_scale(np.zeros((2, 2), np.float32), fmt) == 1.0


@pytest.mark.parametrize("fmt,top", [("e4m3", 448.0), ("e5m2", 57344.0)])
def test_fp8_scale_is_the_smallest_power_of_two(fmt, top):
    """Brute force over magnitudes spanning many binades, the exact edge
    fmax * 2^k, and the values just beside it: s is a power of two with
    amax / s <= fmax and amax / (s / 2) > fmax."""
    rng = np.random.default_rng(9)
    amaxes = np.concatenate([np.exp2(rng.uniform(-60, 60, 3000)),
                             top * np.exp2(np.arange(-20, 21, dtype=np.float64))]).astype(np.float32)
    amaxes = np.concatenate([amaxes, np.nextafter(amaxes, np.float32(np.inf)),
                             np.nextafter(amaxes, np.float32(0))])
    for a in amaxes:
        s = float(O.fp8_scale(np.array([a, -a / 3], np.float32), fmt))
        m, _ = np.frexp(s)
        assert m == 0.5                                   # a power of two
        assert float(a) / s <= top and float(a) / (s / 2) > top


def test_fp8_scale_floor_for_tiny_tensors():
    # amax = 2^-140 would want s = 2^-149 (e4m3): the floor 2^-126 keeps s
    # normal and amax / s far below 448
    x = np.array([2.0 ** -140], np.float32)
    assert O.fp8_scale(x, "e4m3") == np.float32(2.0 ** -126)


def test_fp8_scale_and_quantize():
    x = np.array([[0.5, -3.0], [1.5, 0.25]], np.float32)
    s = O.fp8_scale(x)
    assert s == np.float32(2.0 ** -7)
    q = O.fp8_quantize(x, s)
    # -3 / 2^-7 = -384 = -1.5 * 2^8: sign 1, exponent field 15, mantissa 4
    assert int(q[0, 1]) == 0xFC
    np.testing.assert_array_equal(O.e4m3_decode(q) * s, x)
    assert O.fp8_scale(np.zeros((2, 2))) == 1.0


def test_swiglu_backward_finite_difference():
    """dZ of sum(swiglu(z) * dY) against central differences, element by
    element, on both halves (a swapped half or a dropped silu' term fails)."""
    rng = np.random.default_rng(21)
    z = rng.normal(0, 2, (3, 8))
    dY = rng.normal(0, 1, (3, 4))
    dZ = O.swiglu_backward(dY, z)
    h = 1e-6
    for i in range(z.shape[0]):
        for j in range(z.shape[1]):
            zp, zm = z.copy(), z.copy()
            zp[i, j] += h
            zm[i, j] -= h
            fd = (np.sum(O.swiglu(zp) * dY) - np.sum(O.swiglu(zm) * dY)) / (2 * h)
            assert abs(dZ[i, j] - fd) <= 1e-7 * max(1.0, abs(fd))


def test_argmax_lowest_brute_force():
    """Small-integer rows with many ties: the first index of the row maximum,
    found by a plain loop."""
    rng = np.random.default_rng(22)
    L = rng.integers(-3, 4, (200, 9)).astype(np.float64)
    got = O.argmax_lowest(L)
    for r in range(L.shape[0]):
        best = 0
        for j in range(1, L.shape[1]):
            if L[r, j] > L[r, best]:
                best = j
        assert got[r] == best
