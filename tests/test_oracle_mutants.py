"""Planted mistakes in the oracle (on the CPU): each mutant replaces one
oracle function with a plausible wrong version, and at least one pin in
test_oracle_pins.py must then fail.  This shows the pins are discriminating,
not restatements of the oracle's own formulas."""
import numpy as np
import pytest

import oracle as O
import oracle.coda_oracle as OC
from tests import test_oracle_pins as P


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(OC, name, fn)
    monkeypatch.setattr(O, name, fn)


def _fails(check, *args):
    with pytest.raises((AssertionError, ValueError, IndexError)):
        check(*args)


def test_mutant_rstd_sum_instead_of_mean(monkeypatch):
    _patch(monkeypatch, "rms_rstd",
           lambda h, eps=1e-5: 1.0 / np.sqrt(np.sum(np.asarray(h) ** 2, axis=1) + eps))
    _fails(P.test_rstd_constant_row, 0.5)


def test_mutant_eps_outside_sqrt(monkeypatch):
    _patch(monkeypatch, "rms_rstd",
           lambda h, eps=1e-5: 1.0 / (np.sqrt(np.mean(np.asarray(h) ** 2, axis=1)) + eps))
    _fails(P.test_rstd_constant_row, 0.0)


def test_mutant_fold_on_wrong_axis(monkeypatch):
    _patch(monkeypatch, "fold_weight",
           lambda W2t, g: np.asarray(W2t) * np.asarray(g)[: np.asarray(W2t).shape[0], None])
    _fails(P.test_fold_and_rowscale_commute)


def test_mutant_swiglu_halves_swapped(monkeypatch):
    def bad(z):
        F = z.shape[1] // 2
        return OC.silu(z[:, F:]) * z[:, :F]
    _patch(monkeypatch, "swiglu", bad)
    _fails(P.test_swiglu_halves)


def test_mutant_matmul_not_transposed(monkeypatch):
    _patch(monkeypatch, "matmul_nt", lambda A, Bt: np.asarray(A) @ np.asarray(Bt))
    _fails(P.test_matmul_bruteforce)


def _bad_block_backward(drop_projection=False, flip_sign=False):
    good = OC.block_backward

    def bad(X, W1t, R, g, W2t, dY, eps=1e-5, swiglu_act=True):
        out = good(X, W1t, R, g, W2t, dY, eps, swiglu_act)
        h, r = out["h"], out["rstd"]
        d = h.shape[1]
        dN = out["dZ"] @ np.asarray(W2t)
        dn = dN * np.asarray(g)[None, :]
        proj = np.sum(dn * h, axis=1)
        if drop_projection:
            dh = r[:, None] * dn
        else:
            dh = r[:, None] * dn + (r ** 3 / d)[:, None] * h * proj[:, None]
        out = dict(out)
        out["dh"] = out["dR"] = dh
        out["dX"] = dh @ np.asarray(W1t)
        out["dW1t"] = dh.T @ np.asarray(X)
        return out
    return bad


def test_mutant_rmsnorm_bwd_missing_projection(monkeypatch):
    _patch(monkeypatch, "block_backward", _bad_block_backward(drop_projection=True))
    _fails(P.test_block_backward_finite_difference, True)


def test_mutant_rmsnorm_bwd_sign(monkeypatch):
    _patch(monkeypatch, "block_backward", _bad_block_backward(flip_sign=True))
    _fails(P.test_block_backward_finite_difference, False)


def test_mutant_c_missing_over_d(monkeypatch):
    good = OC.stage_swiglu_bwd
    _patch(monkeypatch, "stage_swiglu_bwd",
           lambda dY, z, rstd, d: (lambda a: (a[0], a[1] * d))(good(dY, z, rstd, d)))
    _fails(P.test_fused_stages_compose_to_textbook_backward)


def test_mutant_dg_with_extra_g(monkeypatch):
    good = OC.stage_dgrad2_rmsbwd

    def bad(dP, W2t, g, h, c):
        dh, dg = good(dP, W2t, g, h, c)
        return dh, dg * np.asarray(g)
    _patch(monkeypatch, "stage_dgrad2_rmsbwd", bad)
    _fails(P.test_fused_stages_compose_to_textbook_backward)


def test_mutant_lse_combine_unweighted(monkeypatch):
    _patch(monkeypatch, "lse_combine",
           lambda mx, se: np.max(mx, axis=1) + np.log(np.sum(se, axis=1)))
    _fails(P.test_lse_combine_identity, 7)


def test_mutant_argmax_highest_on_tie(monkeypatch):
    _patch(monkeypatch, "argmax_lowest",
           lambda L: (L.shape[1] - 1 - np.argmax(L[:, ::-1], axis=1)).astype(np.int64))
    _fails(P.test_ce_argmax_tie_lowest_index)


def test_mutant_ce_grad_missing_mean(monkeypatch):
    good = OC.ce_backward

    def bad(H, Wt, labels, row_chunk=256):
        out = good(H, Wt, labels, row_chunk)
        M = np.asarray(H).shape[0]
        return {"dH": out["dH"] * M, "dWt": out["dWt"] * M}
    _patch(monkeypatch, "ce_backward", bad)
    _fails(P.test_ce_backward_finite_difference_and_row_sum)


def test_mutant_rope_interleaved_pairs(monkeypatch):
    """pairing (2i, 2i+1) instead of (i, i + D/2) must be caught"""
    def bad(x, positions, head_dim, base=10000.0):
        x = np.asarray(x, np.float64)
        th = OC.rope_angles(positions, head_dim, base)
        out = x.copy()
        for s0 in range(0, x.shape[1], head_dim):
            a = x[:, s0:s0 + head_dim:2]
            b = x[:, s0 + 1:s0 + head_dim:2]
            out[:, s0:s0 + head_dim:2] = a * np.cos(th) - b * np.sin(th)
            out[:, s0 + 1:s0 + head_dim:2] = b * np.cos(th) + a * np.sin(th)
        return out
    _patch(monkeypatch, "rope_rotate_half", bad)
    _fails(P.test_rope_two_dim_closed_form)


def test_mutant_rope_rotation_sign(monkeypatch):
    good = OC.rope_rotate_half
    _patch(monkeypatch, "rope_rotate_half",
           lambda x, positions, head_dim, base=10000.0: good(x, -np.asarray(positions, float), head_dim, base))
    _fails(P.test_rope_two_dim_closed_form)


def test_mutant_rope_exponent(monkeypatch):
    """theta_i = p base^(-i/D) instead of base^(-2i/D)"""
    _patch(monkeypatch, "rope_angles",
           lambda positions, head_dim, base=10000.0: np.asarray(positions, float)[:, None]
           * base ** (-np.arange(head_dim // 2) / head_dim)[None, :])
    _fails(P.test_rope_two_dim_closed_form)


def test_mutant_e4m3_ties_away_from_zero(monkeypatch):
    good = OC.e4m3_round

    def bad(x):
        x = np.asarray(x, np.float64)
        a = np.abs(x)
        e = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6, 8)
        quantum = np.exp2(e - 3)
        q = np.minimum(np.floor(a / quantum + 0.5) * quantum, 448.0)
        return np.where(a > 0, np.sign(x) * q, 0.0 * x)
    _patch(monkeypatch, "e4m3_round", bad)
    _fails(P.test_e4m3_rounding_rules)
    assert good is not bad


def test_mutant_e5m2_ties_away_from_zero(monkeypatch):
    def bad(x):
        x = np.asarray(x, np.float64)
        a = np.abs(x)
        e = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -14, 15)
        quantum = np.exp2(e - 2)
        q = np.minimum(np.floor(a / quantum + 0.5) * quantum, 57344.0)
        return np.where(a > 0, np.sign(x) * q, 0.0 * x)
    _patch(monkeypatch, "e5m2_round", bad)
    _fails(P.test_e5m2_rounding_rules)


def test_mutant_e5m2_exponent_bias(monkeypatch):
    good = OC.e5m2_encode

    def bad(v):
        return good(np.asarray(v, np.float64) * 2.0)     # an exponent bias off by one
    _patch(monkeypatch, "e5m2_encode", bad)
    _fails(lambda: P.test_e5m2_known_encodings(1.0, 0x3C))


def test_mutant_fp8_scale_one_binade_high(monkeypatch):
    good = OC.fp8_scale
    _patch(monkeypatch, "fp8_scale", lambda x, fmt="e4m3": np.float32(2.0 * good(x, fmt)))
    _fails(P.test_fp8_scale_is_the_smallest_power_of_two, "e4m3", 448.0)


def test_mutant_fp8_scale_edge_exclusive(monkeypatch):
    """amax exactly fmax * 2^k must take s = 2^k, not 2^(k+1)."""
    def bad(x, fmt="e4m3"):
        amax = float(np.max(np.abs(np.asarray(x, np.float32))))
        if amax == 0.0:
            return np.float32(1.0)
        k = int(np.floor(np.log2(amax / OC.FP8_FORMATS[fmt][0]))) + 1
        return np.float32(2.0 ** k)
    _patch(monkeypatch, "fp8_scale", bad)
    _fails(P.test_fp8_scale_is_the_smallest_power_of_two, "e5m2", 57344.0)


def test_mutant_fp8_scale_amax_over_fmax(monkeypatch):
    """The plain ratio amax / fmax (not a power of two) fails the pins."""
    _patch(monkeypatch, "fp8_scale", lambda x, fmt="e4m3": np.float32(
        float(np.max(np.abs(np.asarray(x, np.float32)))) / OC.FP8_FORMATS[fmt][0]))
    _fails(P.test_fp8_scale_and_quantize)
