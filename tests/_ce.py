"""Checks shared by the LM-head cross-entropy parity tests: label placement
on the kernels' tile and chunk edges, the argmax rule (lowest column among
maximal logits, either index within the fp32 error), and the per-row label
logit / row loss read back from the workspace (Synced write-up, section
五种积木: the label logit is gathered by the epilogue of the vocabulary tile
that holds the label)."""
import numpy as np
import torch

import oracle as O
from tests._parity import assert_elem, f64

CHUNK = 32768  # vocabulary columns per backward chunk (the library's default)


def edge_labels(V, chunk=CHUNK):
    """Vocabulary columns on the edges the kernels split at: the 128-column
    partials, the 256-column tiles, the backward chunks, and the last tile."""
    cols = {0, 1, 127, 128, 129, 255, 256, 257, V - 1, V - 2, V - 128, V - 129, ((V - 1) // 256) * 256,
            ((V - 1) // 256) * 256 - 1}
    for c0 in range(chunk, V, chunk):
        cols |= {c0 - 1, c0, c0 + 1}
    return sorted(c for c in cols if 0 <= c < V)


def with_edge_labels(labels, V, chunk=CHUNK):
    lab = labels.clone()
    e = edge_labels(V, chunk)
    n = min(len(e), lab.numel())
    lab[:n] = torch.tensor(e[:n], dtype=lab.dtype)
    return lab


def check_argmax(gpu_am, H, Wt, tol_gap=1e-3, L=None):
    L = O.logits_rows(H, Wt) if L is None else L
    ref = O.argmax_lowest(L)
    srt = np.sort(L, axis=1)
    gap = srt[:, -1] - srt[:, -2]
    decided = gap > tol_gap
    got = gpu_am.cpu().numpy().astype(np.int64)
    assert np.array_equal(got[decided], ref[decided])
    # undecided rows: the GPU's choice must be a maximal column within the gap
    for m in np.where(~decided)[0]:
        assert L[m, got[m]] >= srt[m, -1] - tol_gap
    return int(decided.sum())


def check_label_rows(zy_gpu, row_loss_gpu, L, y, lse_ref, rows=None, tol_gap=1e-4):
    """Per row: the gathered label logit is L[m, y_m] (elementwise), the
    column it came from is y_m (the nearest logit of the row to the GPU's
    value is column y_m wherever no other column lies within tol_gap of it;
    returns the number of such rows), and the row loss is lse - L[m, y_m].
    Exactness of the index on every row is the known-answer test's job."""
    y = np.asarray(y, np.int64)
    zy = f64(zy_gpu) if rows is None else f64(zy_gpu)[rows]
    rl = f64(row_loss_gpu) if rows is None else f64(row_loss_gpu)[rows]
    ref_zy = L[np.arange(L.shape[0]), y]
    assert_elem(zy, ref_zy, "label logit")
    check_row_loss(rl, lse_ref, ref_zy)
    dist = np.abs(L - zy[:, None])
    nearest = np.argmin(dist, axis=1)
    dist[np.arange(L.shape[0]), y] = np.inf
    unique = dist.min(axis=1) > tol_gap
    assert np.array_equal(nearest[unique], y[unique])
    return int(unique.sum())


def check_row_loss(row_loss, lse_ref, zy_ref):
    """Row loss lse - L[m, y_m] to 1e-4 relative, plus the fp32 rounding of
    the two terms it is the difference of (it can cancel to near zero when
    the label holds almost all of the row's probability)."""
    rl, lse_ref, zy_ref = f64(row_loss), f64(lse_ref), f64(zy_ref)
    ref = lse_ref - zy_ref
    bound = 1e-4 * np.abs(ref) + 2.0 ** -20 * (np.abs(lse_ref) + np.abs(zy_ref))
    bad = np.abs(rl - ref) > bound
    assert not bad.any(), f"row loss off on {int(bad.sum())} rows, first {np.flatnonzero(bad)[:5]}"


def known_answer_ce(M, d, V, seed, base=128):
    """Integer logits with a known label logit and argmax on every row.

    A fixed permutation pi of [0, V) is written in base `base` into the
    first columns of W (one digit per column, digits < base exact in bf16 for
    base 128, and in e4m3 for base 8 after its power-of-two scale), and row m
    of H holds a_m * base^i there (a_m = +1 on even rows, -1 on odd ones;
    powers of two), zeros elsewhere.  Every logit is then the exact integer
    L[m, v] = a_m pi(v) (|L| < 2^18, so any fp32 summation order is exact):
    the label logit must be a_m pi(y_m) bit for bit, and the argmax
    pi^-1(V - 1) on even rows, pi^-1(0) on odd ones, with no ties."""
    nd = 1
    while base ** nd < V:
        nd += 1
    assert d >= nd and V <= 2 ** 18
    r = np.random.default_rng(seed)
    pi = r.permutation(V)
    W = np.zeros((V, d), np.float32)
    a = np.where(np.arange(M) % 2 == 0, 1.0, -1.0).astype(np.float32)
    H = np.zeros((M, d), np.float32)
    for i in range(nd):
        W[:, i] = (pi // base ** i) % base
        H[:, i] = a * float(base ** i)
    labels = r.integers(0, V, size=M)
    e = edge_labels(V)
    labels[:min(M, len(e))] = e[:min(M, len(e))]
    inv = np.argsort(pi)
    zy = a.astype(np.float64) * pi[labels]
    am = np.where(a > 0, inv[V - 1], inv[0])
    bf = torch.bfloat16
    return (torch.from_numpy(H).to(bf), torch.from_numpy(W).to(bf), torch.from_numpy(labels.astype(np.int32)),
            zy, am)


def known_answer_logits(Wt, M, base=128):
    """The integer logits a_m pi(v) of known_answer_ce, read back from W's
    digit columns."""
    Wf = f64(Wt)
    nd = 1
    while base ** nd < Wf.shape[0]:
        nd += 1
    piv = sum(Wf[:, i] * base ** i for i in range(nd))
    return np.where(np.arange(M) % 2 == 0, 1.0, -1.0)[:, None] * piv[None, :]
