"""Rotation construction for OSCAR (oracle; test infrastructure only).

Source: QbitAI article on OSCAR, section "OSCAR aligns the rotation with
attention": the key rotation is derived from the query covariance Q^T Q, the
value rotation from the score-weighted value covariance V^T S^T S V, both
estimated offline per layer and per head; the final rotation is
R = U * Hadamard * bit-reversal, where U aligns the basis with the directions
attention uses, the Hadamard spreads outlier energy and the bit-reversal
balances the INT2 groups. The v2 abstract (arXiv 2605.17757v2) calls these
"attention-aware covariance targets" and "second-moment structures", and the
title's "spectral" is read as: U is the eigenbasis of that target.

Readings taken where the pages are silent:
* rotation acts on row vectors, x_rot = x @ R;
* U holds eigenvectors as columns, sorted by descending eigenvalue, each column
  signed so its largest-magnitude entry is positive (ties: lowest index);
* Hadamard is the Sylvester matrix of the full head_dim, normalised by
  1/sqrt(d); ``hadamard_block`` selects the block-diagonal alternative;
* the bit-reversal permutation matrix has P[i, bitrev(i)] = 1;
* clip thresholds are per channel: ratio * max over calibration rows of
  |(x @ R)_c|.
"""

import numpy as np


def sylvester_hadamard(n):
    """Unnormalised Sylvester Hadamard matrix: H_1 = [1], H_2m = [[H, H], [H, -H]]."""
    if n < 1 or n & (n - 1):
        raise ValueError("Hadamard order must be a power of two")
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def normalized_hadamard(d, block=None):
    """Orthogonal Hadamard factor of R: H_d / sqrt(d), or block-diagonal H_b / sqrt(b)."""
    b = d if block is None else block
    if d % b:
        raise ValueError("block must divide d")
    hb = sylvester_hadamard(b) / np.sqrt(b)
    out = np.zeros((d, d), dtype=np.float64)
    for s in range(0, d, b):
        out[s:s + b, s:s + b] = hb
    return out


def bit_reverse(i, bits):
    """Reverse the low ``bits`` bits of i."""
    r = 0
    for _ in range(bits):
        r = (r << 1) | (i & 1)
        i >>= 1
    return r


def bit_reversal_indices(d):
    bits = d.bit_length() - 1
    if 1 << bits != d:
        raise ValueError("d must be a power of two")
    return np.array([bit_reverse(i, bits) for i in range(d)], dtype=np.int64)


def bit_reversal_matrix(d):
    """Permutation matrix with P[i, bitrev(i)] = 1, so (x @ P)[bitrev(i)] = x[i]."""
    idx = bit_reversal_indices(d)
    p = np.zeros((d, d), dtype=np.float64)
    p[np.arange(d), idx] = 1.0
    return p


def spectral_basis(c):
    """Eigenvectors of the symmetric target c as columns, by descending eigenvalue.

    Sign convention: each column's largest-magnitude entry is positive.
    """
    c = np.asarray(c, dtype=np.float64)
    c = 0.5 * (c + c.T)
    w, u = np.linalg.eigh(c)
    order = np.argsort(-w, kind="stable")
    w = w[order]
    u = u[:, order].copy()
    for j in range(u.shape[1]):
        k = int(np.argmax(np.abs(u[:, j])))
        if u[k, j] < 0:
            u[:, j] = -u[:, j]
    return w, u


def key_covariance(q_rows):
    """Key target: Q^T Q over the calibration queries of the KV head's query group.

    q_rows: [n, d], the group's query heads stacked as rows.
    """
    q = np.asarray(q_rows, dtype=np.float64)
    return q.T @ q


def attention_scores(q_rows, k_rows, sm_scale):
    """Row-wise softmax of sm_scale * Q K^T (no mask: every key is visible)."""
    q = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k_rows, dtype=np.float64)
    logits = sm_scale * (q @ k.T)
    logits = logits - logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    return e / e.sum(axis=1, keepdims=True)


def value_covariance(q_rows, k_rows, v_rows, sm_scale):
    """Value target: V^T S^T S V = (S V)^T (S V) with S the calibration scores."""
    s = attention_scores(q_rows, k_rows, sm_scale)
    sv = s @ np.asarray(v_rows, dtype=np.float64)
    return sv.T @ sv


def oscar_rotation(target, hadamard_block=None):
    """R = U @ H @ P for one (layer, head) from its covariance target."""
    d = target.shape[0]
    _, u = spectral_basis(target)
    return u @ normalized_hadamard(d, hadamard_block) @ bit_reversal_matrix(d)


def hadamard_only_rotation(d, hadamard_block=None):
    """R = H @ P: the data-oblivious rotation that the pages set OSCAR against.

    The v2 abstract (arXiv 2605.17757v2) contrasts OSCAR with data-oblivious
    Hadamard rotations ("Hadamard-only INT2", "QuaRot-style INT2"), and the
    QbitAI article (section "OSCAR aligns the rotation with attention") says a
    plain Hadamard spreads outliers without knowing which directions attention
    uses. The ablation keeps everything else of OSCAR (bit-reversal, clipping,
    grouping) and drops U, i.e. U = I.
    """
    return normalized_hadamard(d, hadamard_block) @ bit_reversal_matrix(d)


def clip_thresholds(x_rows, r, ratio):
    """Per-channel clip threshold: ratio * max_rows |(x @ R)_c|."""
    xr = np.asarray(x_rows, dtype=np.float64) @ np.asarray(r, dtype=np.float64)
    return ratio * np.abs(xr).max(axis=0)
