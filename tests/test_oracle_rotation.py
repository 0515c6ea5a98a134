"""Pins of oracle.rotation against closed forms, textbook/library routines and hand-worked values.

Source of what is pinned: QbitAI article on OSCAR, section "OSCAR aligns the
rotation with attention" (key target Q^T Q, value target V^T S^T S V,
R = U * Hadamard * bit-reversal); arXiv 2605.17757 abstracts (fixed per-layer
rotations and clipping thresholds).
"""

import os

import numpy as np
import pytest
import scipy.linalg

from oracle import calibrate, rotation

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("d", [1, 2, 4, 8, 16, 64, 128])
def test_hadamard_matches_scipy_and_is_orthogonal(d):
    h = rotation.normalized_hadamard(d)
    np.testing.assert_array_equal(rotation.sylvester_hadamard(d), scipy.linalg.hadamard(d))
    assert np.abs(h @ h.T - np.eye(d)).max() < 1e-12


def test_hadamard_block_variant():
    h = rotation.normalized_hadamard(8, block=4)
    assert np.abs(h[:4, 4:]).max() == 0 and np.abs(h[4:, :4]).max() == 0
    np.testing.assert_allclose(h[:4, :4], scipy.linalg.hadamard(4) / 2.0)


def test_bit_reversal_textbook_values_and_involution():
    assert list(rotation.bit_reversal_indices(8)) == [0, 4, 2, 6, 1, 5, 3, 7]
    assert list(rotation.bit_reversal_indices(4)) == [0, 2, 1, 3]
    for d in (2, 16, 64, 128):
        idx = rotation.bit_reversal_indices(d)
        assert sorted(idx) == list(range(d))
        np.testing.assert_array_equal(idx[idx], np.arange(d))
        p = rotation.bit_reversal_matrix(d)
        np.testing.assert_array_equal(p @ p, np.eye(d))


def test_spectral_basis_order_sign_and_eigen_equation():
    rng = np.random.default_rng(7)
    a = rng.standard_normal((40, 16))
    c = a.T @ a
    w, u = rotation.spectral_basis(c)
    assert np.all(np.diff(w) <= 0)
    assert np.abs(c @ u - u * w[None, :]).max() < 1e-9
    assert np.abs(u.T @ u - np.eye(16)).max() < 1e-12
    for j in range(16):
        k = np.argmax(np.abs(u[:, j]))
        assert u[k, j] > 0


def test_spectral_basis_of_diagonal_is_sorted_permutation():
    w, u = rotation.spectral_basis(np.diag([1.0, 4.0, 2.0, 3.0]))
    np.testing.assert_allclose(w, [4, 3, 2, 1])
    np.testing.assert_array_equal(u, np.eye(4)[:, [1, 3, 2, 0]])


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = np.array([float(x) for x in rest])
    return vals


def test_rotation_hand_worked_d4():
    g = _read_golden("rotation_d4.txt")
    r = rotation.oscar_rotation(np.diag(g["C_diag"]))
    np.testing.assert_allclose(g["x"] @ r, g["x_rot"], atol=1e-12)
    # a transposed U or a transposed product gives a different answer
    u = np.eye(4)[:, [1, 3, 2, 0]]
    wrong = g["x"] @ (u.T @ rotation.normalized_hadamard(4) @ rotation.bit_reversal_matrix(4))
    assert np.abs(wrong - g["x_rot"]).max() > 0.5


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_orthogonal_and_logit_invariant(d):
    rng = np.random.default_rng(d)
    q = rng.standard_normal((256, d))
    k = rng.standard_normal((64, d))
    r = rotation.oscar_rotation(rotation.key_covariance(q))
    assert np.abs(r @ r.T - np.eye(d)).max() < 1e-10
    assert np.abs((q @ r) @ (k @ r).T - q @ k.T).max() < 1e-10


def test_rotation_identity_cases():
    assert rotation.oscar_rotation(np.array([[2.0]])).tolist() == [[1.0]]
    # U = I (diagonal, already sorted) => R = H P exactly
    r = rotation.oscar_rotation(np.diag([8.0, 7, 6, 5, 4, 3, 2, 1]))
    np.testing.assert_allclose(r, rotation.normalized_hadamard(8) @ rotation.bit_reversal_matrix(8), atol=1e-15)


def test_key_covariance_hand_worked():
    np.testing.assert_array_equal(rotation.key_covariance(np.array([[1.0, 2.0], [3.0, 4.0]])),
                                  [[10.0, 14.0], [14.0, 20.0]])


def test_value_covariance_closed_forms():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((5, 4))
    # one key: every score row is [1] so S V repeats v
    v1 = rng.standard_normal((1, 4))
    c = rotation.value_covariance(q, rng.standard_normal((1, 4)), v1, 0.5)
    np.testing.assert_allclose(c, 5 * v1.T @ v1, rtol=1e-12)
    # all keys zero: uniform scores, S V = mean(V) on every row
    v = rng.standard_normal((3, 4))
    c = rotation.value_covariance(q, np.zeros((3, 4)), v, 0.5)
    mu = v.mean(axis=0, keepdims=True)
    np.testing.assert_allclose(c, 5 * mu.T @ mu, rtol=1e-12)
    # two keys, known logits: row score = softmax(sm * [q.k0, q.k1])
    qq = np.array([[2.0, 0.0]])
    kk = np.array([[1.0, 0.0], [0.0, 0.0]])
    vv = np.array([[1.0, 0.0], [0.0, 1.0]])
    s0 = np.exp(1.0) / (np.exp(1.0) + 1.0)   # sm_scale 0.5 -> logits (1, 0)
    c = rotation.value_covariance(qq, kk, vv, 0.5)
    sv = np.array([[s0, 1 - s0]])
    np.testing.assert_allclose(c, sv.T @ sv, rtol=1e-12)


def test_clip_thresholds_hand_worked():
    t = rotation.clip_thresholds(np.array([[1.0, -5.0], [-2.0, 3.0]]), np.eye(2), 0.9)
    np.testing.assert_allclose(t, [1.8, 4.5])


def test_calibrate_layer_groups_queries_by_kv_head():
    rng = np.random.default_rng(11)
    d = 8
    q = rng.standard_normal((50, 4, d))
    k = rng.standard_normal((30, 2, d))
    v = rng.standard_normal((30, 2, d))
    rk, rv, tk, tv = calibrate.calibrate_layer(q, k, v, d ** -0.5, 0.9)
    # KV head 1 serves query heads 2, 3
    q1 = q[:, 2:4, :].reshape(-1, d)
    np.testing.assert_allclose(rk[1], rotation.oscar_rotation(q1.T @ q1), atol=1e-12)
    for h in range(2):
        assert np.abs(rk[h] @ rk[h].T - np.eye(d)).max() < 1e-10
        assert np.abs(rv[h] @ rv[h].T - np.eye(d)).max() < 1e-10
        assert np.all(tk[h] > 0) and np.all(tv[h] > 0)
        assert np.all(tk[h] <= 0.9 * np.abs(k[:, h] @ rk[h]).max(axis=0) + 1e-12)
