"""Offline calibration on the host: per (layer, KV head) rotation R and clip threshold T.

This is the offline stage of OSCAR (QbitAI article on OSCAR, section "OSCAR
aligns the rotation with attention"; arXiv 2605.17757 abstracts). A few
calibration samples give the key target Q^T Q and the value target
V^T S^T S V. Their eigenbasis U, sorted by descending eigenvalue, is composed
with a normalised Sylvester Hadamard matrix and the bit-reversal permutation:
R = U H P. The clip threshold of each rotated channel is clip_ratio times its
calibration maximum |x R|. The results are fixed and reused unchanged at
inference: they are the inputs of ``oscar_calibrate_upload``.

It runs once, offline, with NumPy/LAPACK, outside the write and decode hot
path. Conventions match the library: row vectors, x_rot = x @ R; each
eigenvector column is signed so that its largest-magnitude entry is positive.
"""

import numpy as np


def _hadamard(d):
    h = np.array([[1.0]])
    while h.shape[0] < d:
        h = np.vstack([np.hstack([h, h]), np.hstack([h, -h])])
    return h / np.sqrt(d)


def _bitrev_columns(d):
    bits = d.bit_length() - 1
    return np.array([int(format(i, "0%db" % bits)[::-1], 2) if bits else 0 for i in range(d)])


def rotation_from_target(target):
    """R = U H P for a symmetric positive semi-definite d x d target."""
    d = target.shape[0]
    w, u = np.linalg.eigh(0.5 * (target + target.T))
    u = u[:, np.argsort(-w, kind="stable")]
    lead = np.abs(u).argmax(axis=0)
    u = u * np.where(u[lead, np.arange(d)] < 0, -1.0, 1.0)[None, :]
    uh = u @ _hadamard(d)
    r = np.empty_like(uh)
    r[:, _bitrev_columns(d)] = uh          # column i of U H moves to column bitrev(i)
    return r


def hadamard_rotation(d):
    """R = H P with no covariance basis: the data-oblivious rotation that the v2
    abstract contrasts with OSCAR ("Hadamard-only" / "QuaRot-style" INT2), kept
    for the ablation."""
    r = np.empty((d, d))
    r[:, _bitrev_columns(d)] = _hadamard(d)
    return r


def calibrate_layer(q_cal, k_cal, v_cal, sm_scale, clip_ratio=0.9, kind="oscar"):
    """q_cal [n, H_q, d], k_cal/v_cal [m, H_kv, d] -> fp32 (R_k, R_v, T_k, T_v).

    kind "oscar": R = U H P from the attention-aware targets; kind "hadamard":
    R = H P for K and V (the ablation), with thresholds by the same rule."""
    if kind not in ("oscar", "hadamard"):
        raise ValueError("unknown rotation kind %r" % (kind,))
    n, h_q, d = q_cal.shape
    h_kv = k_cal.shape[1]
    g = h_q // h_kv
    r_k = np.empty((h_kv, d, d), np.float32)
    r_v = np.empty((h_kv, d, d), np.float32)
    t_k = np.empty((h_kv, d), np.float32)
    t_v = np.empty((h_kv, d), np.float32)
    for h in range(h_kv):
        qg = np.asarray(q_cal[:, h * g:(h + 1) * g], np.float64).reshape(n * g, d)
        kh = np.asarray(k_cal[:, h], np.float64)
        vh = np.asarray(v_cal[:, h], np.float64)
        logits = (qg @ kh.T) * sm_scale
        logits -= logits.max(axis=1, keepdims=True)
        s = np.exp(logits)
        s /= s.sum(axis=1, keepdims=True)
        sv = s @ vh
        if kind == "oscar":
            rk = rotation_from_target(qg.T @ qg)
            rv = rotation_from_target(sv.T @ sv)
        else:
            rk = rv = hadamard_rotation(d)
        r_k[h], r_v[h] = rk, rv
        t_k[h] = clip_ratio * np.abs(kh @ rk).max(axis=0)
        t_v[h] = clip_ratio * np.abs(vh @ rv).max(axis=0)
    return r_k, r_v, t_k, t_v


def calibrate_layer_gpu(q_cal, k_cal, v_cal, sm_scale, clip_ratio=0.9, device="cuda"):
    """calibrate_layer with the two covariance targets accumulated on the GPU (fp64,
    ``oscar_calibration_targets``); the eigendecomposition, R = U H P and the thresholds stay on the
    host. Inputs are host arrays [n, H_q, d] and [m, H_kv, d]; returns fp32 (R_k, R_v, T_k, T_v)."""
    import torch
    from . import oscar

    q = torch.as_tensor(np.ascontiguousarray(q_cal, np.float32), device=device)
    k = torch.as_tensor(np.ascontiguousarray(k_cal, np.float32), device=device)
    v = torch.as_tensor(np.ascontiguousarray(v_cal, np.float32), device=device)
    n, h_q, d = q.shape
    h_kv = k.shape[1]
    tk = torch.empty(h_kv, d, d, dtype=torch.float64, device=device)
    tv = torch.empty_like(tk)
    ws = torch.empty(oscar.oscar_calibration_workspace_size(n, h_q, h_kv, d), dtype=torch.uint8, device=device)
    oscar.oscar_calibration_targets(q, k, v, sm_scale, tk, tv, ws)
    tk, tv = tk.cpu().numpy(), tv.cpu().numpy()
    kh_all = np.asarray(k_cal, np.float64)
    vh_all = np.asarray(v_cal, np.float64)
    r_k = np.empty((h_kv, d, d), np.float32)
    r_v = np.empty((h_kv, d, d), np.float32)
    t_k = np.empty((h_kv, d), np.float32)
    t_v = np.empty((h_kv, d), np.float32)
    for h in range(h_kv):
        rk = rotation_from_target(tk[h])
        rv = rotation_from_target(tv[h])
        r_k[h], r_v[h] = rk, rv
        t_k[h] = clip_ratio * np.abs(kh_all[:, h] @ rk).max(axis=0)
        t_v[h] = clip_ratio * np.abs(vh_all[:, h] @ rv).max(axis=0)
    return r_k, r_v, t_k, t_v
