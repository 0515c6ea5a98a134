"""Offline calibration per (layer, KV head) (oracle; test infrastructure only).

Source: QbitAI article on OSCAR, section "OSCAR aligns the rotation with
attention": a few calibration samples give, per layer and per head, the key
target Q^T Q and the value target V^T S^T S V; from them the offline stage makes
a fixed rotation and clipping thresholds that inference reuses unchanged.

Readings taken where the pages are silent: the key target of a KV head stacks the
calibration queries of all query heads of its group as rows; S is the row-wise
softmax of sm_scale * Q K^T over the calibration keys (no mask); thresholds are
``clip_ratio`` times the per-channel calibration maximum of |x @ R|.
"""

import numpy as np

from . import rotation


def calibrate_head(q_rows, k_rows, v_rows, sm_scale, clip_ratio, hadamard_block=None, kind="oscar"):
    """Return (R_k, R_v, T_k, T_v) for one KV head, all fp64.

    q_rows [n_q, d]: the head group's calibration queries stacked as rows.
    k_rows, v_rows [n_kv, d]: calibration keys and values of this KV head.
    kind: "oscar" (R = U H P from the attention-aware targets) or "hadamard"
    (the data-oblivious ablation R = H P; thresholds by the same rule).
    """
    if kind == "oscar":
        c_k = rotation.key_covariance(q_rows)
        c_v = rotation.value_covariance(q_rows, k_rows, v_rows, sm_scale)
        r_k = rotation.oscar_rotation(c_k, hadamard_block)
        r_v = rotation.oscar_rotation(c_v, hadamard_block)
    elif kind == "hadamard":
        d = np.asarray(k_rows).shape[1]
        r_k = rotation.hadamard_only_rotation(d, hadamard_block)
        r_v = r_k.copy()
    else:
        raise ValueError("unknown rotation kind %r" % (kind,))
    t_k = rotation.clip_thresholds(k_rows, r_k, clip_ratio)
    t_v = rotation.clip_thresholds(v_rows, r_v, clip_ratio)
    return r_k, r_v, t_k, t_v


def calibrate_layer(q_cal, k_cal, v_cal, sm_scale, clip_ratio, hadamard_block=None, kind="oscar"):
    """Calibrate all KV heads of a layer.

    q_cal [n, H_q, d]; k_cal, v_cal [m, H_kv, d]. Returns fp64 arrays
    R_k, R_v [H_kv, d, d] and T_k, T_v [H_kv, d].
    """
    h_q, d = q_cal.shape[1], q_cal.shape[2]
    h_kv = k_cal.shape[1]
    g = h_q // h_kv
    rk = np.zeros((h_kv, d, d))
    rv = np.zeros((h_kv, d, d))
    tk = np.zeros((h_kv, d))
    tv = np.zeros((h_kv, d))
    for h in range(h_kv):
        q_rows = np.asarray(q_cal[:, h * g:(h + 1) * g, :], dtype=np.float64).reshape(-1, d)
        rk[h], rv[h], tk[h], tv[h] = calibrate_head(
            q_rows, k_cal[:, h, :], v_cal[:, h, :], sm_scale, clip_ratio, hadamard_block, kind)
    return rk, rv, tk, tv
