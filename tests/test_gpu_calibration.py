"""GPU calibration targets (oscar_calibration_targets) against the oracle's fp64 targets.

The key target Q^T Q and the value target V^T S^T S V (QbitAI article on OSCAR, section "OSCAR aligns
the rotation with attention") are accumulated on the GPU in fp64; they must match the oracle's to
1e-10 of their largest entry. The host then forms R = U H P from them.
"""

import numpy as np
import pytest
import torch

from bit_kv_cache_write_gb300 import calibration, synth
from bit_kv_cache_write_gb300 import oscar as O
from oracle import rotation

pytestmark = pytest.mark.gpu


def gpu_targets(q, k, v, sm, dev):
    qt, kt, vt = (torch.as_tensor(np.ascontiguousarray(a, np.float32), device=dev) for a in (q, k, v))
    n, h_q, d = qt.shape
    h_kv = kt.shape[1]
    tk = torch.full((h_kv, d, d), float("nan"), dtype=torch.float64, device=dev)
    tv = torch.full_like(tk, float("nan"))
    ws = torch.empty(O.oscar_calibration_workspace_size(n, h_q, h_kv, d), dtype=torch.uint8, device=dev)
    O.oscar_calibration_targets(qt, kt, vt, sm, tk, tv, ws)
    torch.cuda.synchronize()
    return tk.cpu().numpy(), tv.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "qwen3_8b_bs1_100k"])
def test_targets_match_the_oracle(cuda, name):
    cfg = dict(synth.WORKLOADS[name])
    li = synth.LayerInputs(cfg, 0)
    q, k, v = li.calibration()
    d, h_q, h_kv = cfg["d"], cfg["h_q"], cfg["h_kv"]
    g = h_q // h_kv
    sm = d ** -0.5
    tk, tv = gpu_targets(q, k, v, sm, cuda)
    for h in range(h_kv):
        q_rows = np.asarray(q[:, h * g:(h + 1) * g, :], np.float64).reshape(-1, d)
        want_k = rotation.key_covariance(q_rows)
        want_v = rotation.value_covariance(q_rows, k[:, h, :], v[:, h, :], sm)
        assert np.abs(tk[h] - want_k).max() <= 1e-10 * np.abs(want_k).max()
        assert np.abs(tv[h] - want_v).max() <= 1e-10 * np.abs(want_v).max()


def test_gpu_calibration_gives_orthogonal_rotations_and_matching_thresholds(cuda):
    cfg = dict(synth.WORKLOADS["tiny"])
    li = synth.LayerInputs(cfg, 0)
    q, k, v = li.calibration()
    rk, rv, tk, tv = calibration.calibrate_layer_gpu(q, k, v, cfg["d"] ** -0.5, cfg["clip_ratio"], device=cuda)
    for h in range(cfg["h_kv"]):
        for r in (rk[h], rv[h]):
            assert np.abs(r.astype(np.float64) @ r.T.astype(np.float64) - np.eye(cfg["d"])).max() < 1e-5
        np.testing.assert_allclose(tk[h], rotation.clip_thresholds(k[:, h], rk[h].astype(np.float64), 0.9), rtol=1e-5)


def test_rejected_sizes(cuda):
    z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device=cuda)
    tk, tv = z(2, 64, 64, dt=torch.float64), z(2, 64, 64, dt=torch.float64)
    ws = z(1 << 20, dt=torch.uint8)
    with pytest.raises(O.OscarError) as e:                  # too many keys
        O.oscar_calibration_targets(z(4, 4, 64), z(8193, 2, 64), z(8193, 2, 64), 0.125, tk, tv, ws)
    assert e.value.status == -2
    with pytest.raises(O.OscarError) as e:                  # workspace too small
        O.oscar_calibration_targets(z(4096, 4, 64), z(16, 2, 64), z(16, 2, 64), 0.125, tk, tv, ws[:1024])
    assert e.value.status == -7
