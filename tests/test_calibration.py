"""The library-side offline calibration agrees with the oracle's (independent implementations)."""

import numpy as np
import pytest

from bit_kv_cache_write_gb300 import calibration, synth
from oracle import calibrate, rotation


@pytest.mark.parametrize("name", ["tiny", "qwen3_4b_b64_32k"])
def test_package_calibration_matches_oracle(name):
    cfg = dict(synth.WORKLOADS[name])
    cfg["n_cal_q"] = 256
    cfg["n_cal_kv"] = 128
    li = synth.LayerInputs(cfg, 0)
    q, k, v = li.calibration()
    sm = cfg["d"] ** -0.5
    got = calibration.calibrate_layer(q, k, v, sm, cfg["clip_ratio"])
    want = calibrate.calibrate_layer(q, k, v, sm, cfg["clip_ratio"])
    for g, w in zip(got, want):
        assert np.abs(g.astype(np.float64) - w).max() <= 1e-5 * max(1.0, np.abs(w).max())


def test_package_rotation_is_u_h_p():
    rng = np.random.default_rng(0)
    a = rng.standard_normal((300, 16))
    c = a.T @ a
    np.testing.assert_allclose(calibration.rotation_from_target(c), rotation.oscar_rotation(c), atol=1e-12)


def test_package_hadamard_only_calibration_matches_oracle():
    cfg = dict(synth.WORKLOADS["tiny"])
    cfg["n_cal_q"] = 256
    cfg["n_cal_kv"] = 128
    li = synth.LayerInputs(cfg, 0)
    q, k, v = li.calibration()
    sm = cfg["d"] ** -0.5
    got = calibration.calibrate_layer(q, k, v, sm, cfg["clip_ratio"], kind="hadamard")
    want = calibrate.calibrate_layer(q, k, v, sm, cfg["clip_ratio"], kind="hadamard")
    for g, w in zip(got, want):
        assert np.abs(g.astype(np.float64) - w).max() <= 1e-6 * max(1.0, np.abs(w).max())
    np.testing.assert_array_equal(calibration.hadamard_rotation(4), rotation.hadamard_only_rotation(4))
