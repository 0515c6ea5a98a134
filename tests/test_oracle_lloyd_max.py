"""Pins of oracle.lloyd_max: the Lloyd-Max 2-bit codebook (the step after the uniform grid that the
QbitAI article on OSCAR mentions in its closing part) against published values and its own
optimality conditions.

The published values are from J. Max, "Quantizing for minimum distortion", IRE Transactions on
Information Theory, 1960: the 4-level quantizer of a unit Gaussian has levels +-0.4528 and +-1.510,
thresholds 0 and +-0.9816, and mean squared error 0.1175. The best uniform 4-level quantizer has
step 0.9957 and mean squared error 0.1188.
"""

import numpy as np
import pytest
from scipy.optimize import minimize_scalar
from scipy.stats import norm

from oracle import lloyd_max, quantize


def test_published_four_level_gaussian_quantizer():
    y, t = lloyd_max.lloyd_max_gaussian(4)
    np.testing.assert_allclose(y, [-1.510, -0.4528, 0.4528, 1.510], atol=5e-4)
    np.testing.assert_allclose(t, [-0.9816, 0.0, 0.9816], atol=1e-4)
    assert abs(lloyd_max.gaussian_distortion(y, t) - 0.1175) < 1e-4


def test_optimality_conditions_and_symmetry():
    y, t = lloyd_max.lloyd_max_gaussian(4)
    np.testing.assert_allclose(t, 0.5 * (y[:-1] + y[1:]), atol=1e-15)          # nearest neighbour
    edges = np.concatenate([[-np.inf], t, [np.inf]])
    centroid = (norm.pdf(edges[:-1]) - norm.pdf(edges[1:])) / (norm.cdf(edges[1:]) - norm.cdf(edges[:-1]))
    np.testing.assert_allclose(y, centroid, atol=1e-12)                          # centroid
    np.testing.assert_allclose(y, -y[::-1], atol=1e-12)


def test_distortion_formula_against_monte_carlo():
    y, t = lloyd_max.lloyd_max_gaussian(4)
    x = np.random.default_rng(3).standard_normal(2_000_000)
    q = y[np.searchsorted(t, x, side="left")]
    assert abs(np.mean((x - q) ** 2) - lloyd_max.gaussian_distortion(y, t)) < 1e-3


def test_beats_the_best_uniform_quantizer():
    def uniform_d(step):
        lv = np.array([-1.5, -0.5, 0.5, 1.5]) * step
        return lloyd_max.gaussian_distortion(lv, [-step, 0.0, step])

    res = minimize_scalar(uniform_d, bounds=(0.5, 1.5), method="bounded", options={"xatol": 1e-10})
    assert abs(res.x - 0.9957) < 1e-3 and abs(res.fun - 0.1188) < 1e-4
    y, t = lloyd_max.lloyd_max_gaussian(4)
    assert lloyd_max.gaussian_distortion(y, t) < res.fun


@pytest.mark.parametrize("n", [2, 3, 8])
def test_other_sizes_converge_from_any_start(n):
    # a log-concave density has one fixed point: the two-level answer is +-sqrt(2/pi)
    y, t = lloyd_max.lloyd_max_gaussian(n)
    assert np.all(np.diff(y) > 0)
    if n == 2:
        np.testing.assert_allclose(y, [-np.sqrt(2 / np.pi), np.sqrt(2 / np.pi)], atol=1e-12)


def test_codes_are_the_brute_force_nearest_level():
    y, _ = lloyd_max.lloyd_max_gaussian(4)
    rng = np.random.default_rng(11)
    d, group = 8, 4
    x = rng.standard_normal((50, d)) * rng.uniform(0.1, 3.0, (50, 1))
    big = np.full(d, 1e6)
    q = lloyd_max.quantize_lloyd_max(x, np.eye(d), big, group, y)
    g = np.asarray(x, np.float32).astype(np.float64).reshape(50, d // group, group)
    mu = g.mean(-1, keepdims=True)
    sd = np.sqrt(((g - mu) ** 2).mean(-1, keepdims=True))
    z = ((g - mu) / sd).reshape(50, d)
    want = np.abs(z[..., None] - y[None, None, :]).argmin(-1)
    np.testing.assert_array_equal(q["codes"], want)
    np.testing.assert_array_equal(q["scale"], sd[..., 0].astype(np.float16))
    np.testing.assert_array_equal(q["zero"], mu[..., 0].astype(np.float16))


def test_degenerate_group_and_clipping():
    y, _ = lloyd_max.lloyd_max_gaussian(4)
    d = 8
    x = np.array([[2.0] * 4 + [1.0, -1.0, 3.0, -3.0]])
    t = np.array([1.0] * 4 + [10.0] * 4)            # the first group clips to a constant 1.0
    q = lloyd_max.quantize_lloyd_max(x, np.eye(d), t, 4, y)
    assert q["scale"][0, 0] == 0 and np.all(q["codes"][0, :4] == 0)
    deq = lloyd_max.dequantize_lloyd_max(q["codes"], q["scale"], q["zero"], 4, y)
    np.testing.assert_array_equal(deq[0, :4], [1.0] * 4)
    assert list(q["codes"][0, 4:]) == [2, 1, 3, 0]   # z = +-0.447, +-1.342 of the second group


def test_gaussian_groups_reach_the_codebook_distortion_and_beat_the_uniform_grid():
    y, t = lloyd_max.lloyd_max_gaussian(4)
    rng = np.random.default_rng(5)
    n, d = 2048, 128
    x = rng.standard_normal((n, d)) * rng.uniform(0.5, 2.0, (n, 1)) + rng.uniform(-1, 1, (n, 1))
    big = np.full(d, 1e6)
    q = lloyd_max.quantize_lloyd_max(x, np.eye(d), big, d, y)
    deq = lloyd_max.dequantize_lloyd_max(q["codes"], q["scale"], q["zero"], d, y)
    x32 = np.asarray(x, np.float32).astype(np.float64)
    sd = x32.std(axis=1, keepdims=True)
    mse_lm = np.mean(((deq - x32) / sd) ** 2)
    u = quantize.quantize(x, np.eye(d), big, d)
    mse_u = np.mean(((quantize.dequantize(u["codes"], u["scale"], u["zero"], d) - x32) / sd) ** 2)
    assert abs(mse_lm - lloyd_max.gaussian_distortion(y, t)) < 0.01
    assert mse_lm < 0.5 * mse_u


def test_lloyd_max_against_the_uniform_grid_in_attention():
    """Both codebooks on the same OSCAR-rotated cache (Qwen3-8B shape recipe, 2,048 history tokens):
    reconstruction and attention errors against exact attention over the unquantized bf16 K/V. The
    numbers are printed for the record; checked: the Lloyd-Max codebook reconstructs K and V better."""
    from test_ablation_rotation import bf16, SINK, RECENT
    from bit_kv_cache_write_gb300 import synth
    from oracle import attention, calibrate

    y, _ = lloyd_max.lloyd_max_gaussian(4)
    cfg = dict(synth.WORKLOADS["qwen3_8b_bs1_100k"])
    li = synth.LayerInputs(cfg, 0)
    q_cal, k_cal, v_cal = li.calibration()
    d, group, h_kv, h_q = cfg["d"], cfg["group"], cfg["h_kv"], cfg["h_q"]
    sm = d ** -0.5
    rk, rv, tk, tv = (np.asarray(a, np.float32).astype(np.float64) for a in
                      calibrate.calibrate_layer(q_cal, k_cal, v_cal, sm, cfg["clip_ratio"]))
    k_hist, v_hist = (bf16(a) for a in li.kv("hist", 2048))
    k_bf, v_bf = (bf16(a) for a in li.kv("bf16", SINK + RECENT))
    q = bf16(li.queries(2))
    g = h_q // h_kv
    err = {name: dict(out=[0.0, 0.0], k=[0.0, 0.0], v=[0.0, 0.0]) for name in ("uniform", "lloyd_max")}
    for kv in range(h_kv):
        for name in err:
            deq = []
            for x, r, t in ((k_hist[:, kv], rk[kv], tk[kv]), (v_hist[:, kv], rv[kv], tv[kv])):
                if name == "uniform":
                    qz = quantize.quantize(x, r, t, group)
                    deq.append(quantize.dequantize(qz["codes"], qz["scale"], qz["zero"], group))
                else:
                    qz = lloyd_max.quantize_lloyd_max(x, r, t, group, y)
                    deq.append(lloyd_max.dequantize_lloyd_max(qz["codes"], qz["scale"], qz["zero"], group, y))
            e = err[name]
            for key, got, want in (("k", deq[0] @ rk[kv].T, k_hist[:, kv]), ("v", deq[1] @ rv[kv].T, v_hist[:, kv])):
                e[key][0] += np.sum((got - want) ** 2)
                e[key][1] += np.sum(want ** 2)
            k_all = np.concatenate([k_bf[:, kv], k_hist[:, kv]])
            v_all = np.concatenate([v_bf[:, kv], v_hist[:, kv]])
            for b in range(2):
                for h in range(kv * g, (kv + 1) * g):
                    got = attention.decode_one(q[b, h], rk[kv], rv[kv], deq[0], deq[1], k_bf[:, kv], v_bf[:, kv], sm)
                    want = attention.softmax_attention(sm * (k_all @ q[b, h]), v_all)
                    e["out"][0] += np.sum((got - want) ** 2)
                    e["out"][1] += np.sum(want ** 2)
    rel = {name: {key: float(np.sqrt(a / b)) for key, (a, b) in e.items()} for name, e in err.items()}
    for name in rel:
        print("%s: out rel-L2 %.3f | K rel %.3f | V rel %.3f" % (name, rel[name]["out"], rel[name]["k"], rel[name]["v"]))
    assert rel["lloyd_max"]["k"] < rel["uniform"]["k"] and rel["lloyd_max"]["v"] < rel["uniform"]["v"]


# ---- the stored ("dyadic") codebook: Lloyd-Max levels rounded to multiples of y_1 / 8

def test_dyadic_codebook_rounds_the_published_levels():
    delta, levels, cut = lloyd_max.dyadic_codebook()
    y, _ = lloyd_max.lloyd_max_gaussian(4)
    assert abs(delta * 8 - 0.4528) < 5e-4                      # inner level kept (Max 1960)
    assert abs(levels[3] - 1.510) < 0.02                       # outer level 27 delta ~ 1.528
    assert round(y[3] / delta) == 27                           # 26.7 rounds to 27
    np.testing.assert_allclose(cut, [-17.5 * delta, 0.0, 17.5 * delta], atol=1e-15)
    # distortion on N(0, 1) within 0.1 % of the unrounded quantizer's 0.1175
    d_dyadic = lloyd_max.gaussian_distortion(levels, cut)
    d_exact = lloyd_max.gaussian_distortion(*lloyd_max.lloyd_max_gaussian(4))
    assert d_exact <= d_dyadic < d_exact * 1.001


def test_dyadic_levels_are_linear_in_the_code_and_its_low_bit():
    # l(c) = -27 + 17.5 c + 1.5 b0: what lets a decoder keep exact integer dot products with one bit plane
    for c in range(4):
        assert lloyd_max.DYADIC_STEPS[c] == -27 + 17.5 * c + 1.5 * (c & 1)


def test_dyadic_quantizer_brute_force_and_degenerate_groups():
    rng = np.random.default_rng(7)
    d, group = 16, 8
    r = np.eye(d)
    t = np.full(d, 50.0)
    x = rng.standard_normal((200, d)) * 3.0 + 1.0
    x[0, :group] = 2.5                                         # a flat group: sigma = 0
    q = lloyd_max.quantize_dyadic(x, r, t, group)
    delta, levels, _ = lloyd_max.dyadic_codebook()
    xh = x.astype(np.float32).astype(np.float64)
    for i in range(1, 200):
        for gi in range(d // group):
            seg = xh[i, gi * group:(gi + 1) * group]
            mu, sigma = seg.mean(), seg.std()
            for j, v in enumerate(seg):
                dist = np.abs((v - mu) / sigma - levels)
                best = int(np.flatnonzero(dist == dist.min())[0])       # ties take the lower level
                assert q["codes"][i, gi * group + j] == best
            assert q["scale"][i, gi] == np.float16(sigma * delta) and q["zero"][i, gi] == np.float16(mu)
    assert (q["codes"][0, :group] == 0).all() and q["scale"][0, 0] == 0
    deq = lloyd_max.dequantize_dyadic(q["codes"], q["scale"], q["zero"], group)
    np.testing.assert_allclose(deq[0, :group], np.float16(2.5))    # flat group dequantizes to its mean


def test_dyadic_mse_on_gaussian_groups_matches_the_codebook_distortion():
    rng = np.random.default_rng(11)
    d = group = 128
    x = rng.standard_normal((4000, d))
    q = lloyd_max.quantize_dyadic(x, np.eye(d), np.full(d, 1e9), group)
    deq = lloyd_max.dequantize_dyadic(q["codes"], q["scale"], q["zero"], group)
    sig = q["sigma"][:, 0:1]
    mse = np.mean(((x - deq) / sig) ** 2)
    delta, levels, cut = lloyd_max.dyadic_codebook()
    assert abs(mse - lloyd_max.gaussian_distortion(levels, cut)) < 0.01
