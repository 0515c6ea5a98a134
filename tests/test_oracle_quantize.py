"""Pins of oracle.quantize and oracle.layout: hand-worked groups, brute force, invariants, bounds.

Source of what is pinned: QbitAI article on OSCAR, serving-pipeline part
(rotate, clip, quantize and pack the demoted token; four levels at 2 bits;
four codes per byte; scale/zero-point dequant); arXiv 2605.17757 abstracts
(offline clipping thresholds).
"""

import os

import numpy as np
import pytest

from oracle import layout, quantize, rotation

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_groups():
    rows = []
    with open(os.path.join(GOLDEN, "quantize_g4.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, x, t, c, s, z = [p.strip() for p in line.split("|")]
            rows.append((name, [float(v) for v in x.split()], [float(v) for v in t.split()],
                         [int(v) for v in c.split()], float(s), float(z)))
    return rows


@pytest.mark.parametrize("case", _golden_groups(), ids=lambda c: c[0])
def test_hand_worked_groups(case):
    _, x, t, codes, s, z = case
    q = quantize.quantize(np.array([x]), np.eye(4), np.array(t), 4)
    assert q["codes"][0].tolist() == codes
    assert float(q["scale"][0, 0]) == s
    assert float(q["zero"][0, 0]) == z


def test_degenerate_group_codes_zero_scale_zero():
    q = quantize.quantize(np.array([[0.75] * 8]), np.eye(8), np.full(8, 10.0), 4)
    assert q["codes"].max() == 0
    assert float(q["scale"][0, 0]) == 0.0 and float(q["zero"][0, 0]) == 0.75


def _random_case(seed, n, d, group, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, d))
    if outliers:
        x[:, rng.choice(d, 3, replace=False)] *= 30
    a = rng.standard_normal((4 * d, d))
    r = rotation.oscar_rotation(a.T @ a)
    t = rotation.clip_thresholds(rng.standard_normal((512, d)) * (np.abs(x).max(0) / 3 + 1), r, 0.9)
    return x, r, t


@pytest.mark.parametrize("d,group", [(64, 32), (128, 128), (128, 64), (128, 32)])
def test_codes_match_brute_force_nearest_level(d, group):
    x, r, t = _random_case(d + group, 200, d, group)
    q = quantize.quantize(x, r, t, group)
    xh = q["x_hat64"].reshape(200, d // group, group)
    mn = xh.min(-1, keepdims=True)
    mx = xh.max(-1, keepdims=True)
    levels = mn[..., None] + (mx - mn)[..., None] * np.arange(4) / 3.0   # [n, ng, 1, 4]
    brute = np.argmin(np.abs(xh[..., None] - levels), axis=-1).reshape(200, d)
    near_tie = np.abs(q["u64"] - np.floor(q["u64"]) - 0.5) < 1e-4
    assert np.array_equal(q["codes"][~near_tie], brute[~near_tie])


@pytest.mark.parametrize("d,group", [(64, 32), (128, 128), (128, 64)])
def test_invariants_and_dequant_bound(d, group):
    x, r, t = _random_case(5 * d + group, 300, d, group)
    q = quantize.quantize(x, r, t, group)
    c = q["codes"]
    assert c.max() <= 3
    ng = d // group
    xh = q["x_hat"].reshape(300, ng, group)
    cg = c.reshape(300, ng, group)
    # the element attaining the group min gets code 0, the max gets code 3
    assert np.all(np.take_along_axis(cg, xh.argmin(-1)[..., None], -1) == 0)
    assert np.all(np.take_along_axis(cg, xh.argmax(-1)[..., None], -1) == 3)
    # clipped values lie in [-T, T]
    assert np.all(np.abs(q["x_hat64"]) <= t[None, :] + 1e-12)
    # dequant error with the unrounded scale/zero: at most scale/2 (plus fp32 slack)
    mn = xh.min(-1, keepdims=True)
    s = (xh.max(-1, keepdims=True) - mn) / 3.0
    deq = cg * s + mn
    assert np.all(np.abs(deq - xh) <= s / 2 * (1 + 1e-5) + 1e-6)
    # with the stored fp16 scale/zero: s/2 + 3|s - s_h| + |z - z_h|
    sh = q["scale"].astype(np.float64)[..., None]
    zh = q["zero"].astype(np.float64)[..., None]
    deq_h = quantize.dequantize(c, q["scale"], q["zero"], group).reshape(300, ng, group)
    bound = s / 2 + 3 * np.abs(s - sh) + np.abs(mn - zh)
    assert np.all(np.abs(deq_h - xh) <= bound * (1 + 1e-5) + 1e-6)


def test_clipping_is_applied_before_group_stats():
    # with T tiny every rotated value is clipped to +-T, so each group spans [-T, T]
    x, r, _ = _random_case(99, 20, 64, 32, outliers=False)
    t = np.full(64, 1e-3)
    q = quantize.quantize(x, r, t, 32)
    np.testing.assert_allclose(q["scale"].astype(np.float64), np.float16(2e-3 / 3), rtol=0)
    clipped = np.abs(quantize.rotate(x, r)) >= 1e-3
    assert clipped.mean() > 0.99
    assert set(np.unique(q["codes"][clipped])) <= {0, 3}
    np.testing.assert_array_equal(q["codes"][clipped], np.where(q["x_hat64"][clipped] > 0, 3, 0))


def test_fp16_scale_zero_round_to_nearest_even():
    q = quantize.quantize(np.array([[-1.0, 0.0, 0.5, 1.0]]), np.eye(4), np.full(4, 9.0), 4)
    assert q["scale"].dtype == np.float16 and float(q["scale"][0, 0]) == float(np.float16(2.0 / 3.0))


# --------------------------------------------------------------------------- layout

def _golden_bits():
    out = []
    with open(os.path.join(GOLDEN, "layout_bits.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kind, d, c, o = line.split()
            out.append((kind, int(d), int(c), int(o)))
    return out


@pytest.mark.parametrize("entry", _golden_bits(), ids=lambda e: "%s%d_c%d" % e[:3])
def test_layout_bits_hand_worked(entry):
    kind, d, c, o = entry
    f = layout.k_bit_offset if kind == "k" else layout.v_bit_offset
    assert f(c, d) == o


@pytest.mark.parametrize("kind", ["k", "v"])
@pytest.mark.parametrize("d", [64, 128])
def test_layout_is_a_bijection_and_roundtrips(kind, d):
    offs = layout.bit_offsets(kind, d)
    assert sorted(offs.tolist()) == list(range(0, 2 * d, 2))
    rng = np.random.default_rng(d)
    codes = rng.integers(0, 4, size=(37, d)).astype(np.uint8)
    rows = layout.pack_rows(codes, kind)
    assert rows.shape == (37, d // 4)
    np.testing.assert_array_equal(layout.unpack_rows(rows, kind, d), codes)
    np.testing.assert_array_equal(layout.pack_row(codes[5], kind), rows[5])
    np.testing.assert_array_equal(layout.unpack_row(rows[5], kind, d), codes[5])


def test_four_codes_per_byte():
    geo = layout.Int2Geometry(128, 128, 8)
    assert geo.code_bytes == 16 * 32          # 16 tokens x 128 channels x 2 bits
    assert geo.segment == 576 and geo.block == 1152 and geo.page_bytes == 9216
    geo = layout.Int2Geometry(128, 64, 8)
    assert geo.segment == 640
    geo = layout.Int2Geometry(64, 32, 2)
    assert geo.segment == 384


def test_pool_write_read_roundtrip_and_sharing():
    rng = np.random.default_rng(1)
    geo = layout.Int2Geometry(64, 32, 2)
    pool = np.zeros(10 * geo.page_bytes, dtype=np.uint8)
    slots = rng.permutation(10 * 16)[:50]
    codes = rng.integers(0, 4, size=(50, 64)).astype(np.uint8)
    sc = rng.random((50, 2)).astype(np.float16)
    ze = rng.standard_normal((50, 2)).astype(np.float16)
    layout.write_int2_rows(pool, geo, slots, 1, "v", codes, sc, ze)
    for i in (0, 17, 49):
        c, s, z = layout.read_int2_token(pool, geo, slots[i], 1, "v")
        np.testing.assert_array_equal(c, codes[i])
        np.testing.assert_array_equal(s, sc[i])
        np.testing.assert_array_equal(z, ze[i])
    # head 0 and the K segment stay untouched
    for s_ in slots:
        c, s, z = layout.read_int2_token(pool, geo, s_, 0, "k")
        assert c.max() == 0 and float(np.abs(s).max()) == 0.0
