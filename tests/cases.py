"""Shared builders for GPU parity tests: seeded inputs, oracle calibration, oracle-written pools.

Inputs come from ``bit_kv_cache_write_gb300.synth``. Expected values come from
``oracle`` only. The GPU side receives the same inputs (and, for decode, the
same oracle-written cache) as torch tensors.
"""

import numpy as np

from oracle import layout
from oracle.paged_case import P, DecodeCase, calibration, workload  # noqa: F401  (re-exported for the tests)


def compare_int2_head(gpu_pool, ref_pool, geo, slots, kind, h, q):
    """Write-path parity of one (kind, head) at the given slots; returns the tolerated flips.

    Codes must match bit-exactly, except off-by-one codes whose oracle ratio u
    lies within 1e-5 of the rounding boundary between the two codes. Scale and
    zero must agree within 1 fp16 ulp.
    """
    slots = np.asarray(slots, np.int64)
    pages, rows = slots // geo.page, slots % geo.page
    base = (pages * geo.h_kv + h) * geo.block + (0 if kind == "k" else geo.segment)
    rb = geo.d // 4
    cidx = (base + rows * rb)[:, None] + np.arange(rb)[None, :]
    g_codes = layout.unpack_rows(gpu_pool[cidx], kind, geo.d)
    r_codes = layout.unpack_rows(ref_pool[cidx], kind, geo.d)
    assert np.array_equal(r_codes, q["codes"])
    ng = geo.d // geo.group
    sidx = (base + geo.code_bytes + rows * ng * 4)[:, None] + np.arange(ng * 4)[None, :]
    g_sz = np.ascontiguousarray(gpu_pool[sidx]).view(np.uint16).reshape(len(slots), ng, 2)
    r_sz = np.ascontiguousarray(ref_pool[sidx]).view(np.uint16).reshape(len(slots), ng, 2)
    def ordered(x):      # fp16 bit patterns on one integer line: adjacent values differ by 1, -0 == +0
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    ok_sz = np.abs(ordered(g_sz) - ordered(r_sz)) <= 1
    if not ok_sz.all():
        bad = np.argwhere(~ok_sz)[:5]
        detail = ["slot %d group %d %s: gpu %r oracle %r" % (
            slots[i], g, "scale" if j == 0 else "zero",
            float(g_sz[i, g, j:j + 1].view(np.float16)[0]), float(r_sz[i, g, j:j + 1].view(np.float16)[0]))
            for i, g, j in bad]
        raise AssertionError("%s head %d: scale/zero differ by more than 1 fp16 ulp at %d places: %s" % (
            kind, h, int((~ok_sz).sum()), "; ".join(detail)))
    diff = g_codes.astype(np.int64) - r_codes.astype(np.int64)
    bad = diff != 0
    if not bad.any():
        return 0
    lo = np.minimum(g_codes, r_codes).astype(np.int64)
    if "thresholds" in q:      # Lloyd-Max: the normalised value z against the cut between the two codes
        cut = np.asarray(q["thresholds"])[np.minimum(lo, 2)]
        near = np.abs(q["z"] - cut) <= 1e-6
    else:
        near = np.abs(q["u"] - (lo + 0.5)) <= 1e-5
    tolerated = bad & (np.abs(diff) == 1) & near
    assert (bad == tolerated).all(), "%s head %d: %d code mismatches outside the boundary band" % (
        kind, h, int((bad & ~tolerated).sum()))
    return int(bad.sum())


def compare_int2(gpu_pool, ref_pool, geo, slots, info, max_flip_frac=1e-3):
    """compare_int2_head over every head and K/V, plus: nothing outside the written rows changed."""
    flips = 0
    for kind in ("k", "v"):
        for h in range(geo.h_kv):
            flips += compare_int2_head(gpu_pool, ref_pool, geo, slots, kind, h, info[kind][h])
    assert flips <= max_flip_frac * 2 * geo.h_kv * len(slots) * geo.d
    written = np.zeros(gpu_pool.size, bool)
    slots = np.asarray(slots, np.int64)
    for h in range(geo.h_kv):
        for kind in ("k", "v"):
            base = (slots // geo.page * geo.h_kv + h) * geo.block + (0 if kind == "k" else geo.segment)
            rows = slots % geo.page
            rb, szb = geo.d // 4, 4 * (geo.d // geo.group)
            written[((base + rows * rb)[:, None] + np.arange(rb)).ravel()] = True
            written[((base + geo.code_bytes + rows * szb)[:, None] + np.arange(szb)).ravel()] = True
    assert np.array_equal(gpu_pool[~written], ref_pool[~written])
    return flips


def check_decode(got, want, max_abs=2e-3, rel_l2=1e-3):
    """Decode tolerance: max-abs 2e-3 and relative L2 1e-3 against the fp64 oracle."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    err = np.abs(got - want).max()
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    assert err <= max_abs and rel <= rel_l2, "max-abs %.3g (<= %.1g), rel-L2 %.3g (<= %.1g)" % (err, max_abs, rel, rel_l2)
    return err, rel
