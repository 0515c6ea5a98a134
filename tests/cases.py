"""Shared builders for GPU parity tests: seeded inputs, oracle calibration, oracle-written pools.

Inputs come from ``bit_kv_cache_write_gb300.synth``. Expected values come from
``oracle`` only. The GPU side receives the same inputs (and, for decode, the
same oracle-written cache) as torch tensors.
"""

import numpy as np

from bit_kv_cache_write_gb300 import synth
from oracle import cache, calibrate, layout

P = 16


def workload(name, **over):
    cfg = dict(synth.WORKLOADS[name])
    cfg.update(over)
    return cfg


def calibration(cfg, layer=0):
    """Oracle calibration of one layer, rounded to the fp32 values both sides consume.

    cfg["rotation"] (default "oscar") may select the Hadamard-only ablation ("hadamard")."""
    li = synth.LayerInputs(cfg, layer)
    q_cal, k_cal, v_cal = li.calibration()
    sm = cfg["d"] ** -0.5
    rk, rv, tk, tv = calibrate.calibrate_layer(q_cal, k_cal, v_cal, sm, cfg["clip_ratio"],
                                               kind=cfg.get("rotation", "oscar"))
    f32 = [np.asarray(a, np.float32) for a in (rk, rv, tk, tv)]
    return li, f32


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


class DecodeCase:
    """A batch of sequences in paged INT2 + BF16 pools, written by the oracle.

    hist_lens / bf16_lens: per-sequence lengths. shared_pages: number of
    leading INT2 pages (and ``shared_bf16_pages`` BF16 pages) that every table
    references (prefix sharing); only sequence 0's data is stored there.
    """

    def __init__(self, cfg, hist_lens, bf16_lens, layer=0, shared_pages=0, shared_bf16_pages=0,
                 extra_pages=3, stride_pad=2):
        self.cfg = cfg
        self.codebook = cfg.get("codebook", "uniform")
        d, group, h_kv, h_q = cfg["d"], cfg["group"], cfg["h_kv"], cfg["h_q"]
        self.li, (self.rk, self.rv, self.tk, self.tv) = calibration(cfg, layer)
        self.geo = layout.Int2Geometry(d, group, h_kv)
        self.hist_lens = np.asarray(hist_lens, np.int32)
        self.bf16_lens = np.asarray(bf16_lens, np.int32)
        B = len(hist_lens)
        seed = self.li.seed

        # ---- INT2 pages: shared prefix pages first, then each sequence's own pages, seeded permutation
        own = [max(0, synth.pages_for(int(h)) - shared_pages) for h in hist_lens]
        n_pages = shared_pages + sum(own) + extra_pages
        perm = synth.page_permutation(seed, "int2", n_pages)
        self.int2_stride = max(1, max(synth.pages_for(int(h)) for h in hist_lens) + stride_pad)
        self.int2_tables = np.full((B, self.int2_stride), -1, np.int32)
        nxt = shared_pages
        for b in range(B):
            np_b = synth.pages_for(int(hist_lens[b]))
            for j in range(np_b):
                if j < shared_pages:
                    self.int2_tables[b, j] = perm[j]
                else:
                    self.int2_tables[b, j] = perm[nxt]
                    nxt += 1
        self.int2_pool = np.zeros(n_pages * self.geo.page_bytes, np.uint8)
        self.int2_pages = n_pages
        for b in range(B):
            n = int(hist_lens[b])
            first = 0 if b == 0 else min(n, shared_pages * P)
            if n - first <= 0:
                continue
            k, v = self.li.kv("hist/%d" % b, n)
            t = np.arange(first, n)
            slots = self.int2_tables[b, t // P].astype(np.int64) * P + t % P
            cache.write_tokens(self.int2_pool, self.geo, k[first:], v[first:], slots,
                               self.rk, self.rv, self.tk, self.tv, keep=False, codebook=self.codebook)

        # ---- BF16 pages
        own_bf = [max(0, synth.pages_for(int(n)) - shared_bf16_pages) for n in bf16_lens]
        n_bf_pages = shared_bf16_pages + sum(own_bf) + extra_pages
        perm_bf = synth.page_permutation(seed, "bf16", n_bf_pages)
        self.bf16_stride = max(1, (cfg.get("sink", synth.SINK) + cfg.get("recent", synth.RECENT)) // P)
        self.bf16_tables = np.full((B, self.bf16_stride), -1, np.int32)
        nxt = shared_bf16_pages
        for b in range(B):
            for j in range(synth.pages_for(int(bf16_lens[b]))):
                if j < shared_bf16_pages:
                    self.bf16_tables[b, j] = perm_bf[j]
                else:
                    self.bf16_tables[b, j] = perm_bf[nxt]
                    nxt += 1
        self.bf16_pages = n_bf_pages
        self.bf16_pool = np.zeros(n_bf_pages * h_kv * 2 * P * d, np.float32)
        for b in range(B):
            n = int(bf16_lens[b])
            first = 0 if b == 0 else min(n, shared_bf16_pages * P)
            if n - first <= 0:
                continue
            k, v = self.li.kv("bf16/%d" % b, n)
            for t in range(first, n):
                pg = int(self.bf16_tables[b, t // P])
                for h in range(h_kv):
                    o = layout.bf16_offset(pg, h, "k", t % P, d, h_kv)
                    self.bf16_pool[o:o + d] = k[t, h]
                    o = layout.bf16_offset(pg, h, "v", t % P, d, h_kv)
                    self.bf16_pool[o:o + d] = v[t, h]
        self.q = self.li.queries(B)
        self.sm_scale = d ** -0.5

    def oracle_out(self, seqs=None, heads=None):
        return cache.decode_batch(self.q, self.int2_pool, self.geo, self.int2_tables, self.hist_lens,
                                  self.bf16_pool, self.bf16_tables, self.bf16_lens, self.rk, self.rv,
                                  self.sm_scale, seqs=seqs, heads=heads, codebook=self.codebook)


def check_decode(got, want, max_abs=2e-3, rel_l2=1e-3):
    """Decode tolerance: max-abs 2e-3 and relative L2 1e-3 against the fp64 oracle."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    err = np.abs(got - want).max()
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    assert err <= max_abs and rel <= rel_l2, "max-abs %.3g (<= %.1g), rel-L2 %.3g (<= %.1g)" % (err, max_abs, rel, rel_l2)
    return err, rel
