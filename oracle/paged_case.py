"""Paged caches written by the oracle from the seeded synthetic inputs (test infrastructure).

The inputs come from ``bit_kv_cache_write_gb300.synth`` (seeded generators, none of the method's
arithmetic); calibration, writes and the expected decode output come from this package only. The
GPU parity tests and the oracle timing of ``bench.py`` build their cases here; the GPU side gets
the same inputs and, for decode, the same oracle-written pools.
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
