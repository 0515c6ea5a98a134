"""Seeded synthetic inputs for the OSCAR write and decode workloads.

This module only draws numbers and builds index structures (block tables, slot
maps, lengths). It holds none of the method's arithmetic: no rotation,
quantization or attention. Both the GPU path (through ``bench.py`` and the
tests) and the CPU oracle consume what it returns.

Distributions follow the workload descriptions: K/V rows are N(0,1) (or
Laplace(0,1)), optionally multiplied per (head, channel) by exp(N(0, sigma)),
with a few fixed outlier channels per head multiplied by a constant; queries
are N(0,1). Everything is rounded to bf16 before use (round to nearest even),
and returned as float32 arrays holding bf16-representable values.
"""

import math

import numpy as np

PAGE = 16
SINK = 64
RECENT = 256


def to_bf16(x):
    """Round float32 values to the nearest bf16 (ties to even); returns float32 holding bf16 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def rng_for(seed, stream):
    """Independent numpy Generator for (seed, named stream)."""
    tag = sum((i + 1) * ord(ch) for i, ch in enumerate(stream))
    return np.random.default_rng([int(seed), tag])


class ChannelProfile:
    """Per (head, channel) multiplier of a K or V tensor: outlier channels and log-normal scales."""

    def __init__(self, seed, stream, n_heads, d, n_outliers, outlier_mult, lognormal_sigma=0.0):
        r = rng_for(seed, "profile/" + stream)
        mult = np.ones((n_heads, d), dtype=np.float64)
        if lognormal_sigma > 0:
            mult *= np.exp(r.normal(0.0, lognormal_sigma, size=(n_heads, d)))
        self.outliers = np.zeros((n_heads, n_outliers), dtype=np.int64)
        for h in range(n_heads):
            ch = r.choice(d, size=n_outliers, replace=False) if n_outliers else np.zeros(0, np.int64)
            self.outliers[h] = np.sort(ch)
            mult[h, ch] *= outlier_mult
        self.mult = mult.astype(np.float32)

    def draw(self, seed, stream, n, dist="normal"):
        """[n, H, d] float32 bf16-valued rows."""
        r = rng_for(seed, "rows/" + stream)
        shape = (n,) + self.mult.shape
        if dist == "normal":
            base = r.standard_normal(size=shape, dtype=np.float32)
        elif dist == "laplace":
            base = r.laplace(0.0, 1.0, size=shape).astype(np.float32)
        else:
            raise ValueError(dist)
        return to_bf16(base * self.mult[None])


# ---------------------------------------------------------------------------
# Workload presets (sizes as in the five workload descriptions).
# ---------------------------------------------------------------------------

WORKLOADS = {
    "tiny": dict(batch=1, layers=1, h_q=4, h_kv=2, d=64, group=32, hist=1024,
                 dist="normal", n_outliers=4, outlier_mult=20.0, lognormal_sigma=0.0,
                 q_outliers=True, n_cal_q=4096, n_cal_kv=1024, clip_ratio=0.9, seed=0),
    "qwen3_8b_bs1_100k": dict(batch=1, layers=36, h_q=32, h_kv=8, d=128, group=128, hist=100_000 - SINK - RECENT,
                              dist="normal", n_outliers=3, outlier_mult=30.0, lognormal_sigma=1.0,
                              q_outliers=False, n_cal_q=1024, n_cal_kv=1024, clip_ratio=0.9, seed=2000),
    "qwen3_4b_b64_32k": dict(batch=64, layers=36, h_q=32, h_kv=8, d=128, group=64, hist=32_768 - SINK - RECENT,
                             dist="laplace", n_outliers=1, outlier_mult=25.0, lognormal_sigma=0.0,
                             q_outliers=False, n_cal_q=1024, n_cal_kv=1024, clip_ratio=0.9, seed=3000),
    "bulk_write_131k": dict(tokens=131_072, h_kv=8, h_q=8, d=128, group=128, demote_batch=256,
                            dist="normal", n_outliers=3, outlier_mult=30.0, lognormal_sigma=0.0,
                            q_outliers=False, n_cal_q=1024, n_cal_kv=1024, clip_ratio=0.9, seed=4000),
    "qwen3_32b_mixed16": dict(batch=16, layers=64, h_q=64, h_kv=8, d=128, group=128,
                              len_lo=4096, len_hi=131_072, shared_prefix=16_384,
                              dist="normal", n_outliers=3, outlier_mult=30.0, lognormal_sigma=1.0,
                              q_outliers=False, n_cal_q=1024, n_cal_kv=1024, clip_ratio=0.9, seed=5000),
}


class LayerInputs:
    """All synthetic tensors of one (workload, layer): calibration samples, K/V profiles, queries."""

    def __init__(self, cfg, layer=0):
        self.cfg = cfg
        seed = cfg["seed"] + layer
        self.seed = seed
        h_kv, h_q, d = cfg["h_kv"], cfg["h_q"], cfg["d"]
        self.k_prof = ChannelProfile(seed, "k", h_kv, d, cfg["n_outliers"], cfg["outlier_mult"], cfg["lognormal_sigma"])
        self.v_prof = ChannelProfile(seed, "v", h_kv, d, cfg["n_outliers"], cfg["outlier_mult"], cfg["lognormal_sigma"])
        if cfg["q_outliers"]:
            self.q_prof = ChannelProfile(seed, "q", h_q, d, cfg["n_outliers"], cfg["outlier_mult"], 0.0)
        else:
            self.q_prof = ChannelProfile(seed, "q", h_q, d, 0, 1.0, 0.0)

    def calibration(self):
        """(q_cal [n, H_q, d], k_cal [m, H_kv, d], v_cal [m, H_kv, d])."""
        c = self.cfg
        q = self.q_prof.draw(self.seed, "cal/q", c["n_cal_q"], "normal")
        k = self.k_prof.draw(self.seed, "cal/k", c["n_cal_kv"], c["dist"])
        v = self.v_prof.draw(self.seed, "cal/v", c["n_cal_kv"], c["dist"])
        return q, k, v

    def kv(self, stream, n):
        """K and V rows [n, H_kv, d] for a named stream (e.g. 'hist', 'bf16')."""
        c = self.cfg
        return (self.k_prof.draw(self.seed, "k/" + stream, n, c["dist"]),
                self.v_prof.draw(self.seed, "v/" + stream, n, c["dist"]))

    def queries(self, batch, stream="q"):
        return self.q_prof.draw(self.seed, stream, batch, "normal")


def page_permutation(seed, stream, n_pages, first=0):
    """A seeded random permutation of physical page ids first .. first+n_pages-1."""
    r = rng_for(seed, "pages/" + stream)
    return (first + r.permutation(n_pages)).astype(np.int32)


def mixed_lengths(seed, n, lo, hi, min_len):
    """Sequence lengths log-uniform in [lo, hi], raised to at least ``min_len``."""
    r = rng_for(seed, "lengths")
    raw = np.exp(r.uniform(math.log(lo), math.log(hi), size=n)).astype(np.int64)
    return raw, np.maximum(raw, min_len)


def pages_for(tokens):
    return (tokens + PAGE - 1) // PAGE
