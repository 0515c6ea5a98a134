#!/usr/bin/env python
"""Benchmark of the OSCAR hot path on GB300: INT2 paged decode, bs1, 100k context, Qwen3-8B shape.

One step = one decode token through every layer of the model shape: per layer
one demote (the oldest BF16 recent token is rotated, clipped, quantized and
packed into an INT2 slot) and one paged decode (query rotation, split-K
attention over the INT2 history and the BF16 sink/recent segment,
online-softmax merge, un-rotation). The history length stays fixed from step
to step: the demoted token lands in a spare slot past the history.

`python bench.py [--gpus N] [--steps K] [--warmup W] [--impl oscar|reference]`
prints one JSON line. Under torchrun (N > 1) every rank runs its own replica
of the workload: there is no data-path collective, only the timing barrier.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT2 paged decode: KV tokens/s and achieved HBM GB/s (bs1, 100k ctx, Qwen3-8B shape)"
UNIT = "KV tokens/s"
P = 16


# --------------------------------------------------------------------------- distributed helpers

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x, device=None):
    """Max of a float across ranks (identity without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, max_seconds):
    """Aggregate throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / max_seconds


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- workload

def workload_cfg(name):
    from bit_kv_cache_write_gb300 import synth
    return dict(synth.WORKLOADS[name])


def demote_bytes(cfg, n):
    d, g, h = cfg["d"], cfg["group"], cfg["h_kv"]
    return n * h * 2 * (d * 2 + d // 4 + 4 * (d // g))


def token_bytes(cfg, int2_tokens, bf16_tokens):
    """Decode bytes: packed INT2 codes + fp16 scale/zero per INT2 token, BF16 K/V per BF16 token."""
    d, g, h = cfg["d"], cfg["group"], cfg["h_kv"]
    return int2_tokens * h * 2 * (d // 4 + 4 * (d // g)) + bf16_tokens * h * 2 * d * 2


class GpuWorkload:
    """Device-resident caches for every layer, written through the library's own write path.

    ``batch`` sequences, each a BF16 sink (64 tokens) + INT2 history + BF16 recent window (256).
    Mixed-length workloads draw lengths log-uniform and share a prefix: the INT2 pages of the first
    ``shared_prefix`` tokens and the sink pages are the same physical pages in every table. Every
    sequence owns one spare INT2 page, outside its history, that receives the per-step demote.
    Physical INT2 pages are a seeded permutation (non-contiguous tables)."""

    def __init__(self, cfg, layers, dev, seed_offset=0, shared_prefix_call=False):
        import numpy as np
        import torch
        from bit_kv_cache_write_gb300 import calibration, synth
        from bit_kv_cache_write_gb300 import oscar as O

        self.cfg, self.layers, self.dev = cfg, layers, dev
        d, h_kv, h_q, group = cfg["d"], cfg["h_kv"], cfg["h_q"], cfg["group"]
        B = cfg.get("batch", 1)
        sink, recent = synth.SINK, synth.RECENT
        self.batch, self.n_bf16 = B, sink + recent
        if "len_lo" in cfg:
            prefix = cfg["shared_prefix"]
            _, lengths = synth.mixed_lengths(cfg["seed"], B, cfg["len_lo"], cfg["len_hi"], prefix + self.n_bf16)
            hist = (lengths - self.n_bf16).astype(np.int64)
            shared_hist = prefix - sink                      # INT2 tokens of the shared prefix
        else:
            hist = np.full(B, cfg["hist"], np.int64)
            shared_hist = 0
        assert shared_hist % P == 0
        self.hist, self.max_hist, self.shared_hist = hist, int(hist.max()), shared_hist
        shared_pages = shared_hist // P
        pages = [synth.pages_for(int(x)) for x in hist]
        unique = [p_ - shared_pages for p_ in pages]
        total = shared_pages + sum(unique) + B
        max_pages = max(pages)
        self.codebook = cfg.get("codebook", "uniform")
        self.ctx = O.Oscar(n_layers=layers, n_q_heads=h_q, n_kv_heads=h_kv, head_dim=d, group=group,
                           codebook=O.OSCAR_CODEBOOK_LLOYD_MAX if self.codebook == "lloyd_max"
                           else O.OSCAR_CODEBOOK_UNIFORM)
        pb = self.ctx.int2_page_bytes()
        # the sink pages belong to the shared prefix when there is one; otherwise every sequence owns its sink
        self.shared_sink = shared_hist > 0
        sink_pages = sink // P
        bf_pages = (sink_pages if self.shared_sink else sink_pages * B) + (recent // P) * B
        gen = torch.Generator(device=dev)
        self.int2_pools, self.bf16_pools, self.tables, self.qs = [], [], [], []
        self.calib = []                                      # fp32 (R_k, R_v) per layer, as uploaded
        laplace = cfg["dist"] == "laplace"

        def rows(n):
            if not laplace:
                return torch.randn(n, h_kv, d, generator=gen, device=dev)
            # Laplace(0, 1) by inversion of a uniform draw: -sign(u) log(1 - 2|u|), u in (-1/2, 1/2)
            u = torch.rand(n, h_kv, d, generator=gen, device=dev) - 0.5
            return -torch.sign(u) * torch.log1p(-2.0 * u.abs().clamp(max=0.5 - 2.0 ** -25))

        chunk = 16384
        for layer in range(layers):
            li = synth.LayerInputs(cfg, layer + seed_offset)
            q_cal, k_cal, v_cal = li.calibration()
            rk, rv, tk, tv = calibration.calibrate_layer(q_cal, k_cal, v_cal, d ** -0.5, cfg["clip_ratio"])
            self.ctx.calibrate_upload(layer, rk, rv, tk, tv)
            self.calib.append((np.asarray(rk, np.float32), np.asarray(rv, np.float32)))
            perm = synth.page_permutation(li.seed, "int2", total).astype(np.int64)
            table = np.zeros((B, max_pages), np.int32)
            spare = np.zeros(B, np.int64)
            o = shared_pages
            for i in range(B):
                table[i, :shared_pages] = perm[:shared_pages]
                table[i, shared_pages:pages[i]] = perm[o:o + unique[i]]
                o += unique[i]
            spare[:] = perm[o:o + B]
            table_d = torch.from_numpy(table).to(dev)
            pool = torch.zeros(total * pb, dtype=torch.uint8, device=dev)
            gen.manual_seed(li.seed)
            km = torch.from_numpy(li.k_prof.mult).to(dev)
            vm = torch.from_numpy(li.v_prof.mult).to(dev)
            # token ranges written: the shared prefix once (through sequence 0's table), then each
            # sequence's own history
            ranges = [(0, 0, shared_hist)] + [(i, shared_hist, int(hist[i])) for i in range(B)]
            for i, t_lo, t_hi in ranges:
                for t0 in range(t_lo, t_hi, chunk):
                    n = min(chunk, t_hi - t0)
                    k = (rows(n) * km).to(torch.bfloat16)
                    v = (rows(n) * vm).to(torch.bfloat16)
                    t = torch.arange(t0, t0 + n, device=dev)
                    slots = table_d[i, t // P].to(torch.int64) * P + t % P
                    self.ctx.write_tokens(layer, k, v, slots, pool)
            bf = torch.stack([rows(bf_pages * P).view(bf_pages, P, h_kv, d).transpose(1, 2) for _ in range(2)], 2)
            bf = bf * torch.stack([km, vm], dim=1)[None, :, :, None, :]
            self.bf16_pools.append(bf.to(torch.bfloat16).contiguous())
            self.int2_pools.append(pool)
            self.tables.append(table_d)
            self.qs.append(torch.randn(B, h_q, d, generator=gen, device=dev).to(torch.bfloat16))
        bt = np.zeros((B, self.n_bf16 // P), np.int32)
        per_seq = (recent // P) + (0 if self.shared_sink else sink_pages)
        first_own = sink_pages if self.shared_sink else 0
        for i in range(B):
            if self.shared_sink:
                bt[i, :sink_pages] = np.arange(sink_pages)
            bt[i, first_own:] = first_own + per_seq * i + np.arange(per_seq)
        self.bf16_table_np = bt
        self.bf16_table = torch.from_numpy(bt).to(dev)
        self.hist_len = torch.from_numpy(hist.astype(np.int32)).to(dev)
        self.bf16_len = torch.full((B,), self.n_bf16, dtype=torch.int32, device=dev)
        # demote: each sequence's oldest recent token (row 0 of its first recent page) -> row 0 of
        # its spare INT2 page (same spare page ids in every layer's pool: the permutation per layer
        # differs, so the spare ids are taken per layer below)
        self.src = torch.from_numpy((bt[:, sink_pages].astype(np.int64)) * P).to(dev)
        self.dsts = []
        for layer in range(layers):
            li = synth.LayerInputs(cfg, layer + seed_offset)
            perm = synth.page_permutation(li.seed, "int2", total).astype(np.int64)
            self.dsts.append(torch.from_numpy(perm[total - B:] * P).to(dev))
        # the shared-prefix call takes the prefix pages once and each sequence's own pages after them
        self.shared_prefix_call = shared_prefix_call and shared_pages > 0
        if self.shared_prefix_call:
            self.prefix_tables = [t[0, :shared_pages].contiguous() for t in self.tables]
            self.own_tables = [t[:, shared_pages:].contiguous() for t in self.tables]
            own = (hist - shared_hist).astype(np.int32)
            self.own_len = torch.from_numpy(own).to(dev)
            self.own_max = int(own.max())
            ws_bytes = self.ctx.decode_shared_prefix_workspace_size(B, shared_pages, self.own_max)
        else:
            ws_bytes = self.ctx.decode_workspace_size(B, self.max_hist)
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        self.out = torch.empty(layers, B, h_q, d, dtype=torch.float32, device=dev)
        self.q_all = torch.stack(self.qs, 0).contiguous()
        self.side = torch.cuda.Stream(device=dev)
        self.demoted = [torch.cuda.Event() for _ in range(layers)]
        # bytes and tokens of one decode of one layer
        self.tokens_per_layer = int(hist.sum()) + B * self.n_bf16
        self.logical_bytes = token_bytes(cfg, int(hist.sum()), B * self.n_bf16)
        self.unique_bytes = token_bytes(cfg, shared_hist + int((hist - shared_hist).sum()),
                                        (sink if self.shared_sink else sink * B) + B * recent)
        torch.cuda.synchronize()

    def step(self):
        """Per layer: demote the oldest recent token of every sequence, then decode. The demotes run
        on a side stream (they depend on nothing the decodes produce); decode(layer) waits for
        demote(layer)."""
        import torch
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)
        for layer in range(self.layers):
            with torch.cuda.stream(self.side):
                self.ctx.demote_recent(layer, self.bf16_pools[layer], self.src, self.int2_pools[layer], self.dsts[layer])
                self.demoted[layer].record(self.side)
            main.wait_event(self.demoted[layer])
            if self.shared_prefix_call:
                self.ctx.decode_shared_prefix(layer, self.q_all[layer], self.int2_pools[layer],
                                              self.prefix_tables[layer], self.own_tables[layer], self.own_len,
                                              self.own_max, self.bf16_pools[layer], self.bf16_table, self.bf16_len,
                                              self.out[layer], self.ws)
            else:
                self.ctx.decode(layer, self.q_all[layer], self.int2_pools[layer], self.tables[layer], self.hist_len,
                                self.max_hist, self.bf16_pools[layer], self.bf16_table, self.bf16_len,
                                self.out[layer], self.ws)
        main.wait_stream(self.side)



def write_bytes(cfg, n):
    """Write-path bytes per call: BF16 K/V rows read + packed INT2 codes and fp16 scale/zero written."""
    d, g, h = cfg["d"], cfg["group"], cfg["h_kv"]
    return n * h * 2 * (d * 2 + d // 4 + 4 * (d // g))


def bench_write(dev, steps, warmup):
    """Bulk write of 131,072 prefill tokens x 8 KV heads (K and V) into a paged INT2 cache, and the
    steady-state demote of one token for each of 256 sequences. Device-resident inputs larger than
    L2; CUDA events on the launching stream."""
    import numpy as np
    import torch
    from bit_kv_cache_write_gb300 import calibration, synth
    from bit_kv_cache_write_gb300 import oscar as O

    cfg = workload_cfg("bulk_write_131k")
    n, d, h_kv, group = cfg["tokens"], cfg["d"], cfg["h_kv"], cfg["group"]
    ctx = O.Oscar(n_layers=1, n_q_heads=cfg["h_q"], n_kv_heads=h_kv, head_dim=d, group=group)
    li = synth.LayerInputs(cfg, 0)
    q_cal, k_cal, v_cal = li.calibration()
    rk, rv, tk, tv = calibration.calibrate_layer(q_cal, k_cal, v_cal, d ** -0.5, cfg["clip_ratio"])
    ctx.calibrate_upload(0, rk, rv, tk, tv)
    gen = torch.Generator(device=dev)
    gen.manual_seed(li.seed)
    km = torch.from_numpy(li.k_prof.mult).to(dev)
    vm = torch.from_numpy(li.v_prof.mult).to(dev)
    k = (torch.randn(n, h_kv, d, generator=gen, device=dev) * km).to(torch.bfloat16)
    v = (torch.randn(n, h_kv, d, generator=gen, device=dev) * vm).to(torch.bfloat16)
    pages = synth.pages_for(n)
    perm = torch.from_numpy(synth.page_permutation(li.seed, "bulk", pages).astype(np.int64)).to(dev)
    t = torch.arange(n, device=dev)
    slots = perm[t // P] * P + t % P
    pool = torch.zeros(pages * ctx.int2_page_bytes(), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def timed(fn, reps):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / reps

    us = timed(lambda: ctx.write_tokens(0, k, v, slots, pool), steps)
    nbytes = write_bytes(cfg, n)
    peak, peak_kind = measured_peak()
    bulk = {"workload": "bulk_write_131k", "tokens": n, "kv_heads": h_kv, "head_dim": d, "group": group,
            "us_per_call": us, "tokens_per_s": n / (us * 1e-6), "algorithmic_bytes": nbytes,
            "roofline": {"bound": "hbm", "achieved": nbytes / (us * 1e-6) / 1e9, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": nbytes / (us * 1e-6) / 1e9 / peak,
                         "traffic": kernel_traffic("write", "bulk_write_131k")},
            "l2": "inputs larger than L2 (%.0f MB of K/V rows)" % (n * h_kv * d * 4 / 1e6)}

    # demote: one token per sequence for 256 sequences, from BF16 recent pages into INT2 slots
    nb = cfg["demote_batch"]
    bf = (torch.randn(nb, h_kv, 2, P, d, generator=gen, device=dev)
          * torch.stack([km, vm], dim=1)[None, :, :, None, :]).to(torch.bfloat16).contiguous()
    src = torch.arange(nb, device=dev, dtype=torch.int64) * P          # row 0 of each sequence's oldest page
    dst = perm[:nb] * P + 3
    us_d = timed(lambda: ctx.demote_recent(0, bf, src, pool, dst), steps)
    demote = {"batch": nb, "us_per_call": us_d, "tokens_per_s": nb / (us_d * 1e-6),
              "algorithmic_bytes": write_bytes(cfg, nb)}
    return {"bulk": bulk, "demote": demote}


def bench_calibration(dev, steps, warmup):
    """GPU calibration targets (Q^T Q and V^T S^T S V per KV head, fp64) at the 1,024-sample calibration
    size of the Qwen3-8B-shape workload: 1,024 queries of each of the 32 query heads and 1,024 keys and
    values of each of the 8 KV heads, d = 128. CUDA events on the launching stream."""
    import torch
    from bit_kv_cache_write_gb300 import oscar as O, synth
    cfg = workload_cfg("qwen3_8b_bs1_100k")
    q_cal, k_cal, v_cal = synth.LayerInputs(cfg, 0).calibration()
    q = torch.from_numpy(q_cal).to(dev)
    k = torch.from_numpy(k_cal).to(dev)
    v = torch.from_numpy(v_cal).to(dev)
    n, h_q, d = q.shape
    m, h_kv = k.shape[0], k.shape[1]
    tk = torch.empty(h_kv, d, d, dtype=torch.float64, device=dev)
    tv = torch.empty_like(tk)
    ws = torch.empty(O.oscar_calibration_workspace_size(n, h_q, h_kv, d), dtype=torch.uint8, device=dev)
    sm = d ** -0.5
    for _ in range(warmup):
        O.oscar_calibration_targets(q, k, v, sm, tk, tv, ws)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    a.record(stream)
    for _ in range(steps):
        O.oscar_calibration_targets(q, k, v, sm, tk, tv, ws)
    b.record(stream)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / steps
    rows = n * (h_q // h_kv)
    # fp64 flops: two full d x d Gram products per KV head, and per (row, head) m x d logits and m x d S.V
    flops = h_kv * (2 * 2.0 * rows * d * d + rows * 2 * 2.0 * m * d)
    peak = 1250.0   # GFLOP/s: the part's nominal fp64 rate (not measured on this machine)
    return {"workload": "calibration targets: %d queries x %d query heads, %d keys x %d KV heads, d = %d"
                        % (n, h_q, m, h_kv, d),
            "us_per_call": us, "fp64_gflop": flops / 1e9,
            "roofline": {"bound": "fp64", "achieved": flops / (us * 1e-6) / 1e9, "peak": peak,
                         "peak_kind": "nominal (fp64 is not in the measured peaks)", "unit": "GFLOP/s",
                         "frac": flops / (us * 1e-6) / 1e9 / peak}}


def kernel_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get("%s/%s" % (kernel, workload))
    if not rec:
        return None
    src = os.path.join(ROOT, "bit_kv_cache_write_gb300", "csrc", rec["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != rec["source_sha"]:
        return None
    return rec["bytes_per_launch"]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        return float(json.load(open(path))["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------------------- CPU oracle baseline

def oracle_sample(cfg, sample_hist, layer=0):
    """Build the oracle-side cache for a bounded sample (one layer, ``sample_hist`` history tokens)."""
    from bit_kv_cache_write_gb300 import synth
    from oracle.paged_case import DecodeCase
    c = dict(cfg)
    c["hist"] = sample_hist
    case = DecodeCase(c, [sample_hist], [synth.SINK + synth.RECENT], layer=layer, extra_pages=1)
    return case


def time_oracle_step(case):
    """One oracle pass of the hot path on the sample: demote one BF16 token, then decode every head."""
    import numpy as np
    from oracle import cache
    geo = case.geo
    spare = np.zeros(geo.page_bytes, np.uint8)
    t0 = time.perf_counter()
    cache.demote(case.bf16_pool, spare, geo, [synth_sink()], [0], case.rk, case.rv, case.tk, case.tv)
    case.oracle_out()
    return time.perf_counter() - t0


def synth_sink():
    from bit_kv_cache_write_gb300 import synth
    return synth.SINK


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, cfg, world, rank):
    """--impl reference: the fp64 CPU oracle timed on the host cores, on a bounded sample of the workload."""
    if rank != 0:
        return 0
    sample_hist = args.oracle_hist
    case = oracle_sample(cfg, sample_hist)
    tokens = sample_hist + case.bf16_lens[0]
    for _ in range(args.warmup):
        time_oracle_step(case)
    times = [time_oracle_step(case) for _ in range(args.steps)]
    total = sum(times)
    value = tokens * args.steps / total
    sample = "1 layer, %d INT2 + %d BF16 tokens, %d Q / %d KV heads, d=%d, G=%d; demote 1 token + decode" % (
        sample_hist, case.bf16_lens[0], cfg["h_q"], cfg["h_kv"], cfg["d"], cfg["group"])
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "batch": 1, "context": cfg.get("hist", sample_hist) + 320,
                       "note": "each step is a bounded sample of the workload"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------- main

def measure_decode(cfg, layers, dev, steps, warmup, local, seed_offset=0, shared_prefix_call=False):
    """Build a workload's caches, capture one step in a CUDA graph and time K replays (max over ranks).

    Returns (workload, graph, metrics). The metrics hold the step time, per-kernel CUDA-event averages
    from an eager pass of the same launches, and the split kernel's achieved GB/s on unique bytes."""
    import torch
    from bit_kv_cache_write_gb300 import oscar as O
    wl = GpuWorkload(cfg, layers, dev, seed_offset=seed_offset, shared_prefix_call=shared_prefix_call)
    stream = torch.cuda.current_stream()

    # ---- capture one step in a CUDA graph (the library launches on the capturing stream)
    wl.step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        wl.step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K graph replays; every step reads more distinct pages than L2 holds
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        stop.record(stream)
        torch.cuda.synchronize()
        barrier()
    sec = start.elapsed_time(stop) / 1e3
    max_sec = max_over_ranks(sec, dev)

    # ---- per-kernel durations (same launches, eager, events around each kernel on its stream)
    wl.ctx.profile_enable(True)
    for _ in range(steps):
        wl.step()
    torch.cuda.synchronize()
    wl.ctx.profile_enable(False)
    kt = {}
    for name, kid in (("write", O.OSCAR_KERNEL_WRITE), ("q_rotate", O.OSCAR_KERNEL_QROT),
                      ("split", O.OSCAR_KERNEL_SPLIT), ("merge", O.OSCAR_KERNEL_MERGE)):
        ms, n = wl.ctx.profile_read(kid)
        kt[name] = {"launches": n, "avg_us": 1e3 * ms / max(n, 1)}
    # roofline on unique bytes (a page shared by several tables counts once: conservative)
    split_bytes = wl.unique_bytes
    achieved = split_bytes / (kt["split"]["avg_us"] * 1e-6) / 1e9
    launches = sum(v["launches"] for v in kt.values()) // max(steps, 1)
    return wl, graph, {"max_sec": max_sec, "kernels": kt, "clocks": clocks.summary(), "achieved": achieved,
                       "split_bytes": split_bytes, "launches_per_step": launches}


def workload_line(name, layers, dev, steps, warmup, local, shared_prefix_call=False, codebook="uniform"):
    """Throughput of one more decode workload at a reduced layer count (its per-layer pages exceed L2).
    shared_prefix_call: decode through oscar_decode_shared_prefix (the prefix pages given once);
    codebook: "uniform" or "lloyd_max" (the cache is written and decoded with it)."""
    import torch
    cfg = workload_cfg(name)
    cfg["codebook"] = codebook
    wl, graph, m = measure_decode(cfg, layers, dev, steps, warmup, local, shared_prefix_call=shared_prefix_call)
    peak, peak_kind = measured_peak()
    us_layer = 1e6 * m["max_sec"] / steps / layers
    split_us = m["kernels"]["split"]["avg_us"]
    res = {"layers": layers, "batch": wl.batch, "h_q": cfg["h_q"], "h_kv": cfg["h_kv"], "group": cfg["group"],
           "int2_history": {"min": int(wl.hist.min()), "max": int(wl.hist.max()), "sum": int(wl.hist.sum())},
           "shared_prefix_int2_tokens": wl.shared_hist,
           "call": "oscar_decode_shared_prefix" if wl.shared_prefix_call else "oscar_decode",
           "codebook": codebook,
           "us_per_layer": us_layer, "kv_tokens_per_s": wl.tokens_per_layer / (us_layer * 1e-6),
           "kernels": m["kernels"],
           "split_roofline": {"bound": "hbm", "achieved": m["achieved"], "peak": peak, "peak_kind": peak_kind,
                              "unit": "GB/s", "frac": m["achieved"] / peak,
                              "algorithmic_bytes_per_launch": wl.unique_bytes,
                              "logical_bytes_per_launch": wl.logical_bytes,
                              "logical_gbs": wl.logical_bytes / (split_us * 1e-6) / 1e9,
                              "traffic": kernel_traffic("split", name + ("_shared_prefix" if shared_prefix_call else "")
                                                        + ("_lloyd_max" if codebook == "lloyd_max" else ""))},
           "step_gbs": (wl.unique_bytes + demote_bytes(cfg, wl.batch)) / (us_layer * 1e-6) / 1e9,
           "clocks": m["clocks"],
           "l2": "inputs larger than L2: %.2f GB of distinct pages per step" % (layers * wl.unique_bytes / 1e9)}
    del graph, wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["oscar", "reference"], default="oscar")
    ap.add_argument("--workload", default="qwen3_8b_bs1_100k")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (0: the workload's)")
    ap.add_argument("--oracle-hist", type=int, default=24_992, help="INT2 tokens in the oracle's bounded sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-write", action="store_true", help="skip the bulk-write / demote measurement")
    ap.add_argument("--only-write", action="store_true", help="print only the bulk-write / demote measurement")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the batch-64 and mixed-batch decode workloads (measured at N = 1 only)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank, world, local = dist_env()
    cfg = workload_cfg(args.workload)
    if args.impl == "reference":
        return run_reference(args, cfg, world, rank)

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from bit_kv_cache_write_gb300 import oscar as O

    if args.only_write:
        if rank == 0:
            print(json.dumps({"write": bench_write(dev, args.steps, args.warmup)}))
        return 0

    layers = args.layers or cfg["layers"]
    wl, graph, m = measure_decode(cfg, layers, dev, args.steps, args.warmup, local, seed_offset=1000 * rank)
    stream = torch.cuda.current_stream()
    max_sec = m["max_sec"]
    tokens_per_step = layers * wl.tokens_per_layer
    value = whole_job_rate(tokens_per_step * args.steps, world, max_sec)
    ms_per_step = 1e3 * max_sec / args.steps
    step_bytes = layers * (wl.unique_bytes + demote_bytes(cfg, wl.batch))
    kt, clocks, achieved, split_bytes = m["kernels"], m["clocks"], m["achieved"], m["split_bytes"]
    peak, peak_kind = measured_peak()

    # ---- end to end through the public API with host buffers: q in (pinned H2D), outputs out (D2H)
    q_host = wl.q_all.cpu().pin_memory()
    out_host = torch.empty(wl.out.shape, dtype=torch.float32).pin_memory()
    for _ in range(2):
        wl.q_all.copy_(q_host, non_blocking=True)
        graph.replay()
        out_host.copy_(wl.out, non_blocking=True)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        wl.q_all.copy_(q_host, non_blocking=True)
        graph.replay()
        out_host.copy_(wl.out, non_blocking=True)
        stream.synchronize()
    e2e_sec = max_over_ranks(time.perf_counter() - t0, dev)
    e2e_value = whole_job_rate(tokens_per_step * args.steps, world, e2e_sec)

    # ---- CPU oracle baseline (rank 0, N = 1 only), bounded sample
    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        case = oracle_sample(cfg, args.oracle_hist)
        time_oracle_step(case)
        reps, spent = 0, 0.0
        while spent < 10.0 and reps < 50:
            spent += time_oracle_step(case)
            reps += 1
        tok = args.oracle_hist + case.bf16_lens[0]
        cpu_baseline = {"value": tok * reps / spent, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                        "sample": "%d oracle steps on 1 layer with %d INT2 + %d BF16 tokens (demote 1 token + "
                                  "decode all %d query heads), fp64 NumPy" % (reps, args.oracle_hist,
                                                                              case.bf16_lens[0], cfg["h_q"])}

    write = bench_write(dev, max(args.steps, 5), args.warmup) if rank == 0 and not args.no_write else None
    calib = bench_calibration(dev, 5, 3) if rank == 0 and not args.no_write else None

    # ---- the batched and mixed-length decode workloads (N = 1), at layer counts whose pages exceed L2
    workloads = None
    if world == 1 and not args.no_workloads:
        workloads = {"qwen3_4b_b64_32k": workload_line("qwen3_4b_b64_32k", 2, dev, args.steps, args.warmup, local),
                     "qwen3_32b_mixed16": workload_line("qwen3_32b_mixed16", 4, dev, args.steps, args.warmup,
                                                        local),
                     "qwen3_32b_mixed16_shared_prefix": workload_line("qwen3_32b_mixed16", 4, dev, args.steps,
                                                                      args.warmup, local, shared_prefix_call=True),
                     "qwen3_8b_bs1_100k_lloyd_max": workload_line("qwen3_8b_bs1_100k", 8, dev, args.steps,
                                                                  args.warmup, local, codebook="lloyd_max")}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload, "batch": wl.batch,
                       "context": int(wl.hist[0]) + wl.n_bf16 if wl.batch == 1 else "per sequence, see int2_history",
                       "int2_history": int(wl.hist[0]) if wl.batch == 1 else
                       {"min": int(wl.hist.min()), "max": int(wl.hist.max()), "sum": int(wl.hist.sum())},
                       "shared_prefix_int2_tokens": wl.shared_hist,
                       "bf16_tokens": wl.n_bf16, "layers": layers, "h_q": cfg["h_q"], "h_kv": cfg["h_kv"],
                       "head_dim": cfg["d"], "group": cfg["group"], "page_size": P,
                       "step": "per layer: demote 1 token per sequence (side stream) + decode after it; "
                               "one CUDA graph per step",
                       "l2": "inputs larger than L2: %.2f GB of distinct pages per step" % (step_bytes / 1e9),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "hbm_gbs_step": step_bytes * args.steps * world / max_sec / 1e9,
            "us_per_layer": 1e6 * max_sec / args.steps / layers,
            "roofline": {"bound": "hbm", "kernel": "split (INT2 history + BF16 segment)", "achieved": achieved,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": kernel_traffic("split", args.workload),
                         "algorithmic_bytes_per_launch": split_bytes,
                         "logical_bytes_per_launch": wl.logical_bytes},
            "kernels": kt,
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": q_host.numel() * 2,
                    "d2h_bytes_per_step": out_host.numel() * 4},
            "gpu_launches": args.steps * m["launches_per_step"],
            "cpu_baseline": cpu_baseline,
            "write": write,
            "workloads": workloads,
            "calibration": calib,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
