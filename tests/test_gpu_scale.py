"""GPU decode parity at the full sizes of the batched and mixed-length workloads.

The caches are built exactly as the bench builds them: seeded K/V rows drawn on
the device and written through the library's own write path into permuted
pages, with the mixed batch's 16,384-token prefix referenced by every table.
The decode then runs over the whole batch, so it takes the launch plan the
bench times (many splits per sequence, several waves of CTAs, the last-CTA or
kernel merge, shared prefix pages read by every sequence). The fp64 oracle
decodes the same GPU-written pages for a sample of sequences and KV heads (all
query heads of each sampled KV head), element by element, against the decode
bar: max-abs 2e-3 and relative L2 1e-3.

Pages: QbitAI article on OSCAR, serving-pipeline part (paged KV, radix prefix
cache, multi-request serving); arXiv 2605.17757 v2 abstract (paged KV-cache
layouts and prefix caching preserved).
"""

import numpy as np
import pytest
import torch

import bench
import cases
from bit_kv_cache_write_gb300 import synth
from oracle import cache, layout

pytestmark = pytest.mark.gpu
P = 16


def decode_and_sample(name, dev, seqs, kv_heads):
    cfg = bench.workload_cfg(name)
    wl = bench.GpuWorkload(cfg, 1, dev)
    B, h_q, h_kv, d = wl.batch, cfg["h_q"], cfg["h_kv"], cfg["d"]
    wl.ctx.decode(0, wl.q_all[0], wl.int2_pools[0], wl.tables[0], wl.hist_len, wl.max_hist, wl.bf16_pools[0],
                  wl.bf16_table, wl.bf16_len, wl.out[0], wl.ws)
    torch.cuda.synchronize()
    got = wl.out[0].cpu().numpy()
    assert np.isfinite(got).all()

    geo = layout.Int2Geometry(d, cfg["group"], h_kv)
    rk, rv = wl.calib[0]
    g = h_q // h_kv
    heads = [h for kv in kv_heads for h in range(kv * g, (kv + 1) * g)]
    pb = wl.ctx.int2_page_bytes()
    pool_pages = wl.int2_pools[0].view(-1, pb)
    bf_pages = wl.bf16_pools[0]
    tables = wl.tables[0]
    q = wl.q_all[0].float().cpu().numpy().astype(np.float64)
    for b in seqs:
        n_hist = int(wl.hist[b])
        n_pages = synth.pages_for(n_hist)
        # this sequence's pages, in table order, as a compact pool with the identity table
        pool = pool_pages[tables[b, :n_pages].long()].cpu().numpy().reshape(-1)
        bt = torch.from_numpy(wl.bf16_table_np[b]).to(dev).long()
        bpool = bf_pages[bt].float().cpu().numpy().reshape(-1)
        want = cache.decode_batch(q[b:b + 1], pool, geo, np.arange(n_pages, dtype=np.int32)[None],
                                  np.array([n_hist]), bpool, np.arange(len(bt), dtype=np.int32)[None],
                                  np.array([wl.n_bf16]), rk, rv, d ** -0.5, heads=heads)
        err, rel = cases.check_decode(got[b, heads], want[0, heads])
        print("%s sequence %d (%d INT2 tokens): max-abs %.3g rel-L2 %.3g" % (name, b, n_hist, err, rel))
    return wl


def test_batch64_32k_full_size(cuda):
    """64 sequences x 32,768 tokens (G = 64, Laplace rows), 8 KV heads: 512 units in several waves."""
    wl = decode_and_sample("qwen3_4b_b64_32k", cuda, seqs=[0, 21, 42, 63], kv_heads=[0, 5])
    assert wl.batch == 64 and int(wl.hist.min()) == 32_768 - 320


def test_mixed16_shared_prefix_full_size(cuda):
    """16 log-uniform lengths up to 131,072, GQ 8, every table referencing the 16,384-token prefix."""
    cfg = bench.workload_cfg("qwen3_32b_mixed16")
    _, lengths = synth.mixed_lengths(cfg["seed"], cfg["batch"], cfg["len_lo"], cfg["len_hi"],
                                     cfg["shared_prefix"] + 320)
    order = np.argsort(lengths)
    seqs = sorted({int(order[-1]), int(order[0]), int(order[len(order) // 2]), int(order[-2])})
    wl = decode_and_sample("qwen3_32b_mixed16", cuda, seqs=seqs, kv_heads=[2, 7])
    tables = wl.tables[0].cpu().numpy()
    shared = wl.shared_hist // P
    assert shared == 1020 and (tables[:, :shared] == tables[0, :shared]).all()
