"""GPU parity of the shared-prefix (cascade) decode, oscar_decode_shared_prefix, through the C ABI.

Every sequence of the batch starts with the same INT2 pages (a radix
prefix-cache hit). The call is given those pages once plus each sequence's own
pages; its result must equal the fp64 oracle's decode over the concatenated
tables (max-abs 2e-3, relative L2 1e-3) and agree with oscar_decode over the
same full tables. Cases cover GQ 2, 4 and 8, groups 32, 64 and 128, a batch
that leaves warps of the last prefix group idle, sequences with nothing after
the prefix or without BF16 tokens, a batch of one, and the mixed 16-sequence
workload at full size (16,384-token prefix, lengths up to 131,072).

Pages: QbitAI article on OSCAR, serving-pipeline part (radix prefix cache);
arXiv 2605.17757 v2 abstract (prefix caching preserved).
"""

import numpy as np
import pytest
import torch

import bench
import cases
from bit_kv_cache_write_gb300 import oscar as O
from bit_kv_cache_write_gb300 import synth
from oracle import cache, layout

pytestmark = pytest.mark.gpu
P = 16

CASES = [
    ("tiny", {}, [160 + 40, 160, 160 + 300, 160 + 5, 160 + 64], [320, 17, 0, 320, 100], 10),
    ("tiny", dict(group=64), [512 + 33], [64], 32),
    ("qwen3_8b_bs1_100k", {}, [800 + 300, 800 + 1000, 800], [320, 320, 320], 50),
    ("qwen3_4b_b64_32k", {}, [1024 + 100, 1024 + 555, 1024 + 17, 1024 + 999], [320] * 4, 64),
    ("qwen3_32b_mixed16", {}, [640 + 10, 640 + 700, 640 + 333, 640, 640 + 1200, 640 + 64], [320] * 6, 40),
]


def _decode_both(case, dev, shared):
    cfg = case.cfg
    ctx = O.Oscar(n_layers=1, n_q_heads=cfg["h_q"], n_kv_heads=cfg["h_kv"], head_dim=cfg["d"], group=cfg["group"])
    ctx.calibrate_upload(0, case.rk, case.rv, case.tk, case.tv)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    B = len(case.hist_lens)
    q = t(case.q).to(torch.bfloat16)
    pool = t(case.int2_pool)
    bf = t(case.bf16_pool).to(torch.bfloat16)
    bt, bl = t(case.bf16_tables), t(case.bf16_lens)
    # shared-prefix call: the prefix once, then each sequence's own pages
    prefix = t(case.int2_tables[0, :shared])
    own = t(case.int2_tables[:, shared:])
    own_len = case.hist_lens - shared * P
    assert (own_len >= 0).all()
    mh = int(own_len.max())
    ws = torch.empty(ctx.decode_shared_prefix_workspace_size(B, shared, mh), dtype=torch.uint8, device=dev)
    got = torch.full((B, cfg["h_q"], cfg["d"]), float("nan"), dtype=torch.float32, device=dev)
    ctx.decode_shared_prefix(0, q, pool, prefix, own, t(own_len.astype(np.int32)), mh, bf, bt, bl, got, ws)
    # the plain call over the full tables
    mh_full = int(case.hist_lens.max())
    ws2 = torch.empty(ctx.decode_workspace_size(B, mh_full), dtype=torch.uint8, device=dev)
    plain = torch.empty_like(got)
    ctx.decode(0, q, pool, t(case.int2_tables), t(case.hist_lens), mh_full, bf, bt, bl, plain, ws2)
    torch.cuda.synchronize()
    return got.cpu().numpy(), plain.cpu().numpy()


@pytest.mark.parametrize("name,over,hist,bf,shared", CASES, ids=lambda x: str(x))
def test_shared_prefix_parity(cuda, name, over, hist, bf, shared):
    cfg = cases.workload(name, **over)
    case = cases.DecodeCase(cfg, hist, bf, shared_pages=shared)
    got, plain = _decode_both(case, cuda, shared)
    want = case.oracle_out()
    err, rel = cases.check_decode(got, want)
    cases.check_decode(got, plain)
    print("max-abs %.3g rel-L2 %.3g" % (err, rel))


def test_shared_prefix_of_zero_pages_is_the_plain_decode(cuda):
    cfg = cases.workload("tiny")
    case = cases.DecodeCase(cfg, [300, 41], [320, 64])
    got, plain = _decode_both(case, cuda, 0)
    cases.check_decode(got, case.oracle_out())
    assert np.abs(got - plain).max() <= 1e-6 * max(1.0, np.abs(plain).max())


def test_mixed16_full_size_through_the_shared_prefix_call(cuda):
    """The mixed 16-sequence workload as the bench builds it (GPU-written cache, 1,020 shared INT2 pages),
    decoded through the shared-prefix call; sampled sequences and KV heads against the fp64 oracle."""
    cfg = bench.workload_cfg("qwen3_32b_mixed16")
    wl = bench.GpuWorkload(cfg, 1, cuda)
    shared = wl.shared_hist // P
    tables = wl.tables[0]
    own_len = (wl.hist - wl.shared_hist).astype(np.int32)
    mh = int(own_len.max())
    B, h_q, h_kv, d = wl.batch, cfg["h_q"], cfg["h_kv"], cfg["d"]
    ws = torch.empty(wl.ctx.decode_shared_prefix_workspace_size(B, shared, mh), dtype=torch.uint8, device=cuda)
    out = torch.full((B, h_q, d), float("nan"), dtype=torch.float32, device=cuda)
    wl.ctx.decode_shared_prefix(0, wl.q_all[0], wl.int2_pools[0], tables[0, :shared].contiguous(),
                                tables[:, shared:].contiguous(), torch.from_numpy(own_len).to(cuda), mh,
                                wl.bf16_pools[0], wl.bf16_table, wl.bf16_len, out, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    geo = layout.Int2Geometry(d, cfg["group"], h_kv)
    rk, rv = wl.calib[0]
    g = h_q // h_kv
    order = np.argsort(wl.hist)
    pb = wl.ctx.int2_page_bytes()
    pool_pages = wl.int2_pools[0].view(-1, pb)
    q = wl.q_all[0].float().cpu().numpy().astype(np.float64)
    for b in sorted({int(order[-1]), int(order[0]), int(order[len(order) // 2])}):
        heads = [h for kv in (1, 6) for h in range(kv * g, (kv + 1) * g)]
        n_hist = int(wl.hist[b])
        n_pages = synth.pages_for(n_hist)
        pool = pool_pages[tables[b, :n_pages].long()].cpu().numpy().reshape(-1)
        btab = torch.from_numpy(wl.bf16_table_np[b]).to(cuda).long()
        bpool = wl.bf16_pools[0][btab].float().cpu().numpy().reshape(-1)
        want = cache.decode_batch(q[b:b + 1], pool, geo, np.arange(n_pages, dtype=np.int32)[None],
                                  np.array([n_hist]), bpool, np.arange(len(btab), dtype=np.int32)[None],
                                  np.array([wl.n_bf16]), rk, rv, d ** -0.5, heads=heads)
        err, rel = cases.check_decode(got[b, heads], want[0, heads])
        print("sequence %d (%d INT2 tokens): max-abs %.3g rel-L2 %.3g" % (b, n_hist, err, rel))
