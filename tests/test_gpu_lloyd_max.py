"""GPU parity of the Lloyd-Max codebook (OSCAR_CODEBOOK_LLOYD_MAX) through the C ABI.

The codebook is the rounded Gaussian Lloyd-Max quantizer the oracle defines in
oracle/lloyd_max.py (levels delta (-27, -8, 8, 27), delta = 0.45278 / 8;
(scale, zero) = (fp16(sigma delta), fp16(mu))). Source: QbitAI article on OSCAR,
closing part (the rotation paired with "a stronger Lloyd-Max codebook").

Write bar: codes bit-exact except off-by-one codes whose normalised value lies
within 1e-6 of the cut between the two levels; scale and zero within 1 fp16 ulp;
no byte outside the written rows changes. Decode bar: max-abs 2e-3 and relative
L2 1e-3 against the fp64 oracle on the same pages. Cases cover the write of
many tokens, the demote, d 64 and 128, groups 32, 64 and 128, GQ 1, 2, 4 and 8,
the GPU write feeding the GPU decode, and the shared-prefix call.
"""

import numpy as np
import pytest
import torch

import cases
from bit_kv_cache_write_gb300 import oscar as O
from bit_kv_cache_write_gb300 import synth
from oracle import cache, layout

pytestmark = pytest.mark.gpu
P = 16
LM = O.OSCAR_CODEBOOK_LLOYD_MAX


def _ctx(cfg, rk, rv, tk, tv):
    ctx = O.Oscar(n_layers=1, n_q_heads=cfg["h_q"], n_kv_heads=cfg["h_kv"], head_dim=cfg["d"], group=cfg["group"],
                  codebook=LM)
    ctx.calibrate_upload(0, rk, rv, tk, tv)
    return ctx


def _bf16(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev).to(torch.bfloat16)


@pytest.mark.parametrize("name,over,n", [
    ("tiny", {}, 700),
    ("qwen3_8b_bs1_100k", {}, 1500),
    ("qwen3_4b_b64_32k", {}, 300),
    ("qwen3_8b_bs1_100k", dict(group=32), 129),
    ("tiny", dict(group=64), 3),
], ids=lambda x: str(x))
def test_lloyd_max_write_parity(cuda, name, over, n):
    cfg = cases.workload(name, codebook="lloyd_max", **over)
    li, (rk, rv, tk, tv) = cases.calibration(cfg)
    geo = layout.Int2Geometry(cfg["d"], cfg["group"], cfg["h_kv"])
    n_pages = synth.pages_for(n) + 3
    slots = synth.rng_for(li.seed, "slots").permutation(n_pages * P)[:n].astype(np.int64)
    k, v = li.kv("write", n)
    ref = np.zeros(n_pages * geo.page_bytes, np.uint8)
    info = cache.write_tokens(ref, geo, k, v, slots, rk, rv, tk, tv, codebook="lloyd_max")
    ctx = _ctx(cfg, rk, rv, tk, tv)
    pool = torch.zeros(n_pages * geo.page_bytes, dtype=torch.uint8, device=cuda)
    ctx.write_tokens(0, _bf16(k, cuda), _bf16(v, cuda), torch.from_numpy(slots).to(cuda), pool)
    torch.cuda.synchronize()
    flips = cases.compare_int2(pool.cpu().numpy(), ref, geo, slots, info)
    print("tolerated boundary flips:", flips)


def test_lloyd_max_demote_parity(cuda):
    cfg = cases.workload("qwen3_8b_bs1_100k", codebook="lloyd_max")
    li, (rk, rv, tk, tv) = cases.calibration(cfg)
    d, h_kv = cfg["d"], cfg["h_kv"]
    geo = layout.Int2Geometry(d, cfg["group"], h_kv)
    n, bf_pages, i2_pages = 64, 8, 10
    k, v = li.kv("demote", bf_pages * P)
    bf = np.zeros((bf_pages, h_kv, 2, P, d), np.float32)
    bf[:, :, 0] = k.reshape(bf_pages, P, h_kv, d).transpose(0, 2, 1, 3)
    bf[:, :, 1] = v.reshape(bf_pages, P, h_kv, d).transpose(0, 2, 1, 3)
    rng = synth.rng_for(li.seed, "demote-slots")
    src = rng.permutation(bf_pages * P)[:n].astype(np.int64)
    dst = rng.permutation(i2_pages * P)[:n].astype(np.int64)
    ref = np.zeros(i2_pages * geo.page_bytes, np.uint8)
    info = cache.demote(bf.reshape(-1), ref, geo, src, dst, rk, rv, tk, tv, codebook="lloyd_max")
    ctx = _ctx(cfg, rk, rv, tk, tv)
    pool = torch.zeros(i2_pages * geo.page_bytes, dtype=torch.uint8, device=cuda)
    ctx.demote_recent(0, _bf16(bf, cuda), torch.from_numpy(src).to(cuda), pool, torch.from_numpy(dst).to(cuda))
    torch.cuda.synchronize()
    cases.compare_int2(pool.cpu().numpy(), ref, geo, dst, info)


DECODE_CASES = [
    ("tiny", {}, [1024], [320]),
    ("tiny", dict(group=64), [0, 333], [64, 320]),
    ("qwen3_8b_bs1_100k", {}, [3001], [320]),
    ("qwen3_8b_bs1_100k", dict(group=32), [777], [290]),
    ("qwen3_4b_b64_32k", {}, [2000, 16, 999], [320, 64, 100]),
    ("qwen3_32b_mixed16", {}, [1700, 640], [320, 320]),
    ("qwen3_8b_bs1_100k", dict(h_q=8, h_kv=8), [1200], [320]),
    ("qwen3_8b_bs1_100k", dict(h_q=16, h_kv=8), [640], [200]),
]


def _decode(case, ctx, dev):
    cfg = case.cfg
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    B = len(case.hist_lens)
    mh = int(case.hist_lens.max())
    ws = torch.empty(ctx.decode_workspace_size(B, mh), dtype=torch.uint8, device=dev)
    out = torch.full((B, cfg["h_q"], cfg["d"]), float("nan"), dtype=torch.float32, device=dev)
    ctx.decode(0, t(case.q).to(torch.bfloat16), t(case.int2_pool), t(case.int2_tables), t(case.hist_lens), mh,
               t(case.bf16_pool).to(torch.bfloat16), t(case.bf16_tables), t(case.bf16_lens), out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("name,over,hist,bf", DECODE_CASES, ids=lambda x: str(x))
def test_lloyd_max_decode_parity(cuda, name, over, hist, bf):
    cfg = cases.workload(name, codebook="lloyd_max", **over)
    case = cases.DecodeCase(cfg, hist, bf)
    got = _decode(case, _ctx(cfg, case.rk, case.rv, case.tk, case.tv), cuda)
    err, rel = cases.check_decode(got, case.oracle_out())
    print("max-abs %.3g rel-L2 %.3g" % (err, rel))


def test_lloyd_max_gpu_write_then_decode(cuda):
    """The GPU write of 2,000 history tokens feeding the GPU decode, against the oracle decode of the same
    GPU-written pages."""
    cfg = cases.workload("qwen3_8b_bs1_100k", codebook="lloyd_max")
    case = cases.DecodeCase(cfg, [2000], [320])
    ctx = _ctx(cfg, case.rk, case.rv, case.tk, case.tv)
    k, v = case.li.kv("hist/0", 2000)
    t = np.arange(2000)
    slots = case.int2_tables[0, t // P].astype(np.int64) * P + t % P
    pool = torch.zeros(case.int2_pool.size, dtype=torch.uint8, device=cuda)
    ctx.write_tokens(0, _bf16(k, cuda), _bf16(v, cuda), torch.from_numpy(slots).to(cuda), pool)
    torch.cuda.synchronize()
    case.int2_pool = pool.cpu().numpy()
    got = _decode(case, ctx, cuda)
    cases.check_decode(got, case.oracle_out())


def test_lloyd_max_shared_prefix(cuda):
    cfg = cases.workload("qwen3_8b_bs1_100k", codebook="lloyd_max")
    shared = 30
    case = cases.DecodeCase(cfg, [480 + 100, 480 + 900, 480], [320, 320, 64], shared_pages=shared)
    ctx = _ctx(cfg, case.rk, case.rv, case.tk, case.tv)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda)
    B = len(case.hist_lens)
    own_len = (case.hist_lens - shared * P).astype(np.int32)
    mh = int(own_len.max())
    ws = torch.empty(ctx.decode_shared_prefix_workspace_size(B, shared, mh), dtype=torch.uint8, device=cuda)
    out = torch.full((B, cfg["h_q"], cfg["d"]), float("nan"), dtype=torch.float32, device=cuda)
    ctx.decode_shared_prefix(0, t(case.q).to(torch.bfloat16), t(case.int2_pool), t(case.int2_tables[0, :shared]),
                             t(case.int2_tables[:, shared:]), t(own_len), mh, t(case.bf16_pool).to(torch.bfloat16),
                             t(case.bf16_tables), t(case.bf16_lens), out, ws)
    torch.cuda.synchronize()
    cases.check_decode(out.cpu().numpy(), case.oracle_out())
