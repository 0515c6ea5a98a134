"""GPU parity of paged INT2 decode (through the C ABI) against the fp64 oracle on the same cache.

Bar: max-abs 2e-3 and relative L2 1e-3 against the oracle, which decodes the
same oracle-written INT2/BF16 pools that are uploaded to the GPU.
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


def run_gpu(case, dev, debug=0, ctx=None, max_hist=None):
    cfg = case.cfg
    if ctx is None:
        ctx = O.Oscar(n_layers=1, n_q_heads=cfg["h_q"], n_kv_heads=cfg["h_kv"], head_dim=cfg["d"],
                      group=cfg["group"], debug_bounds=debug)
        ctx.calibrate_upload(0, case.rk, case.rv, case.tk, case.tv)
    B = len(case.hist_lens)
    mh = int(case.hist_lens.max()) if max_hist is None else max_hist
    ws = torch.empty(ctx.decode_workspace_size(B, mh), dtype=torch.uint8, device=dev)
    out = torch.full((B, cfg["h_q"], cfg["d"]), float("nan"), dtype=torch.float32, device=dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    ctx.decode(0, t(case.q).to(torch.bfloat16), t(case.int2_pool), t(case.int2_tables), t(case.hist_lens), mh,
               t(case.bf16_pool).to(torch.bfloat16), t(case.bf16_tables), t(case.bf16_lens), out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ctx


DECODE_CASES = [
    ("tiny", {}, [1024], [320], 0, 0),
    ("tiny", {}, [1000], [301], 0, 0),
    ("tiny", {}, [0, 37, 1024], [320, 0, 17], 0, 0),
    ("tiny", dict(group=64), [513], [64], 0, 0),
    ("qwen3_8b_bs1_100k", {}, [3001], [320], 0, 0),
    ("qwen3_8b_bs1_100k", dict(group=32), [777], [290], 0, 0),
    ("qwen3_4b_b64_32k", {}, [2000, 1500, 16, 999], [320, 320, 64, 100], 0, 0),
    ("qwen3_32b_mixed16", {}, [1700, 2100, 1640], [320, 320, 320], 50, 4),
    ("qwen3_8b_bs1_100k", dict(h_q=8, h_kv=8), [1200], [320], 0, 0),
    ("qwen3_8b_bs1_100k", dict(h_q=16, h_kv=8), [640], [200], 0, 0),
    ("qwen3_8b_bs1_100k", dict(rotation="hadamard"), [2500], [320], 0, 0),      # Hadamard-only ablation
]


@pytest.mark.parametrize("name,over,hist,bf,shared,shared_bf", DECODE_CASES, ids=lambda x: str(x))
def test_decode_parity(cuda, name, over, hist, bf, shared, shared_bf):
    cfg = cases.workload(name, **over)
    case = cases.DecodeCase(cfg, hist, bf, shared_pages=shared, shared_bf16_pages=shared_bf)
    got, _ = run_gpu(case, cuda)
    want = case.oracle_out()
    err, rel = cases.check_decode(got, want)
    print("max-abs %.3g rel-L2 %.3g" % (err, rel))


def test_sequence_without_tokens_gives_zeros(cuda):
    cfg = cases.workload("tiny")
    case = cases.DecodeCase(cfg, [0, 100], [0, 5])
    got, _ = run_gpu(case, cuda)
    assert np.all(got[0] == 0)
    cases.check_decode(got, case.oracle_out())


def test_max_hist_larger_than_lengths(cuda):
    cfg = cases.workload("tiny")
    case = cases.DecodeCase(cfg, [200, 33], [320, 320], stride_pad=40)
    got, _ = run_gpu(case, cuda, max_hist=16 * case.int2_stride)
    cases.check_decode(got, case.oracle_out())


def test_end_to_end_gpu_write_then_decode(cuda):
    """GPU write path feeding GPU decode, against oracle write feeding oracle decode."""
    cfg = cases.workload("tiny")
    case = cases.DecodeCase(cfg, [1024], [320])
    ctx = O.Oscar(n_layers=1, n_q_heads=cfg["h_q"], n_kv_heads=cfg["h_kv"], head_dim=cfg["d"], group=cfg["group"])
    ctx.calibrate_upload(0, case.rk, case.rv, case.tk, case.tv)
    k, v = case.li.kv("hist/0", 1024)
    t = np.arange(1024)
    slots = case.int2_tables[0, t // P].astype(np.int64) * P + t % P
    pool = torch.zeros(case.int2_pool.size, dtype=torch.uint8, device=cuda)
    ctx.write_tokens(0, torch.from_numpy(k).to(cuda).to(torch.bfloat16), torch.from_numpy(v).to(cuda).to(torch.bfloat16),
                     torch.from_numpy(slots).to(cuda), pool)
    torch.cuda.synchronize()
    gpu_pool = pool.cpu().numpy()
    case_gpu_pool = case.int2_pool
    case.int2_pool = gpu_pool
    got, _ = run_gpu(case, cuda, ctx=ctx)
    case.int2_pool = case_gpu_pool
    cases.check_decode(got, case.oracle_out())


def test_debug_bounds_records_bad_page(cuda):
    cfg = cases.workload("tiny")
    case = cases.DecodeCase(cfg, [100], [40])
    case.int2_tables[0, 2] = case.int2_pages + 7      # out of range: skipped and recorded
    got, ctx = run_gpu(case, cuda, debug=1)
    st, kind, index = ctx.debug_error()
    assert st == -5 and kind == 2 and index == case.int2_pages + 7
    assert np.all(np.isfinite(got))


def test_batch_above_the_grid_limit_is_rejected(cuda):
    cfg = cases.workload("tiny")
    ctx = O.Oscar(n_layers=1, n_q_heads=cfg["h_q"], n_kv_heads=cfg["h_kv"], head_dim=cfg["d"], group=cfg["group"])
    li, (rk, rv, tk, tv) = cases.calibration(cfg)
    ctx.calibrate_upload(0, rk, rv, tk, tv)
    B = 65536
    z = lambda *s, dt=torch.int32: torch.zeros(*s, dtype=dt, device=cuda)
    with pytest.raises(O.OscarError) as e:
        ctx.decode(0, z(B, 4, 64, dt=torch.bfloat16), z(4096, dt=torch.uint8), z(B, 4), z(B), 64,
                   z(2 * 2 * 2 * 16 * 64, dt=torch.bfloat16), z(B, 20), z(B), z(B, 4, 64, dt=torch.float32),
                   z(1024, dt=torch.uint8))
    assert e.value.status == -2


def test_workspace_too_small_is_rejected(cuda):
    cfg = cases.workload("tiny")
    ctx = O.Oscar(n_layers=1, n_q_heads=cfg["h_q"], n_kv_heads=cfg["h_kv"], head_dim=cfg["d"], group=cfg["group"])
    li, (rk, rv, tk, tv) = cases.calibration(cfg)
    ctx.calibrate_upload(0, rk, rv, tk, tv)
    need = ctx.decode_workspace_size(1, 1024)
    assert need > 0
    z = lambda *s, dt=torch.int32: torch.zeros(*s, dtype=dt, device=cuda)
    with pytest.raises(O.OscarError) as e:
        ctx.decode(0, z(1, 4, 64, dt=torch.bfloat16), z(4096, dt=torch.uint8), z(1, 64), z(1), 1024,
                   z(2 * 2 * 2 * 16 * 64, dt=torch.bfloat16), z(1, 20), z(1), z(1, 4, 64, dt=torch.float32),
                   z(need - 256, dt=torch.uint8))
    assert e.value.status == -7


def test_merge_one_cta_per_kv_head(cuda):
    """GQA 4, five sequences, one of 66,000 tokens: 33 INT2 splits of up to 128 pages keep 34 partials per
    query head (too many for the last-CTA merge), and 160 query heads exceed one wave of merge CTAs, so the
    merge takes one (sequence, KV head) per CTA. Checked on every head of the long and one short sequence."""
    cfg = cases.workload("qwen3_8b_bs1_100k")
    case = cases.DecodeCase(cfg, [66000, 1000, 1000, 1000, 1000], [320] * 5)
    got, _ = run_gpu(case, cuda)
    want = case.oracle_out(seqs=[0, 3])
    err, rel = cases.check_decode(got[[0, 3]], want[[0, 3]])
    assert np.isfinite(got).all()
    print("max-abs %.3g rel-L2 %.3g" % (err, rel))


def test_qwen3_8b_full_100k_context(cuda):
    """bs1, 100,000-token context (64 sink + 99,680 INT2 + 256 recent), Qwen3-8B shape, all 32 heads."""
    cfg = cases.workload("qwen3_8b_bs1_100k")
    case = cases.DecodeCase(cfg, [cfg["hist"]], [320])
    got, _ = run_gpu(case, cuda)
    err, rel = cases.check_decode(got, case.oracle_out())
    print("max-abs %.3g rel-L2 %.3g" % (err, rel))
