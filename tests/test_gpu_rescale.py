"""GPU parity when the logits of one sequence change by far more than the softmax headroom.

The INT2 decode keeps a lazy running reference per query head: it is set on a warp's first page and
raised only when a logit passes it by more than 2^8 (log2 units), with an exact 2^-k rescale of the
accumulated state (k > 126 rescales to zero). The seeded workloads raise it rarely and by small steps, and a warp only raises it
between its own pages, so the history is long enough for every warp to hold about 7 pages.
These cases put a strong component along the query group's direction into the K rows, with a sign and
size that change along the history, so that:
  - logits climb page after page (many small raises of the reference);
  - logits jump by more than 126 log2 units between two halves of the history (a raise whose rescale
    factor underflows to zero);
  - logits fall after the first pages (no raise; later weights far below the reference).
K clipping is switched off (thresholds 1e30 on both sides) so the keys keep their size; V keeps its
calibrated thresholds, which also set the P.V operand's exponent. Everything else
(oracle, tolerance, C-ABI call) is as in test_gpu_decode.py: max-abs 2e-3 and relative L2 1e-3 against
the fp64 oracle decoding the same pages.

Method page: QbitAI article on OSCAR, serving-pipeline part (online-softmax merge of separately computed
parts).
"""

import numpy as np
import pytest
import torch

import cases
from bit_kv_cache_write_gb300 import oscar as O
from oracle import cache

pytestmark = pytest.mark.gpu
P = 16


def _ramp(kind, n):
    t = np.arange(n)
    if kind == "climb":
        return -30.0 + 110.0 * t / max(1, n - 1)          # about -40 .. +150 log2 units of logit
    if kind == "jump":
        return np.where(t < n // 2, -100.0, 100.0)         # a jump of about 200 log2 units
    return 60.0 - 100.0 * t / max(1, n - 1)                # falling


@pytest.mark.parametrize("kind", ["climb", "jump", "fall"])
@pytest.mark.parametrize("name,over", [("qwen3_8b_bs1_100k", {}), ("qwen3_4b_b64_32k", {}),
                                       ("qwen3_32b_mixed16", {})], ids=lambda x: str(x))
def test_decode_with_large_logit_changes(cuda, name, over, kind):
    cfg = cases.workload(name, **over)
    n_hist = 24_000                    # 1,500 pages: about 7 per warp at the one-wave bs1 plan
    case = cases.DecodeCase(cfg, [n_hist], [320])
    d, h_kv, h_q = cfg["d"], cfg["h_kv"], cfg["h_q"]
    g = h_q // h_kv
    tk = np.full_like(case.tk, 1e30)
    tv = case.tv
    # K rows with a strong component along the mean query direction of each KV head's group
    k, v = case.li.kv("rescale-hist", n_hist)
    k = k.reshape(n_hist, h_kv, d).astype(np.float64)
    c = _ramp(kind, n_hist)
    for kv in range(h_kv):
        u = case.q[0, kv * g:(kv + 1) * g].astype(np.float64).mean(axis=0)
        u /= np.linalg.norm(u)
        k[:, kv] += c[:, None] * u[None, :] * (1.0 / (d ** -0.5 * 1.4426950408889634 * np.linalg.norm(
            case.q[0, kv * g:(kv + 1) * g].astype(np.float64).mean(axis=0)) + 1e-30))
    k = torch.from_numpy(k.astype(np.float32)).to(torch.bfloat16).float().numpy()      # rows stay bf16
    t = np.arange(n_hist)
    slots = case.int2_tables[0, t // P].astype(np.int64) * P + t % P
    case.int2_pool[:] = 0
    cache.write_tokens(case.int2_pool, case.geo, k, v, slots, case.rk, case.rv, tk, tv, keep=False)
    case.tk = tk
    want = case.oracle_out()

    ctx = O.Oscar(n_layers=1, n_q_heads=h_q, n_kv_heads=h_kv, head_dim=d, group=cfg["group"])
    ctx.calibrate_upload(0, case.rk, case.rv, tk, tv)
    dev = cuda
    tt = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    ws = torch.empty(ctx.decode_workspace_size(1, n_hist), dtype=torch.uint8, device=dev)
    out = torch.full((1, h_q, d), float("nan"), dtype=torch.float32, device=dev)
    ctx.decode(0, tt(case.q).to(torch.bfloat16), tt(case.int2_pool), tt(case.int2_tables), tt(case.hist_lens),
               n_hist, tt(case.bf16_pool).to(torch.bfloat16), tt(case.bf16_tables), tt(case.bf16_lens), out, ws)
    torch.cuda.synchronize()
    err, rel = cases.check_decode(out.cpu().numpy(), want)
    print("%s %s: max-abs %.3g rel-L2 %.3g" % (name, kind, err, rel))
