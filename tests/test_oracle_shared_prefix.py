"""Oracle pins for decoding over a shared prefix (radix prefix-cache hit).

Source: QbitAI article on OSCAR, serving-pipeline part (the INT2 cache works
with paged KV and the radix prefix cache; the decode combines separately
computed parts with an online-softmax merge); arXiv 2605.17757 v2 abstract
(paged layouts and prefix caching preserved).

What is pinned, on the CPU, before any GPU comparison:
- block tables that alias the same physical prefix pages decode exactly like
  tables whose prefix pages are separate physical copies of the same bytes
  (aliasing changes where bytes live, never what is computed);
- the cascade decomposition the shared-prefix decode uses: the online-softmax
  merge of the prefix part, the sequence's own INT2 part and its BF16 part
  equals one softmax over the whole sequence, to 1e-12.
"""

import numpy as np

import cases
from oracle import attention, layout, quantize

P = 16


def _case():
    cfg = cases.workload("tiny")
    # 3 sequences sharing 6 prefix pages (96 tokens), one of them with nothing after the prefix
    return cases.DecodeCase(cfg, [96 + 40, 96, 96 + 150], [320, 17, 0], shared_pages=6)


def test_aliased_prefix_pages_decode_like_separate_copies():
    case = _case()
    want = case.oracle_out()
    geo = case.geo
    shared = 6
    # give every sequence but the first its own physical copy of the prefix pages
    pool = case.int2_pool.copy()
    tables = case.int2_tables.copy()
    n_pages = pool.size // geo.page_bytes
    extra = []
    for b in range(1, len(case.hist_lens)):
        for j in range(shared):
            src = int(tables[b, j])
            extra.append(pool[src * geo.page_bytes:(src + 1) * geo.page_bytes].copy())
            tables[b, j] = n_pages + len(extra) - 1
    pool = np.concatenate([pool] + extra)
    assert len(np.unique(tables[:, :shared])) == shared * len(case.hist_lens)
    from oracle import cache
    got = cache.decode_batch(case.q, pool, geo, tables, case.hist_lens, case.bf16_pool, case.bf16_tables,
                             case.bf16_lens, case.rk, case.rv, case.sm_scale)
    assert np.array_equal(got, want)


def test_prefix_suffix_bf16_states_merge_to_one_softmax():
    case = _case()
    geo, d, sm = case.geo, case.geo.d, case.sm_scale
    g = case.q.shape[1] // geo.h_kv
    shared_tok = 6 * P
    for b in range(len(case.hist_lens)):
        n_hist, n_bf = int(case.hist_lens[b]), int(case.bf16_lens[b])
        for kv in range(geo.h_kv):
            ck, sk, zk = layout.read_int2_sequence(case.int2_pool, geo, case.int2_tables[b], n_hist, kv, "k")
            cv, sv, zv = layout.read_int2_sequence(case.int2_pool, geo, case.int2_tables[b], n_hist, kv, "v")
            kd = quantize.dequantize(ck, sk, zk, geo.group)
            vd = quantize.dequantize(cv, sv, zv, geo.group)
            kb = layout.read_bf16_sequence(case.bf16_pool, case.bf16_tables[b], n_bf, kv, "k", d, geo.h_kv, P)
            vb = layout.read_bf16_sequence(case.bf16_pool, case.bf16_tables[b], n_bf, kv, "v", d, geo.h_kv, P)
            rk, rv = case.rk[kv].astype(np.float64), case.rv[kv].astype(np.float64)
            for h in range(kv * g, (kv + 1) * g):
                q = case.q[b, h].astype(np.float64)
                qr = q @ rk
                lg = sm * (kd @ qr)
                # INT2 parts stay in the rotated basis until the merged sum is un-rotated
                st_pre = attention.partial_state(lg[:shared_tok], vd[:shared_tok] @ rv.T)
                st_own = attention.partial_state(lg[shared_tok:], vd[shared_tok:] @ rv.T)
                st_bf = attention.partial_state(sm * (kb @ q), vb)
                merged = attention.merge_states([st_pre, st_own, st_bf])
                direct = attention.decode_one(q, rk, rv, kd, vd, kb, vb, sm)
                assert np.abs(merged - direct).max() < 1e-12 * max(1.0, np.abs(direct).max())
