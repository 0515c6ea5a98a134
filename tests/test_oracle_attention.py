"""Pins of oracle.attention / oracle.cache: brute force, merge equivalence, special cases.

Source of what is pinned: QbitAI article on OSCAR, serving-pipeline part (BF16
sink 64 | INT2 history | BF16 recent 256; INT2 and BF16 parts computed
separately and combined by an online-softmax merge).
"""

import numpy as np
import pytest

from oracle import attention, cache, layout, quantize, rotation


def test_merge_equals_one_softmax_over_concatenation():
    rng = np.random.default_rng(0)
    logits = rng.standard_normal(300) * 3
    vals = rng.standard_normal((300, 16))
    ref = attention.softmax_attention(logits, vals)
    cuts = [0, 64, 64, 200, 300]      # includes an empty segment
    states = [attention.partial_state(logits[a:b], vals[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    assert np.abs(attention.merge_states(states) - ref).max() < 1e-12
    # brute force written out: sum_i exp(l_i) v_i / sum_i exp(l_i)
    e = np.exp(logits)
    assert np.abs((e @ vals) / e.sum() - ref).max() < 1e-12


def test_single_token_and_equal_logits():
    v = np.array([[1.5, -2.0, 3.0]])
    np.testing.assert_allclose(attention.softmax_attention([0.3], v), v[0])
    vals = np.random.default_rng(1).standard_normal((7, 3))
    np.testing.assert_allclose(attention.softmax_attention(np.full(7, 2.0), vals), vals.mean(0), atol=1e-14)


def _orth(rng, d):
    a = rng.standard_normal((3 * d, d))
    return rotation.oscar_rotation(a.T @ a)


def test_decode_one_undoes_rotations_exactly():
    """With exact (unquantized) rotated history, the output equals plain attention on the originals."""
    rng = np.random.default_rng(2)
    d = 32
    rk, rv = _orth(rng, d), _orth(rng, d)
    q = rng.standard_normal(d)
    k_hist, v_hist = rng.standard_normal((40, d)), rng.standard_normal((40, d))
    k_bf, v_bf = rng.standard_normal((9, d)), rng.standard_normal((9, d))
    out = attention.decode_one(q, rk, rv, k_hist @ rk, v_hist @ rv, k_bf, v_bf, d ** -0.5)
    allk = np.concatenate([k_bf, k_hist])
    allv = np.concatenate([v_bf, v_hist])
    ref = attention.softmax_attention(d ** -0.5 * allk @ q, allv)
    assert np.abs(out - ref).max() < 1e-10
    # forgetting the un-rotation (or transposing R_v) is caught
    bad = attention.decode_one(q, rk, rv.T, k_hist @ rk, v_hist @ rv, k_bf, v_bf, d ** -0.5)
    assert np.abs(bad - ref).max() > 1e-3


def test_decode_one_empty_segments():
    rng = np.random.default_rng(3)
    d = 16
    r = np.eye(d)
    q = rng.standard_normal(d)
    k, v = rng.standard_normal((5, d)), rng.standard_normal((5, d))
    e = np.zeros((0, d))
    ref = attention.softmax_attention(d ** -0.5 * k @ q, v)
    assert np.abs(attention.decode_one(q, r, r, k, v, e, e, d ** -0.5) - ref).max() < 1e-12
    assert np.abs(attention.decode_one(q, r, r, e, e, k, v, d ** -0.5) - ref).max() < 1e-12


def test_decode_batch_through_paged_pools_matches_direct():
    """Table indirection: a permuted page table over the pool gives the dense result."""
    rng = np.random.default_rng(4)
    d, group, h_kv, h_q, P = 64, 32, 2, 4, 16
    geo = layout.Int2Geometry(d, group, h_kv)
    hist, n_bf = 70, 20                     # ragged last page in both segments
    n_pages_int2 = 8
    pool = np.zeros(n_pages_int2 * geo.page_bytes, dtype=np.uint8)
    table = rng.permutation(n_pages_int2).astype(np.int32)
    slots = np.array([table[t // P] * P + t % P for t in range(hist)])
    rk = np.stack([_orth(rng, d) for _ in range(h_kv)])
    rv = np.stack([_orth(rng, d) for _ in range(h_kv)])
    tk = np.full((h_kv, d), 50.0)
    tv = np.full((h_kv, d), 50.0)
    k = rng.standard_normal((hist, h_kv, d))
    v = rng.standard_normal((hist, h_kv, d))
    info = cache.write_tokens(pool, geo, k, v, slots, rk, rv, tk, tv)
    bf_pages = 3
    bf_table = np.array([2, 0, 1], dtype=np.int32)
    bf_pool = np.zeros(bf_pages * h_kv * 2 * P * d)
    kb = rng.standard_normal((n_bf, h_kv, d))
    vb = rng.standard_normal((n_bf, h_kv, d))
    for t in range(n_bf):
        for h in range(h_kv):
            o = layout.bf16_offset(bf_table[t // P], h, "k", t % P, d, h_kv)
            bf_pool[o:o + d] = kb[t, h]
            o = layout.bf16_offset(bf_table[t // P], h, "v", t % P, d, h_kv)
            bf_pool[o:o + d] = vb[t, h]
    q = rng.standard_normal((1, h_q, d))
    out = cache.decode_batch(q, pool, geo, [table], [hist], bf_pool, [bf_table], [n_bf], rk, rv, d ** -0.5)
    for h in range(h_q):
        kv = h // 2
        kd = quantize.dequantize(info["k"][kv]["codes"], info["k"][kv]["scale"], info["k"][kv]["zero"], group)
        vd = quantize.dequantize(info["v"][kv]["codes"], info["v"][kv]["scale"], info["v"][kv]["zero"], group)
        ref = attention.decode_one(q[0, h], rk[kv], rv[kv], kd, vd, kb[:, kv], vb[:, kv], d ** -0.5)
        assert np.abs(out[0, h] - ref).max() < 1e-12
    # and the quantized cache approximates full-precision attention
    exact = attention.decode_one(q[0, 0], np.eye(d), np.eye(d), k[:, 0], v[:, 0], kb[:, 0], vb[:, 0], d ** -0.5)
    assert np.abs(out[0, 0] - exact).max() < 1.0


def test_demote_reads_bf16_row_and_writes_int2_slot():
    rng = np.random.default_rng(5)
    d, group, h_kv, P = 64, 32, 2, 16
    geo = layout.Int2Geometry(d, group, h_kv)
    bf_pool = np.zeros(2 * h_kv * 2 * P * d)
    src = [1 * P + 3, 0 * P + 15]
    rows = rng.standard_normal((2, h_kv, 2, d))
    for i, s in enumerate(src):
        for h in range(h_kv):
            for j, kv in enumerate("kv"):
                o = layout.bf16_offset(s // P, h, kv, s % P, d, h_kv)
                bf_pool[o:o + d] = rows[i, h, j]
    int2 = np.zeros(4 * geo.page_bytes, dtype=np.uint8)
    r = np.stack([_orth(rng, d)] * h_kv)
    t = np.full((h_kv, d), 9.0)
    dst = [3 * P + 0, 2 * P + 7]
    cache.demote(bf_pool, int2, geo, src, dst, r, r, t, t)
    for i in range(2):
        for h in range(h_kv):
            c, s, z = layout.read_int2_token(int2, geo, dst[i], h, "v")
            q = quantize.quantize(rows[i, h, 1][None], r[h], t[h], group)
            np.testing.assert_array_equal(c, q["codes"][0])
            np.testing.assert_array_equal(s, q["scale"][0])
