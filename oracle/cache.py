"""End-to-end oracle over paged pools: write tokens, demote, decode a batch (test infrastructure only).

Composes ``quantize``, ``layout`` and ``attention``; see those modules for the
definitions and their sources on the OSCAR pages. Rotation matrices and
thresholds are taken exactly as given (callers pass the fp32 values that are
uploaded to the GPU, so both sides consume identical parameters).
"""

import numpy as np

from . import attention, layout, quantize


def write_tokens(pool, geo, k, v, slots, r_k, r_v, t_k, t_v):
    """Quantize k, v [n, H_kv, d] into the INT2 pool at ``slots`` [n].

    Returns {"k": [per-head quantize dicts], "v": [...]} for tolerance checks.
    """
    info = {"k": [], "v": []}
    for kind, x, r, t in (("k", k, r_k, t_k), ("v", v, r_v, t_v)):
        for h in range(geo.h_kv):
            q = quantize.quantize(np.asarray(x[:, h, :], dtype=np.float64), r[h], t[h], geo.group)
            info[kind].append(q)
            layout.write_int2_rows(pool, geo, slots, h, kind, q["codes"], q["scale"], q["zero"])
    return info


def demote(bf16_pool, int2_pool, geo, src_slots, dst_slots, r_k, r_v, t_k, t_v):
    """Quantize the BF16 rows at ``src_slots`` into INT2 ``dst_slots`` (the pools are modified)."""
    d, h_kv, p = geo.d, geo.h_kv, geo.page
    n = len(src_slots)
    k = np.zeros((n, h_kv, d))
    v = np.zeros((n, h_kv, d))
    for i, s in enumerate(src_slots):
        pg, row = divmod(int(s), p)
        for h in range(h_kv):
            ok = layout.bf16_offset(pg, h, "k", row, d, h_kv, p)
            ov = layout.bf16_offset(pg, h, "v", row, d, h_kv, p)
            k[i, h] = bf16_pool[ok: ok + d]
            v[i, h] = bf16_pool[ov: ov + d]
    return write_tokens(int2_pool, geo, k, v, dst_slots, r_k, r_v, t_k, t_v)


def decode_batch(q, int2_pool, geo, int2_tables, hist_len, bf16_pool, bf16_tables, bf16_len,
                 r_k, r_v, sm_scale, seqs=None):
    """Decode outputs [B, H_q, d] (fp64) for the given batch (or only ``seqs``)."""
    b_total, h_q, d = q.shape
    out = np.zeros((b_total, h_q, d))
    todo = range(b_total) if seqs is None else seqs
    for b in todo:
        kd, vd, kb, vb = [], [], [], []
        for h in range(geo.h_kv):
            ck, sk, zk = layout.read_int2_sequence(int2_pool, geo, int2_tables[b], int(hist_len[b]), h, "k")
            cv, sv, zv = layout.read_int2_sequence(int2_pool, geo, int2_tables[b], int(hist_len[b]), h, "v")
            kd.append(quantize.dequantize(ck, sk, zk, geo.group))
            vd.append(quantize.dequantize(cv, sv, zv, geo.group))
            kb.append(layout.read_bf16_sequence(bf16_pool, bf16_tables[b], int(bf16_len[b]), h, "k", d, geo.h_kv, geo.page))
            vb.append(layout.read_bf16_sequence(bf16_pool, bf16_tables[b], int(bf16_len[b]), h, "v", d, geo.h_kv, geo.page))
        out[b] = attention.decode_heads(np.asarray(q[b], dtype=np.float64), r_k, r_v,
                                        kd, vd, kb, vb, sm_scale)
    return out
