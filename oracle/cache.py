"""End-to-end oracle over paged pools: write tokens, demote, decode a batch (test infrastructure only).

Composes ``quantize``, ``layout`` and ``attention``; see those modules for the
definitions and their sources on the OSCAR pages. Rotation matrices and
thresholds are taken exactly as given (callers pass the fp32 values that are
uploaded to the GPU, so both sides consume identical parameters).
"""

import numpy as np

from . import attention, layout, lloyd_max, quantize

CODEBOOKS = ("uniform", "lloyd_max")


def _quantize(codebook, x, r, t, group):
    if codebook == "lloyd_max":
        return lloyd_max.quantize_dyadic(x, r, t, group)
    return quantize.quantize(x, r, t, group)


def _dequantize(codebook, codes, scale, zero, group):
    if codebook == "lloyd_max":
        return lloyd_max.dequantize_dyadic(codes, scale, zero, group)
    return quantize.dequantize(codes, scale, zero, group)


def write_tokens(pool, geo, k, v, slots, r_k, r_v, t_k, t_v, keep=True, codebook="uniform"):
    """Quantize k, v [n, H_kv, d] into the INT2 pool at ``slots`` [n].

    codebook "uniform" (min/max grid) or "lloyd_max" (the rounded Lloyd-Max levels, see lloyd_max).
    Returns {"k": [per-head quantize dicts], "v": [...]} for tolerance checks
    (or None with keep=False, which holds one head's intermediates at a time).
    """
    info = {"k": [], "v": []}
    for kind, x, r, t in (("k", k, r_k, t_k), ("v", v, r_v, t_v)):
        for h in range(geo.h_kv):
            q = _quantize(codebook, np.asarray(x[:, h, :], dtype=np.float64), r[h], t[h], geo.group)
            layout.write_int2_rows(pool, geo, slots, h, kind, q["codes"], q["scale"], q["zero"])
            if keep:
                info[kind].append(q)
    return info if keep else None


def demote(bf16_pool, int2_pool, geo, src_slots, dst_slots, r_k, r_v, t_k, t_v, codebook="uniform"):
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
    return write_tokens(int2_pool, geo, k, v, dst_slots, r_k, r_v, t_k, t_v, codebook=codebook)


def decode_batch(q, int2_pool, geo, int2_tables, hist_len, bf16_pool, bf16_tables, bf16_len,
                 r_k, r_v, sm_scale, seqs=None, heads=None, codebook="uniform"):
    """Decode outputs [B, H_q, d] (fp64) for the given batch (or only ``seqs`` / query ``heads``).

    Works one (sequence, KV head) at a time so full-length histories fit in host memory.
    """
    b_total, h_q, d = q.shape
    g = h_q // geo.h_kv
    out = np.zeros((b_total, h_q, d))
    todo = range(b_total) if seqs is None else seqs
    want = set(range(h_q)) if heads is None else set(heads)
    for b in todo:
        for kv in range(geo.h_kv):
            hs = [h for h in range(kv * g, (kv + 1) * g) if h in want]
            if not hs:
                continue
            n_hist, n_bf = int(hist_len[b]), int(bf16_len[b])
            ck, sk, zk = layout.read_int2_sequence(int2_pool, geo, int2_tables[b], n_hist, kv, "k")
            cv, sv, zv = layout.read_int2_sequence(int2_pool, geo, int2_tables[b], n_hist, kv, "v")
            kd = _dequantize(codebook, ck, sk, zk, geo.group)
            vd = _dequantize(codebook, cv, sv, zv, geo.group)
            kb = layout.read_bf16_sequence(bf16_pool, bf16_tables[b], n_bf, kv, "k", d, geo.h_kv, geo.page)
            vb = layout.read_bf16_sequence(bf16_pool, bf16_tables[b], n_bf, kv, "v", d, geo.h_kv, geo.page)
            for h in hs:
                out[b, h] = attention.decode_one(np.asarray(q[b, h], dtype=np.float64), r_k[kv], r_v[kv],
                                                 kd, vd, kb, vb, sm_scale)
    return out
