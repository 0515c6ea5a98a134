"""Paged INT2 and BF16 cache layout (oracle; test infrastructure only).

Source: QbitAI article on OSCAR, serving-pipeline part: four 2-bit values are
packed into one byte; the cache stays compatible with paged KV serving and the
radix prefix cache (v1/v2 abstracts: "paged KV-cache layouts", "prefix
caching"). The pages fix nothing else about the layout, so the layout below is
this library's own definition (stated in include/oscar.h) and the
oracle writes it out independently of the CUDA code.

INT2 pool: bytes [num_pages][H_kv][2 (K, V)][segment], page size P.
  segment = codes [P][d/4] bytes, then scale/zero [P][d/G] x (fp16 scale, fp16 zero)
  The code row of one token is a little-endian bit string of 2*d bits; the
  2-bit code of rotated channel c sits at bits [o(c), o(c)+1] (bit b is bit
  b%8 of byte b//8), with n = d/16 and
    K rows:  kk = c//16, t = (c%16)//4, i = c%4
             o_K(c) = 8*n*t + 32*(kk//4) + 16*(i%2) + 2*(2*(kk%4) + i//2)
    V rows:  m = c//16, r = c%16
             o_V(c) = 4*n*(r%8) + 2*n*(r//8) + 2*m
BF16 pool: bf16 [num_pages][H_kv][2 (K, V)][P][d], unrotated.
Slots: slot = page * P + row. Block tables map logical page j of a sequence to
a physical page id; logical token t is at page table[t // P], row t % P.
"""

import numpy as np

PAGE = 16


def k_bit_offset(c, d):
    n = d // 16
    kk, t, i = c // 16, (c % 16) // 4, c % 4
    return 8 * n * t + 32 * (kk // 4) + 16 * (i % 2) + 2 * (2 * (kk % 4) + i // 2)


def v_bit_offset(c, d):
    n = d // 16
    m, r = c // 16, c % 16
    return 4 * n * (r % 8) + 2 * n * (r // 8) + 2 * m


def bit_offsets(kind, d):
    f = k_bit_offset if kind == "k" else v_bit_offset
    return np.array([f(c, d) for c in range(d)], dtype=np.int64)


def pack_row(codes, kind):
    """Pack d codes (0..3) into d/4 bytes following the K or V bit map."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    out = np.zeros(d // 4, dtype=np.uint8)
    for c in range(d):
        o = k_bit_offset(c, d) if kind == "k" else v_bit_offset(c, d)
        out[o // 8] |= np.uint8((int(codes[c]) & 3) << (o % 8))
    return out


def unpack_row(row, kind, d):
    row = np.asarray(row, dtype=np.uint8)
    out = np.zeros(d, dtype=np.uint8)
    for c in range(d):
        o = k_bit_offset(c, d) if kind == "k" else v_bit_offset(c, d)
        out[c] = (int(row[o // 8]) >> (o % 8)) & 3
    return out


def pack_rows(codes, kind):
    """Vectorised pack_row over leading dims: codes [..., d] -> bytes [..., d/4]."""
    codes = np.asarray(codes, dtype=np.uint8)
    d = codes.shape[-1]
    offs = bit_offsets(kind, d)
    lead = codes.shape[:-1]
    out = np.zeros(lead + (d // 4,), dtype=np.uint8)
    for c in range(d):
        o = int(offs[c])
        out[..., o // 8] |= ((codes[..., c] & 3) << (o % 8)).astype(np.uint8)
    return out


def unpack_rows(rows, kind, d):
    rows = np.asarray(rows, dtype=np.uint8)
    offs = bit_offsets(kind, d)
    lead = rows.shape[:-1]
    out = np.zeros(lead + (d,), dtype=np.uint8)
    for c in range(d):
        o = int(offs[c])
        out[..., c] = (rows[..., o // 8] >> (o % 8)) & 3
    return out


class Int2Geometry:
    """Byte geometry of one INT2 page for (d, G, H_kv)."""

    def __init__(self, d, group, n_kv_heads, page=PAGE):
        self.d, self.group, self.h_kv, self.page = d, group, n_kv_heads, page
        self.code_bytes = page * (d // 4)
        self.sz_bytes = page * (d // group) * 4
        self.segment = self.code_bytes + self.sz_bytes
        self.block = 2 * self.segment          # one (page, head)
        self.page_bytes = n_kv_heads * self.block

    def segment_offset(self, page, head, kv):
        return (page * self.h_kv + head) * self.block + (0 if kv == "k" else self.segment)


def write_int2_token(pool, geo, slot, head, kv, codes, scale, zero):
    """Store one quantized row (codes [d], scale/zero [d/G] fp16) at an INT2 slot."""
    page, row = divmod(int(slot), geo.page)
    base = geo.segment_offset(page, head, kv)
    rb = geo.d // 4
    pool[base + row * rb: base + (row + 1) * rb] = pack_row(codes, kv)
    ng = geo.d // geo.group
    sz = np.empty(2 * ng, dtype=np.float16)
    sz[0::2] = np.asarray(scale, dtype=np.float16)
    sz[1::2] = np.asarray(zero, dtype=np.float16)
    s0 = base + geo.code_bytes + row * ng * 4
    pool[s0: s0 + ng * 4] = sz.view(np.uint8)


def write_int2_rows(pool, geo, slots, head, kv, codes, scale, zero):
    """Vectorised write_int2_token for many slots of one head: codes [n, d], scale/zero [n, d/G]."""
    slots = np.asarray(slots, dtype=np.int64)
    page, row = slots // geo.page, slots % geo.page
    base = (page * geo.h_kv + head) * geo.block + (0 if kv == "k" else geo.segment)
    rb = geo.d // 4
    packed = pack_rows(codes, kv)
    idx = (base + row * rb)[:, None] + np.arange(rb)[None, :]
    pool[idx] = packed
    ng = geo.d // geo.group
    sz = np.empty((len(slots), 2 * ng), dtype=np.float16)
    sz[:, 0::2] = np.asarray(scale, dtype=np.float16)
    sz[:, 1::2] = np.asarray(zero, dtype=np.float16)
    sidx = (base + geo.code_bytes + row * ng * 4)[:, None] + np.arange(ng * 4)[None, :]
    pool[sidx] = sz.view(np.uint8).reshape(len(slots), ng * 4)


def read_int2_token(pool, geo, slot, head, kv):
    """Inverse of write_int2_token: (codes [d], scale [d/G] fp16, zero [d/G] fp16)."""
    page, row = divmod(int(slot), geo.page)
    base = geo.segment_offset(page, head, kv)
    rb = geo.d // 4
    codes = unpack_row(pool[base + row * rb: base + (row + 1) * rb], kv, geo.d)
    ng = geo.d // geo.group
    s0 = base + geo.code_bytes + row * ng * 4
    sz = np.frombuffer(pool[s0: s0 + ng * 4].tobytes(), dtype=np.float16)
    return codes, sz[0::2].copy(), sz[1::2].copy()


def read_int2_sequence(pool, geo, table, length, head, kv):
    """All history tokens of one sequence/head: codes [L, d], scale [L, d/G], zero [L, d/G].

    Reads whole pages at once (vectorised) but addresses exactly as the
    per-token reader does.
    """
    d, ng, p = geo.d, geo.d // geo.group, geo.page
    n_pages = (length + p - 1) // p
    rb = d // 4
    pages = np.asarray(table[:n_pages], dtype=np.int64)
    base = (pages * geo.h_kv + head) * geo.block + (0 if kv == "k" else geo.segment)
    cidx = base[:, None] + np.arange(geo.code_bytes)[None, :]
    rows = pool[cidx].reshape(n_pages * p, rb)
    codes = unpack_rows(rows, kv, d)
    sidx = (base + geo.code_bytes)[:, None] + np.arange(geo.sz_bytes)[None, :]
    sz = np.ascontiguousarray(pool[sidx]).view(np.float16).reshape(n_pages * p, 2 * ng)
    return codes[:length], sz[:length, 0::2], sz[:length, 1::2]


def bf16_offset(page, head, kv, row, d, n_kv_heads, page_size=PAGE):
    """Element offset of a BF16 row in the BF16 pool [pages][H_kv][2][P][d]."""
    return (((page * n_kv_heads + head) * 2 + (0 if kv == "k" else 1)) * page_size + row) * d


def read_bf16_sequence(pool, table, length, head, kv, d, n_kv_heads, page_size=PAGE):
    """BF16 segment rows of one sequence/head as fp64 [L, d] (pool holds bf16 values as float)."""
    out = np.zeros((length, d), dtype=np.float64)
    for t in range(length):
        off = bf16_offset(int(table[t // page_size]), head, kv, t % page_size, d, n_kv_heads, page_size)
        out[t] = pool[off: off + d]
    return out
