"""Three-segment decode attention and online-softmax merge (oracle; test infrastructure only).

Source: QbitAI article on OSCAR, serving-pipeline part: the token pool is BF16
sink (64 tokens) | INT2 history | BF16 recent (256 tokens); at decode the INT2
kernel unpacks, dequantizes with scale/zero point and accumulates in floating
point, a BF16 kernel handles sink/recent, and an online-softmax merge combines
the two results.

Definition (fp64 throughout):
  rotated query            q_rot = q @ R_k            (QK^T is invariant under a
                                                        joint orthogonal rotation)
  INT2 logits              sm_scale * q_rot . k_deq   (k_deq in the rotated basis)
  BF16 logits              sm_scale * q . k           (sink/recent are stored unrotated)
  p = one softmax over the concatenation [BF16 segment | INT2 history]
  out = p_bf16 @ V_bf16 + (p_int2 @ V_deq) @ R_v^T    (R_v^T undoes the V rotation)

No causal mask and no positional encoding inside this op: every cached token is
visible to the query, which attends as one of its group's query heads
(KV head of query head h is h // (H_q / H_kv)).
"""

import numpy as np


def softmax_attention(logits, values):
    """Plain softmax(logits) @ values for one query: logits [n], values [n, d]."""
    logits = np.asarray(logits, dtype=np.float64)
    m = logits.max()
    e = np.exp(logits - m)
    return (e / e.sum()) @ np.asarray(values, dtype=np.float64)


def partial_state(logits, values):
    """(m, l, acc) of one segment: m = max logit, l = sum exp(logit - m), acc = sum exp(.) v.

    An empty segment is (-inf, 0, 0).
    """
    logits = np.asarray(logits, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    if logits.size == 0:
        return -np.inf, 0.0, np.zeros(values.shape[-1], dtype=np.float64)
    m = logits.max()
    e = np.exp(logits - m)
    return m, e.sum(), e @ values


def merge_states(states):
    """Online-softmax merge of (m, l, acc) states; returns the normalised output."""
    ms = [s[0] for s in states]
    m = max(ms)
    l_tot = 0.0
    acc = np.zeros_like(states[0][2])
    for mi, li, ai in states:
        if li == 0.0:
            continue
        w = np.exp(mi - m)
        l_tot += li * w
        acc = acc + ai * w
    return acc / l_tot


def decode_one(q, r_k, r_v, k_deq, v_deq, k_bf, v_bf, sm_scale):
    """Decode output for one query head.

    q      [d]       query (unrotated)
    r_k    [d, d]    key rotation of its KV head;  r_v [d, d] value rotation
    k_deq, v_deq [n_hist, d]   dequantized INT2 history, rotated basis
    k_bf, v_bf   [n_bf, d]     BF16 sink + recent rows, unrotated
    """
    q = np.asarray(q, dtype=np.float64)
    q_rot = q @ np.asarray(r_k, dtype=np.float64)
    lg_int2 = sm_scale * (np.asarray(k_deq, dtype=np.float64) @ q_rot)
    lg_bf = sm_scale * (np.asarray(k_bf, dtype=np.float64) @ q)
    logits = np.concatenate([lg_bf, lg_int2])
    if logits.size == 0:                      # no cached token at all: defined as zeros
        return np.zeros(q.shape[0])
    m = logits.max()
    e = np.exp(logits - m)
    p = e / e.sum()
    n_bf = lg_bf.shape[0]
    out_rot = p[n_bf:] @ np.asarray(v_deq, dtype=np.float64)
    return p[:n_bf] @ np.asarray(v_bf, dtype=np.float64) + out_rot @ np.asarray(r_v, dtype=np.float64).T


def decode_heads(q, r_k, r_v, k_deq, v_deq, k_bf, v_bf, sm_scale):
    """Decode output for all query heads of one sequence.

    q [H_q, d]; r_k, r_v [H_kv, d, d]; k_deq/v_deq [H_kv, n_hist, d];
    k_bf/v_bf [H_kv, n_bf, d]. Returns [H_q, d] fp64.
    """
    h_q = q.shape[0]
    h_kv = r_k.shape[0]
    g = h_q // h_kv
    out = np.zeros((h_q, q.shape[1]), dtype=np.float64)
    for h in range(h_q):
        kv = h // g
        out[h] = decode_one(q[h], r_k[kv], r_v[kv], k_deq[kv], v_deq[kv], k_bf[kv], v_bf[kv], sm_scale)
    return out
