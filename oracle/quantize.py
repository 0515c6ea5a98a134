"""Rotate -> clip -> group scale/zero -> 2-bit code, and dequant (oracle; test infrastructure only).

Source: QbitAI article on OSCAR, serving-pipeline part: the oldest recent token
is rotated, clipped, quantized and packed into the INT2 history; 2-bit INT has
four levels; the INT2 decode kernel dequantizes with a scale and a zero point.
The v1/v2 abstracts fix the rotation and clipping thresholds offline.

Definition used here (the pages give no formula; these are readings of them):

  x_rot = x @ R                           exact (fp64), then rounded to fp32
  x_hat = min(max(x_rot, -T), T)          per channel threshold T
  per group of G consecutive rotated channels:
    mn = min x_hat, mx = max x_hat, rng = mx - mn
    if rng < FLT_MIN (smallest normal fp32; includes rng == 0): codes 0
    else: inv = 3 / rng; u = (x_hat - mn) * inv; code = clamp(rint(u), 0, 3)
    scale = fp16(rng / 3), zero = fp16(mn)     (round to nearest even)
  dequant: x_deq = code * scale + zero   with the stored fp16 scale and zero

Every step after the rotation is done in IEEE fp32 with round-to-nearest-even,
in exactly the order written: the code is an integer decided by floating point,
so the oracle takes that decision in the precision the GPU kernel takes it
(fp32). The rotation itself is computed exactly (fp64) and rounded once.
``u64`` (the same ratio in fp64, from the unrounded rotation) is returned for
the boundary-tolerance check of parity tests.
"""

import numpy as np

FLT_MIN = np.float32(np.finfo(np.float32).tiny)


def rotate(x, r):
    """x_rot = x @ R in fp64 (row-vector convention)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(r, dtype=np.float64)


def quantize(x, r, t, group):
    """Quantize rows of x (shape [..., d]) with rotation r [d, d] and thresholds t [d].

    Returns a dict with
      codes  uint8 [..., d]       2-bit codes per rotated channel
      scale  float16 [..., d/G]
      zero   float16 [..., d/G]
      u      float64 [..., d]     fp32 pre-rounding ratio (the value rint sees)
      u64    float64 [..., d]     same ratio from the unrounded fp64 rotation
      x_hat  float64 [..., d]     clipped rotated values (fp32 precision)
      x_hat64 float64 [..., d]    clipped rotated values (fp64)
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    if d % group:
        raise ValueError("group must divide d")
    lead = x.shape[:-1]
    ng = d // group

    xr64 = rotate(x, r)
    xr32 = xr64.astype(np.float32)
    t32 = np.asarray(t, dtype=np.float32)
    xh32 = np.minimum(np.maximum(xr32, -t32), t32)

    g32 = xh32.reshape(lead + (ng, group))
    mn = g32.min(axis=-1)
    mx = g32.max(axis=-1)
    rng = (mx - mn).astype(np.float32)
    degenerate = ~(rng >= FLT_MIN)
    safe = np.where(degenerate, np.float32(1), rng).astype(np.float32)
    inv = (np.float32(3) / safe).astype(np.float32)
    u32 = ((g32 - mn[..., None]).astype(np.float32) * inv[..., None]).astype(np.float32)
    codes = np.clip(np.rint(u32), 0, 3)
    codes = np.where(degenerate[..., None], 0, codes).astype(np.uint8)

    scale = (rng / np.float32(3)).astype(np.float32).astype(np.float16)
    zero = mn.astype(np.float16)

    t64 = np.asarray(t, dtype=np.float64)
    xh64 = np.minimum(np.maximum(xr64, -t64), t64)
    g64 = xh64.reshape(lead + (ng, group))
    mn64 = g64.min(axis=-1)
    rng64 = g64.max(axis=-1) - mn64
    safe64 = np.where(rng64 > 0, rng64, 1.0)
    u64 = 3.0 * (g64 - mn64[..., None]) / safe64[..., None]

    return {
        "codes": codes.reshape(lead + (d,)),
        "scale": scale,
        "zero": zero,
        "u": u32.astype(np.float64).reshape(lead + (d,)),
        "u64": u64.reshape(lead + (d,)),
        "x_hat": xh32.astype(np.float64),
        "x_hat64": xh64,
    }


def dequantize(codes, scale, zero, group):
    """x_deq = code * scale + zero per group, in fp64 from the stored fp16 scale/zero."""
    codes = np.asarray(codes, dtype=np.float64)
    d = codes.shape[-1]
    lead = codes.shape[:-1]
    c = codes.reshape(lead + (d // group, group))
    s = np.asarray(scale, dtype=np.float64)[..., None]
    z = np.asarray(zero, dtype=np.float64)[..., None]
    return (c * s + z).reshape(lead + (d,))
