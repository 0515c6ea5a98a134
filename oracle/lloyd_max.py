"""Lloyd-Max 2-bit codebook: the step after OSCAR's uniform grid (oracle; test infrastructure only).

Source: QbitAI article on OSCAR, closing part. It says the code repository already combines the
attention-aware rotation with a stronger Lloyd-Max codebook to push the compression further. The
pages give nothing else: no level values, no fitting data, no per-group scaling.

Readings taken here, the plainest the sentence supports:
* The codebook is the Lloyd-Max quantizer of a unit Gaussian with four levels (2 bits). After OSCAR's
  Hadamard mixing, the rotated channels of a group are close to Gaussian.
* A group is normalised by its own mean mu and standard deviation sigma (population, over its G
  clipped rotated values). The code is the index of the level nearest to (x_hat - mu) / sigma; a value
  exactly on a threshold takes the lower level.
* The fp16 pair that holds (scale, zero) for the uniform grid holds (sigma, mu) here, so the page
  layout does not change. Dequant is zero + scale * level[code].
* A group with sigma == 0 stores scale 0 and codes 0, so dequant gives mu.
* Rotation and clipping are OSCAR's, unchanged. The statistics and the decision are fp64.

The codebook the library stores ("dyadic" below) rounds the two Lloyd-Max magnitudes to multiples of
delta = y_1 / 8, y_1 the inner Lloyd-Max level: levels delta * (-27, -8, 8, 27) (1.510 / delta = 26.7
rounds to 27). These integers satisfy l(c) = -27 + 17.5 c + 1.5 b0 for code c = b0 + 2 b1, a linear
function of the code and its low bit, so a decoder can keep exact small-integer dot products with
one extra bit plane. The stored fp16 pair is (scale, zero) = (sigma * delta, mu); dequant is
zero + scale * l(code); the decision compares z = (x_hat - mu) / sigma with the midpoints
delta * (-17.5, 0, 17.5), a value on a midpoint taking the lower level.

Lloyd's algorithm for a density p alternates two conditions until the levels stop moving:
  thresholds t_k = (y_k + y_{k+1}) / 2          (nearest neighbour)
  levels     y_k = E[X | t_{k-1} < X <= t_k]     (centroid)
For the standard normal, the conditional mean of a cell (a, b] is
(phi(a) - phi(b)) / (Phi(b) - Phi(a)).
"""

import numpy as np
from scipy.stats import norm

from . import quantize


def lloyd_max_gaussian(n_levels=4, iters=100_000, tol=1e-15):
    """Levels y (ascending) and thresholds t of the n-level Lloyd-Max quantizer of N(0, 1)."""
    y = np.linspace(-1.5, 1.5, n_levels)
    for _ in range(iters):
        t = np.concatenate([[-np.inf], 0.5 * (y[:-1] + y[1:]), [np.inf]])
        y_new = (norm.pdf(t[:-1]) - norm.pdf(t[1:])) / (norm.cdf(t[1:]) - norm.cdf(t[:-1]))
        done = np.max(np.abs(y_new - y)) < tol
        y = y_new
        if done:
            break
    return y, 0.5 * (y[:-1] + y[1:])


def gaussian_distortion(levels, thresholds):
    """E[(X - Q(X))^2] for X ~ N(0, 1), exactly, for levels and the cell edges between them.

    A cell (a, b] contributes M2 - 2 y M1 + y^2 M0 with
    M0 = Phi(b) - Phi(a), M1 = phi(a) - phi(b) and M2 = M0 - (b phi(b) - a phi(a)).
    """
    edges = np.concatenate([[-np.inf], np.asarray(thresholds, np.float64), [np.inf]])
    a, b = edges[:-1], edges[1:]

    def x_phi(x):
        return np.where(np.isfinite(x), np.nan_to_num(x) * norm.pdf(x), 0.0)

    m0 = norm.cdf(b) - norm.cdf(a)
    m1 = norm.pdf(a) - norm.pdf(b)
    m2 = m0 - (x_phi(b) - x_phi(a))
    y = np.asarray(levels, np.float64)
    return float(np.sum(m2 - 2.0 * y * m1 + y * y * m0))


def quantize_lloyd_max(x, r, t, group, levels):
    """Rotate, clip, then code every group against the normalised Gaussian codebook.

    Returns a dict with codes uint8 [..., d], scale (sigma) and zero (mu) as float16 [..., d/G],
    and z float64 [..., d], the normalised values the decision saw.
    """
    levels = np.asarray(levels, np.float64)
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    if d % group:
        raise ValueError("group must divide d")
    lead = x.shape[:-1]
    xr32 = quantize.rotate(x, r).astype(np.float32)
    t32 = np.asarray(t, np.float32)
    xh = np.minimum(np.maximum(xr32, -t32), t32).astype(np.float64)
    g = xh.reshape(lead + (d // group, group))
    mu = g.mean(axis=-1)
    sigma = np.sqrt(((g - mu[..., None]) ** 2).mean(axis=-1))
    flat = ~(sigma > 0)
    z = (g - mu[..., None]) / np.where(flat, 1.0, sigma)[..., None]
    cut = 0.5 * (levels[:-1] + levels[1:])
    codes = np.searchsorted(cut, z, side="left")
    codes = np.where(flat[..., None], 0, codes).astype(np.uint8)
    scale = np.where(flat, 0.0, sigma).astype(np.float16)
    return {"codes": codes.reshape(lead + (d,)), "scale": scale, "zero": mu.astype(np.float16),
            "z": z.reshape(lead + (d,))}


def dequantize_lloyd_max(codes, scale, zero, group, levels):
    """x_deq = zero + scale * level[code] per group, from the stored fp16 scale and zero."""
    levels = np.asarray(levels, np.float64)
    codes = np.asarray(codes)
    d = codes.shape[-1]
    lead = codes.shape[:-1]
    c = levels[codes.reshape(lead + (d // group, group)).astype(np.int64)]
    s = np.asarray(scale, np.float64)[..., None]
    z = np.asarray(zero, np.float64)[..., None]
    return (z + s * c).reshape(lead + (d,))


DYADIC_STEPS = np.array([-27.0, -8.0, 8.0, 27.0])      # levels in units of delta


def dyadic_codebook():
    """(delta, levels, thresholds) of the stored codebook: the Lloyd-Max levels of N(0, 1) rounded
    to multiples of delta = y_1 / 8 (y_1 the inner level), levels delta * (-27, -8, 8, 27)."""
    y, _ = lloyd_max_gaussian(4)
    delta = y[2] / 8.0
    levels = delta * DYADIC_STEPS
    return delta, levels, 0.5 * (levels[:-1] + levels[1:])


def quantize_dyadic(x, r, t, group):
    """Rotate, clip, and code every group against the dyadic codebook (fp64 statistics and decision).

    Returns codes uint8 [..., d], scale = fp16(sigma * delta) and zero = fp16(mu) [..., d/G], z (the
    normalised values the decision saw) and the fp64 sigma."""
    delta, levels, cut = dyadic_codebook()
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    if d % group:
        raise ValueError("group must divide d")
    lead = x.shape[:-1]
    xr32 = quantize.rotate(x, r).astype(np.float32)
    t32 = np.asarray(t, np.float32)
    xh = np.minimum(np.maximum(xr32, -t32), t32).astype(np.float64)
    g = xh.reshape(lead + (d // group, group))
    mu = g.mean(axis=-1)
    sigma = np.sqrt(((g - mu[..., None]) ** 2).mean(axis=-1))
    flat = ~(sigma > 0)
    z = (g - mu[..., None]) / np.where(flat, 1.0, sigma)[..., None]
    codes = np.searchsorted(cut, z, side="left")
    codes = np.where(flat[..., None], 0, codes).astype(np.uint8)
    scale = np.where(flat, 0.0, sigma * delta).astype(np.float16)
    return {"codes": codes.reshape(lead + (d,)), "scale": scale, "zero": mu.astype(np.float16),
            "z": z.reshape(lead + (d,)), "sigma": sigma, "thresholds": cut}


def dequantize_dyadic(codes, scale, zero, group):
    """x_deq = zero + scale * l(code), l = (-27, -8, 8, 27), from the stored fp16 scale and zero."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    lead = codes.shape[:-1]
    c = DYADIC_STEPS[codes.reshape(lead + (d // group, group)).astype(np.int64)]
    s = np.asarray(scale, np.float64)[..., None]
    z = np.asarray(zero, np.float64)[..., None]
    return (z + s * c).reshape(lead + (d,))
