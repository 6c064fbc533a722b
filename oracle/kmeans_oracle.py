"""Plain fp64 CPU oracle of the offline stage that feeds the hot path: key
smoothing calibration, the transform variants, and K-Means codebook training
(test infrastructure only: used by tests/ and by bench.py's CPU baseline,
never by the library).

Sources (cited as page title + section):
  [P1] "VecInfer: Efficient LLM Inference with Low-Bit KV Cache via
       Outlier-Suppressed Vector Quantization", Elamur Research summary page,
       section "Summary": keys are smoothed channel-wise and rotated by a
       Hadamard transform before vector quantization, and the codebook is
       trained offline with K-Means; section "Key points": 2^8 x 4 and
       2^12 x 8 codebook shapes, and the transform ablation (smoothing or
       the rotation alone helps less than both; their order matters little).
Readings where the pages are silent (each also in the readings table):
  * the smoothing factor of key channel c is s_c = sqrt(max_t |K[t, c]|)
    (SmoothQuant's per-channel factor with migration strength 1/2;
    SmoothQuant is in the page's reference list), computed in fp64 and
    rounded to fp32;
  * K-Means is Lloyd's algorithm seeded by k-means++ (Arthur and
    Vassilvitskii, 2007): the first centre is a uniformly drawn point, each
    next centre is point x with probability D(x)^2 / sum D^2, D(x) the
    distance to the nearest centre chosen so far;
  * the random numbers are inputs: u[0] picks the first centre as
    floor(u[0] * n); u[i] picks centre i as the first point whose inclusive
    running sum of D^2 (index order) exceeds u[i] * sum D^2 (when every D^2
    is 0, floor(u[i] * n));
  * an assignment goes to the nearest centroid, distances decided in fp32
    (fp64 value rounded once), ties to the lowest index; a centroid becomes
    the fp64 mean of its points rounded to fp32, an empty cluster keeps its
    centroid; the trained codebook is the fp32 centroids rounded to fp16;
  * a zero channel maximum gives s = 1;
  * the "order" ablation rotates first and smooths the rotated keys with
    their own smoothing vector.
"""
from __future__ import annotations

import numpy as np

HEAD_DIM = 128
VARIANTS = ("none", "smooth", "hadamard", "smooth_hadamard", "hadamard_smooth")


def smoothing_vector(rows: np.ndarray) -> np.ndarray:
    """s_c = sqrt(max_t |x[t, c]|) in fp64, rounded to fp32; zero maxima give 1."""
    m = np.abs(np.asarray(rows, dtype=np.float64)).max(axis=0)
    s = np.sqrt(m).astype(np.float32)
    s[m == 0.0] = 1.0
    return s


def hadamard(n: int = HEAD_DIM) -> np.ndarray:
    """Normalised Sylvester matrix: H[i][k] = (-1)^popcount(i & k) / sqrt(n)."""
    i = np.arange(n)
    bits = np.bitwise_and(i[:, None], i[None, :])
    parity = np.zeros_like(bits)
    while bits.any():
        parity ^= bits & 1
        bits >>= 1
    return np.where(parity == 1, -1.0, 1.0) / np.sqrt(n)


def transform(x: np.ndarray, variant: str, s: np.ndarray | None = None):
    """Key rows (fp16 values) under one transform variant, fp64.

    Returns (x', s_used): x' = x / s, x . Hn, (x / s) . Hn (VecInfer), or,
    for "hadamard_smooth", y / s_y with y = x . Hn and s_y the smoothing
    vector of y.  s defaults to the smoothing vector of x.
    """
    x = np.asarray(x, dtype=np.float64)
    hn = hadamard(x.shape[1])
    if variant == "none":
        return x, None
    if variant in ("smooth", "smooth_hadamard"):
        s = smoothing_vector(x) if s is None else s
        y = x / s.astype(np.float64)
        return (y @ hn if variant == "smooth_hadamard" else y), s
    if variant == "hadamard":
        return x @ hn, None
    if variant == "hadamard_smooth":
        y = x @ hn
        s = smoothing_vector(y) if s is None else s
        return y / s.astype(np.float64), s
    raise ValueError(variant)


def inverse_transform(xq: np.ndarray, variant: str, s: np.ndarray | None) -> np.ndarray:
    """Back to the original key domain (Hn is orthogonal and symmetric)."""
    xq = np.asarray(xq, dtype=np.float64)
    hn = hadamard(xq.shape[1])
    if variant == "none":
        return xq
    if variant == "smooth":
        return xq * s.astype(np.float64)
    if variant == "hadamard":
        return xq @ hn.T
    if variant == "smooth_hadamard":
        return (xq @ hn.T) * s.astype(np.float64)
    if variant == "hadamard_smooth":
        return (xq * s.astype(np.float64)) @ hn.T
    raise ValueError(variant)


def squared_distances(points: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    """||x - c||^2 for every (point, centroid), fp64, from direct differences."""
    x = np.asarray(points, dtype=np.float64)
    c = np.asarray(centroids, dtype=np.float64)
    return ((x[:, None, :] - c[None, :, :]) ** 2).sum(axis=2)


def assign(points: np.ndarray, centroids: np.ndarray):
    """Nearest centroid per point: fp64 distances rounded to fp32, lowest
    index on ties.  Returns (index int64 [n], fp32 distances [n][k])."""
    d32 = squared_distances(points, centroids).astype(np.float32)
    return d32.argmin(axis=1), d32


def assign_near_tie(d32_row: np.ndarray, chosen: int) -> bool:
    """A different choice is a near-tie iff its fp32 distance is within 1e-6
    (relative) of the minimum."""
    best = float(d32_row.min())
    return float(d32_row[chosen]) - best < 1e-6 * max(best, 1e-30)


def update(points: np.ndarray, index: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    """Lloyd update: each centroid becomes the fp64 mean of its points,
    rounded to fp32; an empty cluster keeps its centroid."""
    x = np.asarray(points, dtype=np.float64)
    out = np.array(centroids, dtype=np.float32, copy=True)
    for c in range(out.shape[0]):
        members = x[index == c]
        if len(members):
            out[c] = (members.sum(axis=0) / len(members)).astype(np.float32)
    return out


def seed_next(d2: np.ndarray, u: float) -> int:
    """Next k-means++ centre from the current D^2 (fp64) and one uniform draw."""
    n = len(d2)
    total = float(np.sum(d2))
    if not total > 0.0:
        return min(n - 1, int(np.floor(float(u) * n)))
    cum = np.cumsum(d2)
    return int(min(n - 1, np.searchsorted(cum, float(u) * total, side="right")))


def seed_near_tie(d2: np.ndarray, u: float, a: int, b: int, rel: float = 1e-6) -> bool:
    """Two different picks a, b for the same D^2 and draw are a near-tie iff
    every running-sum boundary between them lies within rel * sum D^2 of the
    threshold u * sum D^2."""
    total = float(np.sum(d2))
    if not total > 0.0:
        return False
    thr = float(u) * total
    cum = np.cumsum(d2)
    lo, hi = min(a, b), max(a, b)
    return bool(np.all(np.abs(cum[lo:hi] - thr) <= rel * total))


def seed(points: np.ndarray, k: int, uniforms: np.ndarray) -> np.ndarray:
    """k-means++ centre indices (int64 [k]) for the given draws u[0..k-1]."""
    x = np.asarray(points, dtype=np.float64)
    n = x.shape[0]
    chosen = [min(n - 1, int(np.floor(float(uniforms[0]) * n)))]
    d2 = ((x - x[chosen[0]]) ** 2).sum(axis=1)
    for i in range(1, k):
        nxt = seed_next(d2, uniforms[i])
        chosen.append(nxt)
        d2 = np.minimum(d2, ((x - x[nxt]) ** 2).sum(axis=1))
    return np.array(chosen, dtype=np.int64)


def seed_d2(points: np.ndarray, chosen) -> np.ndarray:
    """D^2 of every point against the given centres (fp64)."""
    x = np.asarray(points, dtype=np.float64)
    d2 = np.full(x.shape[0], np.inf)
    for c in chosen:
        d2 = np.minimum(d2, ((x - x[c]) ** 2).sum(axis=1))
    return d2


def kmeans(points: np.ndarray, k: int, iters: int, uniforms: np.ndarray):
    """k-means++ seeding then `iters` Lloyd steps.  Returns (fp32 centroids,
    fp16 codebook)."""
    x = np.asarray(points, dtype=np.float32)
    c = x[seed(x, k, uniforms)].copy()
    for _ in range(iters):
        idx, _ = assign(x, c)
        c = update(x, idx, c)
    return c, c.astype(np.float16)


def objective(points: np.ndarray, centroids: np.ndarray) -> float:
    """Mean squared distance of the points to their nearest centroid (fp64)."""
    return float(squared_distances(points, centroids).min(axis=1).mean())


def relative_error(x: np.ndarray, x_hat: np.ndarray) -> float:
    """sum (x - x_hat)^2 / sum x^2, fp64."""
    x = np.asarray(x, dtype=np.float64)
    e = x - np.asarray(x_hat, dtype=np.float64)
    return float((e * e).sum() / (x * x).sum())


def utilization(codes: np.ndarray, k: int):
    """(fraction of the k centroids used, entropy of the code histogram in bits)."""
    counts = np.bincount(np.asarray(codes).ravel(), minlength=k).astype(np.float64)
    p = counts[counts > 0] / counts.sum()
    return float((counts > 0).mean()), float(-(p * np.log2(p)).sum())
