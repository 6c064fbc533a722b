"""Offline calibration that produces the inputs of the hot path: the key
smoothing vector ``s`` and the per-KV-head K/V codebooks.

VecInfer trains its codebooks offline with K-Means on the smoothed,
Hadamard-rotated key subvectors (and on raw value subvectors), VecInfer
paper, "Summary"; the codebook shapes are 2^8 x 4 (2 bit) and 2^12 x 8
(1.5 bit), "Key points".  The smoothing factor per key channel is
``s_c = sqrt(max_t |K[t, c]|)``; the rotation is the normalised 128 x 128
Sylvester Hadamard matrix.

This is the offline stage, not the hot path: it runs once per workload on
the host, and both the CUDA path and the CPU oracle read the fp16 codebook
and fp32 ``s`` it returns as plain data, so no parity result depends on how
good these codebooks are.  It uses library routines for the rotation
(``scipy.linalg.hadamard``) and a plain matrix-product K-Means; it shares no
code with the oracle or with the kernels.
"""
from __future__ import annotations

import numpy as np
import scipy.linalg

from . import synth

HEAD_DIM = synth.HEAD_DIM


def smoothing_vector(k_rows: np.ndarray) -> np.ndarray:
    """s_c = sqrt(max_t |K[t, c]|) over the given key rows; zero channels map to 1."""
    m = np.abs(k_rows.astype(np.float32)).max(axis=0)
    s = np.sqrt(m).astype(np.float32)
    s[s == 0] = 1.0
    return s


def _rotated_key_rows(k_rows: np.ndarray, s: np.ndarray) -> np.ndarray:
    h = scipy.linalg.hadamard(HEAD_DIM).astype(np.float64) / np.sqrt(HEAD_DIM)
    return (k_rows.astype(np.float64) / s.astype(np.float64)) @ h


def kmeans(data: np.ndarray, k: int, iters: int, rng: np.random.Generator,
           init: str = "++") -> np.ndarray:
    """K-Means (Lloyd) on rows of ``data``; returns fp16 centroids [k][dim].

    init "++": k-means++ seeding; init "points": k distinct random rows.
    Empty clusters keep their previous centroid; assignment ties go to the
    lowest index (argmin).  The result is cast to fp16 at the end.
    """
    x = np.ascontiguousarray(data, dtype=np.float32)
    n = x.shape[0]
    if init == "++":
        c = np.empty((k, x.shape[1]), dtype=np.float32)
        c[0] = x[rng.integers(n)]
        d2 = ((x - c[0]) ** 2).sum(axis=1)
        for i in range(1, k):
            tot = d2.sum()
            if tot <= 0:
                c[i] = x[rng.integers(n)]
            else:
                c[i] = x[rng.choice(n, p=d2 / tot)]
            d2 = np.minimum(d2, ((x - c[i]) ** 2).sum(axis=1))
    elif init == "points":
        c = x[rng.choice(n, size=k, replace=False)].copy()
    else:
        raise ValueError(init)
    for _ in range(iters):
        # ||x||^2 is constant per row, so the argmin only needs ||c||^2 - 2 x.c
        cc = (c * c).sum(axis=1)
        a = np.empty(n, dtype=np.int64)
        step = max(1, (1 << 24) // k)
        for r0 in range(0, n, step):
            a[r0:r0 + step] = (cc[None, :] - 2.0 * (x[r0:r0 + step] @ c.T)).argmin(axis=1)
        cnt = np.bincount(a, minlength=k).astype(np.float32)
        sums = np.stack([np.bincount(a, weights=x[:, j], minlength=k)
                         for j in range(x.shape[1])], axis=1)
        nz = cnt > 0
        c[nz] = sums[nz] / cnt[nz, None]
    return c.astype(np.float16)


def calibrate_head(w: synth.Workload, kvh: int, *, sample_tokens: int | None = None,
                   iters: int | None = None, b: int = 0):
    """Returns (s fp32 [128], K codebook fp16 [E][d_sub], V codebook fp16 [E][d_sub]).

    s uses every key row of sequence ``b`` of the workload (its full length);
    the codebooks are trained on ``sample_tokens`` random tokens' subvectors
    (all of them when the sequence is short).  2-bit codebooks use k-means++
    and 20 Lloyd iterations; 1.5-bit codebooks default to random-row seeding
    and fewer iterations, which only changes codebook quality, not any
    parity or timing property.
    """
    L = int(synth.seq_lens(w)[b]) if w.prefill == 0 else w.prefill
    k_all = synth.keys(w, b, kvh, 0, L)
    s = smoothing_vector(k_all)
    E, dsub = w.entries, w.d_sub
    if sample_tokens is None:
        sample_tokens = min(L, (65536 * dsub) // HEAD_DIM)
    r = synth.calibration_rng(w, kvh, 0)
    idx = np.sort(r.choice(L, size=min(sample_tokens, L), replace=False))
    kr = _rotated_key_rows(k_all[idx], s).reshape(-1, dsub)
    v_rows = synth.values(w, b, kvh, 0, L)[idx].astype(np.float32).reshape(-1, dsub)
    if iters is None:
        iters = 4 if E == 4096 else 20
    init = "points" if E == 4096 else "++"
    kcb = kmeans(kr, E, iters, synth.kmeans_rng(w, kvh, 0), init)
    vcb = kmeans(v_rows, E, iters, synth.kmeans_rng(w, kvh, 1), init)
    return s, kcb, vcb


def calibrate(w: synth.Workload, **kw):
    """Per-KV-head calibration: s [Hkv][128] fp32, codebooks [Hkv][E][d_sub] fp16."""
    out = [calibrate_head(w, h, **kw) for h in range(w.Hkv)]
    s = np.stack([o[0] for o in out])
    kcb = np.stack([o[1] for o in out])
    vcb = np.stack([o[2] for o in out])
    return s, kcb, vcb
