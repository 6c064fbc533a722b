"""Seeded synthetic workloads for the VQ KV-cache decode path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no smoothing, rotation, nearest-centroid search, packing
or attention).  Both the CUDA path (through the tests and the benchmark) and
the CPU oracle consume what it returns.

Workloads follow the shapes of the models the VecInfer paper evaluates
(VecInfer: Efficient LLM Inference with Low-Bit KV Cache via
Outlier-Suppressed Vector Quantization, "Key points": Llama-3.1-8B,
Qwen2.5-14B, Mistral-7B; 196k-token context; codebooks of 2^8 x 4 and
2^12 x 8 entries).  The paper's datasets and model weights are not used:
keys, values and queries are Gaussian, with a few key channels scaled up to
act as the outlier channels the paper's smoothing targets ("Summary").

Every stream comes from ``numpy.random.default_rng([seed, config_id,
stream_id, ...])`` so that any slice can be regenerated independently.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

HEAD_DIM = 128

# stream ids (independent substreams per config and tensor)
_S_Q, _S_K, _S_V, _S_OUTLIER, _S_SEQLEN, _S_CODES, _S_CALIB, _S_KMEANS, _S_APPEND = range(1, 10)

MODE_VQ2 = 0
MODE_VQ15 = 1
MODE_VQ4 = 2
MODE_VQ3 = 3
MODE_VQ125 = 4

# codebook geometry per mode: (entries, subvector dims)
MODE_GEOMETRY = {MODE_VQ2: (256, 4), MODE_VQ15: (4096, 8), MODE_VQ4: (256, 2), MODE_VQ3: (4096, 4),
                 MODE_VQ125: (1024, 8)}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode (or encode+decode) workload."""

    config_id: int
    name: str
    mode: int              # MODE_VQ2, MODE_VQ15, MODE_VQ4, MODE_VQ3 or MODE_VQ125
    B: int
    Hq: int
    Hkv: int
    cap_len: int           # cache capacity per sequence (tokens)
    seq_len: int           # tokens per sequence (upper bound when ragged)
    ragged: Optional[tuple] = None   # (lo, hi) inclusive when lengths are drawn
    outliers: str = "random4"        # "fixed4", "random4" (x U[8,20]), "random6x16"
    prefill: int = 0                 # encode workloads: prefill rows per sequence
    append: int = 0                  # encode workloads: appended rows per sequence
    seed: int = 0

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def entries(self) -> int:
        return MODE_GEOMETRY[self.mode][0]

    @property
    def d_sub(self) -> int:
        return MODE_GEOMETRY[self.mode][1]

    @property
    def n_sub(self) -> int:
        return HEAD_DIM // self.d_sub

    def with_mode(self, mode: int) -> "Workload":
        return dataclasses.replace(self, mode=mode)

    def scaled(self, **kw) -> "Workload":
        """Same recipe at other sizes (parity cases the oracle finishes quickly)."""
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny correctness case, the Llama-3.1-8B-shaped 196k
# decode step, a ragged large batch, a Qwen2.5-14B-shaped 1.5-bit decode, and
# a Mistral-7B-shaped encode-then-decode.
WORKLOADS = {
    0: Workload(0, "tiny_vq2_b1_h1_l1024", MODE_VQ2, B=1, Hq=1, Hkv=1, cap_len=1024,
                seq_len=1024, outliers="fixed4"),
    1: Workload(1, "llama8b_vq2_b1_hq32_hkv8_l196608", MODE_VQ2, B=1, Hq=32, Hkv=8,
                cap_len=196608, seq_len=196608),
    2: Workload(2, "ragged_vq2_b32_hq32_hkv8_l16k_32k", MODE_VQ2, B=32, Hq=32, Hkv=8,
                cap_len=32768, seq_len=32768, ragged=(16384, 32768)),
    3: Workload(3, "qwen14b_vq15_b8_hq40_hkv8_l65536", MODE_VQ15, B=8, Hq=40, Hkv=8,
                cap_len=65536, seq_len=65536, outliers="random6x16"),
    4: Workload(4, "mistral7b_b16_hq32_hkv8_prefill16384_append256", MODE_VQ2, B=16, Hq=32,
                Hkv=8, cap_len=16640, seq_len=16640, prefill=16384, append=256),
}


def rng(w: Workload, stream: int, *sub: int) -> np.random.Generator:
    return np.random.default_rng([w.seed, w.config_id, stream, *sub])


def seq_lens(w: Workload) -> np.ndarray:
    """Per-sequence cached lengths, int32 [B]."""
    if w.ragged is None:
        return np.full(w.B, w.seq_len, dtype=np.int32)
    lo, hi = w.ragged
    return rng(w, _S_SEQLEN).integers(lo, hi, size=w.B, endpoint=True).astype(np.int32)


def queries(w: Workload) -> np.ndarray:
    """q, fp16 [B][Hq][128], N(0, 1)."""
    return rng(w, _S_Q).standard_normal((w.B, w.Hq, HEAD_DIM), dtype=np.float32).astype(np.float16)


def outlier_channels(w: Workload, kvh: int):
    """(channels, scales) of the key outlier channels of one KV head."""
    if w.outliers == "fixed4":
        return np.array([3, 17, 64, 101]), np.full(4, 16.0, dtype=np.float32)
    r = rng(w, _S_OUTLIER, kvh)
    if w.outliers == "random4":
        ch = r.choice(HEAD_DIM, size=4, replace=False)
        return np.sort(ch), r.uniform(8.0, 20.0, size=4).astype(np.float32)
    if w.outliers == "random6x16":
        ch = r.choice(HEAD_DIM, size=6, replace=False)
        return np.sort(ch), np.full(6, 16.0, dtype=np.float32)
    raise ValueError(w.outliers)


def keys(w: Workload, b: int, kvh: int, t0: int, n: int, stream: int = _S_K) -> np.ndarray:
    """Rows [t0, t0+n) of the key cache of (b, kvh): fp16 [n][128].

    Rows are generated in blocks of 1024 tokens so that any window is
    reproducible without generating the whole sequence.
    """
    ch, sc = outlier_channels(w, kvh)
    out = _gaussian_rows(w, stream, b, kvh, t0, n)
    out[:, ch] *= sc
    return out.astype(np.float16)


def values(w: Workload, b: int, kvh: int, t0: int, n: int) -> np.ndarray:
    """Rows [t0, t0+n) of the value cache of (b, kvh): fp16 [n][128], N(0, 1)."""
    return _gaussian_rows(w, _S_V, b, kvh, t0, n).astype(np.float16)


def appended_keys(w: Workload, b: int, kvh: int, n: int) -> np.ndarray:
    """Rows of new decode-step tokens (distinct stream from the prefill)."""
    return keys(w, b, kvh, 0, n, stream=_S_APPEND)


_BLOCK = 1024


def _gaussian_rows(w: Workload, stream: int, b: int, kvh: int, t0: int, n: int) -> np.ndarray:
    out = np.empty((n, HEAD_DIM), dtype=np.float32)
    blk0, blk1 = t0 // _BLOCK, (t0 + n - 1) // _BLOCK if n > 0 else t0 // _BLOCK - 1
    pos = 0
    for blk in range(blk0, blk1 + 1):
        rows = rng(w, stream, b, kvh, blk).standard_normal((_BLOCK, HEAD_DIM), dtype=np.float32)
        lo = max(t0, blk * _BLOCK) - blk * _BLOCK
        hi = min(t0 + n, (blk + 1) * _BLOCK) - blk * _BLOCK
        out[pos:pos + hi - lo] = rows[lo:hi]
        pos += hi - lo
    return out


def uniform_codes(w: Workload, b: int, kvh: int, role: int, n: int) -> np.ndarray:
    """Codebook indices for n tokens of one cache stream, drawn uniformly.

    Used where a full-size cache is needed faster than it could be encoded on
    the CPU; int32 [n][n_sub], values in [0, entries).
    """
    r = rng(w, _S_CODES, b, kvh, role)
    return r.integers(0, w.entries, size=(n, w.n_sub), dtype=np.int32)


def calibration_rng(w: Workload, kvh: int, role: int) -> np.random.Generator:
    return rng(w, _S_CALIB, kvh, role)


def kmeans_rng(w: Workload, kvh: int, role: int) -> np.random.Generator:
    return rng(w, _S_KMEANS, kvh, role)
