"""Plain fp64 CPU oracle of VecInfer's hot path (test infrastructure only).

Sources (cited as page title + section):
  [P1] "VecInfer: Efficient LLM Inference with Low-Bit KV Cache via
       Outlier-Suppressed Vector Quantization", Elamur Research summary page,
       sections "Summary" and "Key points".
  [P2] the same title, arXiv 2510.06175 summary page, sections
       "方法详解" (method: preprocessing -> quantization -> fused kernel) and
       "摘要（原文）" (abstract).
What the pages fix:
  * keys are smoothed channel-wise, then rotated by a Hadamard transform;
    the query gets the matching inverse so q.K^T is unchanged [P1 Summary];
  * each subvector of the transformed key (and of the value) is replaced by
    the index of a K-Means centroid; 2-bit = 2^8 entries x 4 dims, 1.5-bit =
    2^12 entries x 8 dims [P1 Key points];
  * attention is computed over the dequantised cache [P1 Summary, P2 方法详解].
Readings where the pages are silent (each also in the readings table):
  * smoothing divides keys by s and multiplies queries by s;
  * the rotation is the normalised Sylvester matrix Hn = H/sqrt(128) with
    H[i][k] = (-1)^popcount(i & k); values are not transformed;
  * one K and one V codebook per KV head, shared by all subvector positions;
  * the transformed key is rounded to fp32 before the nearest-centroid
    search, distances are decided in fp32 with ties to the lowest index;
  * softmax scale 1/sqrt(128); query head h reads KV head h // (Hq/Hkv);
  * the packed-cache byte layout is this library's own (include/vqkv.h).
No function here is used by the CUDA path; nothing here reads CUDA output
except through the comparisons made in tests/.
"""
from __future__ import annotations

import math

import numpy as np

HEAD_DIM = 128
MODE_VQ2 = 0
MODE_VQ15 = 1
MODE_VQ4 = 2
MODE_VQ3 = 3
MODE_VQ125 = 4
ROLE_K = 0
ROLE_V = 1

# (entries, subvector dims) per mode [P1 Key points: 2^8 x 4 and 2^12 x 8]
# and, within the pages' 1.25-4 bit range [P1 Summary], 4 bit = 2^8 x 2,
# 3 bit = 2^12 x 4 and 1.25 bit = 2^10 x 8
GEOMETRY = {MODE_VQ2: (256, 4), MODE_VQ15: (4096, 8), MODE_VQ4: (256, 2), MODE_VQ3: (4096, 4),
            MODE_VQ125: (1024, 8)}
# tokens per layout tile and bytes per tile of one cache stream
TILE_TOKENS = {MODE_VQ2: 16, MODE_VQ15: 64, MODE_VQ4: 16, MODE_VQ3: 16, MODE_VQ125: 16}
TILE_BYTES = {MODE_VQ2: 512, MODE_VQ15: 1536, MODE_VQ4: 1024, MODE_VQ3: 768, MODE_VQ125: 320}
BYTE_CODE_MODES = (MODE_VQ2, MODE_VQ4)   # one byte per code


# ----------------------------------------------------------------------------
# Rotation and smoothing  [P1 Summary: "channel-wise smoothing followed by a
# Hadamard rotation ... matching inverse operations on the queries"]
# ----------------------------------------------------------------------------

def sylvester_hadamard(n: int = HEAD_DIM) -> np.ndarray:
    """H[i][k] = (-1)^popcount(i & k), built entry by entry (fp64, +-1)."""
    h = np.empty((n, n), dtype=np.float64)
    for i in range(n):
        for k in range(n):
            h[i, k] = -1.0 if bin(i & k).count("1") % 2 else 1.0
    return h


_HN = None


def normalized_hadamard() -> np.ndarray:
    """Hn = H / sqrt(128): orthonormal and symmetric."""
    global _HN
    if _HN is None:
        _HN = sylvester_hadamard(HEAD_DIM) / math.sqrt(HEAD_DIM)
    return _HN


def transform_keys(x: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Key rows to the quantisation domain: x' = (x / s) . Hn, fp64 math,
    returned rounded to fp32 (the vector the nearest-centroid search sees).

    x: fp16 [..., 128]; s: fp32 [128] smoothing factors of the KV head.
    """
    y = x.astype(np.float64) / s.astype(np.float64)
    return (y @ normalized_hadamard()).astype(np.float32)


def transform_values(x: np.ndarray) -> np.ndarray:
    """Values are quantised as they are (no smoothing, no rotation)."""
    return x.astype(np.float32)


def transform_query(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """The matching query transform q' = (q * s) . Hn (fp64), so that
    q' . x'^T = q . x^T for an unquantised key x (exactly, up to rounding)."""
    return (q.astype(np.float64) * s.astype(np.float64)) @ normalized_hadamard()


def untransform_keys(xq: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Inverse of the key transform: (x' . Hn^T) * s, fp64."""
    return (xq.astype(np.float64) @ normalized_hadamard().T) * s.astype(np.float64)


# ----------------------------------------------------------------------------
# Nearest centroid  [P1 Summary: K-Means codebook; P2 方法详解 stage 2]
# ----------------------------------------------------------------------------

def subvector_distances(sub: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    """Squared Euclidean distance of every subvector to every centroid.

    sub: fp32 [N][d_sub]; codebook: fp16 [E][d_sub].
    Returns fp64 [N][E], each entry sum_i (sub_i - c_i)^2 by direct
    differences (no expansion), computed in fp64 from the exact fp32/fp16
    operands.
    """
    x = sub.astype(np.float64)[:, None, :]
    c = codebook.astype(np.float64)[None, :, :]
    return ((x - c) ** 2).sum(axis=2)


def nearest_centroid(sub: np.ndarray, codebook: np.ndarray):
    """Index of the nearest centroid of each subvector.

    The decision is taken on distances rounded to fp32; among equal fp32
    distances the lowest index wins.  Returns (codes int64 [N], d32 fp32 [N][E]).
    """
    out_codes = np.empty(sub.shape[0], dtype=np.int64)
    out_d = np.empty((sub.shape[0], codebook.shape[0]), dtype=np.float32)
    step = max(1, (1 << 22) // codebook.shape[0])
    for r0 in range(0, sub.shape[0], step):
        d32 = subvector_distances(sub[r0:r0 + step], codebook).astype(np.float32)
        out_codes[r0:r0 + step] = np.argmin(d32, axis=1)   # first minimum
        out_d[r0:r0 + step] = d32
    return out_codes, out_d


def encode_rows(x: np.ndarray, role: int, s, codebook: np.ndarray):
    """Quantise rows of one KV head.

    x: fp16 [n][128]; role ROLE_K (smooth + rotate) or ROLE_V (as is);
    s: fp32 [128] (keys only); codebook fp16 [E][d_sub].
    Returns (codes int64 [n][n_sub], d32 fp32 [n][n_sub][E]).
    """
    xt = transform_keys(x, s) if role == ROLE_K else transform_values(x)
    dsub = codebook.shape[1]
    n, nsub = xt.shape[0], HEAD_DIM // dsub
    codes, d = nearest_centroid(xt.reshape(n * nsub, dsub), codebook)
    return codes.reshape(n, nsub), d.reshape(n, nsub, -1)


def near_tie(d32_row: np.ndarray, chosen: int) -> bool:
    """True when centroid ``chosen`` is within 1e-6 (relative, fp32
    distances) of the best one, i.e. a tie that rounding may decide."""
    best = float(d32_row.min())
    return abs(float(d32_row[chosen]) - best) < 1e-6 * max(best, 1e-30)


# ----------------------------------------------------------------------------
# Packed cache layout (this library's own byte layout, include/vqkv.h)
# ----------------------------------------------------------------------------

def bits_per_element(mode: int) -> float:
    """log2(entries) / subvector dims [P1 Key points]."""
    e, dsub = GEOMETRY[mode]
    return math.log2(e) / dsub


def code_bytes(mode: int, cap_len: int) -> int:
    """Bytes of one cache stream (one of K or V, one (sequence, KV head))."""
    t = TILE_TOKENS[mode]
    return -(-cap_len // t) * TILE_BYTES[mode]


def vq2_offset(role: int, t: int, j: int) -> int:
    """Byte holding the 8-bit code of subvector j (0..31) of token t."""
    tile, r = divmod(t, 16)
    if role == ROLE_K:
        lane = 4 * (r % 8) + (j % 4)
        return 512 * tile + 16 * lane + 8 * (r // 8) + (j // 4)
    lane = 4 * (j % 8) + (r % 8) // 2
    return 512 * tile + 16 * lane + 4 * (j // 8) + 2 * (r // 8) + (r % 2)


def vq4_offset(role: int, t: int, j: int) -> int:
    """Byte holding the 8-bit code of subvector j (0..63, channels 2j, 2j+1) of token t."""
    tile, r = divmod(t, 16)
    if role == ROLE_K:
        lane = 4 * (r % 8) + (j % 4)
        return 1024 * tile + 512 * (r // 8) + 16 * lane + 2 * (j // 8) + (j // 4) % 2
    lane = 4 * (j % 8) + (r % 8) // 2
    return 1024 * tile + 512 * (j // 32) + 16 * lane + 4 * ((j // 8) % 4) + 2 * (r // 8) + (r % 2)


def byte_offset(mode: int, role: int, t: int, j: int) -> int:
    return vq2_offset(role, t, j) if mode == MODE_VQ2 else vq4_offset(role, t, j)


def vq3_byte(role: int, t: int, pair: int, k: int) -> int:
    """Byte k (0..2) of the 3-byte code pair (pair, pair+16) (pair 0..15) of token t.

    A tile is 32 lanes' 24-byte runs stored as two planes: run bytes 0..15 of
    lane L at 16*L, run bytes 16..23 at 512 + 8*L.  K: lane 4*(r%8) + pair%4,
    run byte 12*(r/8) + 3*(pair/4) + k.  V: lane 4*(pair%8) + (r%8)/2, run
    byte 6*(2*(r/8) + r%2) + 3*(pair/8) + k.
    """
    tile, r = divmod(t, 16)
    if role == ROLE_K:
        lane, b = 4 * (r % 8) + pair % 4, 12 * (r // 8) + 3 * (pair // 4) + k
    else:
        lane, b = 4 * (pair % 8) + (r % 8) // 2, 6 * (2 * (r // 8) + r % 2) + 3 * (pair // 8) + k
    return 768 * tile + (16 * lane + b if b < 16 else 512 + 8 * lane + b - 16)


def vq125_bit(role: int, t: int, j: int, b: int) -> int:
    """Stream bit address (8 * byte + bit, LSB first) of bit b (0..9) of the
    10-bit code of subvector j (0..15, channels 8j..8j+7) of token t.

    A 320-byte tile of 16 tokens is a set of runs, each stored as two planes
    (plane 0 from byte 0, plane 1 from byte 256); run bits are numbered from
    the least significant bit of the run's first byte.  K: 32 runs of 10
    bytes (plane 0: 8 bytes at 8*L, plane 1: 2 bytes at 256 + 2*L), run
    L = 4*(r%8) + j%4, run bit 40*(r/8) + 10*(j/4) + b.  V: 16 runs of 20
    bytes (plane 0: 16 bytes at 16*R, plane 1: 4 bytes at 256 + 4*R), run
    R = 4*((j%8)/2) + (r%8)/2, run bit 40*(2*(r/8) + r%2) + 10*(j%2 + 2*(j/8))
    + b.  Each token's bits of a run fill 5 whole bytes.
    """
    tile, r = divmod(t, 16)
    if role == ROLE_K:
        run, rb, p0, p1 = 4 * (r % 8) + j % 4, 40 * (r // 8) + 10 * (j // 4) + b, 8, 2
    else:
        run, rb, p0, p1 = 4 * ((j % 8) // 2) + (r % 8) // 2, 40 * (2 * (r // 8) + r % 2) + 10 * (j % 2 + 2 * (j // 8)) + b, 16, 4
    n, bit = divmod(rb, 8)
    byte = p0 * run + n if n < p0 else 256 + p1 * run + n - p0
    return 8 * (320 * tile + byte) + bit


def vq15_offset(role: int, t: int, pair: int) -> int:
    """First of the 3 bytes holding the code pair (pair, pair+8) of token t."""
    tile, rem = divmod(t, 64)
    quarter, r = divmod(rem, 16)
    if role == ROLE_K:
        lane = 4 * (r % 8) + (pair % 4)
        return 1536 * tile + 48 * lane + 12 * quarter + 6 * (r // 8) + 3 * (pair // 4)
    lane = 4 * pair + (r % 8) // 2
    return 1536 * tile + 48 * lane + 12 * quarter + 3 * ((r % 2) + 2 * (r // 8))


def pack_pair(c_lo: int, c_hi: int):
    """Two 12-bit codes -> 3 bytes, little-endian nibble order."""
    return (c_lo & 0xFF, (c_lo >> 8) | ((c_hi & 0xF) << 4), c_hi >> 4)


def unpack_pair(b0: int, b1: int, b2: int):
    return b0 | ((b1 & 0xF) << 8), (b1 >> 4) | (b2 << 4)


def pack_stream(codes: np.ndarray, mode: int, role: int, cap_len: int,
                out: np.ndarray | None = None) -> np.ndarray:
    """codes int [L][n_sub] (token t at row t) -> uint8 stream of code_bytes."""
    buf = np.zeros(code_bytes(mode, cap_len), dtype=np.uint8) if out is None else out
    L = codes.shape[0]
    if mode in BYTE_CODE_MODES:
        for t in range(L):
            for j in range(codes.shape[1]):
                buf[byte_offset(mode, role, t, j)] = int(codes[t, j])
    elif mode == MODE_VQ3:
        for t in range(L):
            for p in range(16):
                for k, byte in enumerate(pack_pair(int(codes[t, p]), int(codes[t, p + 16]))):
                    buf[vq3_byte(role, t, p, k)] = byte
    elif mode == MODE_VQ125:
        for t in range(L):
            for j in range(16):
                for b in range(10):
                    a = vq125_bit(role, t, j, b)
                    if (int(codes[t, j]) >> b) & 1:
                        buf[a // 8] |= 1 << (a % 8)
                    else:
                        buf[a // 8] &= ~(1 << (a % 8)) & 0xFF
    else:
        for t in range(L):
            for p in range(8):
                o = vq15_offset(role, t, p)
                buf[o:o + 3] = pack_pair(int(codes[t, p]), int(codes[t, p + 8]))
    return buf


def unpack_stream(buf: np.ndarray, mode: int, role: int, L: int) -> np.ndarray:
    """uint8 stream -> codes int64 [L][n_sub]."""
    if mode in BYTE_CODE_MODES:
        nsub = HEAD_DIM // GEOMETRY[mode][1]
        out = np.empty((L, nsub), dtype=np.int64)
        for t in range(L):
            for j in range(nsub):
                out[t, j] = buf[byte_offset(mode, role, t, j)]
        return out
    if mode == MODE_VQ3:
        out = np.empty((L, 32), dtype=np.int64)
        for t in range(L):
            for p in range(16):
                out[t, p], out[t, p + 16] = unpack_pair(*(int(buf[vq3_byte(role, t, p, k)]) for k in range(3)))
        return out
    if mode == MODE_VQ125:
        out = np.zeros((L, 16), dtype=np.int64)
        for t in range(L):
            for j in range(16):
                for b in range(10):
                    a = vq125_bit(role, t, j, b)
                    out[t, j] |= ((int(buf[a // 8]) >> (a % 8)) & 1) << b
        return out
    out = np.empty((L, 16), dtype=np.int64)
    for t in range(L):
        for p in range(8):
            o = vq15_offset(role, t, p)
            out[t, p], out[t, p + 8] = unpack_pair(int(buf[o]), int(buf[o + 1]), int(buf[o + 2]))
    return out


def offset_table(mode: int, role: int, L: int) -> np.ndarray:
    """Byte offset of every code (VQ2, VQ4) or code pair (VQ15; VQ3: of each
    of its 3 bytes, [L][16][3]) of tokens [0, L), or the stream bit address
    of every code bit (VQ125, [L][16][10]): a vectorised form of the offset
    functions above, for large streams."""
    t = np.arange(L)[:, None]
    if mode == MODE_VQ125:   # [L][16 subvectors][10 bits]: bit addresses
        j = np.arange(16)[None, :, None]
        b = np.arange(10)[None, None, :]
        tt = t[:, :, None]
        tile, r = tt // 16, tt % 16
        if role == ROLE_K:
            run, rb, p0, p1 = 4 * (r % 8) + j % 4, 40 * (r // 8) + 10 * (j // 4) + b, 8, 2
        else:
            run, rb, p0, p1 = (4 * ((j % 8) // 2) + (r % 8) // 2,
                               40 * (2 * (r // 8) + r % 2) + 10 * (j % 2 + 2 * (j // 8)) + b, 16, 4)
        n, bit = rb // 8, rb % 8
        return 8 * (320 * tile + np.where(n < p0, p0 * run + n, 256 + p1 * run + n - p0)) + bit
    if mode == MODE_VQ3:   # [L][16 pairs][3 bytes]
        p = np.arange(16)[None, :, None]
        k = np.arange(3)[None, None, :]
        tt = t[:, :, None]
        tile, r = tt // 16, tt % 16
        if role == ROLE_K:
            lane, b = 4 * (r % 8) + p % 4, 12 * (r // 8) + 3 * (p // 4) + k
        else:
            lane, b = 4 * (p % 8) + (r % 8) // 2, 6 * (2 * (r // 8) + r % 2) + 3 * (p // 8) + k
        return 768 * tile + np.where(b < 16, 16 * lane + b, 512 + 8 * lane + b - 16)
    if mode == MODE_VQ4:
        j = np.arange(64)[None, :]
        tile, r = t // 16, t % 16
        if role == ROLE_K:
            return 1024 * tile + 512 * (r // 8) + 16 * (4 * (r % 8) + j % 4) + 2 * (j // 8) + (j // 4) % 2
        return (1024 * tile + 512 * (j // 32) + 16 * (4 * (j % 8) + (r % 8) // 2) + 4 * ((j // 8) % 4)
                + 2 * (r // 8) + r % 2)
    if mode == MODE_VQ2:
        j = np.arange(32)[None, :]
        tile, r = t // 16, t % 16
        if role == ROLE_K:
            return 512 * tile + 16 * (4 * (r % 8) + j % 4) + 8 * (r // 8) + j // 4
        return 512 * tile + 16 * (4 * (j % 8) + (r % 8) // 2) + 4 * (j // 8) + 2 * (r // 8) + r % 2
    p = np.arange(8)[None, :]
    tile, rem = t // 64, t % 64
    quarter, r = rem // 16, rem % 16
    if role == ROLE_K:
        return 1536 * tile + 48 * (4 * (r % 8) + p % 4) + 12 * quarter + 6 * (r // 8) + 3 * (p // 4)
    return 1536 * tile + 48 * (4 * p + (r % 8) // 2) + 12 * quarter + 3 * ((r % 2) + 2 * (r // 8))


def pack_stream_fast(codes: np.ndarray, mode: int, role: int, cap_len: int) -> np.ndarray:
    buf = np.zeros(code_bytes(mode, cap_len), dtype=np.uint8)
    off = offset_table(mode, role, codes.shape[0])
    if mode in BYTE_CODE_MODES:
        buf[off] = codes.astype(np.uint8)
    elif mode == MODE_VQ125:   # no two code bits share a stream bit, so summing is or-ing
        bits = ((codes.astype(np.int64)[..., None] >> np.arange(10)) & 1) << (off & 7)
        n = int(off.max() >> 3) + 1 if off.size else 0
        buf[:n] = np.bincount((off >> 3).ravel(), weights=bits.ravel(), minlength=n).astype(np.uint8)
    elif mode == MODE_VQ3:
        lo, hi = codes[:, :16].astype(np.int64), codes[:, 16:].astype(np.int64)
        buf[off[..., 0]] = lo & 0xFF
        buf[off[..., 1]] = (lo >> 8) | ((hi & 0xF) << 4)
        buf[off[..., 2]] = hi >> 4
    else:
        lo, hi = codes[:, :8].astype(np.int64), codes[:, 8:].astype(np.int64)
        buf[off] = lo & 0xFF
        buf[off + 1] = (lo >> 8) | ((hi & 0xF) << 4)
        buf[off + 2] = hi >> 4
    return buf


def unpack_stream_fast(buf: np.ndarray, mode: int, role: int, L: int) -> np.ndarray:
    off = offset_table(mode, role, L)
    if mode in BYTE_CODE_MODES:
        return buf[off].astype(np.int64)
    if mode == MODE_VQ3:
        b0, b1, b2 = (buf[off[..., k]].astype(np.int64) for k in range(3))
        return np.concatenate([b0 | ((b1 & 0xF) << 8), (b1 >> 4) | (b2 << 4)], axis=1)
    if mode == MODE_VQ125:
        bits = (buf[off >> 3].astype(np.int64) >> (off & 7)) & 1
        return (bits << np.arange(10)).sum(axis=2)
    b0, b1, b2 = (buf[off + k].astype(np.int64) for k in range(3))
    return np.concatenate([b0 | ((b1 & 0xF) << 8), (b1 >> 4) | (b2 << 4)], axis=1)


# ----------------------------------------------------------------------------
# Decode attention over the quantised cache  [P1 Summary; P2 方法详解 stage 3]
# ----------------------------------------------------------------------------

def dequantize(codes: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    """codes [L][n_sub] -> concatenated centroids [L][128] (fp64)."""
    L = codes.shape[0]
    return codebook.astype(np.float64)[codes].reshape(L, HEAD_DIM)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Single-query softmax attention in fp64: softmax(scale * k.q) . v.
    An empty cache gives a zero row."""
    if k.shape[0] == 0:
        return np.zeros(v.shape[1], dtype=np.float64)
    z = scale * (k @ q.astype(np.float64))
    p = np.exp(z - z.max())
    return (p @ v) / p.sum()


def decode_attention(q, k_codes, v_codes, k_cb, v_cb, s, seq_lens, scale=None,
                     heads=None) -> np.ndarray:
    """O for every (b, query head), in the keys' original domain.

    q fp16 [B][Hq][128]; k_codes/v_codes int [B][Hkv][>=L_b][n_sub];
    k_cb/v_cb fp16 [Hkv][E][d_sub]; s fp32 [Hkv][128]; seq_lens int [B].
    The dequantised rotated keys are mapped back with the inverse rotation
    and smoothing, K = (K' . Hn^T) * s, and plain attention runs on q and K,
    so the query transform is not used here at all.
    ``heads``: optional list of (b, h) to compute (others stay NaN).
    Returns fp64 [B][Hq][128].
    """
    B, Hq, _ = q.shape
    Hkv = k_cb.shape[0]
    g = Hq // Hkv
    scale = 1.0 / math.sqrt(HEAD_DIM) if scale is None else scale
    out = np.full((B, Hq, HEAD_DIM), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    cache = {}
    for b, h in todo:
        kvh = h // g
        L = int(seq_lens[b])
        key = (b, kvh)
        if key not in cache:
            kq = dequantize(k_codes[b][kvh][:L], k_cb[kvh])
            cache.clear()
            cache[key] = (untransform_keys(kq, s[kvh]), dequantize(v_codes[b][kvh][:L], v_cb[kvh]))
        kk, vv = cache[key]
        out[b, h] = attention(q[b, h], kk, vv, scale)
    return out


def decode_attention_multi(q, k_codes, v_codes, k_cb, v_cb, s, seq_lens, scale=None) -> np.ndarray:
    """Several queries per sequence over the same cache (chunked prefill or
    speculative decoding on a VQ cache: attention over the dequantised cache
    [P1 Summary], with M new tokens at the end of each sequence).

    Reading: the M queries of sequence b are the tokens at positions
    L_b - M .. L_b - 1 and attend causally, so query m sees the cached
    tokens t <= L_b - M + m (none when that is negative: a zero row).
    q fp16 [B][M][Hq][128]; returns fp64 [B][M][Hq][128].  Each query is a
    single-query decode over its visible prefix.
    """
    B, M = q.shape[0], q.shape[1]
    out = np.empty(q.shape, dtype=np.float64)
    for m in range(M):
        lens_m = [max(0, int(L) - M + m + 1) for L in seq_lens]
        out[:, m] = decode_attention(q[:, m], k_codes, v_codes, k_cb, v_cb, s, lens_m, scale)
    return out


def decode_attention_rotated(q, k_codes, v_codes, k_cb, v_cb, s, seq_lens, scale=None,
                             heads=None) -> np.ndarray:
    """Same result computed in the rotated domain: scale * q' . K'^T with
    q' = (q * s) . Hn.  Cheaper than decode_attention (no per-token inverse
    rotation); it is checked against decode_attention in the tests."""
    B, Hq, _ = q.shape
    Hkv = k_cb.shape[0]
    g = Hq // Hkv
    scale = 1.0 / math.sqrt(HEAD_DIM) if scale is None else scale
    out = np.full((B, Hq, HEAD_DIM), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in todo:
        kvh = h // g
        L = int(seq_lens[b])
        kq = dequantize(k_codes[b][kvh][:L], k_cb[kvh])
        vv = dequantize(v_codes[b][kvh][:L], v_cb[kvh])
        out[b, h] = attention(transform_query(q[b, h], s[kvh]), kq, vv, scale)
    return out


def o_error(o_gpu: np.ndarray, o_ref: np.ndarray) -> np.ndarray:
    """Per-row error: max_d |O_gpu - O_ref| / max_d |O_ref| (rows of zeros
    compare absolutely)."""
    num = np.abs(o_gpu.astype(np.float64) - o_ref).max(axis=-1)
    den = np.abs(o_ref).max(axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
