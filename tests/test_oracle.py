"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each check is a plain function so that the mutation tests at the end can
plant a plausible mistake in the oracle (on the CPU) and show that at least
one pin fails.  None of these tests touches the CUDA path.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import scipy.spatial.distance
import torch

import oracle
from oracle import vqkv_oracle as vo
from tests.conftest import golden_lines

SCALE = 1.0 / math.sqrt(128)


# --------------------------------------------------------------- rotation

def check_hadamard():
    h = vo.sylvester_hadamard(128)
    # an independent construction (library routine) of the same matrix
    assert np.array_equal(h, scipy.linalg.hadamard(128).astype(np.float64))
    hn = vo.normalized_hadamard()
    assert np.abs(hn @ hn.T - np.eye(128)).max() < 1e-12
    assert np.allclose(np.abs(hn), 1 / math.sqrt(128), rtol=0, atol=1e-15)


def check_score_invariance():
    """q'.K'^T = q.K^T for unquantised keys, to 1e-5 relative (the matching
    inverse transform keeps attention scores unchanged)."""
    r = np.random.default_rng(11)
    q = r.standard_normal((8, 128)).astype(np.float16)
    k = r.standard_normal((64, 128)).astype(np.float32)
    k[:, [5, 40, 77]] *= 15
    k = k.astype(np.float16)
    s = np.sqrt(np.abs(k.astype(np.float32)).max(axis=0)).astype(np.float32)
    qt = vo.transform_query(q, s)
    kt = vo.transform_keys(k, s)
    ref = q.astype(np.float64) @ k.astype(np.float64).T
    got = qt @ kt.astype(np.float64).T
    assert np.abs(got - ref).max() / np.abs(ref).max() < 1e-5
    # and the inverse transform recovers the keys
    assert np.abs(vo.untransform_keys(kt, s) - k.astype(np.float64)).max() < 1e-4


def check_sign_patterns():
    a = [0.70703125, 8.0, 0.353515625]
    cb = np.zeros((48, 4), dtype=np.float16)
    for blk in range(3):
        for e in range(16):
            cb[16 * blk + e] = [-a[blk] if (e >> m) & 1 else a[blk] for m in range(4)]
    for line in golden_lines("hadamard_signs.txt"):
        f = line.split()
        sk, k, rule, codes = float(f[0]), int(f[1]), f[2], [int(c) for c in f[3:]]
        x = np.zeros((1, 128), dtype=np.float16)
        x[0, k] = 8
        s = np.ones(128, dtype=np.float32)
        s[k] = sk
        got, _ = vo.encode_rows(x, vo.ROLE_K, s, cb)
        for j in range(32):
            if rule == "all":
                want = codes[0]
            elif rule == "jbit0":
                want = codes[j & 1]
            else:
                want = codes[(j >> 1) & 1]
            assert got[0, j] == want, (line, j, got[0, j], want)


def test_hadamard():
    check_hadamard()


def test_score_invariance():
    check_score_invariance()


def test_sign_patterns():
    check_sign_patterns()


def test_values_are_not_transformed():
    r = np.random.default_rng(3)
    x = r.standard_normal((5, 128)).astype(np.float16)
    assert np.array_equal(vo.transform_values(x), x.astype(np.float32))


# ------------------------------------------------------- nearest centroid

def check_nearest_golden():
    cent, qs = [], []
    for line in golden_lines("nearest_centroid.txt"):
        f = line.split()
        if f[0] == "C":
            cent.append([float(v) for v in f[1:5]])
        else:
            qs.append(([float(v) for v in f[1:5]], int(f[-1])))
    cb = np.array(cent, dtype=np.float16)
    sub = np.array([q for q, _ in qs], dtype=np.float32)
    codes, d = vo.nearest_centroid(sub, cb)
    assert list(codes) == [w for _, w in qs]
    assert d[5, 1] == 0.0


def check_nearest_bruteforce():
    """Against a library distance routine on random data (away from ties)."""
    r = np.random.default_rng(5)
    for E, dsub in ((256, 4), (4096, 8), (7, 4)):
        cb = r.standard_normal((E, dsub)).astype(np.float16)
        sub = r.standard_normal((300, dsub)).astype(np.float32)
        codes, d = vo.nearest_centroid(sub, cb)
        ref = scipy.spatial.distance.cdist(sub.astype(np.float64), cb.astype(np.float64), "sqeuclidean")
        assert np.allclose(d, ref, rtol=1e-6)
        srt = np.sort(ref, axis=1)
        clear = (srt[:, 1] - srt[:, 0]) > 1e-5 * srt[:, 0]
        assert np.array_equal(codes[clear], ref.argmin(axis=1)[clear])


def test_nearest_golden():
    check_nearest_golden()


def test_nearest_bruteforce():
    check_nearest_bruteforce()


def test_exact_centroid_gives_zero_distance():
    r = np.random.default_rng(9)
    cb = r.standard_normal((256, 4)).astype(np.float16)
    idx = r.integers(0, 256, size=64)
    codes, d = vo.nearest_centroid(cb[idx].astype(np.float32), cb)
    assert np.all(d[np.arange(64), codes] == 0)
    # duplicates in a random fp16 codebook are unlikely; when present the lowest index wins
    first = np.array([np.flatnonzero((cb == cb[i]).all(axis=1))[0] for i in idx])
    assert np.array_equal(codes, first)


def test_near_tie_rule():
    row = np.array([1.0, 1.0 + 5e-7, 1.0 + 2e-6, 3.0], dtype=np.float32)
    assert vo.near_tie(row, 0) and vo.near_tie(row, 1)
    assert not vo.near_tie(row, 2) and not vo.near_tie(row, 3)


# ------------------------------------------------------------ bits/layout

def check_bits():
    assert vo.bits_per_element(vo.MODE_VQ2) == 2.0
    assert vo.bits_per_element(vo.MODE_VQ15) == 1.5
    assert vo.bits_per_element(vo.MODE_VQ4) == 4.0
    assert vo.bits_per_element(vo.MODE_VQ3) == 3.0
    assert vo.bits_per_element(vo.MODE_VQ125) == 1.25
    for mode, cap in ((vo.MODE_VQ2, 16), (vo.MODE_VQ2, 196608), (vo.MODE_VQ15, 64), (vo.MODE_VQ15, 65536),
                      (vo.MODE_VQ4, 16), (vo.MODE_VQ4, 16384), (vo.MODE_VQ3, 16), (vo.MODE_VQ3, 65536),
                      (vo.MODE_VQ125, 16), (vo.MODE_VQ125, 65536)):
        assert vo.code_bytes(mode, cap) * 8 / (cap * 128) == vo.bits_per_element(mode)
    assert vo.code_bytes(vo.MODE_VQ2, 17) == 1024      # rounded up to whole tiles
    assert vo.code_bytes(vo.MODE_VQ15, 65) == 3072
    assert vo.code_bytes(vo.MODE_VQ4, 17) == 2048
    assert vo.code_bytes(vo.MODE_VQ125, 17) == 640


def check_layout_golden():
    for line in golden_lines("layout_vq2.txt"):
        role, t, j, off = line.split()
        r = vo.ROLE_K if role == "K" else vo.ROLE_V
        assert vo.vq2_offset(r, int(t), int(j)) == int(off), line
    for line in golden_lines("layout_vq4.txt"):
        role, t, j, off = line.split()
        r = vo.ROLE_K if role == "K" else vo.ROLE_V
        assert vo.vq4_offset(r, int(t), int(j)) == int(off), line
    for line in golden_lines("layout_vq3.txt"):
        role, t, p, k, off = line.split()
        r = vo.ROLE_K if role == "K" else vo.ROLE_V
        assert vo.vq3_byte(r, int(t), int(p), int(k)) == int(off), line
    for line in golden_lines("layout_vq125.txt"):
        role, t, j, b, addr = line.split()
        r = vo.ROLE_K if role == "K" else vo.ROLE_V
        assert vo.vq125_bit(r, int(t), int(j), int(b)) == int(addr), line
    for line in golden_lines("layout_vq15.txt"):
        role, t, p, off = line.split()
        r = vo.ROLE_K if role == "K" else vo.ROLE_V
        assert vo.vq15_offset(r, int(t), int(p)) == int(off), line
    for line in golden_lines("pair_bytes.txt"):
        lo, hi, b0, b1, b2 = (int(v, 16) for v in line.split())
        assert vo.pack_pair(lo, hi) == (b0, b1, b2), line
        assert vo.unpack_pair(b0, b1, b2) == (lo, hi), line


def check_layout_bijective():
    for role in (0, 1):   # VQ125: bit by bit
        addrs = [vo.vq125_bit(role, t, j, b) for t in range(32) for j in range(16) for b in range(10)]
        assert sorted(addrs) == list(range(8 * 2 * vo.TILE_BYTES[vo.MODE_VQ125]))
        tab = vo.offset_table(vo.MODE_VQ125, role, 32)
        ref = [[[vo.vq125_bit(role, t, j, b) for b in range(10)] for j in range(16)] for t in range(32)]
        assert np.array_equal(tab, np.array(ref))
    for role in (0, 1):   # VQ3: byte by byte
        offs = [vo.vq3_byte(role, t, p, k) for t in range(32) for p in range(16) for k in range(3)]
        assert sorted(offs) == list(range(2 * vo.TILE_BYTES[vo.MODE_VQ3]))
        tab = vo.offset_table(vo.MODE_VQ3, role, 32)
        ref = [[[vo.vq3_byte(role, t, p, k) for k in range(3)] for p in range(16)] for t in range(32)]
        assert np.array_equal(tab, np.array(ref))
    for mode, role in ((0, 0), (0, 1), (1, 0), (1, 1), (2, 0), (2, 1)):
        T = vo.TILE_TOKENS[mode]
        if mode == vo.MODE_VQ4:
            offs = [vo.vq4_offset(role, t, j) for t in range(2 * T) for j in range(64)]
        elif mode == vo.MODE_VQ2:
            offs = [vo.vq2_offset(role, t, j) for t in range(2 * T) for j in range(32)]
        else:
            offs = [vo.vq15_offset(role, t, p) + k for t in range(2 * T) for p in range(8) for k in range(3)]
        assert sorted(offs) == list(range(2 * vo.TILE_BYTES[mode]))
        tab = vo.offset_table(mode, role, 2 * T)
        if mode == vo.MODE_VQ4:
            ref = [[vo.vq4_offset(role, t, j) for j in range(64)] for t in range(2 * T)]
        elif mode == vo.MODE_VQ2:
            ref = [[vo.vq2_offset(role, t, j) for j in range(32)] for t in range(2 * T)]
        else:
            ref = [[vo.vq15_offset(role, t, p) for p in range(8)] for t in range(2 * T)]
        assert np.array_equal(tab, np.array(ref))


def test_bits():
    check_bits()


def test_layout_golden():
    check_layout_golden()


def test_layout_bijective():
    check_layout_bijective()


def test_pack_roundtrip():
    r = np.random.default_rng(1)
    for mode in (vo.MODE_VQ2, vo.MODE_VQ15, vo.MODE_VQ4, vo.MODE_VQ3, vo.MODE_VQ125):
        E, dsub = vo.GEOMETRY[mode]
        for role in (vo.ROLE_K, vo.ROLE_V):
            L = 150
            codes = r.integers(0, E, size=(L, 128 // dsub))
            buf = vo.pack_stream(codes, mode, role, cap_len=200)
            assert buf.size == vo.code_bytes(mode, 200)
            assert np.array_equal(vo.unpack_stream(buf, mode, role, L), codes)
            assert np.array_equal(vo.pack_stream_fast(codes, mode, role, 200), buf)
            assert np.array_equal(vo.unpack_stream_fast(buf, mode, role, L), codes)
    # every 12-bit value survives both positions of a pair
    for c in range(4096):
        assert vo.unpack_pair(*vo.pack_pair(c, 4095 - c)) == (c, 4095 - c)


def test_append_does_not_touch_neighbours():
    """Writing token t changes only token t's bytes (token-local packing)."""
    for mode in (vo.MODE_VQ2, vo.MODE_VQ15, vo.MODE_VQ4, vo.MODE_VQ3, vo.MODE_VQ125):
        E, dsub = vo.GEOMETRY[mode]
        for role in (vo.ROLE_K, vo.ROLE_V):
            codes = np.zeros((64, 128 // dsub), dtype=np.int64)
            a = vo.pack_stream(codes, mode, role, 64)
            codes[37] = E - 1
            b = vo.pack_stream(codes, mode, role, 64)
            changed = np.flatnonzero(a != b)
            assert changed.size > 0
            again = vo.unpack_stream(b, mode, role, 64)
            assert np.array_equal(np.flatnonzero((again != 0).any(axis=1)), [37])


# ------------------------------------------------------------ attention

def _setup(L=33, Hq=4, Hkv=2, E=16, dsub=4, seed=0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((1, Hq, 128)).astype(np.float16)
    kcb = r.standard_normal((Hkv, E, dsub)).astype(np.float16)
    vcb = r.standard_normal((Hkv, E, dsub)).astype(np.float16)
    s = r.uniform(0.5, 4.0, size=(Hkv, 128)).astype(np.float32)
    kc = r.integers(0, E, size=(1, Hkv, L, 128 // dsub))
    vc = r.integers(0, E, size=(1, Hkv, L, 128 // dsub))
    return q, kc, vc, kcb, vcb, s, np.array([L])


def check_attention_vs_sdpa():
    """Plain attention against torch's scaled_dot_product_attention (fp64)."""
    q, kc, vc, kcb, vcb, s, lens = _setup()
    o = vo.decode_attention(q, kc, vc, kcb, vcb, s, lens)
    for h in range(4):
        kvh = h // 2
        k = vo.untransform_keys(vo.dequantize(kc[0, kvh], kcb[kvh]), s[kvh])
        v = vo.dequantize(vc[0, kvh], vcb[kvh])
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[0, h].astype(np.float64))[None, None, None],
            torch.from_numpy(k)[None, None], torch.from_numpy(v)[None, None])[0, 0, 0].numpy()
        assert np.abs(o[0, h] - ref).max() < 1e-12


def check_exact_codebook():
    """When the codebook holds every transformed key subvector exactly, VQ
    attention equals exact attention on the original keys: checks the
    inverse rotation and the smoothing direction end to end."""
    r = np.random.default_rng(4)
    L = 24
    kq = r.standard_normal((L, 128)).astype(np.float16)       # rotated-domain keys
    s = r.uniform(0.5, 3.0, size=128).astype(np.float32)
    k_orig = (kq.astype(np.float64) @ vo.normalized_hadamard().T) * s
    cb = kq.reshape(-1, 4)
    codes = np.arange(L * 32).reshape(L, 32)
    v = r.standard_normal((L, 128)).astype(np.float16)
    vcb = v.reshape(-1, 4)
    q = r.standard_normal((1, 1, 128)).astype(np.float16)
    o = vo.decode_attention(q, codes[None, None], codes[None, None], cb[None], vcb[None],
                            s[None], np.array([L]))
    z = SCALE * (k_orig @ q[0, 0].astype(np.float64))
    p = np.exp(z - z.max())
    ref = (p / p.sum()) @ v.astype(np.float64)
    assert np.abs(o[0, 0] - ref).max() < 1e-12


def check_two_token():
    kcb = np.zeros((1, 2, 4), dtype=np.float16)
    kcb[0, 1] = 1
    vcb = np.zeros((1, 2, 4), dtype=np.float16)
    vcb[0, 1] = [1, 2, 3, 4]
    codes = np.array([[0] * 32, [1] * 32])[None, None]
    s = np.ones((1, 128), dtype=np.float32)
    for line in golden_lines("two_token_decode.txt"):
        c, sig = (float(v) for v in line.split())
        q = np.zeros((1, 1, 128), dtype=np.float16)
        q[0, 0, 0] = c
        o = vo.decode_attention(q, codes, codes, kcb, vcb, s, np.array([2]))
        want = np.tile([1.0, 2.0, 3.0, 4.0], 32) * sig
        assert np.abs(o[0, 0] - want).max() < 1e-12, line


def check_closed_forms():
    q, kc, vc, kcb, vcb, s, lens = _setup(L=40)
    # (i) one cached token: O is its value row
    o = vo.decode_attention(q, kc, vc, kcb, vcb, s, np.array([1]))
    for h in range(4):
        assert np.array_equal(o[0, h], vo.dequantize(vc[0, h // 2, :1], vcb[h // 2])[0])
    # (ii) every value code equal: O is that centroid row whatever q is
    vc2 = np.full_like(vc, 3)
    o = vo.decode_attention(q, kc, vc2, kcb, vcb, s, lens)
    for h in range(4):
        assert np.abs(o[0, h] - np.tile(vcb[h // 2, 3].astype(np.float64), 32)).max() < 1e-12
    # (iii) q = 0: uniform weights, O is the mean value row
    o = vo.decode_attention(np.zeros_like(q), kc, vc, kcb, vcb, s, lens)
    for h in range(4):
        assert np.abs(o[0, h] - vo.dequantize(vc[0, h // 2], vcb[h // 2]).mean(axis=0)).max() < 1e-12
    # (vi) permuting the tokens (codes of K and V together) leaves O unchanged
    perm = np.random.default_rng(2).permutation(40)
    o1 = vo.decode_attention(q, kc, vc, kcb, vcb, s, lens)
    o2 = vo.decode_attention(q, kc[:, :, perm], vc[:, :, perm], kcb, vcb, s, lens)
    assert np.abs(o1 - o2).max() < 1e-12
    # (vii) GQA: query head h reads KV head h // g, so identical queries in a
    # group give identical rows and the two groups differ
    q2 = q.copy()
    q2[0, :] = q[0, 0]
    o = vo.decode_attention(q2, kc, vc, kcb, vcb, s, lens)
    assert np.array_equal(o[0, 0], o[0, 1]) and np.array_equal(o[0, 2], o[0, 3])
    assert not np.allclose(o[0, 1], o[0, 2])
    vconst = np.zeros_like(vcb)
    vconst[0] = 1.0
    vconst[1] = -1.0
    o = vo.decode_attention(q, kc, vc, kcb, vconst, s, lens)
    assert np.allclose(o[0, :2], 1.0) and np.allclose(o[0, 2:], -1.0)
    # empty cache: zero row
    o = vo.decode_attention(q, kc, vc, kcb, vcb, s, np.array([0]))
    assert np.array_equal(o, np.zeros_like(o))


def check_rotated_path():
    q, kc, vc, kcb, vcb, s, lens = _setup(L=57, seed=8)
    a = vo.decode_attention(q, kc, vc, kcb, vcb, s, lens)
    b = vo.decode_attention_rotated(q, kc, vc, kcb, vcb, s, lens)
    assert np.abs(a - b).max() < 1e-9


def test_attention_vs_sdpa():
    check_attention_vs_sdpa()


def test_exact_codebook():
    check_exact_codebook()


def test_two_token():
    check_two_token()


def test_closed_forms():
    check_closed_forms()


def test_rotated_path():
    check_rotated_path()


def test_o_error_metric():
    ref = np.array([[1.0, -2.0, 0.5], [0.0, 0.0, 0.0]])
    got = np.array([[1.0, -2.002, 0.5], [0.0, 1e-3, 0.0]])
    e = vo.o_error(got, ref)
    assert abs(e[0] - 0.001) < 1e-12 and abs(e[1] - 1e-3) < 1e-12


# ------------------------------------------ planted mistakes (mutation tests)

def _fails(check):
    try:
        check()
    except AssertionError:
        return True
    return False


def test_planted_unnormalised_rotation(monkeypatch):
    monkeypatch.setattr(vo, "normalized_hadamard", lambda: vo.sylvester_hadamard(128))
    assert _fails(check_score_invariance) and _fails(check_sign_patterns)


def test_planted_smoothing_direction(monkeypatch):
    hn = vo.normalized_hadamard()
    monkeypatch.setattr(vo, "transform_keys",
                        lambda x, s: ((x.astype(np.float64) * s) @ hn).astype(np.float32))
    assert _fails(check_score_invariance) and _fails(check_sign_patterns)


def test_planted_inverse_without_smoothing(monkeypatch):
    monkeypatch.setattr(vo, "untransform_keys",
                        lambda xq, s: xq.astype(np.float64) @ vo.normalized_hadamard().T)
    assert _fails(check_exact_codebook)


def test_planted_gqa_map(monkeypatch):
    real = vo.decode_attention

    def wrong(q, kc, vc, kcb, vcb, s, lens, scale=None, heads=None):
        # query head h reading KV head h % Hkv instead of h // g
        Hq, Hkv = q.shape[1], kcb.shape[0]
        hp = [h % Hkv * (Hq // Hkv) + h // Hkv for h in range(Hq)]
        qp = np.empty_like(q)
        qp[:, hp] = q
        return real(qp, kc, vc, kcb, vcb, s, lens, scale)[:, hp]
    monkeypatch.setattr(vo, "decode_attention", wrong)
    assert _fails(check_closed_forms)


def test_planted_scale(monkeypatch):
    real = vo.attention
    monkeypatch.setattr(vo, "attention", lambda q, k, v, scale: real(q, k, v, 1.0))
    assert _fails(check_two_token) and _fails(check_attention_vs_sdpa)


def test_planted_tie_break(monkeypatch):
    real = vo.nearest_centroid

    def last_index(sub, cb):
        codes, d = real(sub, cb)
        rev = d.shape[1] - 1 - np.argmin(d[:, ::-1], axis=1)
        return rev, d
    monkeypatch.setattr(vo, "nearest_centroid", last_index)
    assert _fails(check_nearest_golden)


def test_planted_layout(monkeypatch):
    real = vo.vq2_offset
    monkeypatch.setattr(vo, "vq2_offset",
                        lambda role, t, j: real(1 - role, t, j))
    assert _fails(check_layout_golden)


def test_planted_vq4_half_order(monkeypatch):
    """Swapping the two subvectors a K lane's byte pair holds must fail a pin."""
    real = vo.vq4_offset
    monkeypatch.setattr(vo, "vq4_offset",
                        lambda role, t, j: real(role, t, j ^ 4) if role == vo.ROLE_K else real(role, t, j))
    assert _fails(check_layout_golden)


def test_planted_vq3_plane_split(monkeypatch):
    """Storing a run in one 24-byte block instead of two planes must fail a pin."""
    def flat(role, t, pair, k):
        tile, r = divmod(t, 16)
        if role == vo.ROLE_K:
            lane, b = 4 * (r % 8) + pair % 4, 12 * (r // 8) + 3 * (pair // 4) + k
        else:
            lane, b = 4 * (pair % 8) + (r % 8) // 2, 6 * (2 * (r // 8) + r % 2) + 3 * (pair // 8) + k
        return 768 * tile + 24 * lane + b
    monkeypatch.setattr(vo, "vq3_byte", flat)
    assert _fails(check_layout_golden)


def test_planted_vq125_single_plane(monkeypatch):
    """Storing each K run as one 10-byte block instead of two planes must fail a pin."""
    real = vo.vq125_bit

    def flat(role, t, j, b):
        if role != vo.ROLE_K:
            return real(role, t, j, b)
        tile, r = divmod(t, 16)
        return 8 * (320 * tile + 10 * (4 * (r % 8) + j % 4)) + 40 * (r // 8) + 10 * (j // 4) + b
    monkeypatch.setattr(vo, "vq125_bit", flat)
    assert _fails(check_layout_golden)


def test_planted_vq125_slot_order(monkeypatch):
    """Giving V slots 1 and 2 (tokens 2i+1 and 2i+8) each other's bits must fail a pin."""
    real = vo.vq125_bit

    def swapped(role, t, j, b):
        if role == vo.ROLE_V and t % 16 in (1, 8, 3, 10, 5, 12, 7, 14):
            t = t + 7 if t % 2 else t - 7
        return real(role, t, j, b)
    monkeypatch.setattr(vo, "vq125_bit", swapped)
    assert _fails(check_layout_golden)


def test_vq125_token_bits_fill_whole_bytes():
    """Each token's bits of a run occupy 5 whole bytes that hold no other token's bits."""
    for role in (0, 1):
        owner = {}
        for t in range(16):
            for j in range(16):
                for b in range(10):
                    owner.setdefault(vo.vq125_bit(role, t, j, b) // 8, set()).add(t)
        assert all(len(v) == 1 for v in owner.values())
        per_token = np.bincount([next(iter(v)) for v in owner.values()], minlength=16)
        assert (per_token == 20).all()


def test_planted_pair_order(monkeypatch):
    monkeypatch.setattr(vo, "pack_pair",
                        lambda lo, hi: (hi & 0xFF, (hi >> 8) | ((lo & 0xF) << 4), lo >> 4))
    assert _fails(check_layout_golden)


def test_oracle_is_importable_as_package():
    assert oracle.code_bytes(0, 16) == 512


# ---------------------------------------------------------------- multi-query decode

def check_multi_query_vs_sdpa_causal():
    """M queries per sequence against torch SDPA over the dequantised cache
    with an explicit boolean mask: query m sees tokens t <= L - M + m."""
    q1, kc, vc, kcb, vcb, s, lens = _setup()
    L, M = int(lens[0]), 3
    q = np.random.default_rng(11).standard_normal((1, M, q1.shape[1], 128)).astype(np.float16)
    o = vo.decode_attention_multi(q, kc, vc, kcb, vcb, s, lens)
    mask = np.zeros((M, L), dtype=bool)
    for m in range(M):
        mask[m, :L - M + m + 1] = True
    for h in range(q.shape[2]):
        kvh = h // (q.shape[2] // kcb.shape[0])
        k = vo.untransform_keys(vo.dequantize(kc[0, kvh], kcb[kvh]), s[kvh])
        v = vo.dequantize(vc[0, kvh], vcb[kvh])
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[0, :, h].astype(np.float64))[None, None], torch.from_numpy(k)[None, None],
            torch.from_numpy(v)[None, None], attn_mask=torch.from_numpy(mask)[None, None])[0, 0].numpy()
        assert np.abs(o[0, :, h] - ref).max() < 1e-12


def check_multi_query_closed_forms():
    """L = M: query 0 sees only token 0 (O = its value row); with q = 0 every
    query averages the value rows it sees."""
    r = np.random.default_rng(12)
    Hkv, M = 1, 4
    kcb = r.standard_normal((Hkv, 256, 4)).astype(np.float16)
    vcb = r.standard_normal((Hkv, 256, 4)).astype(np.float16)
    s = r.uniform(0.5, 2.0, size=(Hkv, 128)).astype(np.float32)
    kc = r.integers(0, 256, size=(1, Hkv, M, 32))
    vc = r.integers(0, 256, size=(1, Hkv, M, 32))
    q = r.standard_normal((1, M, 2, 128)).astype(np.float16)
    o = vo.decode_attention_multi(q, kc, vc, kcb, vcb, s, [M])
    v_rows = vcb[0][vc[0, 0]].reshape(M, 128).astype(np.float64)
    assert np.array_equal(o[0, 0, 0], v_rows[0]) and np.array_equal(o[0, 0, 1], v_rows[0])
    o0 = vo.decode_attention_multi(np.zeros_like(q), kc, vc, kcb, vcb, s, [M])
    for m in range(M):
        assert np.allclose(o0[0, m, 0], v_rows[:m + 1].mean(axis=0), rtol=0, atol=1e-12)
    # a sequence shorter than its query count: the early queries see nothing
    o1 = vo.decode_attention_multi(q[:, :, :1], kc, vc, kcb, vcb, s, [2])
    assert np.all(o1[0, :2] == 0) and np.array_equal(o1[0, 2, 0], v_rows[0])


def test_multi_query_vs_sdpa_causal():
    check_multi_query_vs_sdpa_causal()


def test_multi_query_closed_forms():
    check_multi_query_closed_forms()


def test_planted_multi_query_off_by_one(monkeypatch):
    real = vo.decode_attention

    def shifted(q, kc, vc, kcb, vcb, s, lens, scale=None, heads=None):
        # each query also sees the token after its own position
        return real(q, kc, vc, kcb, vcb, s, [L + 1 if L < kc[0][0].shape[0] else L for L in lens], scale)
    monkeypatch.setattr(vo, "decode_attention", shifted)
    assert _fails(check_multi_query_vs_sdpa_causal) and _fails(check_multi_query_closed_forms)
