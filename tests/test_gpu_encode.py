"""Encode parity: codes from the CUDA path (through the C ABI) against the
oracle's nearest-centroid codes — bit-exact, except near-ties (oracle fp32
distances within 1e-6 relative), which are counted."""
import numpy as np
import pytest

from oracle import vqkv_oracle as vo
from tests import helpers as H
from vector_quantized_bit_gb300 import _build, _lib, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def unpack_all(mode, role, buf, L):
    B, Hkv = buf.shape[:2]
    return [[vo.unpack_stream_fast(buf[b, h], mode, role, L) for h in range(Hkv)] for b in range(B)]


def compare(name, mode, role, x, s, cb, gpu_buf, pos, n_rows, device_count=None, bounded=True):
    """Oracle-encode every row and compare with the GPU stream bytes: no
    failing mismatch, near-ties recorded and bounded.  Returns the number of
    near-tie mismatches."""
    B, Hkv = x.shape[:2]
    got_all, ref_all, d_all = [], [], []
    for b in range(B):
        for h in range(Hkv):
            ref, d32 = vo.encode_rows(x[b, h], role, s[h] if s is not None else None, cb[h])
            got = vo.unpack_stream_fast(gpu_buf[b, h], mode, role, pos[b] + n_rows)[pos[b]:pos[b] + n_rows]
            got_all.append(got.reshape(-1))
            ref_all.append(ref.reshape(-1))
            d_all.append(d32.reshape(ref.size, -1))
    return H.check_and_record_codes(name, np.concatenate(got_all), np.concatenate(ref_all), np.concatenate(d_all),
                                    device_count, bounded)


def test_tiny_config_keys_and_values():
    w = synth.WORKLOADS[0]
    s, kcb, vcb = H.calibrate(w)
    k = synth.keys(w, 0, 0, 0, w.seq_len)[None, None]
    v = synth.values(w, 0, 0, 0, w.seq_len)[None, None]
    for role, x, cb in ((vo.ROLE_K, k, kcb), (vo.ROLE_V, v, vcb)):
        buf, nties, err = H.gpu_encode(0, role, x, [0], s if role == 0 else None, cb, w.cap_len, with_ties=True)
        assert err == 0
        compare(f"tiny config, role {role}", 0, role, x, s if role == 0 else None, cb, buf, [0], w.seq_len, nties)


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("role", [0, 1])
@pytest.mark.parametrize("n", [37, 3])   # 3 rows: the few-rows launch (candidates split over warps)
def test_ragged_positions_multi_head(mode, role, n):
    w = synth.WORKLOADS[3 if mode == 1 else 1].with_mode(mode).scaled(seq_len=2048, cap_len=2048)
    kw = dict(sample_tokens=512, iters=3) if w.entries == 4096 else dict(sample_tokens=512, iters=5)
    s, kcb, vcb = H.calibrate(w.scaled(Hkv=2), **kw)
    cb = kcb if role == 0 else vcb
    x = np.stack([np.stack([(synth.keys if role == 0 else synth.values)(w, b, h, 100, n) for h in range(2)])
                  for b in range(3)])
    pos = [0, 5, 130]
    cap = 200
    prefill = np.random.default_rng(0).integers(0, 256, size=(3, 2, vo.code_bytes(mode, cap)), dtype=np.uint8)
    buf, nties, _ = H.gpu_encode(mode, role, x, pos, s if role == 0 else None, cb, cap, codes=prefill,
                                 with_ties=True)
    compare(f"ragged positions, mode {mode}, role {role}, {n} rows", mode, role, x, s if role == 0 else None, cb,
            buf, pos, n, nties)
    # bytes of tokens outside [pos, pos+n) are untouched
    for b in range(3):
        for h in range(2):
            L = vo.TILE_TOKENS[mode] * (-(-cap // vo.TILE_TOKENS[mode]))
            off = vo.offset_table(mode, role, L)
            if mode == vo.MODE_VQ125:   # bit addresses -> bytes
                off = off >> 3
            if mode != vo.MODE_VQ15:   # every code byte (VQ3: every pair byte) is listed
                touched = off[pos[b]:pos[b] + n].reshape(-1)
            else:
                touched = (off[pos[b]:pos[b] + n, :, None] + np.arange(3)).reshape(-1)
            mask = np.ones(buf.shape[2], dtype=bool)
            mask[touched] = False
            assert np.array_equal(buf[b, h][mask], prefill[b, h][mask])


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_positions_out_of_range_are_skipped_and_reported(mode):
    s, kcb, vcb = H.random_codebooks(mode, 1, 3)
    x = np.random.default_rng(1).standard_normal((2, 1, 4, 128)).astype(np.float16)
    cap = 64
    prefill = np.full((2, 1, vo.code_bytes(mode, cap)), 0xA5, dtype=np.uint8)
    buf, _, err = H.gpu_encode(mode, 0, x, [62, -3], s, kcb, cap, codes=prefill, with_ties=True)
    assert err & _lib.VQKV_DEVERR_POSITION
    # sequence 0: rows at 62, 63 written; 64, 65 skipped.  sequence 1: rows at -3..-1 skipped, 0 written
    got0 = vo.unpack_stream_fast(buf[0, 0], mode, 0, 64)
    ref0, d0 = vo.encode_rows(x[0, 0], 0, s[0], kcb[0])
    H.check_and_record_codes(f"out-of-range positions, mode {mode}", got0[62:64], ref0[:2], d0[:2])
    changed = np.flatnonzero(buf[1, 0] != 0xA5)
    off = vo.offset_table(mode, 0, 1)
    if mode == vo.MODE_VQ125:   # bit addresses -> bytes
        off = off >> 3
    allowed = off.reshape(-1) if mode != vo.MODE_VQ15 else (off[..., None] + np.arange(3)).reshape(-1)
    assert set(changed.tolist()) <= set(allowed.tolist())


@pytest.mark.parametrize("mode", [0, 2, 3, 4])
def test_encode_then_decode_matches_oracle_pipeline(mode):
    """GPU encode + GPU decode against oracle encode + oracle decode."""
    w = synth.WORKLOADS[1].with_mode(mode).scaled(seq_len=3000, cap_len=3008)
    wh = w.scaled(Hkv=2, Hq=8)
    s, kcb, vcb = H.calibrate(wh, sample_tokens=1024, iters=5)
    k = np.stack([synth.keys(w, 0, h, 0, w.seq_len) for h in range(2)])[None]
    v = np.stack([synth.values(w, 0, h, 0, w.seq_len) for h in range(2)])[None]
    kbuf = H.gpu_encode(mode, 0, k, [0], s, kcb, w.cap_len)
    vbuf = H.gpu_encode(mode, 1, v, [0], None, vcb, w.cap_len)
    q = synth.queries(wh)
    o = H.gpu_decode(mode, q, kbuf, vbuf, [w.seq_len], kcb, vcb, s, w.cap_len, w.seq_len)
    kc = [[vo.encode_rows(k[0, h], 0, s[h], kcb[h])[0] for h in range(2)]]
    vc = [[vo.encode_rows(v[0, h], 1, None, vcb[h])[0] for h in range(2)]]
    ref = vo.decode_attention(q, kc, vc, kcb, vcb, s, [w.seq_len])
    assert vo.o_error(o, ref).max() <= H.O_TOL


def test_near_tie_counter_counts_exact_ties():
    """Two identical centroids make every subvector nearest to them a tie."""
    s, kcb, vcb = H.random_codebooks(0, 1, 5)
    vcb[0, 7] = vcb[0, 3]
    x = np.tile(vcb[0, 3].astype(np.float16), 32)[None, None, None]   # one V row of centroid 3
    buf, nties, err = H.gpu_encode(0, 1, x, [0], None, vcb, 16, with_ties=True)
    assert nties == 32 and err == 0
    assert np.all(vo.unpack_stream_fast(buf[0, 0], 0, 1, 1) == 3)


@pytest.mark.slow
@pytest.mark.parametrize("mode", [0, 1, 3, 4])
def test_full_size_prefill_and_append_sampled(mode):
    """Mistral-7B-shaped encode at full size (16 sequences x 8 KV heads x
    16,384 prefill rows, then 256 appended rows at positions 16,384..16,639),
    launched as one call each (the prefill on the tensor-memory kernel, at
    1.5, 2, 3 and 1.25 bit); the oracle re-encodes sampled rows."""
    w = synth.WORKLOADS[4].with_mode(mode)
    kw = dict(sample_tokens=2048, iters=2) if w.entries >= 1024 else dict(sample_tokens=2048, iters=10)
    s, kcb, vcb = H.calibrate(w, **kw)
    import torch
    sb = vo.code_bytes(mode, w.cap_len)
    kcodes = torch.zeros((w.B, w.Hkv, sb), dtype=torch.uint8, device="cuda")
    r = np.random.default_rng(mode)
    samples = [(int(r.integers(w.B)), int(r.integers(w.Hkv)), int(r.integers(w.prefill))) for _ in range(48)]
    samples += [(w.B - 1, w.Hkv - 1, w.prefill - 1)]
    # generate the prefill one sequence at a time (host memory), encode in one call per sequence batch
    x = np.empty((w.B, w.Hkv, w.prefill, 128), dtype=np.float16)
    with H.pool() as ex:
        futs = {(b, h): ex.submit(synth.keys, w, b, h, 0, w.prefill) for b in range(w.B) for h in range(w.Hkv)}
        for (b, h), f in futs.items():
            x[b, h] = f.result()
    ties = H.torch().zeros(1, dtype=torch.int64, device="cuda")
    _lib.vqkv_encode(mode, 0, H.dev(x), H.dev(np.zeros(w.B, np.int32)), H.dev(s), H.dev(kcb), kcodes, w.cap_len,
                     near_tie_count=ties)
    app = np.stack([np.stack([synth.appended_keys(w, b, h, w.append) for h in range(w.Hkv)]) for b in range(w.B)])
    _lib.vqkv_encode(mode, 0, H.dev(app), H.dev(np.full(w.B, w.prefill, np.int32)), H.dev(s), H.dev(kcb), kcodes,
                     w.cap_len, near_tie_count=ties)
    torch.cuda.synchronize()
    buf = kcodes.cpu().numpy()
    got_all, ref_all, d_all = [], [], []
    for b, h, t in samples:
        for row, tt in ((x[b, h, t:t + 1], t), (app[b, h, t % w.append:t % w.append + 1], w.prefill + t % w.append)):
            ref, d32 = vo.encode_rows(row, 0, s[h], kcb[h])
            got_all.append(vo.unpack_stream_fast(buf[b, h], mode, 0, tt + 1)[tt:tt + 1].reshape(-1))
            ref_all.append(ref.reshape(-1))
            d_all.append(d32.reshape(ref.size, -1))
    # the GPU's own counter covers every row encoded (16 x 8 x 16,640 rows x subvectors)
    n_all = w.B * w.Hkv * (w.prefill + w.append) * (128 // vo.GEOMETRY[mode][1])
    from tests import tie_log
    ntie = int(ties.item())
    H.check_and_record_codes(f"full-size Mistral-shaped key encode, mode {mode} (sampled rows; GPU counter over "
                             f"all {n_all} codes)", np.concatenate(got_all), np.concatenate(ref_all),
                             np.concatenate(d_all))
    tie_log.record(f"full-size Mistral-shaped key encode, mode {mode}: GPU near-tie counter", n_all, 0, 0, ntie)
    assert ntie <= tie_log.bound(n_all)


def _vq15_rows(seed, B, Hkv, n, scale=1.0):
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, Hkv, n, 128)) * scale).astype(np.float16)


@pytest.mark.parametrize("role", [0, 1])
def test_vq15_many_rows_across_tiles_and_sequences(role):
    """The many-rows 1.5-bit path (tensor-core screen in tiles of 8 rows):
    300 rows per sequence, so tiles straddle sequences, ragged positions and
    a partial last tile; every code against the oracle."""
    w = synth.WORKLOADS[3].scaled(seq_len=2048, cap_len=2048, Hkv=2)
    s, kcb, vcb = H.calibrate(w, sample_tokens=1024, iters=3)
    cb = kcb if role == 0 else vcb
    x = np.stack([np.stack([(synth.keys if role == 0 else synth.values)(w, b, h, 7, 300) for h in range(2)])
                  for b in range(3)])
    pos = [0, 19, 1700]
    cap = 2048
    buf, nties, err = H.gpu_encode(1, role, x, pos, s if role == 0 else None, cb, cap, with_ties=True)
    assert err == 0
    compare(f"1.5-bit many rows, role {role}", 1, role, x, s if role == 0 else None, cb, buf, pos, 300, nties)


def test_vq15_many_rows_duplicate_centroids_and_exact_matches():
    """Value rows made of centroids that appear two or three times in the
    codebook (in different groups of 32 centroids): the nearest distance is
    0 and tied, the lowest index must win, and the GPU counts the ties."""
    s, kcb, vcb = H.random_codebooks(1, 1, 9)
    vcb[0, 3000] = vcb[0, 100]
    vcb[0, 2000] = vcb[0, 3] = vcb[0, 4001]
    r = np.random.default_rng(4)
    picks = np.array([100, 3, 3000, 2000, 4001, 17, 3, 100])
    rows = []
    for i in range(40):
        c = picks[r.integers(len(picks), size=16)]
        rows.append(vcb[0][c].reshape(128))
    x = np.stack(rows)[None, None].astype(np.float16)
    buf, nties, err = H.gpu_encode(1, 1, x, [0], None, vcb, 64, with_ties=True)
    assert err == 0
    got = vo.unpack_stream_fast(buf[0, 0], 1, 1, 40)
    ref, d32 = vo.encode_rows(x[0, 0], 1, None, vcb[0])
    assert np.array_equal(got, ref)   # exact matches: no rounding can move them
    assert set(np.unique(got).tolist()) <= {3, 17, 100}
    assert nties == int(np.isin(ref, [3, 100]).sum())
    H.check_and_record_codes("1.5-bit many rows, duplicated centroids", got, ref, d32, nties, bounded=False)


def test_vq15_many_rows_values_beyond_fp16_screening():
    """Keys whose smoothed, rotated values exceed the fp16 range of the
    tensor-core screen (tiny smoothing factors): those subvectors fall back
    to the exhaustive exact search and still match the oracle."""
    s, kcb, vcb = H.random_codebooks(1, 2, 12)
    s[:, :16] = 1e-5
    x = _vq15_rows(5, 2, 2, 30, scale=3.0)
    kcb = (kcb.astype(np.float32) * 50).astype(np.float16)
    buf, nties, err = H.gpu_encode(1, 0, x, [0, 30], s, kcb, 64, with_ties=True)
    assert err == 0
    # distances near 1e11: fp32 rounding alone puts some candidates within
    # 1e-6 relative of each other, so the GPU's near-tie count is not bounded
    compare("1.5-bit many rows, values beyond fp16", 1, 0, x, s, kcb, buf, [0, 30], 30, nties, bounded=False)


@pytest.mark.parametrize("n_rows", [2, 100])
def test_vq15_codebook_beyond_the_screening_tables(n_rows):
    """Centroids of norm up to about 1000: |c|^2 no longer fits the fp16
    screening tables, so the KV head is searched exhaustively from the
    codebook in global memory (few rows: the one-row kernel; many rows: the
    tensor-memory kernel).  Codes still match the oracle."""
    r = np.random.default_rng(13)
    vcb = (r.standard_normal((1, 4096, 8)) * 300.0).astype(np.float16)
    x = (r.standard_normal((2, 1, n_rows, 128)) * 300.0).astype(np.float16)
    buf, nties, err = H.gpu_encode(1, 1, x, [0, 100], None, vcb, 256, with_ties=True)
    assert err == 0
    compare(f"1.5-bit codebook beyond the screen, {n_rows} rows", 1, 1, x, None, vcb, buf, [0, 100], n_rows, nties,
            bounded=False)
