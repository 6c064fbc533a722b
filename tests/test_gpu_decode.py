"""Decode parity: the CUDA path (through the C ABI) against the CPU oracle."""
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


def random_case(mode, B, Hq, Hkv, lens, cap_len, seed):
    r = np.random.default_rng(seed)
    E, dsub = vo.GEOMETRY[mode]
    s, kcb, vcb = H.random_codebooks(mode, Hkv, seed + 1)
    q = r.standard_normal((B, Hq, 128)).astype(np.float16)
    kc = [[r.integers(0, E, size=(cap_len, 128 // dsub)) for _ in range(Hkv)] for _ in range(B)]
    vc = [[r.integers(0, E, size=(cap_len, 128 // dsub)) for _ in range(Hkv)] for _ in range(B)]
    return q, kc, vc, kcb, vcb, s


def oracle_o(q, kc, vc, kcb, vcb, s, lens, heads=None, scale=None):
    return vo.decode_attention(q, kc, vc, kcb, vcb, s, np.asarray(lens), scale=scale, heads=heads)


CASES = [
    # mode, B, Hq, Hkv, lens, cap
    (0, 3, 8, 2, [1, 17, 300], 320),
    (0, 2, 5, 1, [64, 33], 64),
    (0, 1, 8, 1, [257], 260),
    (0, 2, 2, 2, [16, 15], 16),
    (0, 2, 32, 8, [1000, 777], 1024),
    (1, 2, 10, 2, [1, 200], 256),
    (1, 3, 8, 1, [64, 65, 130], 192),
    (1, 1, 4, 4, [100], 100),
    (1, 2, 40, 8, [700, 64], 704),
    (2, 3, 8, 2, [1, 17, 300], 320),
    (2, 2, 5, 1, [64, 33], 64),
    (2, 1, 32, 8, [1000], 1024),
    (2, 2, 16, 2, [16, 15], 16),
    (3, 3, 8, 2, [1, 17, 300], 320),
    (3, 2, 5, 1, [64, 33], 64),
    (3, 1, 32, 8, [1000], 1024),
    (3, 2, 16, 2, [16, 15], 16),
    (3, 1, 8, 1, [257], 260),
    (4, 3, 8, 2, [1, 17, 300], 320),
    (4, 2, 5, 1, [64, 33], 64),
    (4, 1, 32, 8, [1000], 1024),
    (4, 2, 16, 2, [16, 15], 16),
    (4, 1, 8, 1, [257], 260),
]


@pytest.mark.parametrize("case", CASES, ids=[f"m{c[0]}_b{c[1]}_hq{c[2]}_hkv{c[3]}" for c in CASES])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_matches_oracle(case, num_splits):
    mode, B, Hq, Hkv, lens, cap = case
    q, kc, vc, kcb, vcb, s = random_case(mode, B, Hq, Hkv, lens, cap, seed=B * 100 + Hq + mode)
    kbuf = H.pack_cache_role(mode, 0, kc, cap)
    vbuf = H.pack_cache_role(mode, 1, vc, cap)
    o = H.gpu_decode(mode, q, kbuf, vbuf, lens, kcb, vcb, s, cap, max(lens), num_splits=num_splits)
    ref = oracle_o(q, kc, vc, kcb, vcb, s, lens)
    err = vo.o_error(o, ref)
    assert np.isfinite(o).all()
    assert err.max() <= H.O_TOL, err.max()


def test_tiny_config_full_pipeline_codes_from_oracle():
    """Tiny 2-bit workload (batch 1, one head, 1024 tokens): inputs from the
    generator, codebooks from calibration, codes from the oracle's encoder."""
    w = synth.WORKLOADS[0]
    s, kcb, vcb = H.calibrate(w)
    k = synth.keys(w, 0, 0, 0, w.seq_len)
    v = synth.values(w, 0, 0, 0, w.seq_len)
    kc, _ = vo.encode_rows(k, vo.ROLE_K, s[0], kcb[0])
    vc, _ = vo.encode_rows(v, vo.ROLE_V, None, vcb[0])
    q = synth.queries(w)
    kbuf = H.pack_cache_role(0, 0, [[kc]], w.cap_len)
    vbuf = H.pack_cache_role(0, 1, [[vc]], w.cap_len)
    o = H.gpu_decode(0, q, kbuf, vbuf, [w.seq_len], kcb, vcb, s, w.cap_len, w.seq_len)
    ref = oracle_o(q, [[kc]], [[vc]], kcb, vcb, s, [w.seq_len])
    assert vo.o_error(o, ref).max() <= H.O_TOL


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_zero_length_rows_and_empty_cache(mode):
    q, kc, vc, kcb, vcb, s = random_case(mode, 3, 4, 2, [0, 5, 0], 64, seed=7)
    kbuf, vbuf = H.pack_cache_role(mode, 0, kc, 64), H.pack_cache_role(mode, 1, vc, 64)
    o = H.gpu_decode(mode, q, kbuf, vbuf, [0, 5, 0], kcb, vcb, s, 64, 64)
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    ref = oracle_o(q, kc, vc, kcb, vcb, s, [0, 5, 0])
    assert vo.o_error(o[1], ref[1]).max() <= H.O_TOL
    # max_seq_len == 0: every row is zero
    o = H.gpu_decode(mode, q, kbuf, vbuf, [0, 0, 0], kcb, vcb, s, 64, 0)
    assert np.all(o == 0)


def test_empty_batch_is_a_no_op():
    import torch
    out = torch.zeros((0, 4, 128), dtype=torch.float16, device="cuda")
    q = torch.zeros((0, 4, 128), dtype=torch.float16, device="cuda")
    kcb = torch.zeros((1, 256, 4), dtype=torch.float16, device="cuda")
    _lib.vqkv_decode_attn(0, q, None, None, None, kcb, kcb, None, out, None, 16, 16)


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_single_token_is_its_value_row(mode):
    q, kc, vc, kcb, vcb, s = random_case(mode, 1, 4, 1, [1], 16, seed=3)
    kbuf, vbuf = H.pack_cache_role(mode, 0, kc, 16), H.pack_cache_role(mode, 1, vc, 16)
    o = H.gpu_decode(mode, q, kbuf, vbuf, [1], kcb, vcb, s, 16, 1)
    want = vo.dequantize(vc[0][0][:1], vcb[0])[0].astype(np.float16)
    for h in range(4):
        assert np.array_equal(o[0, h], want)


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_constant_value_codes(mode):
    q, kc, vc, kcb, vcb, s = random_case(mode, 1, 8, 2, [333], 400, seed=5)
    vc = [[np.full_like(vc[0][h], 11) for h in range(2)]]
    kbuf, vbuf = H.pack_cache_role(mode, 0, kc, 400), H.pack_cache_role(mode, 1, vc, 400)
    o = H.gpu_decode(mode, q, kbuf, vbuf, [333], kcb, vcb, s, 400, 333)
    for h in range(8):
        want = np.tile(vcb[h // 4, 11].astype(np.float64), 128 // vcb.shape[2])
        assert np.abs(o[0, h] - want).max() <= 1e-3 * np.abs(want).max()


def test_softmax_scale_argument():
    q, kc, vc, kcb, vcb, s = random_case(0, 1, 4, 1, [200], 200, seed=9)
    kbuf, vbuf = H.pack_cache_role(0, 0, kc, 200), H.pack_cache_role(0, 1, vc, 200)
    o = H.gpu_decode(0, q, kbuf, vbuf, [200], kcb, vcb, s, 200, 200, softmax_scale=0.3)
    ref = oracle_o(q, kc, vc, kcb, vcb, s, [200], scale=0.3)
    assert vo.o_error(o, ref).max() <= H.O_TOL


def test_seq_len_above_max_is_clamped_and_reported():
    import torch
    q, kc, vc, kcb, vcb, s = random_case(0, 2, 4, 1, [50, 64], 64, seed=2)
    kbuf, vbuf = H.pack_cache_role(0, 0, kc, 64), H.pack_cache_role(0, 1, vc, 64)
    o, ws = H.gpu_decode(0, q, kbuf, vbuf, [50, 9999], kcb, vcb, s, 64, 64, return_ws=True)
    assert int(ws[:4].view(torch.int32).item()) & _lib.VQKV_DEVERR_SEQ_LEN
    ref = oracle_o(q, kc, vc, kcb, vcb, s, [50, 64])
    assert vo.o_error(o, ref).max() <= H.O_TOL


def test_repeatable_and_workspace_reusable():
    import torch
    q, kc, vc, kcb, vcb, s = random_case(0, 2, 8, 2, [900, 517], 1024, seed=4)
    kbuf, vbuf = H.pack_cache_role(0, 0, kc, 1024), H.pack_cache_role(0, 1, vc, 1024)
    ws = _lib.decode_workspace(0, 2, 8, 2, 1024, 1024)
    a = H.gpu_decode(0, q, kbuf, vbuf, [900, 517], kcb, vcb, s, 1024, 1024, workspace=ws)
    b = H.gpu_decode(0, q, kbuf, vbuf, [900, 517], kcb, vcb, s, 1024, 1024, workspace=ws)
    assert np.array_equal(a, b)
    # the tickets (after the 256-byte header) are back to zero
    t = ws[256:256 + 4 * 4].view(torch.int32).cpu().numpy()
    assert np.all(t == 0)


def test_split_counts_agree():
    q, kc, vc, kcb, vcb, s = random_case(0, 1, 4, 1, [2000], 2048, seed=6)
    kbuf, vbuf = H.pack_cache_role(0, 0, kc, 2048), H.pack_cache_role(0, 1, vc, 2048)
    outs = [H.gpu_decode(0, q, kbuf, vbuf, [2000], kcb, vcb, s, 2048, 2048, num_splits=n).astype(np.float64)
            for n in (1, 2, 5, 16, 125)]
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 2e-3 * np.abs(outs[0]).max()


def test_token_permutation_invariance():
    q, kc, vc, kcb, vcb, s = random_case(0, 1, 4, 1, [96], 96, seed=8)
    perm = np.random.default_rng(1).permutation(96)
    kb1, vb1 = H.pack_cache_role(0, 0, kc, 96), H.pack_cache_role(0, 1, vc, 96)
    kb2 = H.pack_cache_role(0, 0, [[kc[0][0][perm]]], 96)
    vb2 = H.pack_cache_role(0, 1, [[vc[0][0][perm]]], 96)
    a = H.gpu_decode(0, q, kb1, vb1, [96], kcb, vcb, s, 96, 96).astype(np.float64)
    b = H.gpu_decode(0, q, kb2, vb2, [96], kcb, vcb, s, 96, 96).astype(np.float64)
    assert np.abs(a - b).max() <= 2e-3 * np.abs(a).max()


# ------------------------------------------------------------ full sizes

def full_size_uniform_codes(w, b_list=None):
    kc, vc = [], []
    lens = synth.seq_lens(w)
    for b in (b_list if b_list is not None else range(w.B)):
        kc.append([synth.uniform_codes(w, b, h, 0, w.cap_len) for h in range(w.Hkv)])
        vc.append([synth.uniform_codes(w, b, h, 1, w.cap_len) for h in range(w.Hkv)])
    return kc, vc, lens


def _pack_one(args):
    mode, role, codes, cap = args
    return vo.pack_stream_fast(codes, mode, role, cap)


def pack_parallel(mode, role, codes, cap):
    B, Hkv = len(codes), len(codes[0])
    with H.pool() as ex:
        bufs = list(ex.map(_pack_one, [(mode, role, codes[b][h], cap) for b in range(B) for h in range(Hkv)]))
    return np.stack(bufs).reshape(B, Hkv, -1)


@pytest.mark.slow
@pytest.mark.parametrize("mode", [2, 3, 4])
def test_full_size_other_bit_widths_sampled_heads(mode):
    """The 196k-token Llama-shaped workload at 4, 3 and 1.25 bit, launched as
    bench.py --mode launches it; the oracle recomputes a few heads."""
    w = synth.WORKLOADS[1].with_mode(mode)
    kw = {} if mode == 2 else dict(sample_tokens=2048, iters=2)
    s, kcb, vcb = H.calibrate(w, **kw)
    kc, vc, lens = full_size_uniform_codes(w)
    kbuf = pack_parallel(w.mode, 0, kc, w.cap_len)
    vbuf = pack_parallel(w.mode, 1, vc, w.cap_len)
    q = synth.queries(w)
    o = H.gpu_decode(w.mode, q, kbuf, vbuf, lens, kcb, vcb, s, w.cap_len, int(lens.max()))
    assert np.isfinite(o).all()
    r = np.random.default_rng(10 + mode)
    heads = [(0, int(r.integers(w.Hq))) for _ in range(3)] + [(0, w.Hq - 1)]
    ref = vo.decode_attention(q, kc, vc, kcb, vcb, s, lens, heads=heads)
    for b, h in heads:
        e = vo.o_error(o[b, h], ref[b, h])
        assert e <= H.O_TOL, (b, h, e)


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_full_size_sampled_heads(cfg):
    """The benchmarked workloads at full size, launched exactly as bench.py
    launches them (automatic split plan); the oracle recomputes a few heads."""
    w = synth.WORKLOADS[cfg]
    kw = {} if w.mode == 0 else dict(sample_tokens=2048, iters=2)
    s, kcb, vcb = H.calibrate(w, **kw)
    kc, vc, lens = full_size_uniform_codes(w)
    kbuf = pack_parallel(w.mode, 0, kc, w.cap_len)
    vbuf = pack_parallel(w.mode, 1, vc, w.cap_len)
    q = synth.queries(w)
    o = H.gpu_decode(w.mode, q, kbuf, vbuf, lens, kcb, vcb, s, w.cap_len, int(lens.max()))
    assert np.isfinite(o).all()
    # any O row is a convex combination of value rows: bounded by the codebook range
    lo = vcb.astype(np.float32).min(axis=(1, 2))
    hi = vcb.astype(np.float32).max(axis=(1, 2))
    for h in range(w.Hq):
        kvh = h // w.g
        assert (o[:, h] >= lo[kvh] - 1e-2).all() and (o[:, h] <= hi[kvh] + 1e-2).all()
    r = np.random.default_rng(cfg)
    heads = [(int(r.integers(w.B)), int(r.integers(w.Hq))) for _ in range(3)]
    heads.append((w.B - 1, w.Hq - 1))
    ref = vo.decode_attention(q, kc, vc, kcb, vcb, s, lens, heads=heads)
    for b, h in heads:
        e = vo.o_error(o[b, h], ref[b, h])
        assert e <= H.O_TOL, (b, h, e)


# ------------------------------------------------------------ flat plan (batches)

@pytest.mark.parametrize("mode", [0, 2, 3, 4])
def test_flat_plan_ragged_batch(mode):
    """Batches use the flat plan: every CTA of a KV head takes an equal share
    of all sequences' tiles, so a share can start and end inside sequences
    and cover several short ones.  Lengths include 0, 1, a tile edge and the
    capacity."""
    r = np.random.default_rng(40 + mode)
    B, Hq, Hkv, cap = 37, 8, 2, 320
    lens = r.integers(0, cap + 1, size=B)
    lens[:5] = [0, 1, 16, cap, 0]
    q, kc, vc, kcb, vcb, s = random_case(mode, B, Hq, Hkv, lens, cap, seed=400 + mode)
    kbuf, vbuf = H.pack_cache_role(mode, 0, kc, cap), H.pack_cache_role(mode, 1, vc, cap)
    o = H.gpu_decode(mode, q, kbuf, vbuf, lens, kcb, vcb, s, cap, cap)
    ref = oracle_o(q, kc, vc, kcb, vcb, s, lens)
    assert np.isfinite(o).all()
    assert np.all(o[lens == 0] == 0)
    assert vo.o_error(o, ref).max() <= H.O_TOL
    # the split plan (explicit split count) gives the same O up to fp32 regrouping
    o2 = H.gpu_decode(mode, q, kbuf, vbuf, lens, kcb, vcb, s, cap, cap, num_splits=3)
    assert vo.o_error(o2, ref).max() <= H.O_TOL


@pytest.mark.parametrize("mode", [0, 4])
def test_flat_plan_shares_with_merges(mode):
    """More sequences than CTAs per KV head (37 > 152 / 8): the flat plan
    cuts the tiles into equal shares, pieces of a sequence are merged."""
    r = np.random.default_rng(50 + mode)
    B, Hq, Hkv, cap = 37, 8, 8, 320
    lens = r.integers(0, cap + 1, size=B)
    lens[:4] = [0, 1, cap, 17]
    q, kc, vc, kcb, vcb, s = random_case(mode, B, Hq, Hkv, lens, cap, seed=500 + mode)
    kbuf, vbuf = H.pack_cache_role(mode, 0, kc, cap), H.pack_cache_role(mode, 1, vc, cap)
    o = H.gpu_decode(mode, q, kbuf, vbuf, lens, kcb, vcb, s, cap, cap)
    ref = oracle_o(q, kc, vc, kcb, vcb, s, lens)
    assert np.all(o[lens == 0] == 0)
    assert vo.o_error(o, ref).max() <= H.O_TOL


def test_flat_plan_one_long_sequence_among_short_ones():
    """One long sequence and three short ones: the long sequence is cut into
    pieces over many CTAs and merged, the short ones share a CTA."""
    lens = [3000, 10, 10, 10]
    q, kc, vc, kcb, vcb, s = random_case(0, 4, 4, 2, lens, 3008, seed=51)
    kbuf, vbuf = H.pack_cache_role(0, 0, kc, 3008), H.pack_cache_role(0, 1, vc, 3008)
    o = H.gpu_decode(0, q, kbuf, vbuf, lens, kcb, vcb, s, 3008, 3008)
    assert vo.o_error(o, oracle_o(q, kc, vc, kcb, vcb, s, lens)).max() <= H.O_TOL


@pytest.mark.parametrize("mode", [0, 2])
def test_flat_plan_even_lengths_with_an_empty_sequence(mode):
    """Sixteen sequences of (nearly) one length on 19 CTAs per KV head: the
    shares cross sequence boundaries at different tiles in every CTA; an
    empty sequence gives a zero row."""
    lens = [1600] * 16
    lens[5] = 0
    lens[9] = 1599
    q, kc, vc, kcb, vcb, s = random_case(mode, 16, 8, 8, lens, 1600, seed=52 + mode)
    kbuf, vbuf = H.pack_cache_role(mode, 0, kc, 1600), H.pack_cache_role(mode, 1, vc, 1600)
    o = H.gpu_decode(mode, q, kbuf, vbuf, lens, kcb, vcb, s, 1600, 1600)
    assert np.all(o[5] == 0)
    assert vo.o_error(o, oracle_o(q, kc, vc, kcb, vcb, s, lens)).max() <= H.O_TOL
    # one CTA per sequence (an explicit split count of 1) agrees
    o1 = H.gpu_decode(mode, q, kbuf, vbuf, lens, kcb, vcb, s, 1600, 1600, num_splits=1)
    assert vo.o_error(o1, oracle_o(q, kc, vc, kcb, vcb, s, lens)).max() <= H.O_TOL


def test_flat_plan_fewer_tiles_than_ctas():
    """Three one-token sequences: fewer super-tiles than CTAs per KV head."""
    q, kc, vc, kcb, vcb, s = random_case(0, 3, 4, 1, [1, 2, 1], 16, seed=41)
    kbuf, vbuf = H.pack_cache_role(0, 0, kc, 16), H.pack_cache_role(0, 1, vc, 16)
    o = H.gpu_decode(0, q, kbuf, vbuf, [1, 2, 1], kcb, vcb, s, 16, 16)
    ref = oracle_o(q, kc, vc, kcb, vcb, s, [1, 2, 1])
    assert vo.o_error(o, ref).max() <= H.O_TOL


def test_flat_plan_workspace_is_reusable():
    """Tickets of every sequence are back to zero after a flat-plan call."""
    import torch
    lens = [500, 0, 33, 1000, 7]
    q, kc, vc, kcb, vcb, s = random_case(0, 5, 8, 2, lens, 1024, seed=42)
    kbuf, vbuf = H.pack_cache_role(0, 0, kc, 1024), H.pack_cache_role(0, 1, vc, 1024)
    ws = _lib.decode_workspace(0, 5, 8, 2, 1024, 1024)
    a = H.gpu_decode(0, q, kbuf, vbuf, lens, kcb, vcb, s, 1024, 1024, workspace=ws)
    b = H.gpu_decode(0, q, kbuf, vbuf, lens, kcb, vcb, s, 1024, 1024, workspace=ws)
    assert np.array_equal(a, b)
    t = ws[256:256 + 4 * 5 * 2].view(torch.int32).cpu().numpy()
    assert np.all(t == 0)
    assert vo.o_error(a, oracle_o(q, kc, vc, kcb, vcb, s, lens)).max() <= H.O_TOL


def test_batch_beyond_flat_limit_uses_the_split_plan():
    """More sequences than the flat plan takes (1024): the split plan."""
    B = 1100
    r = np.random.default_rng(43)
    lens = r.integers(0, 33, size=B)
    q, kc, vc, kcb, vcb, s = random_case(0, B, 4, 1, lens, 32, seed=43)
    kbuf, vbuf = H.pack_cache_role(0, 0, kc, 32), H.pack_cache_role(0, 1, vc, 32)
    o = H.gpu_decode(0, q, kbuf, vbuf, lens, kcb, vcb, s, 32, 32)
    heads = [(int(b), h) for b in r.integers(B, size=20) for h in range(4)]
    ref = vo.decode_attention(q, kc, vc, kcb, vcb, s, lens, heads=heads)
    for b, h in heads:
        assert vo.o_error(o[b, h], ref[b, h]) <= H.O_TOL
