"""Fused decode step (vqkv_decode_append), through the C ABI.

The call encodes each sequence's new K and V row at position seq_lens[b] - 1
and attends over the updated cache.  Checked against the oracle: the new
codes bit-exact except counted near-ties, every other cache byte untouched,
O within the decode tolerance of the oracle's attention over the updated
cache; and against the unfused sequence vqkv_encode (K) + vqkv_encode (V) +
vqkv_decode_attn, which must give the same cache bytes and the same O."""
import numpy as np
import pytest

from oracle import vqkv_oracle as vo
from tests import helpers as H
from vector_quantized_bit_gb300 import _build, _lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _inputs(B, Hq, Hkv, cap, seed, mode=0):
    r = np.random.default_rng(seed)
    s, kcb, vcb = H.random_codebooks(mode, Hkv, seed + 1)
    sb = vo.code_bytes(mode, cap)
    kbuf = r.integers(0, 256, size=(B, Hkv, sb), dtype=np.uint8)
    vbuf = r.integers(0, 256, size=(B, Hkv, sb), dtype=np.uint8)
    k_new = (r.standard_normal((B, Hkv, 128)) * r.uniform(0.5, 3.0, size=(1, 1, 128))).astype(np.float16)
    v_new = r.standard_normal((B, Hkv, 128)).astype(np.float16)
    q = r.standard_normal((B, Hq, 128)).astype(np.float16)
    return s, kcb, vcb, kbuf, vbuf, k_new, v_new, q


def _fused(q, kbuf, vbuf, lens, kcb, vcb, s, cap, k_new, v_new, num_splits, mode=0):
    t = H.torch()
    B, Hq, _ = q.shape
    Hkv = kcb.shape[0]
    dk, dv = H.dev(kbuf), H.dev(vbuf)
    out = t.full((B, Hq, 128), float("nan"), dtype=t.float16, device="cuda")
    ties = t.zeros(1, dtype=t.int64, device="cuda")
    ws = _lib.decode_workspace(mode, B, Hq, Hkv, cap, cap, num_splits)
    _lib.vqkv_decode_append(mode, H.dev(q), dk, dv, H.dev(np.asarray(lens, dtype=np.int32)), H.dev(kcb), H.dev(vcb),
                            H.dev(s), out, ws, cap, cap, H.dev(k_new), H.dev(v_new), near_tie_count=ties,
                            num_splits=num_splits)
    t.cuda.synchronize()
    return out.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy(), int(ties.item())


def _unfused(q, kbuf, vbuf, lens, kcb, vcb, s, cap, k_new, v_new, num_splits, mode=0):
    pos = [L - 1 if L > 0 else cap for L in lens]    # empty sequences: an out-of-range row, skipped
    kb = H.gpu_encode(mode, 0, k_new[:, :, None], pos, s, kcb, cap, codes=kbuf)
    vb = H.gpu_encode(mode, 1, v_new[:, :, None], pos, None, vcb, cap, codes=vbuf)
    o = H.gpu_decode(mode, q, kb, vb, lens, kcb, vcb, s, cap, cap, num_splits=num_splits)
    return o, kb, vb


CASES = [
    # B, Hq, Hkv, lens, cap, num_splits
    (1, 4, 1, [1000], 1024, 0),
    (2, 8, 2, [1, 517], 1024, 0, 2),         # 4 bit: a sequence holding only the new token
    (3, 8, 2, [32, 33, 640], 704, 5, 2),     # 4 bit: new token first / last of a 32-token step
    (1, 32, 8, [4097], 4112, 0, 2),          # 4 bit, Llama-like GQA
    (2, 8, 2, [1, 517], 1024, 0),            # a sequence holding only the new token
    (3, 8, 2, [48, 49, 640], 704, 5),         # new token first / last of a 48-token step, tile edges
    (2, 16, 2, [0, 300], 320, 3),            # an empty sequence: nothing appended, zero row
    (1, 32, 8, [4097], 4112, 0),             # Llama-like GQA, new token alone in its tile
    (1, 4, 1, [2000], 2048, 1),              # one split: the CTA writes O itself
    (1, 4, 1, [2000], 2048, 7),
    (1, 4, 1, [2000], 2048, 125),            # many splits: the new tile in a late CTA
]


@pytest.mark.parametrize("case", CASES)
def test_fused_step_against_oracle_and_unfused(case):
    B, Hq, Hkv, lens, cap, num_splits = case[:6]
    mode = case[6] if len(case) > 6 else 0
    s, kcb, vcb, kbuf, vbuf, k_new, v_new, q = _inputs(B, Hq, Hkv, cap, seed=7 * B + Hkv + num_splits, mode=mode)
    o, kb, vb, ties = _fused(q, kbuf, vbuf, lens, kcb, vcb, s, cap, k_new, v_new, num_splits, mode)
    assert np.isfinite(o).all()
    got_all, ref_all, d_all = [], [], []
    T = vo.TILE_TOKENS[mode]
    off = {role: vo.offset_table(mode, role, T * (-(-cap // T))) for role in (0, 1)}
    kc, vc = [], []
    for b in range(B):
        L = lens[b]
        kc.append([]), vc.append([])
        for h in range(Hkv):
            for role, got_buf, old_buf, x, cb in ((0, kb, kbuf, k_new, kcb), (1, vb, vbuf, v_new, vcb)):
                mask = np.ones(got_buf.shape[2], dtype=bool)
                if L > 0:
                    ref, d32 = vo.encode_rows(x[b, h][None], role, s[h] if role == 0 else None, cb[h])
                    got = vo.unpack_stream_fast(got_buf[b, h], mode, role, L)[L - 1:L]
                    got_all.append(got.reshape(-1))
                    ref_all.append(ref.reshape(-1))
                    d_all.append(d32.reshape(ref.size, -1))
                    mask[off[role][L - 1]] = False
                # every byte but the new token's is untouched
                assert np.array_equal(got_buf[b, h][mask], old_buf[b, h][mask]), (b, h, role)
            kc[b].append(vo.unpack_stream_fast(kb[b, h], mode, 0, L))
            vc[b].append(vo.unpack_stream_fast(vb[b, h], mode, 1, L))
    if got_all:
        H.check_and_record_codes(f"fused append, mode {mode}, lens {lens}, splits {num_splits}",
                                 np.concatenate(got_all), np.concatenate(ref_all), np.concatenate(d_all), ties)
    ref_o = vo.decode_attention(q, kc, vc, kcb, vcb, s, lens)
    assert vo.o_error(o, ref_o).max() <= H.O_TOL
    # the unfused calls give the same cache, and the same O under the same
    # split plan; the fused call's own plan may shorten the split that holds
    # the new token, which only regroups the fp32 partial sums
    o2, kb2, vb2 = _unfused(q, kbuf, vbuf, lens, kcb, vcb, s, cap, k_new, v_new, num_splits, mode)
    assert np.array_equal(kb, kb2) and np.array_equal(vb, vb2)
    if num_splits > 0:
        assert np.array_equal(o, o2)
    else:
        diff = np.abs(o.astype(np.float32) - o2.astype(np.float32))
        assert diff.max() <= 2e-3 * max(1.0, float(np.abs(o.astype(np.float32)).max()))


def test_near_tie_counter_counts_both_rows():
    """Duplicate centroids make every subvector of the new rows a tie."""
    s, kcb, vcb, kbuf, vbuf, _, _, q = _inputs(1, 4, 1, 64, seed=3)
    vcb[0, 9] = vcb[0, 4]
    v_new = np.tile(vcb[0, 4].astype(np.float16), 32)[None, None]
    k_new = np.zeros((1, 1, 128), dtype=np.float16)
    kcb[0, 11] = kcb[0, 2] = 0      # the zero key row sits on two equal centroids
    o, kb, vb, ties = _fused(q, kbuf, vbuf, [40], kcb, vcb, s, 64, k_new, v_new, 0)
    assert ties == 64
    assert np.all(vo.unpack_stream_fast(vb[0, 0], 0, 1, 40)[39] == 4)
    assert np.all(vo.unpack_stream_fast(kb[0, 0], 0, 0, 40)[39] == 2)
