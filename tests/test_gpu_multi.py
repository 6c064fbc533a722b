"""Multi-query decode (vqkv_decode_attn_multi) through the C ABI against the
oracle: M queries per sequence, query m sees the cached tokens
t <= L - M + m.  Covers both bit-widths, the deferred-merge plan of the
1.5-bit path, sequences shorter than M, and n_queries = 1 against
vqkv_decode_attn."""
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


def _case(mode, B, Hq, Hkv, M, lens, cap, seed):
    r = np.random.default_rng(seed)
    E, dsub = vo.GEOMETRY[mode]
    s, kcb, vcb = H.random_codebooks(mode, Hkv, seed + 1)
    kc = [[r.integers(0, E, size=(cap, 128 // dsub)) for _ in range(Hkv)] for _ in range(B)]
    vc = [[r.integers(0, E, size=(cap, 128 // dsub)) for _ in range(Hkv)] for _ in range(B)]
    q = r.standard_normal((B, M, Hq, 128)).astype(np.float16)
    return q, kc, vc, s, kcb, vcb


def _gpu_multi(mode, q, kc, vc, s, kcb, vcb, lens, cap, num_splits=0):
    t = H.torch()
    B, M, Hq, _ = q.shape
    Hkv = kcb.shape[0]
    kbuf, vbuf = H.pack_cache_role(mode, 0, kc, cap), H.pack_cache_role(mode, 1, vc, cap)
    out = t.full((B, M, Hq, 128), float("nan"), dtype=t.float16, device="cuda")
    ws = _lib.decode_workspace(mode, B, Hq, Hkv, cap, cap, num_splits, n_queries=M)
    _lib.vqkv_decode_attn_multi(mode, H.dev(q), H.dev(kbuf), H.dev(vbuf), H.dev(np.asarray(lens, dtype=np.int32)),
                                H.dev(kcb), H.dev(vcb), H.dev(s), out, ws, cap, cap, num_splits=num_splits)
    t.cuda.synchronize()
    return out.cpu().numpy()


CASES = [
    # mode, B, Hq, Hkv, M, lens, cap, num_splits
    (0, 1, 8, 2, 2, [1000], 1024, 0),          # Llama-like g = 4: 2 queries fill the 8 columns
    (0, 2, 4, 2, 4, [3, 517], 1024, 0),        # a sequence shorter than its 4 queries
    (0, 3, 8, 8, 8, [48, 49, 640], 704, 5),    # g = 1, 8 queries; tails at step edges
    (0, 1, 4, 1, 2, [2000], 2048, 125),        # many splits: the causal tail in one late CTA
    (1, 2, 8, 4, 4, [300, 64], 320, 0),        # 1.5 bit, several sequences per CTA (deferred merge)
    (1, 1, 1, 1, 8, [1000], 1024, 3),         # one head, 8 queries
    (0, 1, 8, 2, 4, [1000], 1024, 0),         # 4 queries x 4 heads: two column groups of 8
    (0, 2, 8, 2, 3, [517, 2], 768, 5),        # 12 columns: groups of 8 and 4; a sequence shorter than M
    (1, 2, 8, 2, 4, [300, 64], 320, 0),       # 1.5 bit, two column groups, deferred merge
    (0, 1, 32, 8, 6, [2000], 2048, 0),        # Llama-like: 6 queries x 4 heads, three groups
    (2, 1, 8, 2, 2, [1000], 1024, 0),         # 4 bit, 2 queries fill the 8 columns
    (2, 2, 8, 2, 3, [517, 2], 768, 5),        # 4 bit, two column groups
    (3, 1, 8, 2, 2, [1000], 1024, 0),         # 3 bit, 2 queries fill the 8 columns
    (3, 2, 8, 2, 3, [517, 2], 768, 5),        # 3 bit, two column groups
    (4, 1, 8, 2, 2, [1000], 1024, 0),         # 1.25 bit, 2 queries fill the 8 columns
    (4, 2, 8, 2, 3, [517, 2], 768, 5),        # 1.25 bit, two column groups
]


@pytest.mark.parametrize("mode,B,Hq,Hkv,M,lens,cap,num_splits", CASES)
def test_multi_query_against_oracle(mode, B, Hq, Hkv, M, lens, cap, num_splits):
    q, kc, vc, s, kcb, vcb = _case(mode, B, Hq, Hkv, M, lens, cap, seed=5 * M + B + mode)
    o = _gpu_multi(mode, q, kc, vc, s, kcb, vcb, lens, cap, num_splits)
    assert np.isfinite(o).all()
    ref = vo.decode_attention_multi(q, kc, vc, kcb, vcb, s, lens)
    err = vo.o_error(o.reshape(B * M, Hq, 128), ref.reshape(B * M, Hq, 128))
    assert err.max() <= H.O_TOL
    # queries that see no token are zero rows
    for b in range(B):
        for m in range(M):
            if lens[b] - M + m + 1 <= 0:
                assert np.all(o[b, m] == 0)


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_one_query_equals_single_query_decode(mode):
    q, kc, vc, s, kcb, vcb = _case(mode, 2, 8, 2, 1, [700, 129], 768, seed=31 + mode)
    o = _gpu_multi(mode, q, kc, vc, s, kcb, vcb, [700, 129], 768)
    kbuf, vbuf = H.pack_cache_role(mode, 0, kc, 768), H.pack_cache_role(mode, 1, vc, 768)
    o1 = H.gpu_decode(mode, q[:, 0], kbuf, vbuf, [700, 129], kcb, vcb, s, 768, 768)
    assert np.array_equal(o[:, 0], o1)
