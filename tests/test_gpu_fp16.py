"""The fp16-KV comparison decode kernel against the oracle's plain attention."""
import math

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


def run(q, k, v, lens, max_len, num_splits=0, scale=0.0):
    import torch
    B, Hq, _ = q.shape
    Hkv, cap = k.shape[1], k.shape[2]
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device="cuda")
    ws = _lib.fp16_decode_workspace(B, Hq, Hkv, cap, max_len, num_splits)
    _lib.vqkv_decode_attn_fp16(H.dev(q), H.dev(k), H.dev(v), H.dev(np.asarray(lens, np.int32)), out, ws, max_len,
                               softmax_scale=scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def oracle(q, k, v, lens, scale=None):
    B, Hq, _ = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    scale = 1 / math.sqrt(128) if scale is None else scale
    o = np.zeros((B, Hq, 128))
    for b in range(B):
        for h in range(Hq):
            L = lens[b]
            o[b, h] = vo.attention(q[b, h], k[b, h // g, :L].astype(np.float64), v[b, h // g, :L].astype(np.float64),
                                   scale)
    return o


@pytest.mark.parametrize("B,Hq,Hkv,lens,cap", [
    (3, 8, 2, [1, 17, 300], 320), (2, 5, 1, [64, 33], 64), (1, 8, 1, [257], 260), (2, 2, 2, [16, 15], 16),
    (2, 32, 8, [1000, 777], 1024), (3, 4, 1, [0, 5, 0], 32),
])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_fp16_decode_matches_oracle(B, Hq, Hkv, lens, cap, num_splits):
    r = np.random.default_rng(B * 7 + Hq)
    q = r.standard_normal((B, Hq, 128)).astype(np.float16)
    k = r.standard_normal((B, Hkv, cap, 128)).astype(np.float16)
    v = r.standard_normal((B, Hkv, cap, 128)).astype(np.float16)
    # rows past each sequence are never read: poison them
    for b in range(B):
        k[b, :, lens[b]:] = np.nan
        v[b, :, lens[b]:] = np.nan
    o = run(q, k, v, lens, max(max(lens), 1), num_splits)
    ref = oracle(q, k, v, lens)
    assert np.isfinite(o).all()
    assert vo.o_error(o, ref).max() <= H.O_TOL


def test_fp16_decode_scale_and_single_token():
    r = np.random.default_rng(3)
    q = r.standard_normal((1, 4, 128)).astype(np.float16)
    k = r.standard_normal((1, 1, 64, 128)).astype(np.float16)
    v = r.standard_normal((1, 1, 64, 128)).astype(np.float16)
    o = run(q, k, v, [1], 64)
    assert np.array_equal(o[0, 0], v[0, 0, 0])
    o = run(q, k, v, [50], 64, scale=0.3)
    assert vo.o_error(o, oracle(q, k, v, [50], scale=0.3)).max() <= H.O_TOL
