"""vqkv_decode_attn_static: decode for callers that cannot allocate device
memory (a serving engine whose pool owns all device memory, a plugin whose
host framework offers no scratch buffer).  Its scratch is an array inside the
library; its results must match vqkv_decode_attn's.

Collected last on purpose (file name), and self-contained so it also passes
alone in a fresh process."""
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


def _case(mode, B, Hq, Hkv, lens, cap, seed):
    import torch
    r = np.random.default_rng(seed)
    E, dsub = vo.GEOMETRY[mode]
    s, kcb, vcb = H.random_codebooks(mode, Hkv, seed + 1)
    kc = [[r.integers(0, E, size=(cap, 128 // dsub)) for _ in range(Hkv)] for _ in range(B)]
    vc = [[r.integers(0, E, size=(cap, 128 // dsub)) for _ in range(Hkv)] for _ in range(B)]
    t = dict(kbuf=H.dev(H.pack_cache_role(mode, 0, kc, cap)), vbuf=H.dev(H.pack_cache_role(mode, 1, vc, cap)),
             lens=H.dev(np.asarray(lens, dtype=np.int32)), kcb=H.dev(kcb), vcb=H.dev(vcb), s=H.dev(s))
    qs = [H.dev(r.standard_normal((B, Hq, 128)).astype(np.float16)) for _ in range(2)]
    return t, qs, torch


@pytest.mark.parametrize("num_splits", [0, 8])
@pytest.mark.parametrize("mode,B,Hq,Hkv,lens,cap", [
    (0, 2, 8, 2, [900, 517], 1024),
    (1, 2, 10, 2, [300, 64], 320),
    (2, 2, 8, 2, [900, 517], 1024),
    (3, 2, 8, 2, [900, 517], 1024),
    (4, 2, 8, 2, [900, 517], 1024),
])
def test_static_scratch_matches_workspace_entry_on_two_calls(mode, B, Hq, Hkv, lens, cap, num_splits):
    """num_splits=8 forces several splits per (sequence, KV head), so the
    tickets and split partials in the library's array are used: the last-CTA
    merge (2, 4, 3, 1.25 bit) or the combine kernel (1.5 bit, whose CTAs
    cover several sequences)."""
    t, qs, torch = _case(mode, B, Hq, Hkv, lens, cap, seed=21 + mode)
    ws = _lib.decode_workspace(mode, B, Hq, Hkv, cap, max(lens), num_splits)
    if num_splits:
        a = _lib.decode_args(mode, qs[0], t["kbuf"], t["vbuf"], t["lens"], t["kcb"], t["vcb"], t["s"], qs[0], ws,
                             cap, max(lens), num_splits=num_splits)
        assert _lib.vqkv_decode_num_splits(a) > 1
        assert _lib.vqkv_decode_kernel_count(a) == (2 if mode == 1 else 1)
    for q in qs:   # two calls in a row; the second sees the first call's scratch contents
        ref = torch.empty((B, Hq, 128), dtype=torch.float16, device="cuda")
        got = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device="cuda")
        _lib.vqkv_decode_attn(mode, q, t["kbuf"], t["vbuf"], t["lens"], t["kcb"], t["vcb"], t["s"], ref, ws,
                              cap, max(lens), num_splits=num_splits)
        _lib.vqkv_decode_attn_static(mode, q, t["kbuf"], t["vbuf"], t["lens"], t["kcb"], t["vcb"], t["s"], got,
                                     cap, max(lens), num_splits=num_splits)
        torch.cuda.synchronize()
        r, g = ref.cpu().numpy(), got.cpu().numpy()
        assert np.isfinite(g).all()
        assert vo.o_error(g, r.astype(np.float64)).max() <= H.O_TOL
        assert _lib.vqkv_decode_static_error() == 0


def test_static_error_word_reports_a_clamped_length_and_clears():
    """An out-of-range sequence length is clamped and reported through the
    error query; the next call starts from a clear error word."""
    import torch
    t, qs, _ = _case(0, 2, 8, 2, [50, 64], 64, seed=5)
    bad = H.dev(np.array([50, 9999], dtype=np.int32))
    out = torch.empty((2, 8, 128), dtype=torch.float16, device="cuda")
    _lib.vqkv_decode_attn_static(0, qs[0], t["kbuf"], t["vbuf"], bad, t["kcb"], t["vcb"], t["s"], out, 64, 64)
    assert _lib.vqkv_decode_static_error() & _lib.VQKV_DEVERR_SEQ_LEN
    _lib.vqkv_decode_attn_static(0, qs[0], t["kbuf"], t["vbuf"], t["lens"], t["kcb"], t["vcb"], t["s"], out, 64,
                                 64)
    assert _lib.vqkv_decode_static_error() == 0


def test_static_scratch_rejects_plans_beyond_its_size():
    import torch
    B, Hq, Hkv, cap = 64, 64, 8, 65536
    q = torch.zeros((B, Hq, 128), dtype=torch.float16, device="cuda")
    cb = torch.zeros((Hkv, 256, 4), dtype=torch.float16, device="cuda")
    buf = torch.zeros(1 << 12, dtype=torch.uint8, device="cuda")
    a = _lib.decode_args(0, q, buf, buf, buf, cb, cb, buf, q, None, cap, cap, num_splits=64)
    assert _lib.vqkv_decode_workspace_bytes(a) > _lib.STATIC_SCRATCH_BYTES
    with pytest.raises(_lib.VqkvError) as e:
        _lib.vqkv_decode_attn_static(0, q, buf, buf, buf, cb, cb, buf, q, cap, cap, num_splits=64)
    assert e.value.status == 3   # VQKV_ERR_WORKSPACE
