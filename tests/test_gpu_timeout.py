"""The bounded on-chip waits of the 2-bit decode, made to run out on purpose.

The test hook withholds every warp's first bulk copy and limits each wait to
a few polls, so every ring wait gives up.  The call must finish, set
VQKV_DEVERR_TIMEOUT in the workspace error word and leave the context
usable: the next ordinary call on the same workspace is correct.  No fault,
trap or hang is involved: nothing waits for more than max_polls polls."""
import ctypes

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


def test_ring_waits_run_out_and_are_reported():
    t = H.torch()
    r = np.random.default_rng(17)
    B, Hq, Hkv, cap, lens = 2, 8, 2, 1024, [1000, 300]
    s, kcb, vcb = H.random_codebooks(0, Hkv, 18)
    kc = [[r.integers(0, 256, size=(cap, 32)) for _ in range(Hkv)] for _ in range(B)]
    vc = [[r.integers(0, 256, size=(cap, 32)) for _ in range(Hkv)] for _ in range(B)]
    q = r.standard_normal((B, Hq, 128)).astype(np.float16)
    dk, dv = H.dev(H.pack_cache_role(0, 0, kc, cap)), H.dev(H.pack_cache_role(0, 1, vc, cap))
    dl = H.dev(np.asarray(lens, dtype=np.int32))
    dq, dkcb, dvcb, ds = H.dev(q), H.dev(kcb), H.dev(vcb), H.dev(s)
    out = t.full((B, Hq, 128), float("nan"), dtype=t.float16, device="cuda")
    ws = _lib.decode_workspace(0, B, Hq, Hkv, cap, cap)
    a = _lib.decode_args(0, dq, dk, dv, dl, dkcb, dvcb, ds, out, ws, cap, cap)
    assert _lib.lib().vqkv_test_decode_ring_timeout(ctypes.byref(a), 64, None) == 0
    t.cuda.synchronize()
    assert int(ws[:4].view(t.int32).item()) & _lib.VQKV_DEVERR_TIMEOUT
    assert np.isfinite(out.cpu().numpy()).all()
    # the context and the workspace still work
    ws[:4] = 0
    _lib.vqkv_decode_attn(0, dq, dk, dv, dl, dkcb, dvcb, ds, out, ws, cap, cap)
    t.cuda.synchronize()
    assert int(ws[:4].view(t.int32).item()) == 0
    ref = vo.decode_attention(q, kc, vc, kcb, vcb, s, lens)
    assert vo.o_error(out.cpu().numpy(), ref).max() <= H.O_TOL
