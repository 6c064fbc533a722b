"""Paged cache (vqkv_encode_paged / vqkv_decode_attn_paged) through the C ABI.

Rows encoded into a shuffled block pool, then decoded through the block
table, must give the same cache bytes (after gathering the blocks back into
streams) and the same O as the contiguous calls, and O within the decode
tolerance of the oracle.  Block ids outside the pool are reported, never
dereferenced."""
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


def _gather(pool, table, mode, block_tokens, cap):
    """Contiguous streams [B][Hkv][code_bytes(cap)] from a paged pool."""
    bb = vo.code_bytes(mode, block_tokens)
    B, nblk = table.shape
    out = np.zeros((B, pool.shape[1], vo.code_bytes(mode, cap)), dtype=np.uint8)
    for b in range(B):
        for i in range(nblk):
            lo = i * bb
            if lo >= out.shape[2]:
                break
            out[b, :, lo:lo + bb] = pool[table[b, i], :, :out.shape[2] - lo][:, :bb]
    return out


@pytest.mark.parametrize("mode,B,Hq,Hkv,lens,cap,block_tokens,num_splits", [
    (0, 3, 8, 2, [1000, 17, 640], 1024, 256, 0),
    (0, 2, 4, 1, [700, 1], 768, 64, 7),       # small blocks: a 48-token step spans two blocks
    (1, 2, 10, 2, [300, 190], 384, 128, 0),   # 1.5 bit, several sequences per CTA
    (1, 1, 4, 1, [1024], 1024, 64, 3),
    (2, 2, 8, 2, [1000, 300], 1024, 64, 5),   # 4 bit: a 32-token step spans two 64-token blocks
    (3, 2, 8, 2, [1000, 300], 1024, 64, 5),   # 3 bit: a 48-token step spans two 64-token blocks
    (4, 2, 8, 2, [1000, 300], 1024, 64, 5),   # 1.25 bit, the same
])
def test_paged_equals_contiguous_and_oracle(mode, B, Hq, Hkv, lens, cap, block_tokens, num_splits):
    t = H.torch()
    r = np.random.default_rng(3 + mode + B)
    s, kcb, vcb = H.random_codebooks(mode, Hkv, 9 + mode)
    k = (r.standard_normal((B, Hkv, cap, 128)) * r.uniform(0.5, 3.0, size=(1, 1, 1, 128))).astype(np.float16)
    v = r.standard_normal((B, Hkv, cap, 128)).astype(np.float16)
    q = r.standard_normal((B, Hq, 128)).astype(np.float16)
    max_blocks = cap // block_tokens
    num_blocks = B * max_blocks + 3
    table = r.permutation(num_blocks)[:B * max_blocks].reshape(B, max_blocks).astype(np.int32)
    bb = vo.code_bytes(mode, block_tokens)
    dtable = H.dev(table)
    pools, streams = [], []
    for role, x, cb in ((0, k, kcb), (1, v, vcb)):
        pool = t.zeros((num_blocks, Hkv, bb), dtype=t.uint8, device="cuda")
        err = t.zeros(1, dtype=t.int32, device="cuda")
        _lib.vqkv_encode_paged(mode, role, H.dev(x), H.dev(np.zeros(B, dtype=np.int32)),
                               H.dev(s) if role == 0 else None, H.dev(cb), pool, cap, dtable, block_tokens,
                               num_blocks, error_flags=err)
        t.cuda.synchronize()
        assert int(err.item()) == 0
        pools.append(pool)
        streams.append(H.gpu_encode(mode, role, x, [0] * B, s if role == 0 else None, cb, cap))
    for role in (0, 1):
        assert np.array_equal(_gather(pools[role].cpu().numpy(), table, mode, block_tokens, cap), streams[role])
    out = t.full((B, Hq, 128), float("nan"), dtype=t.float16, device="cuda")
    ws = _lib.decode_workspace(mode, B, Hq, Hkv, cap, cap, num_splits)
    _lib.vqkv_decode_attn_paged(mode, H.dev(q), pools[0], pools[1], H.dev(np.asarray(lens, dtype=np.int32)),
                                H.dev(kcb), H.dev(vcb), H.dev(s), out, ws, cap, cap, dtable, block_tokens, num_blocks,
                                num_splits=num_splits)
    t.cuda.synchronize()
    o = out.cpu().numpy()
    assert int(ws[:4].view(t.int32).item()) == 0
    o_contig = H.gpu_decode(mode, q, streams[0], streams[1], lens, kcb, vcb, s, cap, cap, num_splits=num_splits)
    assert np.array_equal(o, o_contig)
    kc = [[vo.unpack_stream_fast(streams[0][b, h], mode, 0, lens[b]) for h in range(Hkv)] for b in range(B)]
    vc = [[vo.unpack_stream_fast(streams[1][b, h], mode, 1, lens[b]) for h in range(Hkv)] for b in range(B)]
    assert vo.o_error(o, vo.decode_attention(q, kc, vc, kcb, vcb, s, lens)).max() <= H.O_TOL


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_block_ids_outside_the_pool_are_reported(mode):
    t = H.torch()
    s, kcb, vcb = H.random_codebooks(mode, 1, 4)
    bt, cap = 64, 256
    num_blocks = 4
    table = np.array([[0, 1, 7, 2]], dtype=np.int32)     # block 7 is outside the pool of 4
    bb = vo.code_bytes(mode, bt)
    pool = t.full((num_blocks, 1, bb), 0xA5, dtype=t.uint8, device="cuda")
    err = t.zeros(1, dtype=t.int32, device="cuda")
    x = np.random.default_rng(2).standard_normal((1, 1, cap, 128)).astype(np.float16)
    _lib.vqkv_encode_paged(mode, 1, H.dev(x), H.dev(np.zeros(1, dtype=np.int32)), None, H.dev(vcb), pool, cap,
                           H.dev(table), bt, num_blocks, error_flags=err)
    t.cuda.synchronize()
    assert int(err.item()) & _lib.VQKV_DEVERR_BLOCK
    # logical blocks 0, 1, 3 (physical 0, 1, 2) were written; logical block 2
    # was skipped, and physical block 3 (in no table entry) is untouched
    got = pool.cpu().numpy()
    assert not np.any(np.all(got[:3] == 0xA5, axis=(1, 2))) and np.all(got[3] == 0xA5)
    q = np.random.default_rng(3).standard_normal((1, 4, 128)).astype(np.float16)
    out = t.zeros((1, 4, 128), dtype=t.float16, device="cuda")
    ws = _lib.decode_workspace(mode, 1, 4, 1, cap, cap)
    _lib.vqkv_decode_attn_paged(mode, H.dev(q), pool, pool, H.dev(np.array([cap], dtype=np.int32)), H.dev(kcb),
                                H.dev(vcb), H.dev(s), out, ws, cap, cap, H.dev(table), bt, num_blocks)
    t.cuda.synchronize()
    assert int(ws[:4].view(t.int32).item()) & _lib.VQKV_DEVERR_BLOCK
    assert np.isfinite(out.cpu().numpy()).all()


@pytest.mark.parametrize("mode,block_tokens", [(0, 64), (0, 256), (1, 64), (3, 64), (4, 64)])
def test_table_entries_past_the_sequence_are_not_read(mode, block_tokens):
    """Serving engines leave the entries after a sequence's last block
    unset: they must not be read (no error bit), and O must equal the
    contiguous decode's."""
    t = H.torch()
    r = np.random.default_rng(40 + mode)
    B, Hq, Hkv, cap, lens = 2, 8, 2, 1024, [700, 1]
    E, dsub = vo.GEOMETRY[mode]
    s, kcb, vcb = H.random_codebooks(mode, Hkv, 41)
    max_blocks = cap // block_tokens
    num_blocks = B * max_blocks
    table = r.permutation(num_blocks).reshape(B, max_blocks).astype(np.int32)
    for b in range(B):
        table[b, -(-lens[b] // block_tokens):] = -1          # unset entries
    kc = [[r.integers(0, E, size=(cap, 128 // dsub)) for _ in range(Hkv)] for _ in range(B)]
    vc = [[r.integers(0, E, size=(cap, 128 // dsub)) for _ in range(Hkv)] for _ in range(B)]
    streams = [H.pack_cache_role(mode, role, c, cap) for role, c in ((0, kc), (1, vc))]
    bb = vo.code_bytes(mode, block_tokens)
    pools = []
    for st in streams:
        pool = np.zeros((num_blocks, Hkv, bb), dtype=np.uint8)
        for b in range(B):
            for i in range(max_blocks):
                if table[b, i] >= 0:
                    pool[table[b, i]] = st[b, :, i * bb:(i + 1) * bb]
        pools.append(H.dev(pool))
    q = r.standard_normal((B, Hq, 128)).astype(np.float16)
    out = t.full((B, Hq, 128), float("nan"), dtype=t.float16, device="cuda")
    ws = _lib.decode_workspace(mode, B, Hq, Hkv, cap, cap)
    for num_splits in (0, 7):
        ws[:4] = 0
        _lib.vqkv_decode_attn_paged(mode, H.dev(q), pools[0], pools[1], H.dev(np.asarray(lens, dtype=np.int32)),
                                    H.dev(kcb), H.dev(vcb), H.dev(s), out, ws, cap, cap, H.dev(table), block_tokens,
                                    num_blocks, num_splits=num_splits)
        t.cuda.synchronize()
        assert int(ws[:4].view(t.int32).item()) == 0
        o_contig = H.gpu_decode(mode, q, streams[0], streams[1], lens, kcb, vcb, s, cap, cap, num_splits=num_splits)
        assert np.array_equal(out.cpu().numpy(), o_contig)
