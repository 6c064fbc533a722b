"""Test-side glue: builds inputs (generator + oracle), calls the CUDA path
through the C ABI binding, compares with the oracle."""
from __future__ import annotations

import concurrent.futures
import multiprocessing
import os

import numpy as np

from oracle import vqkv_oracle as vo
from vector_quantized_bit_gb300 import _build, _lib, calib, synth

O_TOL = 2e-3   # max_d |O_gpu - O_ref| / max_d |O_ref| per (b, h) row


def torch():
    import torch as t
    return t


def dev(a, dtype=None):
    t = torch()
    x = t.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        x = x.to(dtype)
    return x.cuda()


def pool(n=None):
    n = n or min(16, os.cpu_count() or 1)
    return concurrent.futures.ProcessPoolExecutor(n, mp_context=multiprocessing.get_context("spawn"))


def _cal(args):
    w, kvh, kw = args
    return calib.calibrate_head(w, kvh, **kw)


def calibrate(w, **kw):
    """calib.calibrate over KV heads in parallel (spawned workers)."""
    if w.Hkv == 1:
        s, k, v = calib.calibrate_head(w, 0, **kw)
        return s[None], k[None], v[None]
    with pool(min(w.Hkv, 16)) as ex:
        out = list(ex.map(_cal, [(w, h, kw) for h in range(w.Hkv)]))
    return np.stack([o[0] for o in out]), np.stack([o[1] for o in out]), np.stack([o[2] for o in out])


def random_codebooks(mode, Hkv, seed):
    E, dsub = vo.GEOMETRY[mode]
    r = np.random.default_rng(seed)
    kcb = (r.standard_normal((Hkv, E, dsub)) * 0.6).astype(np.float16)
    vcb = r.standard_normal((Hkv, E, dsub)).astype(np.float16)
    s = r.uniform(0.5, 4.0, size=(Hkv, 128)).astype(np.float32)
    return s, kcb, vcb


def pack_cache(mode, codes, cap_len):
    """codes: list over b of list over kvh of int arrays [L][n_sub] -> uint8 [B][Hkv][stream]."""
    B, Hkv = len(codes), len(codes[0])
    sb = vo.code_bytes(mode, cap_len)
    out = np.zeros((B, Hkv, sb), dtype=np.uint8)
    for b in range(B):
        for h in range(Hkv):
            role_k = codes[b][h]
            out[b, h] = vo.pack_stream_fast(role_k, mode, 0, cap_len) if role_k is not None else 0
    return out


def pack_cache_role(mode, role, codes, cap_len):
    B, Hkv = len(codes), len(codes[0])
    out = np.zeros((B, Hkv, vo.code_bytes(mode, cap_len)), dtype=np.uint8)
    for b in range(B):
        for h in range(Hkv):
            out[b, h] = vo.pack_stream_fast(codes[b][h], mode, role, cap_len)
    return out


def gpu_decode(mode, q, kbuf, vbuf, lens, kcb, vcb, s, cap_len, max_seq_len, num_splits=0, softmax_scale=0.0,
               workspace=None, return_ws=False):
    t = torch()
    B, Hq, _ = q.shape
    Hkv = kcb.shape[0]
    dq, dk, dv = dev(q), dev(kbuf), dev(vbuf)
    dl = dev(np.asarray(lens, dtype=np.int32))
    dkcb, dvcb, ds = dev(kcb), dev(vcb), dev(s)
    out = t.full((B, Hq, 128), float("nan"), dtype=t.float16, device="cuda")
    ws = workspace if workspace is not None else _lib.decode_workspace(mode, B, Hq, Hkv, cap_len, max_seq_len,
                                                                        num_splits)
    _lib.vqkv_decode_attn(mode, dq, dk, dv, dl, dkcb, dvcb, ds, out, ws, cap_len, max_seq_len,
                          softmax_scale=softmax_scale, num_splits=num_splits)
    t.cuda.synchronize()
    o = out.cpu().numpy()
    return (o, ws) if return_ws else o


def gpu_encode(mode, role, x, pos, s, cb, cap_len, codes=None, with_ties=False):
    t = torch()
    B, Hkv = x.shape[0], x.shape[1]
    sb = vo.code_bytes(mode, cap_len)
    dcodes = dev(codes) if codes is not None else t.zeros((B, Hkv, sb), dtype=t.uint8, device="cuda")
    ties = t.zeros(1, dtype=t.int64, device="cuda")
    err = t.zeros(1, dtype=t.int32, device="cuda")
    _lib.vqkv_encode(mode, role, dev(x), dev(np.asarray(pos, dtype=np.int32)), dev(s) if s is not None else None,
                     dev(cb), dcodes, cap_len, near_tie_count=ties, error_flags=err)
    t.cuda.synchronize()
    res = dcodes.cpu().numpy()
    if with_ties:
        return res, int(ties.item()), int(err.item())
    return res


def check_codes(gpu_codes, ref_codes, d32):
    """Bit-exact except near-ties (oracle fp32 distances within 1e-6 relative).
    Returns (#near-tie mismatches, #failing mismatches)."""
    gpu_codes = np.asarray(gpu_codes).reshape(-1)
    ref_codes = np.asarray(ref_codes).reshape(-1)
    d = d32.reshape(gpu_codes.size, -1)
    bad = np.flatnonzero(gpu_codes != ref_codes)
    ties = sum(1 for i in bad if vo.near_tie(d[i], int(gpu_codes[i])))
    return ties, len(bad) - ties


def check_and_record_codes(name, gpu_codes, ref_codes, d32, device_count=None, bounded=True):
    """check_codes, recorded in the near-tie log (tests/tie_log.py), with the
    failing count asserted zero and, for natural data, the near-tie count
    bounded.  Returns the number of near-tie mismatches."""
    from tests import tie_log
    ties, fails = check_codes(gpu_codes, ref_codes, d32)
    n = int(np.asarray(gpu_codes).size)
    tie_log.record(name, n, ties, fails, device_count)
    assert fails == 0, (name, ties, fails)
    if bounded:
        assert ties <= tie_log.bound(n), (name, ties, n)
        if device_count is not None:
            assert device_count <= tie_log.bound(n), (name, device_count, n)
    return ties


def library_loaded() -> bool:
    return os.path.exists(_build.LIB)
