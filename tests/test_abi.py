"""The C-ABI library builds, loads and exports what include/vqkv.h declares;
argument validation that happens before any CUDA call.  No GPU needed."""
import ctypes
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT
from vector_quantized_bit_gb300 import _build, _lib

HEADER = os.path.join(ROOT, "include", "vqkv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vqkv_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTED), names
    nm = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (vqkv_\w+)", nm))
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_struct_layout_matches_header(tmp_path):
    """ctypes mirrors of the argument structs have the C layout (gcc offsetof)."""
    fields = {"vqkv_encode_args": _lib.EncodeArgs, "vqkv_decode_args": _lib.DecodeArgs,
              "vqkv_fp16_decode_args": _lib.Fp16DecodeArgs, "vqkv_decode_append_args": _lib.DecodeAppendArgs,
              "vqkv_decode_multi_args": _lib.DecodeMultiArgs, "vqkv_paging": _lib.Paging,
              "vqkv_kmeans_args": _lib.KmeansArgs}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "vqkv.h"', "int main(void){"]
    for cname, cls in fields.items():
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0;}")
    c = tmp_path / "layout.c"
    c.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(c), "-o", str(exe)], check=True)
    out = dict(line.rsplit(" ", 1) for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                              check=True).stdout.split("\n") if line)
    for cname, cls in fields.items():
        assert int(out[cname]) == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert int(out[f"{cname}.{f}"]) == getattr(cls, f).offset, (cname, f)


def test_code_bytes(lib):
    assert lib.vqkv_code_bytes(2, 16384) == 16384 * 64
    assert lib.vqkv_code_bytes(2, 17) == 2048
    assert lib.vqkv_code_bytes(0, 196608) == 196608 * 32
    assert lib.vqkv_code_bytes(1, 65536) == 65536 * 24
    assert lib.vqkv_code_bytes(0, 1) == 512
    assert lib.vqkv_code_bytes(1, 65) == 3072
    assert lib.vqkv_code_bytes(3, 65536) == 65536 * 48
    assert lib.vqkv_code_bytes(3, 17) == 1536
    assert lib.vqkv_code_bytes(4, 65536) == 65536 * 20
    assert lib.vqkv_code_bytes(4, 17) == 640
    assert lib.vqkv_code_bytes(7, 16) == 0
    assert lib.vqkv_code_bytes(0, -1) == 0


def _dec(**kw):
    a = _lib.DecodeArgs(mode=0, B=1, Hq=4, Hkv=1, head_dim=128, cap_len=64, max_seq_len=64,
                        q=0x1000, k_codes=0x2000, v_codes=0x3000, seq_lens=0x4000, k_codebook=0x5000,
                        v_codebook=0x6000, s=0x7000, softmax_scale=0.0, num_splits=0, workspace=0x8000,
                        workspace_bytes=1 << 20, out=0x9000)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _enc(**kw):
    a = _lib.EncodeArgs(mode=0, role=0, B=1, Hkv=1, head_dim=128, n_rows=4, cap_len=64, x=0x1000,
                        pos=0x2000, s=0x3000, codebook=0x4000, codes=0x5000)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), 2), (dict(mode=5), 2), (dict(Hq=36, Hkv=4), 2), (dict(Hq=6, Hkv=4), 1),
    (dict(Hkv=0), 1), (dict(B=-1), 1), (dict(max_seq_len=65), 1), (dict(max_seq_len=-1), 1),
    (dict(cap_len=0, max_seq_len=0), 1), (dict(q=None), 1), (dict(k_codes=None), 1), (dict(s=None), 1),
    (dict(out=None), 1), (dict(k_codes=0x2008), 1), (dict(k_codebook=0x5004), 1), (dict(q=0x1002), 1),
    (dict(num_splits=-2), 1), (dict(softmax_scale=float("nan")), 1),
])
def test_decode_validation(lib, kw, status):
    assert lib.vqkv_decode_attn(ctypes.byref(_dec(**kw)), None) == status
    pointer_only = all(k in ("q", "k_codes", "v_codes", "s", "out", "k_codebook", "softmax_scale") for k in kw)
    if not pointer_only:   # the size queries read sizes only
        assert lib.vqkv_decode_workspace_bytes(ctypes.byref(_dec(**kw))) == 0
        assert lib.vqkv_decode_num_splits(ctypes.byref(_dec(**kw))) == -1
        assert lib.vqkv_decode_kernel_count(ctypes.byref(_dec(**kw))) == -1


def test_decode_empty_batch_is_a_no_op(lib):
    # B == 0: nothing to validate beyond the sizes, nothing launched
    assert lib.vqkv_decode_attn(ctypes.byref(_dec(B=0, q=None, out=None)), None) == 0


def test_null_args(lib):
    assert lib.vqkv_decode_attn(None, None) == 1
    assert lib.vqkv_encode(None, None) == 1
    assert lib.vqkv_decode_workspace_bytes(None) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=256), 2), (dict(mode=5), 2), (dict(role=2), 1), (dict(Hkv=0), 1), (dict(n_rows=-1), 1),
    (dict(cap_len=0), 1), (dict(x=None), 1), (dict(pos=None), 1), (dict(codebook=None), 1),
    (dict(codes=None), 1), (dict(s=None), 1), (dict(x=0x1004), 1), (dict(codebook=0x4008), 1),
])
def test_encode_validation(lib, kw, status):
    assert lib.vqkv_encode(ctypes.byref(_enc(**kw)), None) == status


def test_encode_empty_is_a_no_op(lib):
    assert lib.vqkv_encode(ctypes.byref(_enc(n_rows=0, x=None)), None) == 0
    assert lib.vqkv_encode(ctypes.byref(_enc(B=0, x=None)), None) == 0
    # values need no smoothing vector
    assert lib.vqkv_encode(ctypes.byref(_enc(role=1, s=None, n_rows=0)), None) == 0


def test_status_strings(lib):
    for st in range(6):
        assert lib.vqkv_status_string(st)
    assert lib.vqkv_status_string(99) == b"unknown status"


def test_product_path_has_no_cpu_fallback(monkeypatch, tmp_path):
    """Without the built library the binding raises instead of computing."""
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib(str(tmp_path / "missing.so"))
    src = open(_lib.__file__).read() + open(os.path.join(ROOT, "vector_quantized_bit_gb300", "__init__.py")).read()
    assert "oracle" not in src.replace("no fallback", "")


def test_decode_append_validation(lib):
    # checked on the host before anything is launched (no device needed)
    a = _lib.DecodeAppendArgs()
    a.decode = _dec(mode=1)
    assert lib.vqkv_decode_append(ctypes.byref(a), None) == 2    # 2-bit only
    a.decode = _dec(mode=3)
    assert lib.vqkv_decode_append(ctypes.byref(a), None) == 2    # nor 3 bit (12-bit code pairs)
    a.decode = _dec(mode=4)
    assert lib.vqkv_decode_append(ctypes.byref(a), None) == 2    # nor 1.25 bit (10-bit codes)
    a.decode = _dec(mode=2)
    assert lib.vqkv_decode_append(ctypes.byref(a), None) == 1    # 4 bit too: no new rows
    a.decode = _dec()
    assert lib.vqkv_decode_append(ctypes.byref(a), None) == 1    # no new rows
    a.k_new, a.v_new = 0x10000, 0x10004                             # v_new not 8-byte aligned
    assert lib.vqkv_decode_append(ctypes.byref(a), None) == 1
    assert lib.vqkv_decode_append(None, None) == 1
    a.decode = _dec(B=0, q=None, out=None)
    assert lib.vqkv_decode_append(ctypes.byref(a), None) == 0    # empty batch: a no-op


def test_decode_multi_validation(lib):
    a = _lib.DecodeMultiArgs()
    a.decode = _dec(Hq=4, Hkv=1)
    a.n_queries = 0
    assert lib.vqkv_decode_attn_multi(ctypes.byref(a), None) == 1    # at least one query
    a.n_queries = 17
    assert lib.vqkv_decode_attn_multi(ctypes.byref(a), None) == 2    # 17 queries x 4 heads > 64 columns
    assert lib.vqkv_decode_attn_multi(None, None) == 1
    a.decode = _dec(B=0, q=None, out=None)
    a.n_queries = 2
    assert lib.vqkv_decode_attn_multi(ctypes.byref(a), None) == 0    # empty batch: a no-op


@pytest.mark.parametrize("kw", [dict(block_tokens=100), dict(block_tokens=192), dict(block_tokens=0), dict(max_blocks=0),
                                dict(num_blocks=0), dict(max_blocks=1)])   # 1 x 64 tokens < cap_len 128
def test_paging_validation(lib, kw):
    pg = _lib.Paging(block_table=0x1000, max_blocks=2, block_tokens=64, num_blocks=4)
    for k, v in kw.items():
        setattr(pg, k, v)
    d = _dec(cap_len=128, max_seq_len=128)
    assert lib.vqkv_decode_attn_paged(ctypes.byref(d), ctypes.byref(pg), None) == 1
    assert lib.vqkv_encode_paged(ctypes.byref(_enc(cap_len=128)), ctypes.byref(pg), None) == 1


def test_paging_required_and_empty_batch(lib):
    assert lib.vqkv_decode_attn_paged(ctypes.byref(_dec()), None, None) == 1
    assert lib.vqkv_encode_paged(ctypes.byref(_enc()), None, None) == 1
    pg = _lib.Paging(block_table=None, max_blocks=1, block_tokens=64, num_blocks=1)
    assert lib.vqkv_decode_attn_paged(ctypes.byref(_dec()), ctypes.byref(pg), None) == 1   # no table
    assert lib.vqkv_decode_attn_paged(ctypes.byref(_dec(B=0, q=None, out=None)), ctypes.byref(pg), None) == 0


def test_ring_timeout_hook_validation(lib):
    assert lib.vqkv_test_decode_ring_timeout(ctypes.byref(_dec(mode=1)), 64, None) == 2   # 2-bit only
    assert lib.vqkv_test_decode_ring_timeout(ctypes.byref(_dec(mode=2)), 64, None) == 2
    assert lib.vqkv_test_decode_ring_timeout(ctypes.byref(_dec(mode=3)), 64, None) == 2
    assert lib.vqkv_test_decode_ring_timeout(ctypes.byref(_dec(mode=4)), 64, None) == 2
    assert lib.vqkv_test_decode_ring_timeout(ctypes.byref(_dec()), 0, None) == 1
    assert lib.vqkv_test_decode_ring_timeout(ctypes.byref(_dec()), 5000, None) == 1
    assert lib.vqkv_test_decode_ring_timeout(None, 64, None) == 1


def _km(**kw):
    base = dict(n=1000, dim=4, k=256, iters=20, points=0x1000, uniforms=0x2000, centroids=0x3000,
                workspace=0x10000, workspace_bytes=1 << 24)
    base.update(kw)
    return _lib.KmeansArgs(**base)


@pytest.mark.parametrize("kw", [dict(n=0), dict(dim=3), dict(dim=16), dict(k=0), dict(k=4097), dict(k=1001),
                                dict(iters=-1), dict(iters=1001)])
def test_kmeans_size_validation(lib, kw):
    a = _km(**kw)
    assert lib.vqkv_kmeans_workspace_bytes(ctypes.byref(a)) == 0
    assert lib.vqkv_kmeans(ctypes.byref(a), None) == 1


def test_kmeans_workspace_layout(lib):
    # D^2 [n] fp32 | assignment [n] int32 | second centroid buffer [k][dim], each padded to 256 bytes
    # ... then the update's sort scratch: H [k][blocks of 1024] | start [k + 1] | perm [n] | tot [k] int32, + 256
    upd = lambda n, k: (4 * (k * max(1, -(-n // 1024)) + k + 1 + n + k) + 256 + 255) // 256 * 256
    assert lib.vqkv_kmeans_update_workspace_bytes(1000, 256) == upd(1000, 256)
    assert lib.vqkv_kmeans_workspace_bytes(ctypes.byref(_km(n=1000, dim=4, k=256))) == 3 * 4096 + upd(1000, 256)
    assert lib.vqkv_kmeans_workspace_bytes(ctypes.byref(_km(n=65536, dim=8, k=4096))) == (
        2 * 262144 + 131072 + upd(65536, 4096))
    assert lib.vqkv_kmeans_update_workspace_bytes(10, 0) == 0


def test_kmeans_pointer_and_workspace_validation(lib):
    assert lib.vqkv_kmeans(ctypes.byref(_km(points=None)), None) == 1
    assert lib.vqkv_kmeans(ctypes.byref(_km(points=0x1004)), None) == 1          # 16-byte alignment
    assert lib.vqkv_kmeans(ctypes.byref(_km(workspace_bytes=100)), None) == 3    # VQKV_ERR_WORKSPACE
    assert lib.vqkv_kmeans(ctypes.byref(_km(workspace=0x10010)), None) == 1      # 256-byte alignment
    assert lib.vqkv_kmeans_seed(ctypes.byref(_km(seeds=None)), None) == 1        # seeding needs its picks
    assert lib.vqkv_kmeans(None, None) == 1


def test_kmeans_step_validation(lib):
    assert lib.vqkv_kmeans_assign(0x1000, 10, 5, 0x2000, 4, 0x3000, None, None) == 1      # dim
    assert lib.vqkv_kmeans_assign(0x1000, 10, 4, 0x2000, 0, 0x3000, None, None) == 1      # k
    assert lib.vqkv_kmeans_assign(0x1008, 10, 4, 0x2000, 4, 0x3000, None, None) == 1      # alignment
    assert lib.vqkv_kmeans_assign(None, 0, 4, None, 4, None, None, None) == 0              # nothing to do
    ws = 0x100000
    assert lib.vqkv_kmeans_update(0x1000, 10, 4, 0x3000, 4, 0x2000, 0x2020, ws, 1 << 20, None) == 1   # overlap
    assert lib.vqkv_kmeans_update(0x1000, 10, 4, 0x3000, 5000, 0x2000, 0x90000, ws, 1 << 20, None) == 1
    assert lib.vqkv_kmeans_update(0x1000, 10, 4, 0x3000, 4, 0x2000, 0x9000, ws, 8, None) == 3        # workspace
    assert lib.vqkv_kmeans_update(0x1000, 10, 4, 0x3000, 4, 0x2000, 0x9000, ws + 8, 1 << 20, None) == 1


def test_calibration_validation(lib):
    assert lib.vqkv_smoothing(0x1000, 2, 10, 0x2000, None) == 1        # dtype
    assert lib.vqkv_smoothing(0x1000, 0, -1, 0x2000, None) == 1        # n_rows
    assert lib.vqkv_smoothing(0x1000, 0, 10, None, None) == 1          # s
    assert lib.vqkv_smoothing(0x1000, 0, 10, 0x2004, None) == 1        # s alignment
    assert lib.vqkv_calib_transform(0x1000, 0, 10, None, 1, None, 0x2008, None) == 1   # out alignment
    assert lib.vqkv_calib_transform(0x1000, 3, 10, None, 1, None, 0x2000, None) == 1   # dtype
    assert lib.vqkv_calib_transform(None, 0, 0, None, 1, None, None, None) == 0        # no rows
