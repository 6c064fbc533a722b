"""ctypes binding of libvqkv (include/vqkv.h): argument marshalling only.

Every function here forwards to the C ABI; all arithmetic of the hot path
runs in the CUDA kernels of the library.  The library must have been built
(``vector_quantized_bit_gb300._build.build()``): there is no fallback, and a
missing library raises on first use.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

VQKV_MODE_VQ2 = 0
VQKV_MODE_VQ15 = 1
VQKV_MODE_VQ4 = 2
VQKV_MODE_VQ3 = 3
VQKV_MODE_VQ125 = 4
VQKV_ROLE_K = 0
VQKV_ROLE_V = 1
VQKV_DEVERR_SEQ_LEN = 0x1
VQKV_DEVERR_POSITION = 0x2
VQKV_DEVERR_TIMEOUT = 0x4
VQKV_DEVERR_BLOCK = 0x8

STATUS = {0: "VQKV_OK", 1: "VQKV_ERR_INVALID_ARG", 2: "VQKV_ERR_UNSUPPORTED", 3: "VQKV_ERR_WORKSPACE",
          4: "VQKV_ERR_CUDA", 5: "VQKV_ERR_NO_DEVICE"}

EXPORTED = ["vqkv_code_bytes", "vqkv_decode_workspace_bytes", "vqkv_decode_num_splits", "vqkv_decode_kernel_count",
            "vqkv_encode", "vqkv_decode_attn", "vqkv_decode_attn_multi", "vqkv_decode_append",
            "vqkv_decode_attn_static", "vqkv_decode_static_error", "vqkv_encode_paged", "vqkv_decode_attn_paged", "vqkv_test_decode_ring_timeout",
            "vqkv_fp16_decode_workspace_bytes", "vqkv_decode_attn_fp16", "vqkv_smoothing", "vqkv_calib_transform",
            "vqkv_kmeans_workspace_bytes", "vqkv_kmeans", "vqkv_kmeans_seed", "vqkv_kmeans_assign",
            "vqkv_kmeans_update_workspace_bytes", "vqkv_kmeans_update", "vqkv_status_string"]
STATIC_SCRATCH_BYTES = 8 << 20


class VqkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({string(status)})")


class EncodeArgs(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("role", ctypes.c_int32), ("B", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("n_rows", ctypes.c_int32),
                ("cap_len", ctypes.c_int32), ("x", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("s", ctypes.c_void_p), ("codebook", ctypes.c_void_p), ("codes", ctypes.c_void_p),
                ("near_tie_count", ctypes.c_void_p), ("error_flags", ctypes.c_void_p)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("B", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("cap_len", ctypes.c_int32),
                ("max_seq_len", ctypes.c_int32), ("q", ctypes.c_void_p), ("k_codes", ctypes.c_void_p),
                ("v_codes", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p), ("k_codebook", ctypes.c_void_p),
                ("v_codebook", ctypes.c_void_p), ("s", ctypes.c_void_p), ("softmax_scale", ctypes.c_float),
                ("num_splits", ctypes.c_int32), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("out", ctypes.c_void_p)]


class Fp16DecodeArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("cap_len", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("softmax_scale", ctypes.c_float),
                ("num_splits", ctypes.c_int32), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("out", ctypes.c_void_p)]


class Paging(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("max_blocks", ctypes.c_int32), ("block_tokens", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32)]


class DecodeMultiArgs(ctypes.Structure):
    _fields_ = [("decode", DecodeArgs), ("n_queries", ctypes.c_int32)]


class KmeansArgs(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("dim", ctypes.c_int32), ("k", ctypes.c_int32), ("iters", ctypes.c_int32),
                ("points", ctypes.c_void_p), ("uniforms", ctypes.c_void_p), ("centroids", ctypes.c_void_p),
                ("codebook", ctypes.c_void_p), ("seeds", ctypes.c_void_p), ("assign", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class DecodeAppendArgs(ctypes.Structure):
    _fields_ = [("decode", DecodeArgs), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("near_tie_count", ctypes.c_void_p)]


_lib = None


def lib(path: str | None = None) -> ctypes.CDLL:
    """The loaded library (built in-tree); raises if it is missing."""
    global _lib
    if _lib is None:
        path = path or _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libvqkv is not built ({path} missing); run __graft_entry__.build()")
        # make sure the CUDA runtime PyTorch ships is loaded first, so the
        # library binds to the same libcudart (one runtime per process)
        try:
            import torch  # noqa: F401
        except ImportError:
            pass
        L = ctypes.CDLL(path)
        L.vqkv_code_bytes.restype = ctypes.c_size_t
        L.vqkv_code_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32]
        L.vqkv_decode_workspace_bytes.restype = ctypes.c_size_t
        L.vqkv_decode_workspace_bytes.argtypes = [ctypes.POINTER(DecodeArgs)]
        L.vqkv_decode_num_splits.restype = ctypes.c_int32
        L.vqkv_decode_num_splits.argtypes = [ctypes.POINTER(DecodeArgs)]
        L.vqkv_decode_kernel_count.restype = ctypes.c_int32
        L.vqkv_decode_kernel_count.argtypes = [ctypes.POINTER(DecodeArgs)]
        L.vqkv_encode.restype = ctypes.c_int
        L.vqkv_encode.argtypes = [ctypes.POINTER(EncodeArgs), ctypes.c_void_p]
        L.vqkv_decode_attn.restype = ctypes.c_int
        L.vqkv_decode_attn.argtypes = [ctypes.POINTER(DecodeArgs), ctypes.c_void_p]
        L.vqkv_test_decode_ring_timeout.restype = ctypes.c_int
        L.vqkv_test_decode_ring_timeout.argtypes = [ctypes.POINTER(DecodeArgs), ctypes.c_uint32, ctypes.c_void_p]
        L.vqkv_encode_paged.restype = ctypes.c_int
        L.vqkv_encode_paged.argtypes = [ctypes.POINTER(EncodeArgs), ctypes.POINTER(Paging), ctypes.c_void_p]
        L.vqkv_decode_attn_paged.restype = ctypes.c_int
        L.vqkv_decode_attn_paged.argtypes = [ctypes.POINTER(DecodeArgs), ctypes.POINTER(Paging), ctypes.c_void_p]
        L.vqkv_decode_attn_multi.restype = ctypes.c_int
        L.vqkv_decode_attn_multi.argtypes = [ctypes.POINTER(DecodeMultiArgs), ctypes.c_void_p]
        L.vqkv_decode_append.restype = ctypes.c_int
        L.vqkv_decode_append.argtypes = [ctypes.POINTER(DecodeAppendArgs), ctypes.c_void_p]
        L.vqkv_decode_attn_static.restype = ctypes.c_int
        L.vqkv_decode_attn_static.argtypes = [ctypes.POINTER(DecodeArgs), ctypes.c_void_p]
        L.vqkv_decode_static_error.restype = ctypes.c_int
        L.vqkv_decode_static_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
        L.vqkv_fp16_decode_workspace_bytes.restype = ctypes.c_size_t
        L.vqkv_fp16_decode_workspace_bytes.argtypes = [ctypes.POINTER(Fp16DecodeArgs)]
        L.vqkv_decode_attn_fp16.restype = ctypes.c_int
        L.vqkv_decode_attn_fp16.argtypes = [ctypes.POINTER(Fp16DecodeArgs), ctypes.c_void_p]
        L.vqkv_smoothing.restype = ctypes.c_int
        L.vqkv_smoothing.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                                     ctypes.c_void_p]
        L.vqkv_calib_transform.restype = ctypes.c_int
        L.vqkv_calib_transform.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.vqkv_kmeans_workspace_bytes.restype = ctypes.c_size_t
        L.vqkv_kmeans_workspace_bytes.argtypes = [ctypes.POINTER(KmeansArgs)]
        for name in ("vqkv_kmeans", "vqkv_kmeans_seed"):
            getattr(L, name).restype = ctypes.c_int
            getattr(L, name).argtypes = [ctypes.POINTER(KmeansArgs), ctypes.c_void_p]
        L.vqkv_kmeans_assign.restype = ctypes.c_int
        L.vqkv_kmeans_assign.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                         ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.vqkv_kmeans_update_workspace_bytes.restype = ctypes.c_size_t
        L.vqkv_kmeans_update_workspace_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32]
        L.vqkv_kmeans_update.restype = ctypes.c_int
        L.vqkv_kmeans_update.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                         ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_size_t, ctypes.c_void_p]
        L.vqkv_status_string.restype = ctypes.c_char_p
        L.vqkv_status_string.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def string(status: int) -> str:
    return lib().vqkv_status_string(status).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def vqkv_code_bytes(mode: int, cap_len: int) -> int:
    return int(lib().vqkv_code_bytes(mode, cap_len))


def encode_args(mode, role, x, pos, s, codebook, codes, cap_len, near_tie_count=None, error_flags=None):
    B, Hkv, n_rows, D = (x.shape if x is not None else (0, codebook.shape[0], 0, 128))
    return EncodeArgs(mode=mode, role=role, B=B, Hkv=Hkv, head_dim=D, n_rows=n_rows, cap_len=cap_len,
                      x=_ptr(x), pos=_ptr(pos), s=_ptr(s), codebook=_ptr(codebook), codes=_ptr(codes),
                      near_tie_count=_ptr(near_tie_count), error_flags=_ptr(error_flags))


def vqkv_encode(mode, role, x, pos, s, codebook, codes, cap_len, near_tie_count=None, error_flags=None,
                stream=None) -> None:
    """Quantise rows x [B][Hkv][n_rows][128] (fp16, device) into ``codes``.

    pos int32 [B]; s fp32 [Hkv][128] (keys) or None; codebook fp16 [Hkv][E][d_sub];
    codes uint8 [B][Hkv][vqkv_code_bytes(mode, cap_len)].
    """
    a = encode_args(mode, role, x, pos, s, codebook, codes, cap_len, near_tie_count, error_flags)
    st = lib().vqkv_encode(ctypes.byref(a), _stream(stream))
    if st != 0:
        raise VqkvError(st, "vqkv_encode")


def paging(block_table, block_tokens, num_blocks) -> Paging:
    """Block table int32 [B][max_blocks] (device) of a paged cache."""
    return Paging(block_table=_ptr(block_table), max_blocks=block_table.shape[1], block_tokens=block_tokens,
                  num_blocks=num_blocks)


def vqkv_encode_paged(mode, role, x, pos, s, codebook, pool, cap_len, block_table, block_tokens, num_blocks,
                      near_tie_count=None, error_flags=None, stream=None) -> None:
    """vqkv_encode into a paged pool uint8 [num_blocks][Hkv][vqkv_code_bytes(mode, block_tokens)]."""
    a = encode_args(mode, role, x, pos, s, codebook, pool, cap_len, near_tie_count, error_flags)
    pg = paging(block_table, block_tokens, num_blocks)
    st = lib().vqkv_encode_paged(ctypes.byref(a), ctypes.byref(pg), _stream(stream))
    if st != 0:
        raise VqkvError(st, "vqkv_encode_paged")


def vqkv_decode_attn_paged(mode, q, k_pool, v_pool, seq_lens, k_codebook, v_codebook, s, out, workspace, cap_len,
                           max_seq_len, block_table, block_tokens, num_blocks, softmax_scale=0.0, num_splits=0,
                           stream=None) -> None:
    """vqkv_decode_attn over paged pools (see vqkv_encode_paged)."""
    a = decode_args(mode, q, k_pool, v_pool, seq_lens, k_codebook, v_codebook, s, out, workspace, cap_len,
                    max_seq_len, softmax_scale, num_splits)
    pg = paging(block_table, block_tokens, num_blocks)
    st = lib().vqkv_decode_attn_paged(ctypes.byref(a), ctypes.byref(pg), _stream(stream))
    if st != 0:
        raise VqkvError(st, "vqkv_decode_attn_paged")


def decode_args(mode, q, k_codes, v_codes, seq_lens, k_codebook, v_codebook, s, out, workspace, cap_len,
                max_seq_len, softmax_scale=0.0, num_splits=0, workspace_bytes=None):
    B, Hq, D = q.shape
    Hkv = k_codebook.shape[0]
    wb = workspace_bytes if workspace_bytes is not None else (
        workspace.numel() * workspace.element_size() if workspace is not None else 0)
    return DecodeArgs(mode=mode, B=B, Hq=Hq, Hkv=Hkv, head_dim=D, cap_len=cap_len, max_seq_len=max_seq_len,
                      q=_ptr(q), k_codes=_ptr(k_codes), v_codes=_ptr(v_codes), seq_lens=_ptr(seq_lens),
                      k_codebook=_ptr(k_codebook), v_codebook=_ptr(v_codebook), s=_ptr(s),
                      softmax_scale=softmax_scale, num_splits=num_splits, workspace=_ptr(workspace),
                      workspace_bytes=wb, out=_ptr(out))


def vqkv_decode_workspace_bytes(args: DecodeArgs) -> int:
    return int(lib().vqkv_decode_workspace_bytes(ctypes.byref(args)))


def vqkv_decode_num_splits(args: DecodeArgs) -> int:
    return int(lib().vqkv_decode_num_splits(ctypes.byref(args)))


def vqkv_decode_kernel_count(args: DecodeArgs) -> int:
    return int(lib().vqkv_decode_kernel_count(ctypes.byref(args)))


def vqkv_decode_attn(mode, q, k_codes, v_codes, seq_lens, k_codebook, v_codebook, s, out, workspace,
                     cap_len, max_seq_len, softmax_scale=0.0, num_splits=0, stream=None) -> None:
    """O = decode attention of q [B][Hq][128] (fp16) over the packed cache.

    Writes ``out`` (fp16 [B][Hq][128]).  ``workspace``: a device buffer of
    at least vqkv_decode_workspace_bytes bytes; its first word is the sticky
    device error word (zero it before reading it).
    """
    a = decode_args(mode, q, k_codes, v_codes, seq_lens, k_codebook, v_codebook, s, out, workspace, cap_len,
                    max_seq_len, softmax_scale, num_splits)
    st = lib().vqkv_decode_attn(ctypes.byref(a), _stream(stream))
    if st != 0:
        raise VqkvError(st, "vqkv_decode_attn")


def vqkv_decode_attn_multi(mode, q, k_codes, v_codes, seq_lens, k_codebook, v_codebook, s, out, workspace,
                           cap_len, max_seq_len, softmax_scale=0.0, num_splits=0, stream=None) -> None:
    """M queries per sequence: q and out fp16 [B][M][Hq][128]; query m sees
    the cached tokens t <= seq_lens[b] - M + m."""
    B, M, Hq, D = q.shape
    a = DecodeMultiArgs(decode=decode_args(mode, q.view(B, M * Hq, D), k_codes, v_codes, seq_lens, k_codebook,
                                           v_codebook, s, out, workspace, cap_len, max_seq_len, softmax_scale,
                                           num_splits), n_queries=M)
    a.decode.Hq = Hq
    st = lib().vqkv_decode_attn_multi(ctypes.byref(a), _stream(stream))
    if st != 0:
        raise VqkvError(st, "vqkv_decode_attn_multi")


def vqkv_decode_append(mode, q, k_codes, v_codes, seq_lens, k_codebook, v_codebook, s, out, workspace,
                       cap_len, max_seq_len, k_new, v_new, near_tie_count=None, softmax_scale=0.0, num_splits=0,
                       stream=None) -> None:
    """One fused decode step: encodes k_new / v_new (fp16 [B][Hkv][128]) at
    position seq_lens[b] - 1 of the caches, then writes O as vqkv_decode_attn."""
    a = DecodeAppendArgs(decode=decode_args(mode, q, k_codes, v_codes, seq_lens, k_codebook, v_codebook, s, out,
                                            workspace, cap_len, max_seq_len, softmax_scale, num_splits),
                         k_new=_ptr(k_new), v_new=_ptr(v_new), near_tie_count=_ptr(near_tie_count))
    st = lib().vqkv_decode_append(ctypes.byref(a), _stream(stream))
    if st != 0:
        raise VqkvError(st, "vqkv_decode_append")


def vqkv_decode_attn_static(mode, q, k_codes, v_codes, seq_lens, k_codebook, v_codebook, s, out, cap_len,
                            max_seq_len, softmax_scale=0.0, num_splits=0, stream=None) -> None:
    """vqkv_decode_attn without a workspace: for callers that cannot allocate
    device memory.  The split-KV scratch is an 8 MiB array inside the library,
    shared by all calls on a device (calls must not overlap on the GPU)."""
    a = decode_args(mode, q, k_codes, v_codes, seq_lens, k_codebook, v_codebook, s, out, None, cap_len,
                    max_seq_len, softmax_scale, num_splits)
    st = lib().vqkv_decode_attn_static(ctypes.byref(a), _stream(stream))
    if st != 0:
        raise VqkvError(st, "vqkv_decode_attn_static")


def vqkv_decode_static_error(stream=None) -> int:
    """Device error word (VQKV_DEVERR_* bits) of the last
    vqkv_decode_attn_static call on the current device; waits for `stream`."""
    flags = ctypes.c_uint32(0)
    st = lib().vqkv_decode_static_error(ctypes.byref(flags), _stream(stream))
    if st != 0:
        raise VqkvError(st, "vqkv_decode_static_error")
    return int(flags.value)


def decode_workspace(mode, B, Hq, Hkv, cap_len, max_seq_len, num_splits=0, device="cuda", n_queries=1):
    """A zero-filled workspace tensor of the size the decode call needs
    (n_queries > 1: for vqkv_decode_attn_multi)."""
    import torch
    a = DecodeArgs(mode=mode, B=B, Hq=Hq, Hkv=Hkv, head_dim=128, cap_len=cap_len, max_seq_len=max_seq_len,
                   num_splits=num_splits)
    n = vqkv_decode_workspace_bytes(a) * n_queries
    if n == 0:
        raise VqkvError(1, "vqkv_decode_workspace_bytes")
    return torch.zeros((n + 255) // 256 * 256, dtype=torch.uint8, device=device)


def fp16_decode_args(q, k, v, seq_lens, out, workspace, max_seq_len, softmax_scale=0.0, num_splits=0):
    B, Hq, D = q.shape
    Hkv, cap = k.shape[1], k.shape[2]
    wb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return Fp16DecodeArgs(B=B, Hq=Hq, Hkv=Hkv, head_dim=D, cap_len=cap, max_seq_len=max_seq_len, q=_ptr(q),
                          k=_ptr(k), v=_ptr(v), seq_lens=_ptr(seq_lens), softmax_scale=softmax_scale,
                          num_splits=num_splits, workspace=_ptr(workspace), workspace_bytes=wb, out=_ptr(out))


def vqkv_decode_attn_fp16(q, k, v, seq_lens, out, workspace, max_seq_len, softmax_scale=0.0, num_splits=0,
                          stream=None) -> None:
    """Decode attention over a plain fp16 cache k, v [B][Hkv][cap][128] (the
    comparison kernel for the quantised path)."""
    a = fp16_decode_args(q, k, v, seq_lens, out, workspace, max_seq_len, softmax_scale, num_splits)
    st = lib().vqkv_decode_attn_fp16(ctypes.byref(a), _stream(stream))
    if st != 0:
        raise VqkvError(st, "vqkv_decode_attn_fp16")


def fp16_decode_workspace(B, Hq, Hkv, cap_len, max_seq_len, num_splits=0, device="cuda"):
    import torch
    a = Fp16DecodeArgs(B=B, Hq=Hq, Hkv=Hkv, head_dim=128, cap_len=cap_len, max_seq_len=max_seq_len,
                       num_splits=num_splits)
    n = int(lib().vqkv_fp16_decode_workspace_bytes(ctypes.byref(a)))
    if n == 0:
        raise VqkvError(1, "vqkv_fp16_decode_workspace_bytes")
    return torch.zeros((n + 255) // 256 * 256, dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- calibration

def _check(st: int, what: str) -> None:
    if st != 0:
        raise VqkvError(st, what)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return 0
    if t.dtype == torch.float32:
        return 1
    raise TypeError(f"rows must be fp16 or fp32, not {t.dtype}")


def vqkv_smoothing(rows, s, stream=None) -> None:
    """s fp32 [128] <- sqrt(max_t |rows[t]|) (0 -> 1); rows fp16 or fp32 [n][128] (device)."""
    _check(lib().vqkv_smoothing(_ptr(rows), _dtype_code(rows), rows.shape[0], _ptr(s), _stream(stream)),
           "vqkv_smoothing")


def vqkv_calib_transform(x, out, s_pre=None, rotate=False, s_post=None, stream=None) -> None:
    """out fp32 [n][128] <- R(x / s_pre) / s_post (R: the normalised Hadamard rotation if ``rotate``)."""
    _check(lib().vqkv_calib_transform(_ptr(x), _dtype_code(x), x.shape[0], _ptr(s_pre), int(bool(rotate)),
                                      _ptr(s_post), _ptr(out), _stream(stream)), "vqkv_calib_transform")


def kmeans_args(points, uniforms, centroids, iters=0, codebook=None, seeds=None, assign=None, workspace=None):
    n, dim = points.shape
    a = KmeansArgs(n=n, dim=dim, k=centroids.shape[0], iters=iters, points=_ptr(points), uniforms=_ptr(uniforms),
                   centroids=_ptr(centroids), codebook=_ptr(codebook), seeds=_ptr(seeds), assign=_ptr(assign))
    if workspace is not None:
        a.workspace = _ptr(workspace)
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def kmeans_workspace(n, dim, k, device="cuda"):
    """A workspace tensor of the size vqkv_kmeans needs."""
    import torch
    a = KmeansArgs(n=n, dim=dim, k=k)
    nbytes = int(lib().vqkv_kmeans_workspace_bytes(ctypes.byref(a)))
    if nbytes == 0:
        raise VqkvError(1, "vqkv_kmeans_workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def vqkv_kmeans(points, uniforms, centroids, iters, codebook=None, seeds=None, assign=None, workspace=None,
                stream=None) -> None:
    """k-means++ seeding and ``iters`` Lloyd steps: points fp32 [n][dim] -> centroids fp32 [k][dim]
    (codebook fp16 [k][dim], seeds int32 [k], assign int32 [n] optional)."""
    if workspace is None:
        workspace = kmeans_workspace(points.shape[0], points.shape[1], centroids.shape[0], points.device)
    a = kmeans_args(points, uniforms, centroids, iters, codebook, seeds, assign, workspace)
    _check(lib().vqkv_kmeans(ctypes.byref(a), _stream(stream)), "vqkv_kmeans")


def vqkv_kmeans_seed(points, uniforms, centroids, seeds, workspace=None, stream=None) -> None:
    """k-means++ seeding only: seeds int32 [k], centroids fp32 [k][dim] = the picked points."""
    if workspace is None:
        workspace = kmeans_workspace(points.shape[0], points.shape[1], centroids.shape[0], points.device)
    a = kmeans_args(points, uniforms, centroids, 0, None, seeds, None, workspace)
    _check(lib().vqkv_kmeans_seed(ctypes.byref(a), _stream(stream)), "vqkv_kmeans_seed")


def vqkv_kmeans_assign(points, centroids, assign, dist=None, stream=None) -> None:
    """assign int32 [n] (and dist fp32 [n]) <- nearest centroid of each point."""
    n, dim = points.shape
    _check(lib().vqkv_kmeans_assign(_ptr(points), n, dim, _ptr(centroids), centroids.shape[0], _ptr(assign),
                                    _ptr(dist), _stream(stream)), "vqkv_kmeans_assign")


def vqkv_kmeans_update(points, assign, c_in, c_out, workspace=None, stream=None) -> None:
    """c_out <- per-cluster fp64 means of the points (c_in for empty clusters)."""
    import torch
    n, dim = points.shape
    k = c_in.shape[0]
    if workspace is None:
        nbytes = int(lib().vqkv_kmeans_update_workspace_bytes(n, k))
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=c_in.device)
    _check(lib().vqkv_kmeans_update(_ptr(points), n, dim, _ptr(assign), k, _ptr(c_in), _ptr(c_out),
                                    _ptr(workspace), workspace.numel(), _stream(stream)), "vqkv_kmeans_update")
