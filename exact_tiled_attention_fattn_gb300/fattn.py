"""Thin Python binding of libfattn (ctypes): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
checks tensor shapes/dtypes, allocates outputs with PyTorch when the caller
does not pass them, and forwards raw device pointers and the current CUDA
stream. There is no fallback: if ``libfattn.so`` is missing or fails to load,
every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfattn.so")

FATTN_OK = 0
FATTN_ERR_INVALID_ARG = 1
FATTN_ERR_UNSUPPORTED = 2
FATTN_ERR_WORKSPACE = 3
FATTN_ERR_CUDA = 4
FATTN_ERR_TIMEOUT = 5
FATTN_ERR_DEVICE_CHECK = 6
FATTN_BF16 = 0
FATTN_FP32 = 1

# Every entry point declared in include/fattn.h: name -> (restype, argtypes)
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fattn_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _i, _i, _vp]),
    "fattn_fwd_block_sparse": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _i, _vp]),
    "fattn_fwd_masked": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, ctypes.c_longlong,
                              ctypes.c_longlong, _i, _vp]),
    "fattn_fwd_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _f, _f, _f, _vp]),
    "fattn_fwd_paged": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f,
                             _vp]),
    "fattn_bwd_workspace_size": (_sz, [_i, _i, _i]),
    "fattn_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "fattn_decode_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fattn_decode_paged": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _sz,
                                _vp]),
    "fattn_decode_paged_static": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f,
                                       _vp]),
    "fattn_merge_partials": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "fattn_status_string": (ctypes.c_char_p, [_i]),
    "fattn_debug_read_status": (_i, [_vp]),
    "fattn_debug_set_wait_limit": (None, [ctypes.c_ulonglong, _i]),
}

_lib = None


class FattnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} (status {status})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfattn.so and declare its C signatures; raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libfattn.so not found at {path}: build it with __graft_entry__.build() "
                           "or python -m exact_tiled_attention_fattn_gb300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().fattn_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != FATTN_OK:
        raise FattnError(fn, status)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    elif stream.device.index != torch.cuda.current_device():
        raise ValueError(f"stream is on {stream.device} but the current CUDA device is cuda:{torch.cuda.current_device()}")
    return int(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(dt) -> int:
    if dt == torch.bfloat16:
        return FATTN_BF16
    if dt == torch.float32:
        return FATTN_FP32
    raise TypeError(f"unsupported dtype {dt}: bf16 or fp32 only")


def _need_cuda(*ts):
    """All given tensors are contiguous CUDA tensors on one device, the current one
    (the library launches on the current device, so a tensor elsewhere would be an
    invalid address there)."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"all tensors must be on one device (got {dev} and {t.device})")
    if dev is not None and dev.index != torch.cuda.current_device():
        raise ValueError(f"tensors are on {dev} but the current CUDA device is cuda:{torch.cuda.current_device()}; "
                         f"call under torch.cuda.device({dev.index})")


def _expect(t, shape, name, dtype=None):
    """Shape (and dtype) check of an argument the library will read or write in full."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def fwd(q, k, v, causal: bool = False, scale: float | None = None, cu_seqlens=None, max_seqlen: int | None = None,
        out=None, lse=None, want_lse: bool = True, stream=None):
    """Prefill attention. Dense q [B,N,Hq,d] / k,v [B,N,Hkv,d]; varlen q [T,Hq,d] with
    int32 ``cu_seqlens`` [B+1] on the device and ``max_seqlen`` (host int).
    Returns (O, lse): lse is [B,Hq,N] (dense) or [Hq,T] (varlen), fp32, natural log.
    """
    lib = load_library()
    _need_cuda(q, k, v, cu_seqlens, out, lse)
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share a dtype")
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if cu_seqlens is None:
        if q.dim() != 4:
            raise ValueError("dense q must be [B, N, Hq, d]")
        B, N, Hq, _ = q.shape
        if k.dim() != 4:
            raise ValueError("dense k must be [B, N, Hkv, d]")
        Hkv = k.shape[2]
        kv_shape, o_shape = (B, N, Hkv, d), (B, N, Hq, d)
        T = B * N
        lse_shape = (B, Hq, N)
    else:
        if q.dim() != 3 or max_seqlen is None:
            raise ValueError("varlen q must be [T, Hq, d] and max_seqlen must be given")
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
        T, Hq, _ = q.shape
        if k.dim() != 3:
            raise ValueError("varlen k must be [T, Hkv, d]")
        Hkv = k.shape[1]
        kv_shape, o_shape = (T, Hkv, d), (T, Hq, d)
        B = cu_seqlens.numel() - 1
        N = int(max_seqlen)
        lse_shape = (Hq, T)
    _expect(k, kv_shape, "k")
    _expect(v, kv_shape, "v")
    _expect(out, o_shape, "out", q.dtype)
    _expect(lse, lse_shape, "lse", torch.float32)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    st = lib.fattn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d, 1 if causal else 0,
                       float(scale), _ptr(cu_seqlens), T if cu_seqlens is not None else 0, _dtype_code(q.dtype),
                       ctypes.c_void_p(_stream_handle(stream)))
    _check("fattn_fwd", st)
    return out, lse


SPARSE_BLOCK = 128  # FATTN_SPARSE_BLOCK: rows/keys per block-mask entry


def fwd_block_sparse(q, k, v, block_mask, causal: bool = False, scale: float | None = None, out=None, lse=None,
                     want_lse: bool = True, stream=None):
    """Prefill restricted by a block mask. q [B,N,Hq,d], k/v [B,N,Hkv,d] bf16;
    block_mask uint8 [mask_heads, nb, nb] on the device, nb = ceil(N/128), mask_heads 1 or Hq.
    Returns (O, lse [B,Hq,N]); rows that keep no key get O = 0, lse = -inf."""
    lib = load_library()
    _need_cuda(q, k, v, block_mask, out, lse)
    if not (q.dtype == k.dtype == v.dtype == torch.bfloat16):
        raise TypeError("block-sparse prefill takes bf16 q, k, v")
    if block_mask.dtype != torch.uint8 or block_mask.dim() != 3:
        raise TypeError("block_mask must be uint8 [mask_heads, nb, nb]")
    B, N, Hq, d = q.shape
    if k.dim() != 4:
        raise ValueError("k must be [B, N, Hkv, d]")
    _expect(k, (B, N, k.shape[2], d), "k")
    _expect(v, k.shape, "v")
    _expect(out, q.shape, "out", q.dtype)
    _expect(lse, (B, Hq, N), "lse", torch.float32)
    nb = -(-N // SPARSE_BLOCK)
    if block_mask.shape[1] != nb or block_mask.shape[2] != nb:
        raise ValueError(f"block_mask must be [mask_heads, {nb}, {nb}]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    st = lib.fattn_fwd_block_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, k.shape[2], N, d,
                                    1 if causal else 0, float(scale), _ptr(block_mask), block_mask.shape[0],
                                    ctypes.c_void_p(_stream_handle(stream)))
    _check("fattn_fwd_block_sparse", st)
    return out, lse


def fwd_masked(q, k, v, mask, causal: bool = False, scale: float | None = None, out=None, lse=None,
               want_lse: bool = True, stream=None):
    """Prefill with an additive bf16 mask: O = softmax(scale Q K^T + M) V.
    q [B,N,Hq,d], k/v [B,N,Hkv,d] bf16; mask [Bm, Hm, N, L] bf16 on the device with
    Bm in {1, B}, Hm in {1, Hq} (size 1 is shared) and row length L >= N, L a multiple of 8
    (entries past N are ignored). Returns (O, lse [B,Hq,N]); a row with no key gets
    O = 0, lse = -inf."""
    lib = load_library()
    _need_cuda(q, k, v, mask, out, lse)
    if not (q.dtype == k.dtype == v.dtype == mask.dtype == torch.bfloat16):
        raise TypeError("masked prefill takes bf16 q, k, v and mask")
    if q.dim() != 4 or k.dim() != 4 or mask.dim() != 4:
        raise ValueError("q [B,N,Hq,d], k [B,N,Hkv,d] and mask [Bm,Hm,N,L] expected")
    B, N, Hq, d = q.shape
    _expect(k, (B, N, k.shape[2], d), "k")
    _expect(v, k.shape, "v")
    _expect(out, q.shape, "out", q.dtype)
    _expect(lse, (B, Hq, N), "lse", torch.float32)
    Bm, Hm, Nm, L = mask.shape
    if Bm not in (1, B) or Hm not in (1, Hq) or Nm != N or L < N or L % 8:
        raise ValueError(f"mask must be [1 or {B}, 1 or {Hq}, {N}, L] with L >= {N}, L % 8 == 0")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    sb = 0 if Bm == 1 else Hm * N * L
    sh = 0 if Hm == 1 else N * L
    st = lib.fattn_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, k.shape[2], N, d,
                              1 if causal else 0, float(scale), _ptr(mask), sb, sh, L,
                              ctypes.c_void_p(_stream_handle(stream)))
    _check("fattn_fwd_masked", st)
    return out, lse


def fwd_fp8(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float, causal: bool = False,
            scale: float | None = None, out=None, lse=None, want_lse: bool = True, stream=None):
    """FP8 prefill. q8 [B,N,Hq,d], k8/v8 [B,N,Hkv,d] E4M3 (torch.float8_e4m3fn or uint8 codes),
    d = 128; the inputs are descale * e4m3. Returns (O bf16 [B,N,Hq,d], lse [B,Hq,N])."""
    lib = load_library()
    _need_cuda(q8, k8, v8, out, lse)
    for t in (q8, k8, v8):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise TypeError("fp8 prefill takes E4M3 tensors (float8_e4m3fn or uint8 codes)")
    if q8.dim() != 4 or k8.dim() != 4:
        raise ValueError("q [B,N,Hq,d] and k [B,N,Hkv,d] expected")
    B, N, Hq, d = q8.shape
    _expect(k8, (B, N, k8.shape[2], d), "k")
    _expect(v8, k8.shape, "v")
    _expect(out, q8.shape, "out", torch.bfloat16)
    _expect(lse, (B, Hq, N), "lse", torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q8.shape, dtype=torch.bfloat16, device=q8.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q8.device)
    st = lib.fattn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(out), _ptr(lse), B, Hq, k8.shape[2], N, d,
                           1 if causal else 0, float(scale), float(q_descale), float(k_descale), float(v_descale),
                           ctypes.c_void_p(_stream_handle(stream)))
    _check("fattn_fwd_fp8", st)
    return out, lse


def fwd_paged(q, kcache, vcache, block_table, seqlens_k, cu_seqlens_q, max_seqlen_q: int, causal: bool = True,
              scale: float | None = None, out=None, lse=None, want_lse: bool = True, stream=None):
    """Prefill of query chunks against a paged KV cache. q [Tq,Hq,d] bf16 packed by
    int32 ``cu_seqlens_q`` [B+1]; chunk b holds the last Lq_b positions of sequence b's
    ``seqlens_k[b]`` context tokens; kcache/vcache [pages, page_size, Hkv, d] bf16;
    block_table int32 [B, max_pages_per_seq]. Returns (O [Tq,Hq,d], lse [Hq,Tq])."""
    lib = load_library()
    _need_cuda(q, kcache, vcache, block_table, seqlens_k, cu_seqlens_q, out, lse)
    if not (q.dtype == kcache.dtype == vcache.dtype == torch.bfloat16):
        raise TypeError("paged prefill takes bf16 q and caches")
    if block_table.dtype != torch.int32 or seqlens_k.dtype != torch.int32 or cu_seqlens_q.dtype != torch.int32:
        raise TypeError("block_table, seqlens_k and cu_seqlens_q must be int32")
    if q.dim() != 3 or kcache.dim() != 4:
        raise ValueError("q must be [Tq, Hq, d] and kcache [pages, page_size, Hkv, d]")
    Tq, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = kcache.shape
    B = cu_seqlens_q.numel() - 1
    _expect(kcache, (num_pages, page_size, Hkv, d), "kcache")
    _expect(vcache, kcache.shape, "vcache")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError(f"block_table must be [{B}, max_pages_per_seq]")
    _expect(seqlens_k, (B,), "seqlens_k")
    _expect(out, q.shape, "out", q.dtype)
    _expect(lse, (Hq, Tq), "lse", torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    st = lib.fattn_fwd_paged(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(block_table), _ptr(seqlens_k),
                             _ptr(cu_seqlens_q), _ptr(out), _ptr(lse), B, Hq, Hkv, d, page_size,
                             block_table.shape[1], num_pages, Tq, int(max_seqlen_q), 1 if causal else 0,
                             float(scale), ctypes.c_void_p(_stream_handle(stream)))
    _check("fattn_fwd_paged", st)
    return out, lse


def bwd_workspace_size(B: int, Hq: int, N: int) -> int:
    return int(load_library().fattn_bwd_workspace_size(B, Hq, N))


def bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
        workspace=None, stream=None):
    """Attention backward. q, o, dout [B,N,Hq,d], k, v [B,N,Hkv,d] bf16; lse [B,Hq,N] fp32 from
    ``fwd`` on the same inputs. Returns (dq, dk, dv) in the input layouts (bf16)."""
    lib = load_library()
    _need_cuda(q, k, v, o, lse, dout, dq, dk, dv, workspace)
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype == torch.bfloat16):
        raise TypeError("backward takes bf16 q, k, v, o and dout")
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, N, Hq, d] and k [B, N, Hkv, d]")
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    _expect(k, (B, N, Hkv, d), "k")
    _expect(v, k.shape, "v")
    _expect(o, q.shape, "o")
    _expect(dout, q.shape, "dout")
    _expect(lse, (B, Hq, N), "lse", torch.float32)
    _expect(dq, q.shape, "dq", q.dtype)
    _expect(dk, k.shape, "dk", q.dtype)
    _expect(dv, k.shape, "dv", q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = bwd_workspace_size(B, Hq, N)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = lib.fattn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                       B, Hq, Hkv, N, d, 1 if causal else 0, float(scale), _ptr(workspace),
                       workspace.numel() * workspace.element_size(), ctypes.c_void_p(_stream_handle(stream)))
    _check("fattn_bwd", st)
    return dq, dk, dv


def decode_workspace_size(B: int, Hq: int, d: int, num_splits: int) -> int:
    return int(load_library().fattn_decode_workspace_size(B, Hq, d, num_splits))


def choose_num_splits(batch: int, hkv: int, max_pages_per_seq: int, num_sms: int | None = None,
                      chunk_pages: int = 256) -> int:
    """A split count that cuts contexts into ~``chunk_pages``-page chunks and gives at
    least two work items per SM over the batch. Larger chunks amortise each item's
    fixed cost (Q load, pipeline fill, partial write); smaller ones balance better.
    On the 8 x 64k-context decode workload, 256-page chunks (16 splits) read the KV
    cache at 85.6 % of the measured HBM bandwidth against 81 % for 128-page chunks
    (32 splits), 83 % for 12 splits and 63 % for 8."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    by_chunk = -(-max_pages_per_seq // chunk_pages)
    by_fill = -(-2 * num_sms // max(1, batch * hkv))
    return max(1, min(max_pages_per_seq, max(by_chunk, by_fill)))


def decode_paged(q, kcache, vcache, block_table, seqlens, num_splits: int, scale: float | None = None,
                 out=None, lse=None, workspace=None, want_lse: bool = True, stream=None):
    """Split-KV paged decode. q [B,Hq,d] bf16; kcache/vcache [pages, page_size, Hkv, d] bf16;
    block_table int32 [B, max_pages_per_seq]; seqlens int32 [B]. Returns (O [B,Hq,d], lse [B,Hq])."""
    lib = load_library()
    _need_cuda(q, kcache, vcache, block_table, seqlens, out, lse, workspace)
    if block_table.dtype != torch.int32 or seqlens.dtype != torch.int32:
        raise TypeError("block_table and seqlens must be int32")
    if not (q.dtype == kcache.dtype == vcache.dtype == torch.bfloat16):
        raise TypeError("q, kcache and vcache must be bfloat16 (the decode kernels read bf16 only)")
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = kcache.shape
    _expect(kcache, (num_pages, page_size, Hkv, d), "kcache")
    _expect(vcache, kcache.shape, "vcache")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError(f"block_table must be [{B}, max_pages_per_seq]")
    _expect(seqlens, (B,), "seqlens")
    _expect(out, q.shape, "out", q.dtype)
    _expect(lse, (B, Hq), "lse", torch.float32)
    maxp = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = decode_workspace_size(B, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.fattn_decode_paged(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(block_table), _ptr(seqlens), num_splits,
                                _ptr(out), _ptr(lse), B, Hq, Hkv, d, page_size, maxp, num_pages, float(scale),
                                _ptr(workspace), ws_bytes, ctypes.c_void_p(_stream_handle(stream)))
    _check("fattn_decode_paged", st)
    return out, lse


# Size of the fixed device scratch behind decode_paged_static (FATTN_DECODE_STATIC_SCRATCH_BYTES).
DECODE_STATIC_SCRATCH_BYTES = 32 << 20


def decode_paged_static(q, kcache, vcache, block_table, seqlens, num_splits: int, scale: float | None = None,
                        out=None, lse=None, want_lse: bool = True, stream=None):
    """decode_paged for callers that cannot allocate a device workspace: the split
    partials live in the library's fixed 32 MiB device scratch. Calls share that
    scratch, so calls that overlap on the GPU race; the first call on a device
    looks up the scratch address and should come before any stream capture."""
    lib = load_library()
    _need_cuda(q, kcache, vcache, block_table, seqlens, out, lse)
    if block_table.dtype != torch.int32 or seqlens.dtype != torch.int32:
        raise TypeError("block_table and seqlens must be int32")
    if not (q.dtype == kcache.dtype == vcache.dtype == torch.bfloat16):
        raise TypeError("q, kcache and vcache must be bfloat16 (the decode kernels read bf16 only)")
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = kcache.shape
    _expect(kcache, (num_pages, page_size, Hkv, d), "kcache")
    _expect(vcache, kcache.shape, "vcache")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError(f"block_table must be [{B}, max_pages_per_seq]")
    _expect(seqlens, (B,), "seqlens")
    _expect(out, q.shape, "out", q.dtype)
    _expect(lse, (B, Hq), "lse", torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    st = lib.fattn_decode_paged_static(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(block_table), _ptr(seqlens),
                                       num_splits, _ptr(out), _ptr(lse), B, Hq, Hkv, d, page_size,
                                       block_table.shape[1], num_pages, float(scale),
                                       ctypes.c_void_p(_stream_handle(stream)))
    _check("fattn_decode_paged_static", st)
    return out, lse


def split_workspace(workspace, B: int, Hq: int, d: int, num_splits: int):
    """Views (lse_part [B,Hq,S], o_part [B,Hq,S,d]) of a decode workspace (fp32)."""
    rows = B * Hq * num_splits
    lse_bytes = (rows * 4 + 255) // 256 * 256
    flat = workspace.view(torch.uint8)
    lse_part = flat[: rows * 4].view(torch.float32).view(B, Hq, num_splits)
    o_part = flat[lse_bytes: lse_bytes + rows * d * 4].view(torch.float32).view(B, Hq, num_splits, d)
    return lse_part, o_part


def merge_partials(o_part, lse_part, out_dtype=torch.bfloat16, out=None, lse=None, want_lse: bool = True,
                   stream=None):
    """Merge split partials: o_part [B,Hq,S,d] fp32, lse_part [B,Hq,S] fp32 -> (O [B,Hq,d], lse [B,Hq])."""
    lib = load_library()
    _need_cuda(o_part, lse_part, out, lse)
    B, Hq, S, d = o_part.shape
    _expect(lse_part, (B, Hq, S), "lse_part", torch.float32)
    if o_part.dtype != torch.float32:
        raise TypeError("o_part must be float32")
    _expect(out, (B, Hq, d), "out")
    _expect(lse, (B, Hq), "lse", torch.float32)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=out_dtype, device=o_part.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=o_part.device)
    st = lib.fattn_merge_partials(_ptr(o_part), _ptr(lse_part), _ptr(out), _ptr(lse), B, Hq, S, d,
                                  _dtype_code(out.dtype), ctypes.c_void_p(_stream_handle(stream)))
    _check("fattn_merge_partials", st)
    return out, lse


def debug_read_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the device status word."""
    return int(load_library().fattn_debug_read_status(ctypes.c_void_p(_stream_handle(stream))))


def debug_set_wait_limit(limit_ns: int = 0, stall: bool = False) -> None:
    """Test hook: limit of every pipeline wait in later tensor-core launches (0 = the
    default, 2 s); with ``stall`` their softmax / element-wise warps first wait on a
    barrier nothing arrives on, so each launch times out (FATTN_ERR_TIMEOUT) and
    returns without writing its outputs. Reset with debug_set_wait_limit(0, False)."""
    load_library().fattn_debug_set_wait_limit(int(limit_ns), 1 if stall else 0)
