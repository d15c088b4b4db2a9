"""fp64 CPU oracle for MiniMax Sparse Attention (MSA).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code
with the CUDA library and never imports it.

Each function here marshals numpy / CPU torch arrays into ``liboracle.so``
(built from ``oracle.cpp``), whose functions each cite the documentation
passage they follow. Results are fp64 numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None

BF16, FP16, E4M3, F64 = 0, 1, 2, 3


def _load():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build())
        i32p = C.POINTER(C.c_int32)
        f64p = C.POINTER(C.c_double)
        vp = C.c_void_p
        ci = C.c_int
        _lib.oracle_sparse_attention.argtypes = [
            vp, ci, vp, vp, ci, i32p, ci, i32p, i32p, i32p, ci, ci, i32p, ci, ci, ci, ci, ci,
            ci, C.c_double, i32p, ci, f64p, f64p, ci]
        _lib.oracle_proxy_score.argtypes = [
            vp, ci, vp, ci, i32p, i32p, i32p, ci, ci, i32p, ci, ci, ci, ci, ci, ci, ci, ci,
            i32p, ci, f64p, ci]
        _lib.oracle_topk_select.argtypes = [
            C.POINTER(C.c_float), ci, ci, ci, ci, ci, i32p, ci, i32p]
        _lib.oracle_build_union.argtypes = [
            i32p, ci, i32p, i32p, i32p, ci, ci, ci, ci, ci, ci, ci, ci, i32p, i32p,
            C.POINTER(C.c_uint32)]
        _lib.oracle_e4m3_decode.argtypes = [C.POINTER(C.c_uint8), C.c_longlong, f64p]
        _lib.oracle_bf16_decode.argtypes = [C.POINTER(C.c_uint16), C.c_longlong, f64p]
        _lib.oracle_fp16_decode.argtypes = [C.POINTER(C.c_uint16), C.c_longlong, f64p]
        _lib.oracle_e2m1_decode.argtypes = [C.POINTER(C.c_uint8), C.c_longlong, f64p]
        _lib.oracle_nvfp4_dequant.argtypes = [
            C.POINTER(C.c_uint8), C.c_longlong, ci, ci, ci, C.c_double, C.c_double, f64p, f64p]
        for f in ("oracle_sparse_attention", "oracle_proxy_score", "oracle_topk_select",
                  "oracle_build_union"):
            getattr(_lib, f).restype = ci
    return _lib


def _threads(threads):
    return int(threads) if threads else (os.cpu_count() or 1)


def _raw(x):
    """Contiguous numpy view of the raw element bits of a CPU tensor/array.

    Returns (array, dtype code). bf16 and fp16 are passed as their 16-bit
    patterns, E4M3 as bytes; the oracle decodes them itself. fp64 numpy
    arrays (already decoded values, e.g. from ``nvfp4_dequant``) pass as is.
    """
    if isinstance(x, np.ndarray) and x.dtype == np.float64:
        return np.ascontiguousarray(x), F64
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), BF16
        if x.dtype == torch.float16:
            return x.view(torch.int16).numpy().view(np.uint16), FP16
        if x.dtype == torch.float8_e4m3fn:
            return x.view(torch.uint8).numpy(), E4M3
        if x.dtype == torch.uint8:
            return x.numpy(), E4M3
        raise TypeError(f"unsupported oracle input dtype {x.dtype}")
    raise TypeError("oracle inputs are torch CPU tensors")


def _i32(x):
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(C.POINTER(ctype))


def sparse_attention(q, k, v, q2k_indices, cu_seqlens_q, cu_seqlens_k=None, *, causal=False,
                     softmax_scale=None, page_table=None, seqused_k=None, num_pages=None,
                     rows=None, threads=None):
    """Plain per-query MSA forward (fp64). Returns (out[n_rows,Hq,d], lse[n_rows,Hq]).

    Follows "flashinfer.msa_ops.msa_sparse_attention" (Parameters; Returns).
    ``rows`` selects packed query rows (default: all). ``softmax_scale`` defaults
    to head_dim**-0.5 evaluated in fp64.
    """
    lib = _load()
    qa, qdt = _raw(q)
    ka, kdt = _raw(k)
    va, vdt = _raw(v)
    assert kdt == vdt
    total_q, Hq, d = q.shape
    q2k = _i32(q2k_indices)
    Hkv, tq2, topk = q2k.shape
    assert tq2 == total_q
    cu_q = _i32(cu_seqlens_q)
    batch = cu_q.shape[0] - 1
    cu_k = _i32(cu_seqlens_k)
    pt = _i32(page_table)
    su = _i32(seqused_k)
    if pt is not None:
        max_pages = pt.shape[1]
        npages = int(num_pages if num_pages is not None else k.shape[0])
    else:
        max_pages, npages = 0, 0
    rws = _i32(rows) if rows is not None else None
    n_rows = total_q if rws is None else rws.shape[0]
    scale = float(softmax_scale) if softmax_scale is not None else d ** -0.5
    out = np.zeros((n_rows, Hq, d), dtype=np.float64)
    lse = np.zeros((n_rows, Hq), dtype=np.float64)
    rc = lib.oracle_sparse_attention(
        qa.ctypes.data, qdt, ka.ctypes.data, va.ctypes.data, kdt, _ptr(q2k, C.c_int32), topk,
        _ptr(cu_q, C.c_int32), _ptr(cu_k, C.c_int32), _ptr(pt, C.c_int32), max_pages, npages,
        _ptr(su, C.c_int32), batch, total_q, Hq, Hkv, d, int(bool(causal)), scale,
        _ptr(rws, C.c_int32), n_rows, _ptr(out, C.c_double), _ptr(lse, C.c_double),
        _threads(threads))
    if rc != 0:
        raise ValueError(f"oracle_sparse_attention rejected its arguments ({rc})")
    return out, lse


def proxy_score(q, k, cu_seqlens_q, cu_seqlens_k=None, *, page_table=None, seqused_k=None,
                num_pages=None, causal=True, max_k_tiles=None, reduce_heads=False, rows=None,
                threads=None):
    """Per-128-block max of unscaled, causally masked q.k (fp64).

    Follows "flashinfer.msa_ops.msa_proxy_score". Returns
    (Hq or 1, max_k_tiles, n_rows) fp64 with -inf for blocks with no visible key.
    """
    lib = _load()
    qa, qdt = _raw(q)
    ka, kdt = _raw(k)
    total_q, Hq, d = q.shape
    Hkv = k.shape[1]
    cu_q = _i32(cu_seqlens_q)
    batch = cu_q.shape[0] - 1
    cu_k = _i32(cu_seqlens_k)
    pt = _i32(page_table)
    su = _i32(seqused_k)
    if pt is not None:
        max_pages = pt.shape[1]
        npages = int(num_pages if num_pages is not None else k.shape[0])
        lens = su
    else:
        max_pages, npages = 0, 0
        lens = np.diff(cu_k)
    if max_k_tiles is None:
        max_k_tiles = int(max(1, max((int(x) + 127) // 128 for x in lens)))
    rws = _i32(rows) if rows is not None else None
    n_rows = total_q if rws is None else rws.shape[0]
    out = np.zeros(((1 if reduce_heads else Hq), max_k_tiles, n_rows), dtype=np.float64)
    rc = lib.oracle_proxy_score(
        qa.ctypes.data, qdt, ka.ctypes.data, kdt, _ptr(cu_q, C.c_int32), _ptr(cu_k, C.c_int32),
        _ptr(pt, C.c_int32), max_pages, npages, _ptr(su, C.c_int32), batch, total_q, Hq, Hkv, d,
        max_k_tiles, int(bool(causal)), int(bool(reduce_heads)), _ptr(rws, C.c_int32), n_rows,
        _ptr(out, C.c_double), _threads(threads))
    if rc != 0:
        raise ValueError(f"oracle_proxy_score rejected its arguments ({rc})")
    return out


def topk_select(scores, topk, num_kv_heads_out, rows=None):
    """Top-k block ids per query from fp32 scores (Hs, max_k_tiles, total_q).

    Ties go to the lower block id; the result is ascending and -1 padded;
    -inf and NaN are never selected. Returns int32 (num_kv_heads_out, n_rows, topk).
    """
    lib = _load()
    try:
        import torch
        if isinstance(scores, torch.Tensor):
            scores = scores.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float32))
    Hs, T, total_q = s.shape
    rws = _i32(rows) if rows is not None else None
    n_rows = total_q if rws is None else rws.shape[0]
    out = np.zeros((num_kv_heads_out, n_rows, topk), dtype=np.int32)
    rc = lib.oracle_topk_select(_ptr(s, C.c_float), Hs, T, total_q, int(topk),
                                int(num_kv_heads_out), _ptr(rws, C.c_int32), n_rows,
                                _ptr(out, C.c_int32))
    if rc != 0:
        raise ValueError(f"oracle_topk_select rejected its arguments ({rc})")
    return out


def num_tiles(cu_seqlens_q, tile_tokens):
    cu = _i32(cu_seqlens_q)
    return int(sum((int(cu[b + 1] - cu[b]) + tile_tokens - 1) // tile_tokens
                   for b in range(cu.shape[0] - 1)))


def build_union(q2k_indices, cu_seqlens_q, cu_seqlens_k=None, *, seqused_k=None, max_pages=0,
                causal=True, tile_tokens=16, cap=None):
    """Per-tile union metadata in the canonical format (see ``oracle.cpp``).

    Returns (union_len[Hkv, T], union_blocks[Hkv, T, cap], member[Hkv, T, W, cap/32]).
    """
    lib = _load()
    q2k = _i32(q2k_indices)
    Hkv, total_q, topk = q2k.shape
    cu_q = _i32(cu_seqlens_q)
    batch = cu_q.shape[0] - 1
    cu_k = _i32(cu_seqlens_k)
    su = _i32(seqused_k)
    if cap is None:
        cap = tile_tokens * topk
    words = (cap + 31) // 32
    T = num_tiles(cu_q, tile_tokens)
    ulen = np.zeros((Hkv, T), dtype=np.int32)
    ublk = np.zeros((Hkv, T, cap), dtype=np.int32)
    mem = np.zeros((Hkv, T, tile_tokens, words), dtype=np.uint32)
    rc = lib.oracle_build_union(_ptr(q2k, C.c_int32), topk, _ptr(cu_q, C.c_int32),
                                _ptr(cu_k, C.c_int32), _ptr(su, C.c_int32), int(max_pages), batch,
                                total_q, Hkv, int(bool(causal)), tile_tokens, cap, T,
                                _ptr(ulen, C.c_int32), _ptr(ublk, C.c_int32),
                                _ptr(mem, C.c_uint32))
    if rc != 0:
        raise ValueError(f"oracle_build_union rejected its arguments ({rc})")
    return ulen, ublk, mem


def e4m3_decode(codes):
    lib = _load()
    a = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.zeros(a.shape, dtype=np.float64)
    lib.oracle_e4m3_decode(_ptr(a, C.c_uint8), a.size, _ptr(out, C.c_double))
    return out


def bf16_decode(bits):
    lib = _load()
    a = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.zeros(a.shape, dtype=np.float64)
    lib.oracle_bf16_decode(_ptr(a, C.c_uint16), a.size, _ptr(out, C.c_double))
    return out


def fp16_decode(bits):
    """Values of IEEE binary16 bit patterns, decoded from the bits in fp64."""
    lib = _load()
    a = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.zeros(a.shape, dtype=np.float64)
    lib.oracle_fp16_decode(_ptr(a, C.c_uint16), a.size, _ptr(out, C.c_double))
    return out


def e2m1_decode(codes):
    """Values of E2M1 codes (the low nibble of each byte)."""
    lib = _load()
    a = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.zeros(a.shape, dtype=np.float64)
    lib.oracle_e2m1_decode(_ptr(a, C.c_uint8), a.size, _ptr(out, C.c_double))
    return out


def nvfp4_dequant(pool, num_kv_heads, head_dim=128, k_global_scale=1.0, v_global_scale=1.0):
    """fp64 K and V, (num_pages, Hkv, 128, d) each, of a planar NVFP4 page pool.

    ``pool`` is (num_pages, page_stride) bytes; each page holds [K data | K
    scales | V data | V scales] as "msa_sparse_attention" (k, k_scale, v_scale,
    k_global_scale, v_global_scale) describes; see oracle_nvfp4_dequant for
    the nibble and scale-order readings.
    """
    lib = _load()
    try:
        import torch
        if isinstance(pool, torch.Tensor):
            pool = pool.detach().cpu().contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(np.asarray(pool, dtype=np.uint8))
    npg, stride = a.shape
    kk = np.zeros((npg, num_kv_heads, 128, head_dim), dtype=np.float64)
    vv = np.zeros_like(kk)
    lib.oracle_nvfp4_dequant(_ptr(a, C.c_uint8), stride, npg, num_kv_heads, head_dim,
                             float(k_global_scale), float(v_global_scale),
                             _ptr(kk, C.c_double), _ptr(vv, C.c_double))
    return kk, vv
