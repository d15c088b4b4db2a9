"""MiniMax Sparse Attention (MSA) forward on GB300 (sm_103a).

Thin Python binding over the C ABI of ``libmsa.so`` (declared in
``include/msa.h``). Every function here only marshals torch CUDA tensors into
raw device pointers and sizes and calls the C entry point of the same name;
all computation happens in the library's CUDA kernels. There is no fallback:
if the library has not been built, every call raises.

Convenience defaults that need information the C ABI takes explicitly
(``max_seqlen_q``, ``max_k_tiles``) are derived here from ``cu_seqlens`` /
``seqused_k`` when omitted. That derivation READS THE DEVICE (except
``max_seqlen_q`` of a single sequence, which is ``total_q``): a
device-to-host copy that synchronises the host with the GPU and launches
two small torch kernels on every such call. Code that must not synchronise
(CUDA-graph capture, pipelined serving loops) passes them explicitly; the C
ABI itself never synchronises. Output and workspace buffers are allocated
with torch when not supplied.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

MSA_OK, MSA_INVALID_ARG, MSA_UNSUPPORTED, MSA_WORKSPACE_TOO_SMALL, MSA_CUDA_ERROR = range(5)
MSA_BF16, MSA_FP16, MSA_FP8_E4M3 = 0, 1, 2

_lib = None


class MSAError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def build(force: bool = False) -> str:
    """Compile libmsa.so in-tree with nvcc (sm_103a)."""
    from . import buildlib as _b
    return _b.build(force=force)


def lib():
    """The loaded C library. Raises if it was never built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libmsa.so is not built ({LIB_PATH}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = C.CDLL(LIB_PATH)
        vp, i32, f32, sz = C.c_void_p, C.c_int, C.c_float, C.c_size_t
        L.msa_status_string.restype = C.c_char_p
        L.msa_status_string.argtypes = [i32]
        L.msa_sparse_attention_workspace_size.restype = sz
        L.msa_sparse_attention_workspace_size.argtypes = [i32] * 8
        L.msa_sparse_attention_workspace_size_kv.restype = sz
        L.msa_sparse_attention_workspace_size_kv.argtypes = [i32] * 10
        L.msa_sparse_attention_nvfp4_workspace_size.restype = sz
        L.msa_sparse_attention_nvfp4_workspace_size.argtypes = [i32] * 8
        L.msa_sparse_attention_fwd.restype = i32
        L.msa_sparse_attention_fwd.argtypes = [
            vp, i32, vp, vp, i32, vp, i32, vp, vp, vp, i32, i32, vp, i32, i32, i32, i32, i32,
            i32, i32, i32, f32, vp, vp, vp, sz, vp]
        L.msa_sparse_attention_prepare.restype = i32
        L.msa_sparse_attention_prepare.argtypes = [
            vp, i32, vp, vp, i32, vp, i32, vp, vp, vp, i32, i32, vp, i32, i32, i32, i32, i32,
            i32, i32, i32, f32, vp, vp, vp, sz, C.POINTER(vp)]
        L.msa_sparse_attention_run.restype = i32
        L.msa_sparse_attention_run.argtypes = [vp, vp]
        L.msa_sparse_attention_plan_free.restype = None
        L.msa_sparse_attention_plan_free.argtypes = [vp]
        fp4 = [vp, i32, vp, vp, vp, vp, C.c_longlong, f32, f32, vp, i32, vp, vp, i32, i32, vp, i32,
               i32, i32, i32, i32, i32, f32, vp, vp, vp, sz]
        L.msa_sparse_attention_nvfp4_paged.restype = i32
        L.msa_sparse_attention_nvfp4_paged.argtypes = fp4 + [vp]
        L.msa_sparse_attention_nvfp4_prepare.restype = i32
        L.msa_sparse_attention_nvfp4_prepare.argtypes = fp4 + [C.POINTER(vp)]
        L.msa_proxy_score.restype = i32
        L.msa_proxy_score.argtypes = [
            vp, i32, vp, i32, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
            i32, vp, vp]
        L.msa_topk_select.restype = i32
        L.msa_topk_select.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp]
        L.msa_build_union.restype = i32
        L.msa_build_union.argtypes = [
            vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp]
        L.msa_union_tile_tokens.restype = i32
        L.msa_union_tile_tokens.argtypes = [i32, i32]
        L.msa_build_union_block_members.restype = i32
        L.msa_build_union_block_members.argtypes = [
            vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.msa_prefill_tile_tokens.restype = i32
        L.msa_prefill_tile_tokens.argtypes = [i32] * 7
        L.msa_set_prefill_route.restype = i32
        L.msa_set_prefill_route.argtypes = [i32]
        L.msa_sparse_decode_noalloc.restype = i32
        L.msa_sparse_decode_noalloc.argtypes = [
            vp, vp, vp, vp, i32, vp, vp, i32, i32, vp, i32, i32, i32, i32, i32, i32, i32, f32,
            vp, vp, vp]
        L.msa_sparse_decode_noalloc_scratch_limit.restype = sz
        L.msa_sparse_decode_noalloc_scratch_limit.argtypes = []
        L.msa_set_timing_events.restype = i32
        L.msa_set_timing_events.argtypes = [C.POINTER(C.c_void_p), i32]
        L.msa_selftest_wait_timeout.restype = i32
        L.msa_selftest_wait_timeout.argtypes = [C.c_uint, vp]
        L.msa_read_device_fault.restype = i32
        L.msa_read_device_fault.argtypes = [C.POINTER(C.c_uint), vp]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().msa_status_string(int(status)).decode()


def _check(fn, status):
    if status != MSA_OK:
        raise MSAError(fn, status)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MSA_BF16
    if t.dtype == torch.float16:
        return MSA_FP16
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return MSA_FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _cuda_contig(name, t, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _max_len(cu: torch.Tensor) -> int:
    return int((cu[1:] - cu[:-1]).max().item()) if cu.numel() > 1 else 0


def _q_bound(cu_q: torch.Tensor, total_q: int) -> int:
    """A bound on every query run: total_q itself for one sequence (no device
    read), else the longest run read back from the device (a host sync)."""
    return total_q if cu_q.numel() == 2 else _max_len(cu_q)


def msa_union_tile_tokens(num_qo_heads: int, num_kv_heads: int) -> int:
    return int(lib().msa_union_tile_tokens(num_qo_heads, num_kv_heads))


def msa_prefill_tile_tokens(batch, total_q, num_qo_heads, num_kv_heads, topk, max_seqlen_q,
                            kv_dtype=MSA_BF16) -> int:
    """Tokens per query tile of the attention kernel the forward picks; see
    include/msa.h. ``kv_dtype`` is a torch dtype or an MSA_* code."""
    code = kv_dtype if isinstance(kv_dtype, int) else _dtype_code(torch.empty(0, dtype=kv_dtype))
    return int(lib().msa_prefill_tile_tokens(batch, total_q, num_qo_heads, num_kv_heads, topk,
                                             max_seqlen_q, code))


def msa_set_prefill_route(route: int) -> None:
    """0: pick the attention kernel by shape (default); 1: always the
    union-tile kernel; 2: the swapped-orientation kernel wherever it applies.
    Process-wide (include/msa.h)."""
    _check("msa_set_prefill_route", lib().msa_set_prefill_route(int(route)))


def msa_sparse_attention_workspace_size(batch, total_q, num_qo_heads, num_kv_heads, head_dim,
                                        topk, max_seqlen_q, paged) -> int:
    return int(lib().msa_sparse_attention_workspace_size(
        batch, total_q, num_qo_heads, num_kv_heads, head_dim, topk, max_seqlen_q, int(bool(paged))))


def msa_sparse_attention_workspace_size_kv(batch, total_q, num_qo_heads, num_kv_heads, head_dim,
                                           topk, max_seqlen_q, paged, kv_dtype, total_k) -> int:
    """``kv_dtype`` is a torch dtype or an MSA_* code."""
    code = kv_dtype if isinstance(kv_dtype, int) else _dtype_code(torch.empty(0, dtype=kv_dtype))
    return int(lib().msa_sparse_attention_workspace_size_kv(
        batch, total_q, num_qo_heads, num_kv_heads, head_dim, topk, max_seqlen_q, int(bool(paged)),
        code, total_k))


def msa_sparse_attention_nvfp4_workspace_size(batch, total_q, num_qo_heads, num_kv_heads,
                                              head_dim, topk, max_seqlen_q, max_pages) -> int:
    return int(lib().msa_sparse_attention_nvfp4_workspace_size(
        batch, total_q, num_qo_heads, num_kv_heads, head_dim, topk, max_seqlen_q, max_pages))


def msa_sparse_attention_fwd(q, k, v, q2k_indices, cu_seqlens_q, cu_seqlens_k=None, *,
                             causal=False, softmax_scale=None, page_table=None, seqused_k=None,
                             max_seqlen_q=None, return_softmax_lse=False, out=None, lse=None,
                             workspace=None, stream=None):
    """Sparse attention forward; see ``msa_sparse_attention_fwd`` in include/msa.h.

    Returns ``out`` or ``(out, lse)``. With ``max_seqlen_q=None`` and more
    than one sequence the longest query run is read back from
    ``cu_seqlens_q`` on the device, which synchronises the host; pass it to
    keep the call asynchronous (one sequence needs no read: its run is
    ``total_q``).
    """
    L = lib()
    args, out, lse, workspace = _forward_args(
        q, k, v, q2k_indices, cu_seqlens_q, cu_seqlens_k, causal, softmax_scale, page_table,
        seqused_k, max_seqlen_q, return_softmax_lse, out, lse, workspace)
    st = L.msa_sparse_attention_fwd(*args, _stream(stream))
    _check("msa_sparse_attention_fwd", st)
    return (out, lse) if lse is not None else out


def _forward_args(q, k, v, q2k_indices, cu_seqlens_q, cu_seqlens_k, causal, softmax_scale,
                  page_table, seqused_k, max_seqlen_q, return_softmax_lse, out, lse, workspace):
    """The C arguments of a forward (all but the stream), allocating out, lse
    and workspace when not given."""
    _cuda_contig("q", q)
    _cuda_contig("k", k)
    _cuda_contig("v", v)
    _cuda_contig("q2k_indices", q2k_indices, torch.int32)
    _cuda_contig("cu_seqlens_q", cu_seqlens_q, torch.int32)
    _cuda_contig("cu_seqlens_k", cu_seqlens_k, torch.int32)
    _cuda_contig("page_table", page_table, torch.int32)
    _cuda_contig("seqused_k", seqused_k, torch.int32)
    total_q, hq, d = q.shape
    hkv = k.shape[1]
    topk = q2k_indices.shape[2]
    batch = cu_seqlens_q.shape[0] - 1
    paged = page_table is not None
    if max_seqlen_q is None:
        max_seqlen_q = _q_bound(cu_seqlens_q, total_q)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_softmax_lse:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = msa_sparse_attention_workspace_size_kv(
            batch, total_q, hq, hkv, d, topk, max(1, max_seqlen_q), paged, _dtype_code(k),
            page_table.shape[1] if paged else k.shape[0])
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    args = (_p(q), _dtype_code(q), _p(k), _p(v), _dtype_code(k), _p(q2k_indices), topk,
            _p(cu_seqlens_q), _p(cu_seqlens_k), _p(page_table),
            page_table.shape[1] if paged else 0, k.shape[0] if paged else 0, _p(seqused_k),
            batch, total_q, 0 if paged else k.shape[0], hq, hkv, d, int(max_seqlen_q),
            int(bool(causal)), float(softmax_scale) if softmax_scale is not None else 0.0,
            _p(out), _p(lse), _p(workspace), workspace.numel())
    return args, out, lse, workspace


class SparseAttentionRunner:
    """A forward prepared once (``msa_sparse_attention_prepare``) and launched
    by ``run()`` (``msa_sparse_attention_run``): no allocation, no host
    synchronisation and no argument processing per launch; capturable into a
    CUDA graph. The tensors given here are bound by address: refill them in
    place between runs. ``out`` and ``lse`` hold the results."""

    def __init__(self, q, k, v, q2k_indices, cu_seqlens_q, cu_seqlens_k=None, *, causal=False,
                 softmax_scale=None, page_table=None, seqused_k=None, max_seqlen_q=None,
                 return_softmax_lse=False, out=None, lse=None, workspace=None):
        L = lib()
        args, self.out, self.lse, self.workspace = _forward_args(
            q, k, v, q2k_indices, cu_seqlens_q, cu_seqlens_k, causal, softmax_scale, page_table,
            seqused_k, max_seqlen_q, return_softmax_lse, out, lse, workspace)
        # Keep every bound buffer alive as long as the plan.
        self._bound = (q, k, v, q2k_indices, cu_seqlens_q, cu_seqlens_k, page_table, seqused_k)
        plan = C.c_void_p()
        _check("msa_sparse_attention_prepare",
               L.msa_sparse_attention_prepare(*args, C.byref(plan)))
        self._plan = plan
        self._lib = L

    def run(self, stream=None):
        _check("msa_sparse_attention_run",
               self._lib.msa_sparse_attention_run(self._plan, _stream(stream)))
        return (self.out, self.lse) if self.lse is not None else self.out

    def close(self):
        if getattr(self, "_plan", None):
            self._lib.msa_sparse_attention_plan_free(self._plan)
            self._plan = None

    def __del__(self):
        self.close()


def nvfp4_views(kv_pool: torch.Tensor, num_kv_heads: int, head_dim: int = 128):
    """(k, k_scale, v, v_scale) strided uint8 views of a planar NVFP4 page pool
    (num_pages, page_stride) laid out [K data | K scales | V data | V scales]
    per page: (num_pages, Hkv, 128, d/2) codes and (num_pages, Hkv, 128, d/16)
    scales ("msa_sparse_attention": k, k_scale, v_scale)."""
    npg, stride = kv_pool.shape
    data, sc = num_kv_heads * 128 * head_dim // 2, num_kv_heads * 128 * head_dim // 16
    flat = kv_pool.reshape(-1)

    def view(off, inner):
        return flat.as_strided((npg, num_kv_heads, 128, inner),
                               (stride, 128 * inner, inner, 1), off)
    return (view(0, head_dim // 2), view(data, head_dim // 16), view(data + sc, head_dim // 2),
            view(2 * data + sc, head_dim // 16))


def _fp4_args(q, k, k_scale, v, v_scale, q2k_indices, cu_seqlens_q, page_table, seqused_k,
              k_global_scale, v_global_scale, max_seqlen_q, softmax_scale, return_softmax_lse,
              out, lse, workspace):
    _cuda_contig("q", q)
    for name, t in (("q2k_indices", q2k_indices), ("cu_seqlens_q", cu_seqlens_q),
                    ("page_table", page_table), ("seqused_k", seqused_k)):
        _cuda_contig(name, t, torch.int32)
    views = (k, k_scale, v, v_scale)
    for name, t in zip(("k", "k_scale", "v", "v_scale"), views):
        if not t.is_cuda or t.dtype not in (torch.uint8, torch.float8_e4m3fn) or t.dim() != 4:
            raise ValueError(f"{name} must be a 4-d uint8 CUDA view of the page pool")
        inner = t.shape[3]
        if t.stride()[1:] != (128 * inner, inner, 1):
            raise ValueError(f"{name}: (head, token, byte) must be contiguous within a page")
    stride = k.stride(0)
    if any(t.stride(0) != stride for t in views):
        raise ValueError("k, k_scale, v and v_scale must share one page stride")
    total_q, hq, d = q.shape
    hkv, topk = k.shape[1], q2k_indices.shape[2]
    batch = cu_seqlens_q.shape[0] - 1
    if max_seqlen_q is None:
        max_seqlen_q = _q_bound(cu_seqlens_q, total_q)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_softmax_lse:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = msa_sparse_attention_nvfp4_workspace_size(batch, total_q, hq, hkv, d, topk,
                                                         max(1, max_seqlen_q), page_table.shape[1])
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    args = (_p(q), _dtype_code(q), _p(k), _p(k_scale), _p(v), _p(v_scale), stride,
            float(k_global_scale), float(v_global_scale), _p(q2k_indices), topk, _p(cu_seqlens_q),
            _p(page_table), page_table.shape[1], k.shape[0], _p(seqused_k), batch, total_q, hq,
            hkv, d, int(max_seqlen_q),
            float(softmax_scale) if softmax_scale is not None else 0.0, _p(out), _p(lse),
            _p(workspace), workspace.numel())
    return args, out, lse, workspace


def msa_sparse_attention_nvfp4_paged(q, k, k_scale, v, v_scale, q2k_indices, cu_seqlens_q, *,
                                     page_table, seqused_k, k_global_scale, v_global_scale,
                                     max_seqlen_q=None, softmax_scale=None,
                                     return_softmax_lse=False, out=None, lse=None,
                                     workspace=None, stream=None):
    """Packed NVFP4 paged forward; see ``msa_sparse_attention_nvfp4_paged`` in
    include/msa.h. ``k`` .. ``v_scale`` are the views ``nvfp4_views`` returns.
    Returns ``out`` or ``(out, lse)``."""
    L = lib()
    args, out, lse, _ = _fp4_args(q, k, k_scale, v, v_scale, q2k_indices, cu_seqlens_q,
                                  page_table, seqused_k, k_global_scale, v_global_scale,
                                  max_seqlen_q, softmax_scale, return_softmax_lse, out, lse,
                                  workspace)
    _check("msa_sparse_attention_nvfp4_paged",
           L.msa_sparse_attention_nvfp4_paged(*args, _stream(stream)))
    return (out, lse) if lse is not None else out


class Nvfp4AttentionRunner(SparseAttentionRunner):
    """The packed NVFP4 paged forward prepared once
    (``msa_sparse_attention_nvfp4_prepare``) and launched by ``run()``."""

    def __init__(self, q, k, k_scale, v, v_scale, q2k_indices, cu_seqlens_q, *, page_table,
                 seqused_k, k_global_scale, v_global_scale, max_seqlen_q=None,
                 softmax_scale=None, return_softmax_lse=False, out=None, lse=None,
                 workspace=None):
        L = lib()
        args, self.out, self.lse, self.workspace = _fp4_args(
            q, k, k_scale, v, v_scale, q2k_indices, cu_seqlens_q, page_table, seqused_k,
            k_global_scale, v_global_scale, max_seqlen_q, softmax_scale, return_softmax_lse,
            out, lse, workspace)
        self._bound = (q, k, k_scale, v, v_scale, q2k_indices, cu_seqlens_q, page_table,
                       seqused_k)
        plan = C.c_void_p()
        _check("msa_sparse_attention_nvfp4_prepare",
               L.msa_sparse_attention_nvfp4_prepare(*args, C.byref(plan)))
        self._plan = plan
        self._lib = L


def msa_proxy_score(q, k, cu_seqlens_q, cu_seqlens_k=None, *, causal=True, max_k_tiles=None,
                    reduce_heads=False, output=None, max_seqlen_q=None, page_table=None,
                    seqused_k=None, stream=None):
    """Per-block max of unscaled causal q.k; see ``msa_proxy_score`` in include/msa.h.

    Flat K (Tk, Hkv, 128) with cu_seqlens_k, or a paged pool
    (num_pages, Hkv, 128, 128) with page_table and seqused_k.
    """
    L = lib()
    _cuda_contig("q", q)
    _cuda_contig("k", k)
    _cuda_contig("cu_seqlens_q", cu_seqlens_q, torch.int32)
    _cuda_contig("cu_seqlens_k", cu_seqlens_k, torch.int32)
    _cuda_contig("page_table", page_table, torch.int32)
    _cuda_contig("seqused_k", seqused_k, torch.int32)
    total_q, hq, d = q.shape
    hkv = k.shape[1]
    batch = cu_seqlens_q.shape[0] - 1
    if max_k_tiles is None:
        longest = (int(seqused_k.max().item()) if page_table is not None
                   else _max_len(cu_seqlens_k))
        max_k_tiles = max(1, (longest + 127) // 128)
    if max_seqlen_q is None:
        max_seqlen_q = 0
    if output is None:
        output = torch.empty(((1 if reduce_heads else hq), max_k_tiles, total_q),
                             dtype=torch.float32, device=q.device)
    _cuda_contig("output", output, torch.float32)
    max_pages = page_table.shape[1] if page_table is not None else 0
    st = L.msa_proxy_score(_p(q), _dtype_code(q), _p(k), _dtype_code(k), _p(cu_seqlens_q),
                           _p(cu_seqlens_k), _p(page_table), max_pages, _p(seqused_k), batch,
                           total_q, k.shape[0], hq, hkv, d, int(max_seqlen_q), int(max_k_tiles),
                           int(bool(causal)), int(bool(reduce_heads)), _p(output), _stream(stream))
    _check("msa_proxy_score", st)
    return output


def msa_topk_select(scores, topk, num_kv_heads_out, *, out=None, stream=None):
    """Top-k block ids per query (ascending, -1 padded); see include/msa.h."""
    L = lib()
    _cuda_contig("scores", scores, torch.float32)
    hs, T, total_q = scores.shape
    if out is None:
        out = torch.empty((num_kv_heads_out, total_q, topk), dtype=torch.int32,
                          device=scores.device)
    _cuda_contig("out", out, torch.int32)
    st = L.msa_topk_select(_p(scores), hs, T, total_q, int(topk), int(num_kv_heads_out), _p(out),
                           _stream(stream))
    _check("msa_topk_select", st)
    return out


def msa_build_union(q2k_indices, cu_seqlens_q, cu_seqlens_k=None, *, seqused_k=None,
                    max_pages=0, causal=True, tile_tokens=16, max_tiles=None, stream=None):
    """Per-tile union metadata in the canonical format; see include/msa.h.

    Returns (union_len, union_blocks, member, tile_info) sized for max_tiles
    (default ceil(total_q / tile_tokens) + batch).
    """
    L = lib()
    _cuda_contig("q2k_indices", q2k_indices, torch.int32)
    hkv, total_q, topk = q2k_indices.shape
    batch = cu_seqlens_q.shape[0] - 1
    if max_tiles is None:
        max_tiles = (total_q + tile_tokens - 1) // tile_tokens + batch
    cap = tile_tokens * topk
    words = (cap + 31) // 32
    dev = q2k_indices.device
    ulen = torch.empty((hkv, max_tiles), dtype=torch.int32, device=dev)
    ublk = torch.empty((hkv, max_tiles, cap), dtype=torch.int32, device=dev)
    mem = torch.empty((hkv, max_tiles, tile_tokens, words), dtype=torch.int32, device=dev)
    info = torch.empty((max_tiles, 2), dtype=torch.int32, device=dev)
    st = L.msa_build_union(_p(q2k_indices), topk, _p(cu_seqlens_q), _p(cu_seqlens_k),
                           _p(seqused_k), int(max_pages), batch, total_q, hkv, int(bool(causal)),
                           int(tile_tokens), int(max_tiles), _p(ulen), _p(ublk), _p(mem),
                           _p(info), _stream(stream))
    _check("msa_build_union", st)
    return ulen, ublk, mem, info


def msa_build_union_block_members(q2k_indices, cu_seqlens_q, cu_seqlens_k=None, *,
                                  seqused_k=None, max_pages=0, causal=True, tile_tokens=32,
                                  max_tiles=None, stream=None):
    """msa_build_union plus the per-union-block member-token masks
    (tile_tokens <= 32); returns (union_len, union_blocks, member,
    block_members, tile_info)."""
    L = lib()
    _cuda_contig("q2k_indices", q2k_indices, torch.int32)
    hkv, total_q, topk = q2k_indices.shape
    batch = cu_seqlens_q.shape[0] - 1
    if max_tiles is None:
        max_tiles = (total_q + tile_tokens - 1) // tile_tokens + batch
    cap = tile_tokens * topk
    words = (cap + 31) // 32
    dev = q2k_indices.device
    ulen = torch.empty((hkv, max_tiles), dtype=torch.int32, device=dev)
    ublk = torch.empty((hkv, max_tiles, cap), dtype=torch.int32, device=dev)
    mem = torch.empty((hkv, max_tiles, tile_tokens, words), dtype=torch.int32, device=dev)
    bmem = torch.empty((hkv, max_tiles, cap), dtype=torch.int32, device=dev)
    info = torch.empty((max_tiles, 2), dtype=torch.int32, device=dev)
    st = L.msa_build_union_block_members(
        _p(q2k_indices), topk, _p(cu_seqlens_q), _p(cu_seqlens_k), _p(seqused_k),
        int(max_pages), batch, total_q, hkv, int(bool(causal)), int(tile_tokens), int(max_tiles),
        _p(ulen), _p(ublk), _p(mem), _p(bmem), _p(info), _stream(stream))
    _check("msa_build_union_block_members", st)
    return ulen, ublk, mem, bmem, info


def msa_read_device_fault(stream=None) -> int:
    """Synchronise the stream, return and clear the library's device fault word."""
    v = C.c_uint(0)
    _check("msa_read_device_fault", lib().msa_read_device_fault(C.byref(v), _stream(stream)))
    return int(v.value)


def msa_set_timing_events(events=None):
    """Record three torch.cuda.Event objects around the forward's launches
    (before, after the metadata step, after attention); None turns it off."""
    if not events:
        _check("msa_set_timing_events", lib().msa_set_timing_events(None, 0))
        return
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on first record
            e.record()
    arr = (C.c_void_p * 3)(*[C.c_void_p(e.cuda_event) for e in events])
    _check("msa_set_timing_events", lib().msa_set_timing_events(arr, 3))


def msa_sparse_decode_noalloc(q, k, v, q2k_indices, cu_seqlens_q, page_table, seqused_k, *,
                              max_seqlen_q, causal=True, softmax_scale=None, out=None, lse=None,
                              stream=None):
    """Paged decode that uses the library's fixed device scratch instead of a
    workspace (for callers that cannot allocate); see include/msa.h."""
    L = lib()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_contig(name, t, torch.bfloat16)
    _cuda_contig("q2k_indices", q2k_indices, torch.int32)
    _cuda_contig("cu_seqlens_q", cu_seqlens_q, torch.int32)
    _cuda_contig("page_table", page_table, torch.int32)
    _cuda_contig("seqused_k", seqused_k, torch.int32)
    if k.dim() != 4 or tuple(k.shape[2:]) != (128, 128) or k.shape != v.shape:
        raise ValueError("k and v must be paged pools of shape (num_pages, Hkv, 128, 128)")
    total_q, hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, torch.bfloat16)
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have q's shape")
    _cuda_contig("lse", lse, torch.float32)
    if lse is not None and tuple(lse.shape) != (total_q, hq):
        raise ValueError("lse must have shape (total_q, num_qo_heads)")
    st = L.msa_sparse_decode_noalloc(
        _p(q), _p(k), _p(v), _p(q2k_indices), q2k_indices.shape[2], _p(cu_seqlens_q),
        _p(page_table), page_table.shape[1], k.shape[0], _p(seqused_k),
        cu_seqlens_q.shape[0] - 1, total_q, hq, k.shape[1], d, int(max_seqlen_q),
        int(bool(causal)), float(softmax_scale) if softmax_scale is not None else 0.0, _p(out),
        _p(lse), _stream(stream))
    _check("msa_sparse_decode_noalloc", st)
    return (out, lse) if lse is not None else out


def msa_selftest_wait_timeout(timeout_us, stream=None):
    """Run the bounded-wait self-test kernel (see include/msa.h)."""
    _check("msa_selftest_wait_timeout", lib().msa_selftest_wait_timeout(int(timeout_us),
                                                                        _stream(stream)))
