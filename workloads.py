"""Seeded synthetic inputs for MSA workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. Both the CUDA library's tests/benchmark and the CPU oracle
consume exactly the tensors produced here.

Shapes, distributions and selection structure follow the workloads the MSA
documentation pages describe ("msa_sparse_attention": q (total_q, Hq, d),
k/v flat (total_k, Hkv, d) or paged (num_pages, Hkv, 128, d), q2k_indices
(Hkv, total_q, topk) int32 ascending and -1 padded; "msa_proxy_score": proxy
q and index k; "prepare_msa_nvfp4_sparse_decode": decode rows b*seqlen_q ..
(b+1)*seqlen_q, right-aligned token positions). All values are N(0, 1);
E4M3 tensors hold N(0, 1) rounded to nearest-even by torch's float8_e4m3fn cast
after clamping to +-448 (unit scale).

Every generator takes a ``seed`` and a ``device``; a torch.Generator on that
device makes the draws, so a given (seed, device) always yields the same data.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

BLOCK = 128  # KV block / page size in tokens


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def randn_e4m3(shape, g, device):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)


def randn_chunked(shape, g, device, dtype):
    """N(0,1) in ``dtype`` drawn in slabs along dim 0 to bound fp32 scratch."""
    out = torch.empty(shape, dtype=dtype, device=device)
    per = max(1, (1 << 26) // max(1, math.prod(shape[1:])))
    for s in range(0, shape[0], per):
        e = min(shape[0], s + per)
        x = torch.randn((e - s,) + tuple(shape[1:]), generator=g, device=device,
                        dtype=torch.float32)
        if dtype == torch.float8_e4m3fn:
            x.clamp_(-448.0, 448.0)
        out[s:e] = x.to(dtype)
    return out


def nvfp4_page_stride(num_kv_heads: int, head_dim: int = 128) -> int:
    """Bytes of one planar NVFP4 page: [K data | K scales | V data | V scales],
    each (Hkv, 128, d/2) packed codes or (Hkv, 128, d/16) scales."""
    return 2 * num_kv_heads * BLOCK * (head_dim // 2 + head_dim // 16)


def nvfp4_pool(num_pages: int, num_kv_heads: int, g, device, head_dim: int = 128):
    """A planar NVFP4 page pool (num_pages, page_stride) of uint8: uniform
    random E2M1 nibbles and positive E4M3 block scales with exponent field
    5..8 (2^-2 .. 2^1 times 1 + m/8), so no scale is zero, NaN or huge."""
    stride = nvfp4_page_stride(num_kv_heads, head_dim)
    pool = torch.empty((num_pages, stride), dtype=torch.uint8, device=device)
    data = num_kv_heads * BLOCK * head_dim // 2
    scales = num_kv_heads * BLOCK * head_dim // 16
    per = max(1, (1 << 28) // stride)
    for s in range(0, num_pages, per):
        e = min(num_pages, s + per)
        slab = pool[s:e]
        slab.copy_(torch.randint(0, 256, (e - s, stride), generator=g, device=device,
                                 dtype=torch.int32).to(torch.uint8))
        for off in (data, 2 * data + scales):
            ex = torch.randint(5, 9, (e - s, scales), generator=g, device=device, dtype=torch.int32)
            ma = torch.randint(0, 8, (e - s, scales), generator=g, device=device, dtype=torch.int32)
            slab[:, off:off + scales] = (ex * 8 + ma).to(torch.uint8)
    return pool


def cu_from_lengths(lengths: Sequence[int], device="cpu") -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def select_blocks(positions: torch.Tensor, num_kv_heads: int, topk: int, g: torch.Generator,
                  *, first: bool = False, prev: bool = False, chunk: int = 4096) -> torch.Tensor:
    """Random block selections, one row per (kv head, query).

    ``positions`` (n,) int64 holds each query's right-aligned key position
    (negative: sees nothing). For a query at position p the causally visible
    blocks are 0 .. p // 128. The row always holds the diagonal block p // 128,
    plus block 0 when ``first`` and block p//128 - 1 when ``prev``; the rest are
    distinct visible blocks drawn uniformly, up to ``topk``. When fewer than
    ``topk`` blocks are visible, all of them are taken. Rows are ascending and
    -1 padded. Returns int32 (num_kv_heads, n, topk).
    """
    device = positions.device
    n = positions.shape[0]
    out = torch.full((num_kv_heads, n, topk), -1, dtype=torch.int32, device=device)
    if n == 0:
        return out
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        pos = positions[s:e]
        diag = torch.where(pos >= 0, pos // BLOCK, torch.full_like(pos, -1))
        nvis = diag + 1  # 0 when nothing is visible
        width = int(max(1, int(nvis.max().item())))
        col = torch.arange(width, device=device)
        for h in range(num_kv_heads):
            key = torch.rand((e - s, width), generator=g, device=device)
            key = torch.where(col[None, :] < nvis[:, None], key, torch.full_like(key, -1.0))
            forced = col[None, :] == diag[:, None]
            if first:
                forced |= (col[None, :] == 0) & (nvis[:, None] > 0)
            if prev:
                forced |= col[None, :] == (diag[:, None] - 1)
            key = torch.where(forced & (key >= 0), torch.full_like(key, 2.0), key)
            k = min(topk, width)
            val, idx = torch.topk(key, k, dim=1)
            idx = torch.where(val >= 0, idx, torch.full_like(idx, 1 << 30))
            idx, _ = torch.sort(idx, dim=1)
            idx = torch.where(idx >= (1 << 30), torch.full_like(idx, -1), idx)
            out[h, s:e, :k] = idx.to(torch.int32)
    return out


def query_positions(cu_q: torch.Tensor, k_lengths: Sequence[int]) -> torch.Tensor:
    """Right-aligned key position of every packed query row (int64)."""
    cu = cu_q.tolist()
    parts = []
    for b in range(len(cu) - 1):
        lq = cu[b + 1] - cu[b]
        parts.append(torch.arange(lq, dtype=torch.int64) + (int(k_lengths[b]) - lq))
    return torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int64)


# --------------------------------------------------------------------------
# Prefill (flat K/V)
# --------------------------------------------------------------------------
@dataclasses.dataclass
class PrefillSpec:
    name: str
    seqlens: Optional[List[int]]       # Lq = Lk per sequence; None -> drawn
    num_qo_heads: int
    num_kv_heads: int
    topk: int
    kv_dtype: str = "bf16"             # "bf16" | "e4m3"
    causal: bool = True
    return_lse: bool = True
    first_prev: bool = False           # force block 0 and the previous block
    head_dim: int = 128
    draw_lengths: Optional[tuple] = None  # (count, lo, hi) uniform inclusive


def prefill_lengths(spec: PrefillSpec, seed: int) -> List[int]:
    if spec.seqlens is not None:
        return list(spec.seqlens)
    count, lo, hi = spec.draw_lengths
    g = _gen(seed + 7919, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (count,), generator=g).tolist()]


def make_prefill(spec: PrefillSpec, seed: int, device="cpu"):
    """q, k, v, q2k_indices, cu_seqlens_q, cu_seqlens_k for a flat prefill."""
    lens = prefill_lengths(spec, seed)
    g = _gen(seed, device)
    total = sum(lens)
    d = spec.head_dim
    q = randn_chunked((total, spec.num_qo_heads, d), g, device, torch.bfloat16)
    kvdt = torch.float8_e4m3fn if spec.kv_dtype == "e4m3" else torch.bfloat16
    k = randn_chunked((total, spec.num_kv_heads, d), g, device, kvdt)
    v = randn_chunked((total, spec.num_kv_heads, d), g, device, kvdt)
    cu = cu_from_lengths(lens, device)
    pos = query_positions(cu.cpu(), lens).to(device)
    q2k = select_blocks(pos, spec.num_kv_heads, spec.topk, g, first=spec.first_prev,
                        prev=spec.first_prev)
    return dict(q=q, k=k, v=v, q2k_indices=q2k, cu_seqlens_q=cu, cu_seqlens_k=cu.clone(),
                causal=spec.causal, softmax_scale=d ** -0.5, lengths=lens)


def make_paged_prefill_nvfp4(spec: PrefillSpec, seed: int, device="cpu",
                             k_global_scale=0.25, v_global_scale=0.125):
    """A paged prefill over a planar NVFP4 page pool: each sequence's pages are
    a random permutation of the pool; selections as make_prefill."""
    lens = prefill_lengths(spec, seed)
    gl = _gen(seed + 7919, "cpu")
    pages_per = [(n + BLOCK - 1) // BLOCK for n in lens]
    num_pages = sum(pages_per)
    perm = torch.randperm(num_pages, generator=gl).to(torch.int32)
    page_table = torch.zeros((len(lens), max(pages_per)), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per):
        page_table[b, :n] = perm[off:off + n]
        off += n
    g = _gen(seed, device)
    d = spec.head_dim
    q = randn_chunked((sum(lens), spec.num_qo_heads, d), g, device, torch.bfloat16)
    pool = nvfp4_pool(num_pages, spec.num_kv_heads, g, device, d)
    cu = cu_from_lengths(lens, device)
    pos = query_positions(cu.cpu(), lens).to(device)
    q2k = select_blocks(pos, spec.num_kv_heads, spec.topk, g, first=spec.first_prev,
                        prev=spec.first_prev)
    return dict(q=q, kv_pool=pool, q2k_indices=q2k, cu_seqlens_q=cu,
                page_table=page_table.to(device),
                seqused_k=torch.tensor(lens, dtype=torch.int32, device=device),
                softmax_scale=d ** -0.5, lengths=lens, k_global_scale=k_global_scale,
                v_global_scale=v_global_scale)


# --------------------------------------------------------------------------
# Paged decode
# --------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeSpec:
    name: str
    batch: int
    seqused_range: tuple               # uniform inclusive
    num_qo_heads: int
    num_kv_heads: int
    topk: int
    seqlen_q: int = 1
    head_dim: int = 128
    kv_dtype: str = "bf16"
    k_global_scale: float = 1.0
    v_global_scale: float = 1.0


def make_decode(spec: DecodeSpec, seed: int, device="cpu", seqlen_q: Optional[int] = None):
    """Paged decode inputs: pages in a shared pool, page_table a random permutation.

    Query token i of request b sits at key position seqused_k[b] - seqlen_q + i.
    Each token selects the page holding its own position plus random visible
    pages (reading of "the last page plus 15 random visible pages" for
    seqlen_q > 1: the own-position page per token).
    """
    sq = seqlen_q if seqlen_q is not None else spec.seqlen_q
    gl = _gen(seed + 104729, "cpu")
    lo, hi = spec.seqused_range
    seqused = torch.randint(lo, hi + 1, (spec.batch,), generator=gl)
    pages_per = [(int(x) + BLOCK - 1) // BLOCK for x in seqused.tolist()]
    num_pages = sum(pages_per)
    max_pages = max(pages_per)
    perm = torch.randperm(num_pages, generator=gl).to(torch.int32)
    page_table = torch.zeros((spec.batch, max_pages), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per):
        page_table[b, :n] = perm[off:off + n]
        off += n
    g = _gen(seed, device)
    d = spec.head_dim
    extra = {}
    if spec.kv_dtype == "nvfp4":
        # K and V live in one planar page pool; k / v stay None.
        k = v = None
        extra = dict(kv_pool=nvfp4_pool(num_pages, spec.num_kv_heads, g, device, d),
                     k_global_scale=spec.k_global_scale, v_global_scale=spec.v_global_scale)
    else:
        kvdt = torch.float8_e4m3fn if spec.kv_dtype == "e4m3" else torch.bfloat16
        k = randn_chunked((num_pages, spec.num_kv_heads, BLOCK, d), g, device, kvdt)
        v = randn_chunked((num_pages, spec.num_kv_heads, BLOCK, d), g, device, kvdt)
    q = randn_chunked((spec.batch * sq, spec.num_qo_heads, d), g, device, torch.bfloat16)
    cu_q = torch.arange(0, spec.batch * sq + 1, sq, dtype=torch.int32)
    pos = query_positions(cu_q, seqused.tolist())
    gs = _gen(seed + 1, "cpu")
    q2k = select_blocks(pos, spec.num_kv_heads, spec.topk, gs)
    return dict(q=q, k=k, v=v, q2k_indices=q2k.to(device), cu_seqlens_q=cu_q.to(device),
                page_table=page_table.to(device), seqused_k=seqused.to(torch.int32).to(device),
                causal=True, softmax_scale=d ** -0.5, seqlen_q=sq, num_pages=num_pages, **extra)


# --------------------------------------------------------------------------
# Two-stage pipeline: proxy score -> top-k -> sparse attention
# --------------------------------------------------------------------------
@dataclasses.dataclass
class TwoStageSpec:
    name: str
    seqlens: List[int]
    proxy_heads: int
    num_qo_heads: int
    num_kv_heads: int
    topk: int
    head_dim: int = 128


def make_two_stage(spec: TwoStageSpec, seed: int, device="cpu"):
    g = _gen(seed, device)
    total = sum(spec.seqlens)
    d = spec.head_dim
    cu = cu_from_lengths(spec.seqlens, device)
    return dict(
        proxy_q=randn_chunked((total, spec.proxy_heads, d), g, device, torch.bfloat16),
        index_k=randn_chunked((total, spec.num_kv_heads, d), g, device, torch.bfloat16),
        q=randn_chunked((total, spec.num_qo_heads, d), g, device, torch.bfloat16),
        k=randn_chunked((total, spec.num_kv_heads, d), g, device, torch.bfloat16),
        v=randn_chunked((total, spec.num_kv_heads, d), g, device, torch.bfloat16),
        cu_seqlens_q=cu, cu_seqlens_k=cu.clone(), causal=True, softmax_scale=d ** -0.5,
        lengths=list(spec.seqlens))


# --------------------------------------------------------------------------
# The five workloads of the MSA forward (tiny flat, flat varlen, mixed dtype,
# paged decode, two-stage)
# --------------------------------------------------------------------------
TINY_FLAT = PrefillSpec("tiny_flat_prefill_1x1024_h4kv1_top4", [1024], 4, 1, 4)
FLAT_VARLEN = PrefillSpec("flat_varlen_prefill_2x32768_h64kv8_top16", [32768, 32768], 64, 8, 16,
                          first_prev=True)
MIXED_E4M3 = PrefillSpec("e4m3kv_varlen_prefill_8xU[4096,65536]_h32kv4_top16", None, 32, 4, 16,
                         kv_dtype="e4m3", draw_lengths=(8, 4096, 65536))
PAGED_DECODE = DecodeSpec("paged_decode_b128_U[8192,131072]_h64kv4_top16", 128, (8192, 131072),
                          64, 4, 16)
# Global scales chosen so that the decoded K and V have about unit RMS (the
# pool's E2M1 x block-scale values have RMS about 5), like the N(0,1) values
# of the other workloads.
PAGED_PREFILL_NVFP4 = PrefillSpec("nvfp4_paged_prefill_4x16384_h32kv4_top16", [16384] * 4, 32, 4,
                                  16, first_prev=True)
PAGED_DECODE_NVFP4 = DecodeSpec("nvfp4_paged_decode_b128_U[8192,131072]_h64kv4_top16", 128,
                                (8192, 131072), 64, 4, 16, kv_dtype="nvfp4",
                                k_global_scale=0.25, v_global_scale=0.125)
TWO_STAGE = TwoStageSpec("two_stage_proxy_top16_attn_1x65536_h32kv4", [65536], 32, 32, 4, 16)


def parity_rows(cu_q: torch.Tensor, tile_tokens: int, target: int, seed: int) -> torch.Tensor:
    """Sampled packed query rows for oracle parity at full size.

    Always contains the first and the last tile of every sequence and every row
    of one tile per 8192 tokens; the rest is uniform, up to ``target`` rows.
    """
    cu = [int(x) for x in cu_q.cpu().tolist()]
    rows = set()
    g = _gen(seed + 31337, "cpu")
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        if e <= s:
            continue
        rows.update(range(s, min(e, s + tile_tokens)))
        last0 = s + ((e - s - 1) // tile_tokens) * tile_tokens
        rows.update(range(last0, e))
        for c in range(s, e, 8192):
            span = min(8192, e - c)
            ntile = (span + tile_tokens - 1) // tile_tokens
            t = int(torch.randint(0, ntile, (1,), generator=g).item())
            rows.update(range(c + t * tile_tokens, min(e, c + (t + 1) * tile_tokens)))
    total = cu[-1]
    while len(rows) < min(target, total):
        for x in torch.randint(0, total, (min(target, total) - len(rows),), generator=g).tolist():
            rows.add(int(x))
    return torch.tensor(sorted(rows), dtype=torch.int32)
