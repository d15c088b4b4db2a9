"""GPU parity at the full sizes of the five MSA workloads, in the launch
configuration the benchmark times.

Inputs are drawn on the GPU by the seeded generators in ``workloads`` and
copied to the host for the oracle. The tiny prefill and the paged decode are
compared in full; the large prefill workloads and the two-stage pipeline on a
seeded sample of query rows (first and last tile of every sequence, one full
tile per 8192 tokens, the rest uniform) with every head.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import check_attention, check_proxy, f32, fault_clear, to_cpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def msa():
    import block_sparse_top_msa_gb300 as m
    m.build()
    m.lib()
    return m


def _fwd(msa, g, max_sq=None, paged=False):
    return msa.msa_sparse_attention_fwd(
        g["q"], g["k"], g["v"], g["q2k_indices"], g["cu_seqlens_q"], g.get("cu_seqlens_k"),
        causal=True, softmax_scale=g["softmax_scale"], page_table=g.get("page_table"),
        seqused_k=g.get("seqused_k"), max_seqlen_q=max_sq, return_softmax_lse=True)


def _oracle(c, rows=None):
    return oracle.sparse_attention(c["q"], c["k"], c["v"], c["q2k_indices"], c["cu_seqlens_q"],
                                   c.get("cu_seqlens_k"), causal=True,
                                   softmax_scale=f32(c["softmax_scale"]),
                                   page_table=c.get("page_table"), seqused_k=c.get("seqused_k"),
                                   rows=rows)


@pytest.mark.parametrize("spec", [workloads.TINY_FLAT, workloads.FLAT_VARLEN,
                                  workloads.MIXED_E4M3], ids=lambda s: s.name)
def test_prefill_workload(msa, spec):
    g = workloads.make_prefill(spec, seed=0, device=DEV)
    out, lse = _fwd(msa, g, max_sq=max(g["lengths"]))
    torch.cuda.synchronize()
    fault_clear(msa)
    c = to_cpu(g)
    tq = c["q"].shape[0]
    W = msa.msa_union_tile_tokens(c["q"].shape[1], c["k"].shape[1])
    rows = None if tq <= 4096 else workloads.parity_rows(c["cu_seqlens_q"], W, 4096, seed=0)
    ref_out, ref_lse = _oracle(c, rows)
    check_attention(out, lse, ref_out, ref_lse, rows=rows, label=spec.name)


def _compact_pages(g):
    """Host copy of the paged inputs holding only the pages the selections read.

    The pool (about 18.6 GB) is gathered on the device down to the referenced
    pages and the page table is renumbered; unreferenced entries point past the
    compact pool, which the oracle treats as unmapped (they are never read).
    """
    pt, q2k, cu = g["page_table"], g["q2k_indices"], g["cu_seqlens_q"]
    B = pt.shape[0]
    req = torch.repeat_interleave(torch.arange(B, device=pt.device),
                                  (cu[1:] - cu[:-1]).long())
    ids = q2k.long()
    ok = (ids >= 0) & (ids < pt.shape[1])
    pages = pt[req[None, :, None].expand_as(ids)[ok], ids[ok]]
    used = torch.unique(pages[(pages >= 0) & (pages < g["k"].shape[0])])
    remap = torch.full((g["k"].shape[0],), used.numel(), dtype=torch.int32, device=pt.device)
    remap[used] = torch.arange(used.numel(), dtype=torch.int32, device=pt.device)
    c = to_cpu({k: v for k, v in g.items() if k not in ("k", "v", "page_table")})
    c["k"] = g["k"].index_select(0, used).cpu()
    c["v"] = g["v"].index_select(0, used).cpu()
    c["page_table"] = remap[pt.long()].cpu()
    return c


@pytest.mark.parametrize("sq", [1, 4])
def test_decode_workload(msa, sq):
    spec = workloads.PAGED_DECODE
    g = workloads.make_decode(spec, seed=0, device=DEV, seqlen_q=sq)
    out, lse = _fwd(msa, g, max_sq=sq)
    torch.cuda.synchronize()
    fault_clear(msa)
    c = _compact_pages(g)
    ref_out, ref_lse = _oracle(c)
    check_attention(out, lse, ref_out, ref_lse, label=f"{spec.name}_sq{sq}")


@pytest.mark.parametrize("sq", [1, 4])
def test_nvfp4_decode_workload(msa, sq):
    """The packed NVFP4 paged decode at its benchmark size, in the benchmark's
    launch configuration; every query row of a sample of requests (every
    16th) is compared with every head. The oracle decodes only the pages
    those rows can read (renumbered into a compact pool)."""
    spec = workloads.PAGED_DECODE_NVFP4
    g = workloads.make_decode(spec, seed=0, device=DEV, seqlen_q=sq)
    q2k, pt, cu = g["q2k_indices"], g["page_table"], g["cu_seqlens_q"]
    hkv = q2k.shape[0]
    k, ks, v, vs = msa.nvfp4_views(g["kv_pool"], hkv)
    out, lse = msa.msa_sparse_attention_nvfp4_paged(
        g["q"], k, ks, v, vs, q2k, cu, page_table=pt, seqused_k=g["seqused_k"],
        k_global_scale=spec.k_global_scale, v_global_scale=spec.v_global_scale, max_seqlen_q=sq,
        return_softmax_lse=True)
    torch.cuda.synchronize()
    fault_clear(msa)
    B = pt.shape[0]
    reqs = torch.arange(0, B, 16, device=pt.device)
    rows = (reqs[:, None] * sq + torch.arange(sq, device=pt.device)).flatten()
    ids = q2k[:, rows, :].long()
    req = (rows // sq)[None, :, None].expand_as(ids)
    ok = (ids >= 0) & (ids < pt.shape[1])
    pages = pt[req[ok], ids[ok]].long()
    npg = g["kv_pool"].shape[0]
    used = torch.unique(pages[(pages >= 0) & (pages < npg)])
    remap = torch.full((npg,), used.numel(), dtype=torch.int32, device=pt.device)
    remap[used] = torch.arange(used.numel(), dtype=torch.int32, device=pt.device)
    pool = g["kv_pool"].index_select(0, used).cpu()
    kf, vf = oracle.nvfp4_dequant(pool, hkv, 128, spec.k_global_scale, spec.v_global_scale)
    ref_out, ref_lse = oracle.sparse_attention(
        g["q"].cpu(), kf, vf, q2k.cpu(), cu.cpu(), causal=True,
        softmax_scale=f32(g["softmax_scale"]), page_table=remap[pt.long()].cpu(),
        seqused_k=g["seqused_k"].cpu(), num_pages=used.numel(), rows=rows.to(torch.int32).cpu())
    check_attention(out, lse, ref_out, ref_lse, rows=rows.cpu(), label=f"{spec.name}_sq{sq}")


def test_two_stage_workload(msa):
    spec = workloads.TWO_STAGE
    g = workloads.make_two_stage(spec, seed=0, device=DEV)
    L = spec.seqlens[0]
    T = (L + 127) // 128
    scores = msa.msa_proxy_score(g["proxy_q"], g["index_k"], g["cu_seqlens_q"],
                                 g["cu_seqlens_k"], causal=True, max_k_tiles=T, reduce_heads=True)
    q2k = msa.msa_topk_select(scores, spec.topk, spec.num_kv_heads)
    g2 = dict(g, q2k_indices=q2k)
    out, lse = _fwd(msa, g2, max_sq=L)
    torch.cuda.synchronize()
    fault_clear(msa)
    c = to_cpu(g2)
    s_gpu = scores.cpu().numpy()
    # Top-k: bit-exact against the oracle run on the GPU's own scores (all queries).
    assert np.array_equal(q2k.cpu().numpy(), oracle.topk_select(s_gpu, spec.topk,
                                                                spec.num_kv_heads))
    # Proxy: sampled queries against the fp64 oracle.
    prow = torch.tensor(sorted({0, 1, 127, 128, 129, 4095, 4096, 30000, L // 2, L - 129,
                                L - 2, L - 1}), dtype=torch.int32)
    ref = oracle.proxy_score(c["proxy_q"], c["index_k"], c["cu_seqlens_q"], c["cu_seqlens_k"],
                             causal=True, max_k_tiles=T, reduce_heads=True, rows=prow)
    check_proxy(s_gpu[:, :, prow.long().numpy()], ref, label="proxy")
    # Selection from fp64 scores may differ only at near-ties of the 16th/17th score.
    for j, r in enumerate(prow.tolist()):
        col = ref[0, :, j]
        fin = np.isfinite(col)
        if fin.sum() <= spec.topk:
            continue
        order = sorted(np.nonzero(fin)[0].tolist(), key=lambda t: (-col[t], t))
        exp = sorted(order[:spec.topk])
        got = [x for x in q2k[0, r].tolist() if x >= 0]
        if got != exp:
            gap = col[order[spec.topk - 1]] - col[order[spec.topk]]
            assert gap < 1e-4 * abs(col[order[spec.topk - 1]]), (r, got, exp, gap)
    # Attention with the GPU-selected blocks, sampled rows.
    rows = workloads.parity_rows(c["cu_seqlens_q"], 16, 4096, seed=5)
    ref_out, ref_lse = _oracle(c, rows)
    check_attention(out, lse, ref_out, ref_lse, rows=rows, label=spec.name)
