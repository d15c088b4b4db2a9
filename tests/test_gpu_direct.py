"""GPU parity of one-token-tile launches without the union kernel.

When a launch's query tiles hold one token (seqlen_q 1 decode, or G = 128),
the attention kernel builds each tile's block list from the token's own
q2k_indices row ("flashinfer.msa_ops.msa_sparse_attention", Parameters
`q2k_indices`: int32 block ids, ascending, -1 padded): usable ids only,
ascending, each once. These cases feed it rows the pages do not promise
(unsorted, repeated, -1 in the middle, ids past the sequence or above the
causal limit, empty rows), empty query sequences, split work items whose
partials the merge kernel combines, and topk at both ends of the direct
range; every result is compared with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import check_attention, f32, fault_clear, to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def msa():
    import block_sparse_top_msa_gb300 as m
    m.build()
    m.lib()
    return m


def _run(msa, inp, causal=True, max_seqlen_q=1):
    g = to_dev(inp, DEV)
    out, lse = msa.msa_sparse_attention_fwd(
        g["q"], g["k"], g["v"], g["q2k_indices"], g["cu_seqlens_q"], g.get("cu_seqlens_k"),
        causal=causal, page_table=g.get("page_table"), seqused_k=g.get("seqused_k"),
        max_seqlen_q=max_seqlen_q, return_softmax_lse=True)
    torch.cuda.synchronize()
    fault_clear(msa)
    return out, lse


def _oracle(inp, causal=True):
    return oracle.sparse_attention(inp["q"], inp["k"], inp["v"], inp["q2k_indices"],
                                   inp["cu_seqlens_q"], inp.get("cu_seqlens_k"), causal=causal,
                                   softmax_scale=f32(128 ** -0.5),
                                   page_table=inp.get("page_table"),
                                   seqused_k=inp.get("seqused_k"))


def _paged_decode(g, seqused, hq, hkv, topk, lens_q=None, unmapped=True):
    """Paged inputs, lens_q query tokens per request (default one each)."""
    lens_q = lens_q if lens_q is not None else [1] * len(seqused)
    cu_q = workloads.cu_from_lengths(lens_q)
    pages = [(n + 127) // 128 for n in seqused]
    npg = sum(pages) + 3
    perm = torch.randperm(npg, generator=g).to(torch.int32)
    pt = torch.zeros(len(seqused), max(pages), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, :n] = perm[off:off + n]
        off += n
    if unmapped and len(seqused) > 1 and pages[1] > 1:
        pt[1, 0] = npg + 7  # an unmapped page: reads as no keys
    k = torch.randn(npg, hkv, 128, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(npg, hkv, 128, 128, generator=g).to(torch.bfloat16)
    q = torch.randn(sum(lens_q), hq, 128, generator=g).to(torch.bfloat16)
    q2k = workloads.select_blocks(workloads.query_positions(cu_q, seqused), hkv, topk, g)
    return dict(q=q, k=k, v=v, q2k_indices=q2k, cu_seqlens_q=cu_q, page_table=pt,
                seqused_k=torch.tensor(seqused, dtype=torch.int32))


def test_direct_decode_irregular_rows(msa):
    g = torch.Generator().manual_seed(101)
    seqused = [8192, 3000, 129, 128, 1, 1000, 5000]
    inp = _paged_decode(g, seqused, 32, 2, 8)
    q2k = inp["q2k_indices"]                                 # (hkv, tokens, topk)
    q2k[0, 0] = torch.tensor([60, 3, 60, 7, -1, 3, 0, 63])    # unsorted, repeated, -1 inside
    q2k[1, 0] = torch.tensor([-1, -1, 5, -1, 2, -1, -1, 9])   # padding first
    q2k[0, 1] = torch.tensor([0, 23, 24, 100, 5000, 2, 1, 1])  # ids past the sequence (24 pages)
    q2k[1, 2] = -1                                           # an empty row: out 0, lse -inf
    q2k[0, 3] = torch.tensor([0, 0, 0, 0, 0, 0, 0, 0])        # one block, eight times
    q2k[1, 4] = torch.tensor([0, 1, 2, 3, 4, 5, 6, 7])        # 1-token sequence: only block 0
    q2k[0, 6] = torch.arange(39, 31, -1)                     # strictly descending
    out, lse = _run(msa, inp)
    ref_out, ref_lse = _oracle(inp)
    assert np.isneginf(ref_lse[2, 16:]).all()  # KV head 1 serves query heads 16-31
    check_attention(out, lse, ref_out, ref_lse, label="direct_irregular")


@pytest.mark.parametrize("topk", [1, 32])
def test_direct_decode_topk_range(msa, topk):
    g = torch.Generator().manual_seed(200 + topk)
    seqused = [20000, 4500, 129, 9000]
    inp = _paged_decode(g, seqused, 16, 1, topk)
    if topk == 32:
        # a full-width unsorted row with repeats
        inp["q2k_indices"][0, 0] = torch.randint(0, 157, (32,), generator=g).to(torch.int32)
    out, lse = _run(msa, inp)
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label=f"direct_topk{topk}")


def test_union_kernel_route_above_direct_topk(msa):
    """topk 40 at one token per tile keeps the union kernel."""
    g = torch.Generator().manual_seed(7)
    inp = _paged_decode(g, [12000, 6000, 300], 16, 2, 40)
    out, lse = _run(msa, inp)
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label="union_topk40")


def test_direct_empty_query_sequences(msa):
    """Requests without query tokens between others (cu_seqlens_q repeats):
    the equal-length guess for a token's sequence misses and the search
    decides."""
    g = torch.Generator().manual_seed(31)
    seqused = [3000, 700, 129, 5000, 64, 2000]
    inp = _paged_decode(g, seqused, 32, 4, 16, lens_q=[1, 0, 0, 1, 1, 0], unmapped=False)
    out, lse = _run(msa, inp)
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label="direct_empty_seqs")


def test_direct_split_items(msa):
    """160 (request, KV head) units on 152 SMs: the 8 tail units are split
    across CTAs, each of which rebuilds the unit's list, and the merge kernel
    reads the lists written during the attention launch."""
    g = torch.Generator().manual_seed(47)
    seqused = [int(x) for x in torch.randint(2500, 9000, (40,), generator=g)]
    inp = _paged_decode(g, seqused, 16, 4, 16)
    out, lse = _run(msa, inp)
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label="direct_split")
    out2, lse2 = _run(msa, inp)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("causal", [True, False])
def test_direct_flat_decode(msa, causal):
    """Flat K/V (cu_seqlens_k), one query token per request; non-causal rows
    may use every block of their sequence."""
    g = torch.Generator().manual_seed(5 + causal)
    lens_k = [900, 128, 2000, 1]
    cu_q = workloads.cu_from_lengths([1] * len(lens_k))
    cu_k = workloads.cu_from_lengths(lens_k)
    hq, hkv, topk = 16, 2, 6
    q = torch.randn(len(lens_k), hq, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(sum(lens_k), hkv, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(sum(lens_k), hkv, 128, generator=g).to(torch.bfloat16)
    q2k = workloads.select_blocks(workloads.query_positions(cu_q, lens_k), hkv, topk, g)
    q2k[0, 1] = torch.tensor([0, 1, 1, -1, 0, 3])  # block 1 has no keys (128-token request)
    inp = dict(q=q, k=k, v=v, q2k_indices=q2k, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
    out, lse = _run(msa, inp, causal=causal)
    ref_out, ref_lse = _oracle(inp, causal=causal)
    check_attention(out, lse, ref_out, ref_lse, label=f"direct_flat_causal{causal}")


def test_direct_group128_prefill(msa):
    """G = 128 prefill: one token per tile, many tiles per sequence, causal
    limits per token, rows reversed."""
    g = torch.Generator().manual_seed(13)
    lens = [300, 0, 200]
    cu = workloads.cu_from_lengths(lens)
    q = torch.randn(sum(lens), 128, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(sum(lens), 1, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(sum(lens), 1, 128, generator=g).to(torch.bfloat16)
    q2k = workloads.select_blocks(workloads.query_positions(cu, lens), 1, 3, g)
    q2k = torch.flip(q2k, dims=[2]).contiguous()
    inp = dict(q=q, k=k, v=v, q2k_indices=q2k, cu_seqlens_q=cu, cu_seqlens_k=cu)
    out, lse = _run(msa, inp, max_seqlen_q=max(lens))
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label="direct_g128")
