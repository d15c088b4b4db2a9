"""GPU parity of every kernel against the fp64 oracle on small seeded inputs.

Sizes are chosen so the oracle runs in seconds while every case spans several
query tiles and KV blocks with ragged tails. All calls go through the C ABI
(via the thin binding).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import check_attention, check_proxy, f32, fault_clear, to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def msa():
    import block_sparse_top_msa_gb300 as m
    m.build()
    m.lib()
    return m


def _prefill_inputs(lens_q, lens_k, hq, hkv, topk, seed, kv="bf16", first_prev=False):
    g = torch.Generator().manual_seed(seed)
    d = 128
    tq, tk = sum(lens_q), sum(lens_k)
    q = torch.randn(tq, hq, d, generator=g).to(torch.float16 if kv == "f16" else torch.bfloat16)
    if kv == "f16":
        k = torch.randn(tk, hkv, d, generator=g).to(torch.float16)
        v = torch.randn(tk, hkv, d, generator=g).to(torch.float16)
    elif kv == "e4m3":
        k = torch.randn(tk, hkv, d, generator=g).to(torch.float8_e4m3fn)
        v = torch.randn(tk, hkv, d, generator=g).to(torch.float8_e4m3fn)
    else:
        k = torch.randn(tk, hkv, d, generator=g).to(torch.bfloat16)
        v = torch.randn(tk, hkv, d, generator=g).to(torch.bfloat16)
    cu_q = workloads.cu_from_lengths(lens_q)
    cu_k = workloads.cu_from_lengths(lens_k)
    pos = workloads.query_positions(cu_q, lens_k)
    q2k = workloads.select_blocks(pos, hkv, topk, g, first=first_prev, prev=first_prev)
    return dict(q=q, k=k, v=v, q2k_indices=q2k, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)


def _run_prefill(msa, inp, causal=True, scale=None, max_seqlen_q=None, workspace=None):
    g = to_dev(inp, DEV)
    out, lse = msa.msa_sparse_attention_fwd(
        g["q"], g["k"], g["v"], g["q2k_indices"], g["cu_seqlens_q"], g.get("cu_seqlens_k"),
        causal=causal, softmax_scale=scale, page_table=g.get("page_table"),
        seqused_k=g.get("seqused_k"), max_seqlen_q=max_seqlen_q, return_softmax_lse=True,
        workspace=workspace)
    torch.cuda.synchronize()
    fault_clear(msa)
    return out, lse


def _oracle(inp, causal=True, scale=None, rows=None):
    s = f32(scale if scale is not None else 128 ** -0.5)
    return oracle.sparse_attention(inp["q"], inp["k"], inp["v"], inp["q2k_indices"],
                                   inp["cu_seqlens_q"], inp.get("cu_seqlens_k"), causal=causal,
                                   softmax_scale=s, page_table=inp.get("page_table"),
                                   seqused_k=inp.get("seqused_k"), rows=rows)


# ---------------------------------------------------------------- union metadata
@pytest.mark.parametrize("W,topk,lens", [(16, 16, [300, 45, 1000]), (32, 4, [1024]),
                                         (1, 3, [77, 300]), (128, 8, [600, 129]),
                                         (10, 5, [333]), (128, 16, [2000, 129]),
                                         (64, 40, [3000])])
def test_union_bit_exact(msa, W, topk, lens):
    g = torch.Generator().manual_seed(W * 7 + topk)
    hkv = 3
    cu = workloads.cu_from_lengths(lens)
    pos = workloads.query_positions(cu, lens)
    q2k = workloads.select_blocks(pos, hkv, topk, g, first=True, prev=True)
    q2k[0, 5, 0] = 1000          # beyond the sequence
    q2k[1, 7, -1] = q2k[1, 7, 0]  # duplicate
    q2k[2, 9, :] = -1             # empty row
    ref_len, ref_blk, ref_mem = oracle.build_union(q2k, cu, cu, causal=True, tile_tokens=W)
    T = ref_len.shape[1]
    ulen, ublk, mem, info = msa.msa_build_union(q2k.to(DEV), cu.to(DEV), cu.to(DEV), causal=True,
                                                tile_tokens=W)
    torch.cuda.synchronize()
    assert np.array_equal(ulen[:, :T].cpu().numpy(), ref_len)
    assert np.array_equal(ublk[:, :T].cpu().numpy(), ref_blk)
    assert np.array_equal(mem[:, :T].cpu().numpy().view(np.uint32), ref_mem)
    assert np.all(ulen[:, T:].cpu().numpy() == 0)
    infos = info.cpu().numpy()
    assert np.all(infos[T:] == -1)
    starts = [s for b, L in enumerate(lens) for s in range(int(cu[b]), int(cu[b]) + L, W)]
    assert infos[:T, 0].tolist() == starts


def test_union_paged_lengths(msa):
    g = torch.Generator().manual_seed(3)
    lens_q, seqused = [3, 200], [900, 260]
    cu = workloads.cu_from_lengths(lens_q)
    pos = workloads.query_positions(cu, seqused)
    q2k = workloads.select_blocks(pos, 2, 6, g)
    su = torch.tensor(seqused, dtype=torch.int32)
    ref = oracle.build_union(q2k, cu, seqused_k=su, max_pages=5, causal=True, tile_tokens=16)
    got = msa.msa_build_union(q2k.to(DEV), cu.to(DEV), seqused_k=su.to(DEV), max_pages=5,
                              causal=True, tile_tokens=16)
    T = ref[0].shape[1]
    for r, x in zip(ref, got[:3]):
        assert np.array_equal(x[:, :T].cpu().numpy().view(r.dtype), r)


# ---------------------------------------------------------------- top-k
@pytest.mark.parametrize("topk,hs,hkv,n", [(16, 1, 4, 1000), (1, 1, 2, 1000), (5, 3, 3, 1000),
                                           (33, 1, 1, 1000), (64, 2, 2, 1000),
                                           (16, 2, 2, 1003),  # unaligned rows: scalar loads
                                           (8, 1, 1, 37)])    # fewer queries than a CTA
def test_topk_bit_exact(msa, topk, hs, hkv, n):
    rng = np.random.default_rng(topk + hs + n)
    T = 97
    s = rng.integers(-20, 20, size=(hs, T, n)).astype(np.float32) / 4  # many ties
    s[rng.random(s.shape) < 0.1] = -np.inf
    s[rng.random(s.shape) < 0.02] = np.nan
    s[:, :, 0] = -np.inf  # a query with nothing selectable
    s[:, 5:, 1] = -np.inf  # fewer than topk selectable
    ref = oracle.topk_select(s, topk, hkv)
    got = msa.msa_topk_select(torch.from_numpy(s).to(DEV), topk, hkv)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), ref)


# ---------------------------------------------------------------- prefill attention
PREFILL_CASES = [
    # name, lens_q, lens_k, hq, hkv, topk, kv, first_prev
    ("gqa4_varlen_ragged", [300, 129, 517], [300, 129, 517], 8, 2, 5, "bf16", True),
    ("gqa8_lq_lt_lk", [64, 200, 1], [700, 333, 129], 16, 2, 6, "bf16", False),
    ("gqa16", [400], [400], 16, 1, 4, "bf16", True),
    ("mha", [260, 300], [260, 300], 2, 2, 3, "bf16", False),
    ("gqa2_w64", [500], [500], 4, 2, 4, "bf16", False),
    ("gqa3_padded_rows", [270, 90], [270, 90], 6, 2, 4, "bf16", False),
    ("group128_w1", [40], [300], 128, 1, 2, "bf16", False),
    ("e4m3_gqa4", [300, 517], [300, 517], 8, 2, 5, "e4m3", True),
    ("e4m3_mha_lq_lt_lk", [100], [900], 2, 2, 7, "e4m3", False),
    ("topk1", [300], [300], 8, 1, 1, "bf16", False),
    ("topk64", [1200], [1200], 8, 1, 64, "bf16", False),
    ("mha_topk16_wide_union", [700, 260], [700, 260], 2, 2, 16, "bf16", True),
    ("f16_gqa8_varlen", [300, 517, 64], [300, 517, 900], 16, 2, 8, "f16", True),
    ("f16_gqa4_split", [200], [200], 8, 2, 4, "f16", False),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_prefill_parity(msa, case):
    name, lq, lk, hq, hkv, topk, kv, fp = case
    inp = _prefill_inputs(lq, lk, hq, hkv, topk, seed=len(name), kv=kv, first_prev=fp)
    out, lse = _run_prefill(msa, inp)
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label=name)


def _plain_workspace(msa, inp, hq, hkv, topk):
    """A workspace of the plain size query: E4M3 K/V then convert in-kernel."""
    lq = inp["cu_seqlens_q"]
    n = msa.msa_sparse_attention_workspace_size(
        lq.numel() - 1, inp["q"].shape[0], hq, hkv, 128, topk,
        int((lq[1:] - lq[:-1]).max()), False)
    return torch.empty(n, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("route", ["bf16_copy", "in_kernel"])
def test_prefill_e4m3_every_code(msa, route):
    """K takes every non-NaN E4M3 code (zeros, subnormals, the largest
    magnitudes) and V every code below 2 in magnitude, scattered at random,
    so the E4M3 -> bf16 decode is checked code by code through the attention
    result, on both routes: the decode pass into the workspace's bf16 copy
    (prefill-sized call, full workspace) and the conversion inside the
    attention kernel (plain-size workspace)."""
    inp = _prefill_inputs([300, 200], [300, 200], 8, 2, 4, seed=11, kv="e4m3")
    g = torch.Generator().manual_seed(3)
    k_codes = torch.tensor([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=torch.uint8)
    v_codes = torch.tensor([c for c in range(256) if (c & 0x78) <= 0x38], dtype=torch.uint8)

    def fill(codes, like):
        n = like.numel()
        rep = codes.repeat((n + codes.numel() - 1) // codes.numel())[:n]
        return rep[torch.randperm(n, generator=g)].view(like.shape).view(torch.float8_e4m3fn)

    inp["k"] = fill(k_codes, inp["k"])
    inp["v"] = fill(v_codes, inp["v"])
    inp["q"] = (inp["q"].float() / 64).to(torch.bfloat16)  # keeps logits moderate
    ws = _plain_workspace(msa, inp, 8, 2, 4) if route == "in_kernel" else None
    out, lse = _run_prefill(msa, inp, workspace=ws)
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label=f"e4m3_every_code_{route}")


def test_e4m3_bf16_copy_bit_exact(msa):
    """The decode pass writes K and V as bf16 right after the layout's regions
    of the workspace: bit-identical to torch's exact E4M3 -> bf16 cast for
    every code, NaN codes included (compared as NaN)."""
    lens = [700, 333]
    inp = _prefill_inputs(lens, lens, 8, 2, 4, seed=21, kv="e4m3")
    n = inp["k"].numel()
    codes = torch.arange(n, dtype=torch.int64) % 256
    inp["k"] = codes.to(torch.uint8).view(inp["k"].shape).view(torch.float8_e4m3fn)
    inp["v"] = (255 - codes).to(torch.uint8).view(inp["v"].shape).view(torch.float8_e4m3fn)
    inp["q"] = torch.zeros_like(inp["q"])
    tq = inp["q"].shape[0]
    base = msa.msa_sparse_attention_workspace_size(2, tq, 8, 2, 128, 4, max(lens), False)
    full = msa.msa_sparse_attention_workspace_size_kv(2, tq, 8, 2, 128, 4, max(lens), False,
                                                      torch.float8_e4m3fn, sum(lens))
    copy = (n * 2 + 255) // 256 * 256
    assert full == base + 2 * copy
    ws = torch.zeros(full, dtype=torch.uint8, device=DEV)
    _run_prefill(msa, inp, workspace=ws)
    for name, off in (("k", base), ("v", base + copy)):
        got = ws[off:off + 2 * n].view(torch.bfloat16).cpu().view(torch.int16)
        want = inp[name].to(torch.bfloat16).view(torch.int16)
        nan = torch.isnan(inp[name].to(torch.float32)).flatten()
        assert torch.isnan(got.view(torch.bfloat16)[nan]).all(), name
        assert torch.equal(got[~nan], want.flatten()[~nan]), name


def test_prefill_non_causal_and_scale(msa):
    inp = _prefill_inputs([200, 300], [200, 300], 8, 2, 4, seed=9)
    out, lse = _run_prefill(msa, inp, causal=False, scale=0.05)
    ref_out, ref_lse = _oracle(inp, causal=False, scale=0.05)
    check_attention(out, lse, ref_out, ref_lse, label="non_causal")


def test_prefill_edge_selections(msa):
    """Empty rows, duplicates, out-of-range ids, ids above the causal limit,
    -1 not at the tail, and an empty sequence in the batch."""
    inp = _prefill_inputs([300, 0, 257], [300, 0, 257], 8, 2, 4, seed=4)
    q2k = inp["q2k_indices"]
    q2k[0, 0:20, :] = -1                        # empty rows
    q2k[1, 30, :] = torch.tensor([1, 1, 1, 1])  # duplicates of a block above the limit
    q2k[0, 200, :] = torch.tensor([0, -1, 2, 77])
    q2k[1, 299, :] = torch.tensor([2, 1, 0, 0])  # descending, with a duplicate
    q2k[0, 310, :] = torch.tensor([5, 6, 7, 8])  # all beyond the sequence
    out, lse = _run_prefill(msa, inp)
    ref_out, ref_lse = _oracle(inp)
    assert np.isneginf(ref_lse[0:20, :4]).all()  # KV head 0 serves query heads 0-3
    check_attention(out, lse, ref_out, ref_lse, label="edges")


def _paged(inp_flat, lens_k, extra_pages=5, seed=0, bad_page=False):
    """Scatter flat K/V into a permuted page pool (tails filled with other values)."""
    g = torch.Generator().manual_seed(seed)
    k, v = inp_flat["k"], inp_flat["v"]
    hkv, d = k.shape[1], k.shape[2]
    pages = [(n + 127) // 128 for n in lens_k]
    npg = sum(pages) + extra_pages
    perm = torch.randperm(npg, generator=g)
    kp = torch.randn(npg, hkv, 128, d, generator=g).to(k.dtype)
    vp = torch.randn(npg, hkv, 128, d, generator=g).to(v.dtype)
    pt = torch.zeros(len(lens_k), max(pages) + 1, dtype=torch.int32)
    c = off = 0
    for b, n in enumerate(lens_k):
        for t in range(pages[b]):
            p = int(perm[off])
            off += 1
            pt[b, t] = p
            seg = slice(c + 128 * t, c + min(n, 128 * (t + 1)))
            kp[p, :, :seg.stop - seg.start] = k[seg].permute(1, 0, 2)
            vp[p, :, :seg.stop - seg.start] = v[seg].permute(1, 0, 2)
        c += n
    if bad_page:
        pt[0, 1] = npg + 100  # unmapped page: contributes no keys
    out = dict(inp_flat)
    out.update(k=kp, v=vp, page_table=pt, seqused_k=torch.tensor(lens_k, dtype=torch.int32))
    out.pop("cu_seqlens_k")
    return out


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_prefill_paged(msa, kv):
    lens_q, lens_k = [40, 300], [700, 300]
    flat = _prefill_inputs(lens_q, lens_k, 8, 2, 5, seed=12, kv=kv)
    inp = _paged(flat, lens_k, seed=3, bad_page=True)
    out, lse = _run_prefill(msa, inp)
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label=f"paged_{kv}")


def test_prefill_deterministic(msa):
    inp = _prefill_inputs([700, 300], [700, 300], 8, 2, 6, seed=2)
    o1, l1 = _run_prefill(msa, inp)
    o2, l2 = _run_prefill(msa, inp)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ---------------------------------------------------------------- paged decode
DECODE_CASES = [
    # name, seqlen_q, seqused, hq, hkv, topk
    ("sq1_g16", 1, [8192, 300, 129, 128, 1000], 32, 2, 16),
    ("sq4_g16", 4, [5000, 300, 130, 4], 32, 2, 16),
    ("sq2_g8", 2, [2000, 700], 16, 2, 8),
    ("sq3_g4", 3, [1500, 257, 10], 8, 2, 5),
    ("sq1_mha", 1, [600, 128], 4, 4, 3),
    ("sq4_g16_topk64", 4, [20000], 16, 1, 64),
    # multi-token decode: 5..32 query tokens per request (one or several tiles)
    ("sq5_g16", 5, [3000, 400], 32, 2, 16),
    ("sq8_g16", 8, [4000, 130], 32, 2, 16),
    ("sq8_g8", 8, [2500, 900, 260], 16, 2, 16),
    ("sq16_g16", 16, [5000], 32, 2, 16),
    ("sq32_g16", 32, [6000, 1000], 32, 2, 16),
    # G above 16 on the decode route (any G up to 128 is accepted)
    ("sq1_g32", 1, [9000, 300, 129, 4000], 64, 2, 16),
    ("sq4_g32", 4, [7000, 260, 2000], 64, 2, 12),
    ("sq2_g64", 2, [5000, 130, 3000], 128, 2, 8),
    ("sq1_g128", 1, [4000, 700, 129], 128, 1, 16),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_decode_parity(msa, case):
    name, sq, seqused, hq, hkv, topk = case
    spec = workloads.DecodeSpec(name, len(seqused), (1, 1), hq, hkv, topk, seqlen_q=sq)
    g = torch.Generator().manual_seed(len(name))
    cu_q = torch.arange(0, len(seqused) * sq + 1, sq, dtype=torch.int32)
    pages = [(n + 127) // 128 for n in seqused]
    npg = sum(pages) + 3
    perm = torch.randperm(npg, generator=g).to(torch.int32)
    pt = torch.zeros(len(seqused), max(pages), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, :n] = perm[off:off + n]
        off += n
    k = torch.randn(npg, hkv, 128, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(npg, hkv, 128, 128, generator=g).to(torch.bfloat16)
    q = torch.randn(len(seqused) * sq, hq, 128, generator=g).to(torch.bfloat16)
    pos = workloads.query_positions(cu_q, seqused)
    q2k = workloads.select_blocks(pos, hkv, topk, g)
    q2k[0, 0, 0] = q2k[0, 0, 0]
    if len(seqused) > 1:
        pt[1, 0] = npg + 7  # an unmapped page
    inp = dict(q=q, k=k, v=v, q2k_indices=q2k, cu_seqlens_q=cu_q, page_table=pt,
               seqused_k=torch.tensor(seqused, dtype=torch.int32))
    out, lse = _run_prefill(msa, inp, max_seqlen_q=sq)
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label=name)


def _decode_inputs(g, seqused, sq, hq, hkv, topk, npg_extra=3, dtype=torch.bfloat16):
    cu_q = torch.arange(0, len(seqused) * sq + 1, sq, dtype=torch.int32)
    pages = [(n + 127) // 128 for n in seqused]
    npg = sum(pages) + npg_extra
    perm = torch.randperm(npg, generator=g).to(torch.int32)
    pt = torch.zeros(len(seqused), max(pages), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, :n] = perm[off:off + n]
        off += n
    k = torch.randn(npg, hkv, 128, 128, generator=g).to(dtype)
    v = torch.randn(npg, hkv, 128, 128, generator=g).to(dtype)
    q = torch.randn(len(seqused) * sq, hq, 128, generator=g).to(dtype)
    q2k = workloads.select_blocks(workloads.query_positions(cu_q, seqused), hkv, topk, g)
    return dict(q=q, k=k, v=v, q2k_indices=q2k, cu_seqlens_q=cu_q, page_table=pt,
                seqused_k=torch.tensor(seqused, dtype=torch.int32))


# ---------------------------------------------------------------- packed NVFP4 paged K/V
# Global scales (K folds into the softmax scale, V into out), chosen so that
# the decoded K and V have about unit RMS like the bf16 cases (the pool's
# E2M1 x block-scale values have RMS about 5): the absolute output
# tolerance assumes outputs of order one.
NVFP4_KGS, NVFP4_VGS = 0.25, 0.125


def _nvfp4_inputs(g, seqused, lens_q, hq, hkv, topk, bad_page=False):
    cu_q = workloads.cu_from_lengths(lens_q)
    pages = [(n + 127) // 128 for n in seqused]
    npg = sum(pages) + 3
    perm = torch.randperm(npg, generator=g).to(torch.int32)
    pt = torch.zeros(len(seqused), max(pages) + 1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, :n] = perm[off:off + n]
        off += n
    if bad_page:
        pt[0, 1] = npg + 100  # unmapped: neither read nor attended
    pool = workloads.nvfp4_pool(npg, hkv, g, "cpu")
    q = torch.randn(int(cu_q[-1]), hq, 128, generator=g).to(torch.bfloat16)
    q2k = workloads.select_blocks(workloads.query_positions(cu_q, seqused), hkv, topk, g)
    return dict(q=q, pool=pool, q2k_indices=q2k, cu_seqlens_q=cu_q, page_table=pt,
                seqused_k=torch.tensor(seqused, dtype=torch.int32)), npg


def _nvfp4_run(msa, dev, hkv, runner=False, plain_workspace=False):
    k, ks, v, vs = msa.nvfp4_views(dev["pool"], hkv)
    kw = dict(page_table=dev["page_table"], seqused_k=dev["seqused_k"],
              k_global_scale=NVFP4_KGS, v_global_scale=NVFP4_VGS, return_softmax_lse=True)
    if plain_workspace:  # the paged size only: NVFP4 is decoded inside the attention kernel
        cu = dev["cu_seqlens_q"]
        n = msa.msa_sparse_attention_workspace_size(
            cu.numel() - 1, dev["q"].shape[0], dev["q"].shape[1], hkv, 128,
            dev["q2k_indices"].shape[2], int((cu[1:] - cu[:-1]).max()), True)
        kw["workspace"] = torch.empty(n, dtype=torch.uint8, device=DEV)
    if runner:
        r = msa.Nvfp4AttentionRunner(dev["q"], k, ks, v, vs, dev["q2k_indices"],
                                     dev["cu_seqlens_q"], **kw)
        out, lse = r.run()
        out, lse = out.clone(), lse.clone()
        r.close()
    else:
        out, lse = msa.msa_sparse_attention_nvfp4_paged(dev["q"], k, ks, v, vs, dev["q2k_indices"],
                                                        dev["cu_seqlens_q"], **kw)
    torch.cuda.synchronize()
    fault_clear(msa)
    return out, lse


NVFP4_CASES = [
    # name, seqused, lens_q, hq, hkv, topk, bad_page
    ("sq1_g16", [3000, 900, 129, 128, 4000], [1] * 5, 32, 2, 16, False),
    ("sq4_g16_unmapped", [2000, 300, 130], [4] * 3, 32, 2, 16, True),
    ("sq3_g4", [1500, 257, 10], [3, 3, 3], 8, 2, 5, False),
    ("prefill_lq_le_lk", [700, 300], [40, 300], 8, 2, 6, True),
    # prefill-sized: the default workspace takes the bf16 page-pool route
    ("prefill_pool_route", [700, 300], [700, 300], 8, 2, 6, True),
]


@pytest.mark.parametrize("case", NVFP4_CASES, ids=[c[0] for c in NVFP4_CASES])
def test_nvfp4_paged_parity(msa, case):
    """Packed NVFP4 paged K/V against the oracle on the decoded values (E2M1
    nibbles x E4M3 block scales x global scales), decode and prefill shapes,
    with an unmapped page."""
    name, seqused, lens_q, hq, hkv, topk, bad = case
    g = torch.Generator().manual_seed(len(name) * 31 + topk)
    host, npg = _nvfp4_inputs(g, seqused, lens_q, hq, hkv, topk, bad_page=bad)
    out, lse = _nvfp4_run(msa, to_dev(host, DEV), hkv)
    kf, vf = oracle.nvfp4_dequant(host["pool"], hkv, 128, NVFP4_KGS, NVFP4_VGS)
    ref_out, ref_lse = oracle.sparse_attention(
        host["q"], kf, vf, host["q2k_indices"], host["cu_seqlens_q"], causal=True,
        page_table=host["page_table"], seqused_k=host["seqused_k"], num_pages=npg)
    check_attention(out, lse, ref_out, ref_lse, label=f"nvfp4_{name}")


def test_nvfp4_routes_agree(msa):
    """A prefill-sized call on both routes, the bf16 page pool (default
    workspace) and the in-kernel decode (paged workspace size only), each
    against the oracle."""
    g = torch.Generator().manual_seed(23)
    host, npg = _nvfp4_inputs(g, [1100, 260, 129], [1100, 260, 129], 8, 2, 8, bad_page=True)
    dev = to_dev(host, DEV)
    kf, vf = oracle.nvfp4_dequant(host["pool"], 2, 128, NVFP4_KGS, NVFP4_VGS)
    ref_out, ref_lse = oracle.sparse_attention(
        host["q"], kf, vf, host["q2k_indices"], host["cu_seqlens_q"], causal=True,
        page_table=host["page_table"], seqused_k=host["seqused_k"], num_pages=npg)
    for plain in (False, True):
        out, lse = _nvfp4_run(msa, dev, 2, plain_workspace=plain)
        check_attention(out, lse, ref_out, ref_lse, label=f"nvfp4_route_plain{plain}")


def test_e4m3_paged_pool_route(msa):
    """Prefill-sized paged E4M3: the default workspace decodes the pages into
    a bf16 pool (renumbered table, one unmapped page); the paged size keeps
    the in-kernel conversion; both against the oracle."""
    lens = [700, 300]
    flat = _prefill_inputs(lens, lens, 8, 2, 5, seed=31, kv="e4m3")
    inp = _paged(flat, lens, seed=5, bad_page=True)
    ref_out, ref_lse = _oracle(inp)
    out, lse = _run_prefill(msa, inp)
    check_attention(out, lse, ref_out, ref_lse, label="e4m3_paged_pool")
    n = msa.msa_sparse_attention_workspace_size(2, sum(lens), 8, 2, 128, 5, max(lens), True)
    out2, lse2 = _run_prefill(msa, inp, workspace=torch.empty(n, dtype=torch.uint8, device=DEV))
    check_attention(out2, lse2, ref_out, ref_lse, label="e4m3_paged_in_kernel")


def test_nvfp4_pool_route_graph_replay(msa):
    """The prepared NVFP4 forward on its page-pool route (page decode, union
    and attention kernels) captured once into a CUDA graph; each replay reads
    the pool and queries refilled in place."""
    g = torch.Generator().manual_seed(71)
    seqused = [900, 300]
    host, npg = _nvfp4_inputs(g, seqused, seqused, 8, 2, 6)
    dev = to_dev(host, DEV)
    k, ks, v, vs = msa.nvfp4_views(dev["pool"], 2)
    r = msa.Nvfp4AttentionRunner(dev["q"], k, ks, v, vs, dev["q2k_indices"], dev["cu_seqlens_q"],
                                 page_table=dev["page_table"], seqused_k=dev["seqused_k"],
                                 k_global_scale=NVFP4_KGS, v_global_scale=NVFP4_VGS,
                                 return_softmax_lse=True)
    r.run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            r.run(stream=stream)
    torch.cuda.synchronize()
    for trial in range(2):
        gt = torch.Generator().manual_seed(500 + trial)
        new_pool = workloads.nvfp4_pool(npg, 2, gt, "cpu")
        new_q = torch.randn(host["q"].shape, generator=gt).to(torch.bfloat16)
        dev["pool"].copy_(new_pool)
        dev["q"].copy_(new_q)
        graph.replay()
        torch.cuda.synchronize()
        fault_clear(msa)
        kf, vf = oracle.nvfp4_dequant(new_pool, 2, 128, NVFP4_KGS, NVFP4_VGS)
        ref_out, ref_lse = oracle.sparse_attention(
            new_q, kf, vf, host["q2k_indices"], host["cu_seqlens_q"], causal=True,
            page_table=host["page_table"], seqused_k=host["seqused_k"], num_pages=npg)
        check_attention(r.out, r.lse, ref_out, ref_lse, label=f"nvfp4_graph_{trial}")
    r.close()


def test_nvfp4_runner_matches_forward(msa):
    """The prepared NVFP4 forward (prepare once, run) gives the direct call's bits."""
    g = torch.Generator().manual_seed(5)
    host, _ = _nvfp4_inputs(g, [2500, 700, 129], [1, 1, 1], 32, 2, 16)
    dev = to_dev(host, DEV)
    o1, l1 = _nvfp4_run(msa, dev, 2)
    o2, l2 = _nvfp4_run(msa, dev, 2, runner=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_graph_replay(msa):
    """The forward is captured once into a CUDA graph with caller-owned out, lse
    and workspace and explicit sizes (no allocation, no host read-back); each
    replay computes on whatever inputs were copied into the captured buffers."""
    seqused, sq, hq, hkv, topk = [3000, 900, 129], 1, 32, 2, 16
    g = torch.Generator().manual_seed(7)
    host = _decode_inputs(g, seqused, sq, hq, hkv, topk)
    dev = to_dev(host, DEV)
    out = torch.empty_like(dev["q"])
    lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device=DEV)
    need = msa.msa_sparse_attention_workspace_size(len(seqused), dev["q"].shape[0], hq, hkv, 128,
                                                   topk, sq, True)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)

    def call():
        msa.msa_sparse_attention_fwd(dev["q"], dev["k"], dev["v"], dev["q2k_indices"],
                                     dev["cu_seqlens_q"], None, causal=True,
                                     page_table=dev["page_table"], seqused_k=dev["seqused_k"],
                                     max_seqlen_q=sq, out=out, lse=lse, workspace=ws)

    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            call()
    torch.cuda.synchronize()
    for trial in range(2):
        new = _decode_inputs(torch.Generator().manual_seed(100 + trial), seqused, sq, hq, hkv,
                             topk)
        for key in ("q", "k", "v", "q2k_indices", "page_table"):
            dev[key].copy_(new[key])
        graph.replay()
        torch.cuda.synchronize()
        fault_clear(msa)
        ref_out, ref_lse = _oracle(new)
        check_attention(out, lse, ref_out, ref_lse, label=f"graph_replay_{trial}")


@pytest.mark.parametrize("sq", [1, 4])
def test_decode_f16(msa, sq):
    seqused = [4000, 700, 129]
    inp = _decode_inputs(torch.Generator().manual_seed(40 + sq), seqused, sq, 32, 2, 16,
                         dtype=torch.float16)
    out, lse = _run_prefill(msa, inp, max_seqlen_q=sq)
    assert out.dtype == torch.float16
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label=f"f16_decode_sq{sq}")


@pytest.mark.parametrize("sq", [1, 4])
def test_decode_e4m3(msa, sq):
    """Paged E4M3 K/V at decode size: the converter-warp instance with the
    union split over work items and the merge of the partials."""
    seqused = [4000, 700, 129, 2600]
    inp = _decode_inputs(torch.Generator().manual_seed(60 + sq), seqused, sq, 32, 2, 16)
    inp["k"] = inp["k"].float().clamp(-448, 448).to(torch.float8_e4m3fn)
    inp["v"] = inp["v"].float().clamp(-448, 448).to(torch.float8_e4m3fn)
    out, lse = _run_prefill(msa, inp, max_seqlen_q=sq)
    ref_out, ref_lse = _oracle(inp)
    check_attention(out, lse, ref_out, ref_lse, label=f"e4m3_decode_sq{sq}")


def test_prepared_runner_matches_forward(msa):
    """A prepared forward gives the plain forward's bits, refilled inputs give
    fresh results, and its run captures into a CUDA graph."""
    seqused, sq, hq, hkv, topk = [2500, 900, 129], 4, 32, 2, 16
    host = _decode_inputs(torch.Generator().manual_seed(21), seqused, sq, hq, hkv, topk)
    dev = to_dev(host, DEV)
    kw = dict(causal=True, page_table=dev["page_table"], seqused_k=dev["seqused_k"],
              max_seqlen_q=sq, return_softmax_lse=True)
    ref_o, ref_l = msa.msa_sparse_attention_fwd(dev["q"], dev["k"], dev["v"], dev["q2k_indices"],
                                                dev["cu_seqlens_q"], None, **kw)
    runner = msa.SparseAttentionRunner(dev["q"], dev["k"], dev["v"], dev["q2k_indices"],
                                       dev["cu_seqlens_q"], None, **kw)
    o, l = runner.run()
    torch.cuda.synchronize()
    fault_clear(msa)
    assert torch.equal(o, ref_o) and torch.equal(l, ref_l)
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            runner.run()
    new = _decode_inputs(torch.Generator().manual_seed(22), seqused, sq, hq, hkv, topk)
    for key in ("q", "k", "v", "q2k_indices"):
        dev[key].copy_(new[key])
    graph.replay()
    torch.cuda.synchronize()
    fault_clear(msa)
    new["page_table"], new["seqused_k"] = host["page_table"], host["seqused_k"]
    ref_out, ref_lse = _oracle(new)
    check_attention(runner.out, runner.lse, ref_out, ref_lse, label="runner_graph")
    runner.close()


def test_decode_deterministic(msa):
    g = torch.Generator().manual_seed(0)
    seqused = [3000, 900]
    cu_q = torch.arange(0, 2 * 4 + 1, 4, dtype=torch.int32)
    pt = torch.arange(0, 48, dtype=torch.int32).view(2, 24)
    k = torch.randn(48, 1, 128, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(48, 1, 128, 128, generator=g).to(torch.bfloat16)
    q = torch.randn(8, 16, 128, generator=g).to(torch.bfloat16)
    q2k = workloads.select_blocks(workloads.query_positions(cu_q, seqused), 1, 16, g)
    inp = dict(q=q, k=k, v=v, q2k_indices=q2k, cu_seqlens_q=cu_q, page_table=pt,
               seqused_k=torch.tensor(seqused, dtype=torch.int32))
    o1, l1 = _run_prefill(msa, inp, max_seqlen_q=4)
    o2, l2 = _run_prefill(msa, inp, max_seqlen_q=4)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ---------------------------------------------------------------- proxy score
PAGED_PROXY_CASES = [
    # name, seqused, query tokens per request (None: as many as keys), hq, hkv, reduce,
    # pass max_seqlen_q (decode: one M tile per query tile)
    ("decode_sq1_reduce_g16", [8192, 300, 129, 128, 3000], 1, 32, 2, True, True),
    ("decode_sq4_perhead_g8", [5000, 700], 4, 16, 2, False, True),
    ("decode_sq1_reduce_long", [40000, 20000], 1, 64, 4, True, True),
    ("decode_sq2_reduce_two_m_tiles", [3000, 900, 128], 2, 32, 2, True, False),
    ("paged_prefill_reduce_g8", [300, 517], None, 16, 2, True, False),
]


@pytest.mark.parametrize("case", PAGED_PROXY_CASES, ids=[c[0] for c in PAGED_PROXY_CASES])
def test_proxy_paged_parity(msa, case):
    """Paged K (one page per block, a page table, seqused_k), including an
    unmapped page; decode-sized cases run with their block columns split over
    many CTAs."""
    name, seqused, sq, hq, hkv, red, pass_sq = case
    g = torch.Generator().manual_seed(len(name) + 300)
    lens_q = list(seqused) if sq is None else [sq] * len(seqused)
    cu_q = workloads.cu_from_lengths(lens_q)
    pages = [(n + 127) // 128 for n in seqused]
    npg = sum(pages) + 2
    perm = torch.randperm(npg, generator=g).to(torch.int32)
    pt = torch.zeros(len(seqused), max(pages), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, :n] = perm[off:off + n]
        off += n
    pt[1, 0] = npg + 5  # an unmapped page: its block holds no key
    k = torch.randn(npg, hkv, 128, 128, generator=g).to(torch.bfloat16)
    q = torch.randn(sum(lens_q), hq, 128, generator=g).to(torch.bfloat16)
    su = torch.tensor(seqused, dtype=torch.int32)
    T = max(pages) + 1
    got = msa.msa_proxy_score(q.to(DEV), k.to(DEV), cu_q.to(DEV), None, causal=True,
                              max_k_tiles=T, reduce_heads=red, page_table=pt.to(DEV),
                              seqused_k=su.to(DEV), max_seqlen_q=max(lens_q) if pass_sq else None)
    torch.cuda.synchronize()
    fault_clear(msa)
    rows = None
    if q.shape[0] > 600:
        rows = torch.tensor(sorted(set([0, 1, 127, 128, 129, q.shape[0] - 1] +
                                       list(range(0, q.shape[0], 97)))), dtype=torch.int32)
    ref = oracle.proxy_score(q, k, cu_q, None, page_table=pt, seqused_k=su, causal=True,
                             max_k_tiles=T, reduce_heads=red, rows=rows)
    gpu = got.cpu().numpy()
    if rows is not None:
        gpu = gpu[:, :, rows.long().numpy()]
    check_proxy(gpu, ref, label=name)


PROXY_CASES = [
    # name, lens_q, lens_k, hq, hkv, reduce, causal, extra_tiles
    ("reduce_g8", [300, 517], [300, 517], 16, 2, True, True, 0),
    ("perhead_g8", [300], [300], 16, 2, False, True, 2),
    ("reduce_g4_lq_lt_lk", [50, 129], [700, 129], 8, 2, True, True, 1),
    ("reduce_mha", [400], [400], 2, 2, True, True, 0),
    ("perhead_g3", [200], [260], 6, 2, False, True, 0),
    ("reduce_g32", [300], [300], 32, 1, True, False, 0),
]


@pytest.mark.parametrize("case", PROXY_CASES, ids=[c[0] for c in PROXY_CASES])
def test_proxy_parity(msa, case):
    name, lq, lk, hq, hkv, red, causal, extra = case
    g = torch.Generator().manual_seed(len(name) + 100)
    q = torch.randn(sum(lq), hq, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(sum(lk), hkv, 128, generator=g).to(torch.bfloat16)
    cu_q, cu_k = workloads.cu_from_lengths(lq), workloads.cu_from_lengths(lk)
    T = max((n + 127) // 128 for n in lk) + extra
    ref = oracle.proxy_score(q, k, cu_q, cu_k, causal=causal, max_k_tiles=T, reduce_heads=red)
    got = msa.msa_proxy_score(q.to(DEV), k.to(DEV), cu_q.to(DEV), cu_k.to(DEV), causal=causal,
                              max_k_tiles=T, reduce_heads=red)
    torch.cuda.synchronize()
    fault_clear(msa)
    check_proxy(got, ref, label=name)
