"""GPU parity of the swapped-orientation prefill kernel, and right-aligned edge
cases of both attention kernels, against the fp64 oracle.

The forward picks one of two kernels that compute the same result (see
msa_prefill_tile_tokens in include/msa.h); msa_set_prefill_route forces one,
so each case here runs through both where both apply. The swapped kernel's
union metadata adds one mask of member tokens per union block, checked bit
for bit against the oracle's membership bits (transposed here).
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
    yield m
    m.msa_set_prefill_route(0)


def _inputs(lens_q, lens_k, hq, hkv, topk, seed, kv="bf16", first_prev=False):
    g = torch.Generator().manual_seed(seed)
    d = 128
    dt = torch.float16 if kv == "f16" else torch.bfloat16
    tq, tk = sum(lens_q), sum(lens_k)
    q = torch.randn(tq, hq, d, generator=g).to(dt)
    k = torch.randn(tk, hkv, d, generator=g).to(dt)
    v = torch.randn(tk, hkv, d, generator=g).to(dt)
    cu_q = workloads.cu_from_lengths(lens_q)
    cu_k = workloads.cu_from_lengths(lens_k)
    pos = workloads.query_positions(cu_q, lens_k)
    q2k = workloads.select_blocks(pos, hkv, topk, g, first=first_prev, prev=first_prev)
    return dict(q=q, k=k, v=v, q2k_indices=q2k, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)


def _run(msa, inp, route, causal=True, scale=None):
    msa.msa_set_prefill_route(route)
    try:
        g = to_dev(inp, DEV)
        out, lse = msa.msa_sparse_attention_fwd(
            g["q"], g["k"], g["v"], g["q2k_indices"], g["cu_seqlens_q"], g.get("cu_seqlens_k"),
            causal=causal, softmax_scale=scale, page_table=g.get("page_table"),
            seqused_k=g.get("seqused_k"), return_softmax_lse=True)
        torch.cuda.synchronize()
        fault_clear(msa)
    finally:
        msa.msa_set_prefill_route(0)
    return out, lse


def _oracle(inp, causal=True, scale=None):
    s = f32(scale if scale is not None else 128 ** -0.5)
    return oracle.sparse_attention(inp["q"], inp["k"], inp["v"], inp["q2k_indices"],
                                   inp["cu_seqlens_q"], inp.get("cu_seqlens_k"), causal=causal,
                                   softmax_scale=s, page_table=inp.get("page_table"),
                                   seqused_k=inp.get("seqused_k"))


def _both(msa, inp, label, causal=True, scale=None):
    ref_out, ref_lse = _oracle(inp, causal=causal, scale=scale)
    for route, name in ((1, "union_tile"), (2, "swapped")):
        out, lse = _run(msa, inp, route, causal=causal, scale=scale)
        check_attention(out, lse, ref_out, ref_lse, label=f"{label}/{name}")
    return ref_out, ref_lse


# ---------------------------------------------------------------- union member masks
@pytest.mark.parametrize("W,topk,lens", [(32, 16, [700, 45, 1000]), (32, 64, [1500]),
                                         (16, 8, [300, 17]), (8, 3, [129, 400]),
                                         (1, 4, [50])])
def test_block_members_bit_exact(msa, W, topk, lens):
    g = torch.Generator().manual_seed(W + topk)
    hkv = 2
    cu = workloads.cu_from_lengths(lens)
    pos = workloads.query_positions(cu, lens)
    q2k = workloads.select_blocks(pos, hkv, topk, g, first=True, prev=True)
    q2k[0, 3, 0] = 999            # beyond the sequence
    q2k[1, 9, -1] = q2k[1, 9, 0]  # duplicate
    q2k[0, 11, :] = -1            # empty row
    ref_len, ref_blk, ref_mem = oracle.build_union(q2k, cu, cu, causal=True, tile_tokens=W)
    T = ref_len.shape[1]
    # Transpose of the oracle's membership bits: bit w of entry j.
    want = np.zeros(ref_blk.shape, dtype=np.uint32)
    for h in range(hkv):
        for t in range(T):
            for j in range(int(ref_len[h, t])):
                for w in range(W):
                    if (int(ref_mem[h, t, w, j >> 5]) >> (j & 31)) & 1:
                        want[h, t, j] |= np.uint32(1 << w)
    ulen, ublk, mem, bmem, info = msa.msa_build_union_block_members(
        q2k.to(DEV), cu.to(DEV), cu.to(DEV), causal=True, tile_tokens=W)
    torch.cuda.synchronize()
    assert np.array_equal(ulen[:, :T].cpu().numpy(), ref_len)
    assert np.array_equal(ublk[:, :T].cpu().numpy(), ref_blk)
    assert np.array_equal(mem[:, :T].cpu().numpy().view(np.uint32), ref_mem)
    assert np.array_equal(bmem[:, :T].cpu().numpy().view(np.uint32), want)


def test_block_members_paged(msa):
    g = torch.Generator().manual_seed(5)
    lens_q, seqused = [40, 200], [900, 260]
    cu = workloads.cu_from_lengths(lens_q)
    pos = workloads.query_positions(cu, seqused)
    q2k = workloads.select_blocks(pos, 2, 6, g)
    su = torch.tensor(seqused, dtype=torch.int32)
    ref_len, ref_blk, ref_mem = oracle.build_union(q2k, cu, seqused_k=su, max_pages=5,
                                                   causal=True, tile_tokens=32)
    got = msa.msa_build_union_block_members(q2k.to(DEV), cu.to(DEV), seqused_k=su.to(DEV),
                                            max_pages=5, causal=True, tile_tokens=32)
    T = ref_len.shape[1]
    bm = got[3][:, :T].cpu().numpy().view(np.uint32)
    for h in range(2):
        for t in range(T):
            for j in range(int(ref_len[h, t])):
                for w in range(32):
                    bit = (int(ref_mem[h, t, w, j >> 5]) >> (j & 31)) & 1
                    assert ((int(bm[h, t, j]) >> w) & 1) == bit


# ---------------------------------------------------------------- parity
SWAPPED_CASES = [
    # name, lens_q, lens_k, hq, hkv, topk, kv, first_prev
    ("g8_varlen_ragged", [300, 129, 517, 33], [300, 129, 517, 33], 16, 2, 6, "bf16", True),
    ("g8_lq_lt_lk", [64, 200, 1], [700, 333, 129], 16, 2, 6, "bf16", False),
    ("g8_topk16", [1300], [1300], 8, 1, 16, "bf16", True),
    ("g8_topk1", [400], [400], 8, 1, 1, "bf16", False),
    ("g8_topk64", [1500], [1500], 8, 1, 64, "bf16", False),
    ("g16", [450, 100], [450, 100], 32, 2, 5, "bf16", True),
    ("g24", [333], [333], 24, 1, 3, "bf16", False),
    ("g32", [260, 300], [260, 300], 32, 1, 4, "bf16", False),
    ("g64", [300], [300], 64, 1, 3, "bf16", True),
    ("f16_g8", [300, 517], [300, 900], 16, 2, 8, "f16", True),
]


@pytest.mark.parametrize("case", SWAPPED_CASES, ids=[c[0] for c in SWAPPED_CASES])
def test_swapped_parity(msa, case):
    name, lq, lk, hq, hkv, topk, kv, fp = case
    msa.msa_set_prefill_route(2)
    try:
        tiles = msa.msa_prefill_tile_tokens(len(lq), sum(lq), hq, hkv, topk, max(lq))
    finally:
        msa.msa_set_prefill_route(0)
    assert tiles == min(32, 256 // (hq // hkv), max(lq))  # route 2 runs the swapped kernel
    inp = _inputs(lq, lk, hq, hkv, topk, seed=len(name) + 100, kv=kv, first_prev=fp)
    _both(msa, inp, name)


def test_swapped_non_causal_scale(msa):
    inp = _inputs([200, 333], [200, 333], 16, 2, 4, seed=31)
    _both(msa, inp, "non_causal", causal=False, scale=0.05)


def test_swapped_edge_selections(msa):
    """Empty rows, duplicates, ids beyond the sequence or above the causal
    limit, -1 before valid ids, and an empty sequence in the batch."""
    inp = _inputs([300, 0, 257], [300, 0, 257], 16, 2, 4, seed=4)
    q2k = inp["q2k_indices"]
    q2k[0, 0:40, :] = -1
    q2k[1, 30, :] = torch.tensor([1, 1, 1, 1])
    q2k[0, 200, :] = torch.tensor([0, -1, 2, 77])
    q2k[1, 299, :] = torch.tensor([2, 1, 0, 0])
    q2k[0, 310, :] = torch.tensor([5, 6, 7, 8])
    ref_out, ref_lse = _both(msa, inp, "edges")
    assert np.isneginf(ref_lse[0:40, :8]).all()


def test_swapped_whole_tile_empty(msa):
    """A 32-token tile whose tokens selected nothing: out 0, lse -inf."""
    inp = _inputs([128, 64], [128, 64], 8, 1, 2, seed=8)
    inp["q2k_indices"][0, 32:64, :] = -1
    ref_out, ref_lse = _both(msa, inp, "empty_tile")
    assert np.isneginf(ref_lse[32:64]).all()


def _paged(inp, lens_k, seed, bad_page):
    g = torch.Generator().manual_seed(seed)
    k, v = inp["k"], inp["v"]
    hkv = k.shape[1]
    pages = [(n + 127) // 128 for n in lens_k]
    npg = sum(pages) + 4
    perm = torch.randperm(npg, generator=g)
    kp = torch.randn(npg, hkv, 128, 128, generator=g).to(k.dtype)
    vp = torch.randn(npg, hkv, 128, 128, generator=g).to(v.dtype)
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
        pt[0, 1] = npg + 50  # unmapped: contributes no keys
    out = dict(inp)
    out.update(k=kp, v=vp, page_table=pt, seqused_k=torch.tensor(lens_k, dtype=torch.int32))
    out.pop("cu_seqlens_k")
    return out


def test_swapped_paged(msa):
    lens_q, lens_k = [100, 300], [700, 300]
    flat = _inputs(lens_q, lens_k, 16, 2, 5, seed=12)
    _both(msa, _paged(flat, lens_k, seed=3, bad_page=True), "paged")


def test_swapped_deterministic(msa):
    inp = _inputs([700, 300], [700, 300], 16, 2, 6, seed=2)
    o1, l1 = _run(msa, inp, 2)
    o2, l2 = _run(msa, inp, 2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ---------------------------------------------------------------- right-aligned edges
def test_causal_lq_gt_lk(msa):
    """Causal with more queries than keys: rows at a negative position
    (Lk - Lq + i < 0) see nothing and give out 0, lse -inf, even with block
    ids planted in their rows; the rest see the right-aligned prefix."""
    lens_q, lens_k = [300, 200], [100, 330]
    inp = _inputs(lens_q, lens_k, 16, 2, 4, seed=41)
    inp["q2k_indices"][:, 0:150, 0] = 0  # rows of sequence 0 at negative positions
    ref_out, ref_lse = _both(msa, inp, "lq_gt_lk")
    assert np.isneginf(ref_lse[:200]).all() and not np.isneginf(ref_lse[200:300]).any()


def test_non_causal_lq_ne_lk(msa):
    """Non-causal with Lq != Lk in both directions: every selected block
    within the sequence is visible to every query row."""
    lens_q, lens_k = [300, 90, 40], [120, 700, 40]
    g = torch.Generator().manual_seed(43)
    inp = _inputs(lens_q, lens_k, 16, 2, 4, seed=43)
    # Selections drawn over all of each sequence's blocks (not only the causal prefix).
    heads = []
    for _h in range(2):
        rows = []
        for lq, lk in zip(lens_q, lens_k):
            nb = (lk + 127) // 128
            for _ in range(lq):
                sel = torch.randperm(nb, generator=g)[:4].sort().values
                rows.append(torch.cat([sel, torch.full((4 - sel.numel(),), -1)]))
        heads.append(torch.stack(rows))
    inp["q2k_indices"] = torch.stack(heads).to(torch.int32)
    _both(msa, inp, "non_causal_lq_ne_lk", causal=False)


def test_g1_topk64_wide_union(msa):
    """G = 1 with top-64: the union-tile kernel's tiles are 128 tokens, so a
    tile's union can reach 128 * 64 = 8192 entries (membership words and
    union lists at full capacity)."""
    lens = [4096, 300]
    inp = _inputs(lens, lens, 2, 2, 64, seed=44)
    assert msa.msa_prefill_tile_tokens(2, sum(lens), 2, 2, 64, max(lens)) == 128
    ref_out, ref_lse = _oracle(inp)
    out, lse = _run(msa, inp, 0)
    check_attention(out, lse, ref_out, ref_lse, label="g1_topk64")
