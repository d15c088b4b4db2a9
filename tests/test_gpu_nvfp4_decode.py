"""GPU parity of the packed-NVFP4 decode kernel (decode-shaped calls: G <= 16
query heads per KV head, at most 16 query tokens per request).

"flashinfer.msa_ops.msa_sparse_attention", the packed-NVFP4 paged route:
K = e2m1 * block scale * k_global_scale, V likewise; "prepare_msa_nvfp4_sparse_
decode". Each (token, KV head) attends over the usable blocks of its own q2k
row, each once. The cases feed rows the pages do not promise (unsorted,
repeated, -1 in the middle, ids past the sequence or above the causal limit,
empty rows), topk 64, every G from 1 to 16, several query tokens per request
with causal limits inside the last block, NaN codes planted in the bytes past
the end of a sequence (never attended, so they must not reach the output),
requests without query tokens, more work units than the kernel's CTAs, and a
page pool whose pages are padded beyond the planar regions. Every result is
compared with the fp64 oracle on the decoded values.
"""
import pytest
import torch

import oracle
import workloads
from parity_util import check_attention, fault_clear, to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
KGS, VGS = 0.25, 0.125


@pytest.fixture(scope="module")
def msa():
    import block_sparse_top_msa_gb300 as m
    m.build()
    m.lib()
    return m


def _inputs(g, seqused, lens_q, hq, hkv, topk, pad=0, unmapped=False):
    """Paged NVFP4 inputs; `pad` extra bytes per page after the planar regions."""
    cu_q = workloads.cu_from_lengths(lens_q)
    pages = [(n + 127) // 128 for n in seqused]
    npg = sum(pages) + 2
    perm = torch.randperm(npg, generator=g).to(torch.int32)
    pt = torch.zeros(len(seqused), max(pages) + 1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, :n] = perm[off:off + n]
        off += n
    if unmapped and len(pages) > 1 and pages[1] > 1:
        pt[1, 0] = npg + 9  # an unmapped page: neither read nor attended
    pool = workloads.nvfp4_pool(npg, hkv, g, "cpu")
    if pad:
        wide = torch.randint(0, 256, (npg, pool.shape[1] + pad), generator=g,
                             dtype=torch.int32).to(torch.uint8)
        wide[:, :pool.shape[1]] = pool
        pool = wide
    q = torch.randn(int(cu_q[-1]), hq, 128, generator=g).to(torch.bfloat16)
    q2k = workloads.select_blocks(workloads.query_positions(cu_q, seqused), hkv, topk, g)
    return dict(q=q, pool=pool, q2k_indices=q2k, cu_seqlens_q=cu_q, page_table=pt,
                seqused_k=torch.tensor(seqused, dtype=torch.int32)), npg


def _views(pool, hkv):
    """(k, k_scale, v, v_scale) views of a planar pool whose rows may be padded."""
    npg, stride = pool.shape
    data, sc = hkv * 128 * 64, hkv * 128 * 8
    flat = pool.reshape(-1)

    def view(off, inner):
        return flat.as_strided((npg, hkv, 128, inner), (stride, 128 * inner, inner, 1), off)
    return view(0, 64), view(data, 8), view(data + sc, 64), view(2 * data + sc, 8)


def _run_and_check(msa, host, npg, hkv, label, max_seqlen_q=None):
    dev = to_dev(host, DEV)
    k, ks, v, vs = _views(dev["pool"], hkv)
    out, lse = msa.msa_sparse_attention_nvfp4_paged(
        dev["q"], k, ks, v, vs, dev["q2k_indices"], dev["cu_seqlens_q"],
        page_table=dev["page_table"], seqused_k=dev["seqused_k"], k_global_scale=KGS,
        v_global_scale=VGS, max_seqlen_q=max_seqlen_q, return_softmax_lse=True)
    torch.cuda.synchronize()
    fault_clear(msa)
    stride = host["pool"].shape[1]
    pool = host["pool"][:, :workloads.nvfp4_page_stride(hkv)].contiguous()
    assert pool.shape[1] <= stride
    kf, vf = oracle.nvfp4_dequant(pool, hkv, 128, KGS, VGS)
    ref_out, ref_lse = oracle.sparse_attention(
        host["q"], kf, vf, host["q2k_indices"], host["cu_seqlens_q"], causal=True,
        page_table=host["page_table"], seqused_k=host["seqused_k"], num_pages=npg)
    check_attention(out, lse, ref_out, ref_lse, label=label)
    return out, lse, ref_lse


def test_irregular_rows(msa):
    g = torch.Generator().manual_seed(401)
    seqused = [8192, 3000, 129, 128, 1, 1000, 5000]
    host, npg = _inputs(g, seqused, [1] * len(seqused), 32, 2, 8, unmapped=True)
    q2k = host["q2k_indices"]                                   # (hkv, tokens, topk)
    q2k[0, 0] = torch.tensor([60, 3, 60, 7, -1, 3, 0, 63])       # unsorted, repeated, -1 inside
    q2k[1, 0] = torch.tensor([-1, -1, 5, -1, 2, -1, -1, 9])      # padding first
    q2k[0, 1] = torch.tensor([0, 23, 24, 100, 5000, 2, 1, 1])    # ids past the sequence
    q2k[1, 2] = -1                                              # empty row: out 0, lse -inf
    q2k[0, 3] = torch.zeros(8, dtype=torch.int32)               # one block, eight times
    q2k[1, 4] = torch.arange(8, dtype=torch.int32)              # 1-token request: block 0 only
    q2k[0, 6] = torch.arange(39, 31, -1, dtype=torch.int32)     # strictly descending
    _, _, ref_lse = _run_and_check(msa, host, npg, 2, "fp4dec_irregular")
    assert torch.isinf(torch.as_tensor(ref_lse[2, 16:])).all()


def test_topk64_duplicates_across_halves(msa):
    g = torch.Generator().manual_seed(402)
    seqused = [20000, 9000, 12000]
    host, npg = _inputs(g, seqused, [1, 1, 1], 16, 2, 64)
    q2k = host["q2k_indices"]
    q2k[0, 0, 32:] = q2k[0, 0, :32]   # the second half repeats the first
    q2k[1, 1, 40] = q2k[1, 1, 3]
    q2k[1, 2, 63] = -1
    _run_and_check(msa, host, npg, 2, "fp4dec_topk64")


@pytest.mark.parametrize("G", [1, 2, 3, 8, 12, 16])
def test_group_sizes(msa, G):
    g = torch.Generator().manual_seed(410 + G)
    hkv = 2 if G > 1 else 4
    seqused = [4000, 777, 2049]
    host, npg = _inputs(g, seqused, [2, 1, 3], G * hkv, hkv, 12)
    _run_and_check(msa, host, npg, hkv, f"fp4dec_G{G}")


def test_multi_token_causal_tail(msa):
    """Eight query tokens per request: each token's last visible block is cut
    at its own position, so the visible-key count differs per token."""
    g = torch.Generator().manual_seed(420)
    seqused = [1000, 135, 4101, 640]
    host, npg = _inputs(g, seqused, [8, 8, 5, 16], 16, 2, 10, unmapped=True)
    _run_and_check(msa, host, npg, 2, "fp4dec_sq8_causal")


def test_nan_bytes_past_the_sequence(msa):
    """NaN block scales and arbitrary codes on the keys past seqused in the
    last page of each request: those keys are never attended, and neither a
    NaN K score nor 0 * NaN in PV may reach the output."""
    g = torch.Generator().manual_seed(430)
    seqused = [1000, 300, 129, 4000]
    hkv = 2
    host, npg = _inputs(g, seqused, [1, 2, 1, 3], 16, hkv, 8)
    pool = host["pool"]
    data, sc = hkv * 128 * 64, hkv * 128 * 8
    for b, n in enumerate(seqused):
        last = (n + 127) // 128 - 1
        page = int(host["page_table"][b, last])
        for h in range(hkv):
            for t in range(n - last * 128, 128):
                pool[page, data + h * 1024 + t * 8:data + h * 1024 + t * 8 + 8] = 0x7F  # K scales
                for s in range(8):  # V scales, 4 x 4 (token, scale) tiles
                    pool[page, 2 * data + sc + h * 1024 + 32 * (t // 4) + 16 * (s // 4)
                         + 4 * (s % 4) + t % 4] = 0xFF
    out, _, _ = _run_and_check(msa, host, npg, hkv, "fp4dec_nan_tail")
    assert torch.isfinite(out.float()).all()


def test_empty_requests_and_many_units(msa):
    """Requests with no query tokens between others, and more (token, KV head)
    units than the kernel runs CTAs, so each CTA takes several units."""
    g = torch.Generator().manual_seed(440)
    n = 420
    seqused = [int(x) for x in torch.randint(130, 3000, (n,), generator=g)]
    lens_q = [0 if i % 7 == 3 else 1 for i in range(n)]
    host, npg = _inputs(g, seqused, lens_q, 16, 2, 16)
    out, lse, _ = _run_and_check(msa, host, npg, 2, "fp4dec_many_units", max_seqlen_q=1)
    # the same launch again gives the same bits
    dev = to_dev(host, DEV)
    k, ks, v, vs = _views(dev["pool"], 2)
    out2, lse2 = msa.msa_sparse_attention_nvfp4_paged(
        dev["q"], k, ks, v, vs, dev["q2k_indices"], dev["cu_seqlens_q"],
        page_table=dev["page_table"], seqused_k=dev["seqused_k"], k_global_scale=KGS,
        v_global_scale=VGS, max_seqlen_q=1, return_softmax_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_padded_page_stride(msa):
    """Pages padded by 4 KB beyond the four planar regions (the stride is
    taken from the views)."""
    g = torch.Generator().manual_seed(450)
    host, npg = _inputs(g, [3000, 800, 2222], [1, 4, 2], 32, 4, 16, pad=4096)
    _run_and_check(msa, host, npg, 4, "fp4dec_padded_stride")


def test_negative_block_scales(msa):
    """E4M3 block scales with the sign bit set decode to negative scales on
    both sides."""
    g = torch.Generator().manual_seed(460)
    hkv = 2
    host, npg = _inputs(g, [2500, 900], [1, 1], 16, hkv, 12)
    pool = host["pool"]
    data, sc = hkv * 128 * 64, hkv * 128 * 8
    flip = torch.rand(npg, sc, generator=g) < 0.3
    for off in (data, 2 * data + sc):
        region = pool[:, off:off + sc]
        region[flip] |= 0x80
    _run_and_check(msa, host, npg, hkv, "fp4dec_negative_scales")


def test_decode_route_graph_replay(msa):
    """The prepared decode route (list and decode launches) captured once into
    a CUDA graph. Units are split over several CTAs each (100 units x 16 list
    positions over the CTAs), so every replay goes through the per-unit merge
    counters, which the list launch zeroes; each replay reads q, the pool and
    the selection refilled in place."""
    g = torch.Generator().manual_seed(480)
    seqused = [int(x) for x in torch.randint(1500, 6000, (50,), generator=g)]
    hkv = 2
    host, npg = _inputs(g, seqused, [1] * len(seqused), 16 * hkv, hkv, 16)
    dev = to_dev(host, DEV)
    k, ks, v, vs = _views(dev["pool"], hkv)
    r = msa.Nvfp4AttentionRunner(dev["q"], k, ks, v, vs, dev["q2k_indices"], dev["cu_seqlens_q"],
                                 page_table=dev["page_table"], seqused_k=dev["seqused_k"],
                                 k_global_scale=KGS, v_global_scale=VGS, max_seqlen_q=1,
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
    for trial in range(3):
        gt = torch.Generator().manual_seed(900 + trial)
        new_pool = workloads.nvfp4_pool(npg, hkv, gt, "cpu")
        new_q = torch.randn(host["q"].shape, generator=gt).to(torch.bfloat16)
        new_sel = workloads.select_blocks(
            workloads.query_positions(host["cu_seqlens_q"], seqused), hkv, 16, gt)
        dev["pool"].copy_(new_pool)
        dev["q"].copy_(new_q)
        dev["q2k_indices"].copy_(new_sel)
        graph.replay()
        torch.cuda.synchronize()
        fault_clear(msa)
        kf, vf = oracle.nvfp4_dequant(new_pool, hkv, 128, KGS, VGS)
        ref_out, ref_lse = oracle.sparse_attention(
            new_q, kf, vf, new_sel, host["cu_seqlens_q"], causal=True,
            page_table=host["page_table"], seqused_k=host["seqused_k"], num_pages=npg)
        check_attention(r.out, r.lse, ref_out, ref_lse, label=f"fp4dec_graph_{trial}")
    r.close()


@pytest.mark.parametrize("case", [
    # name, seqused, lens_q, topk
    ("topk1", [3000, 700, 129], [1, 3, 2], 1),
    ("sq16_max_decode_shape", [5000, 2100], [16, 16], 16),
    # 2 units x 2 list positions: fewer positions than CTAs, so each CTA takes
    # one position and every unit is combined from several CTAs' partials
    ("fewer_positions_than_ctas", [900], [1], 2),
])
def test_small_and_boundary_shapes(msa, case):
    name, seqused, lens_q, topk = case
    g = torch.Generator().manual_seed(len(name) + 600)
    host, npg = _inputs(g, seqused, lens_q, 32, 2, topk)
    _run_and_check(msa, host, npg, 2, f"fp4dec_{name}", max_seqlen_q=max(lens_q))
