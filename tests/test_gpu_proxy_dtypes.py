"""GPU parity of the proxy pass with fp16 q and E4M3 index-K.

"flashinfer.msa_ops.msa_proxy_score", Parameters: q is bf16 or fp16, and K
may be fp8 E4M3, upconverted in the kernel. The kernel converts each E4M3 K
tile exactly to q's 16-bit type before the tensor-core QK^T; the fp64 oracle
decodes the same codes. Flat and paged K, per head and reduced over heads,
prefill-shaped and decode-shaped (column-sliced) launches, an unmapped page,
and a context long enough that a tile's block columns take several passes.
"""
import pytest
import torch

import oracle
import workloads
from parity_util import check_proxy, fault_clear

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DT = {"bf16": torch.bfloat16, "f16": torch.float16, "e4m3": torch.float8_e4m3fn}


@pytest.fixture(scope="module")
def msa():
    import block_sparse_top_msa_gb300 as m
    m.build()
    m.lib()
    return m


FLAT_CASES = [
    # name, q dtype, k dtype, lens_q, lens_k, hq, hkv, reduce, causal
    ("bf16q_e4m3k_reduce", "bf16", "e4m3", [300, 517], [300, 517], 16, 2, True, True),
    ("bf16q_e4m3k_perhead_lq_lt_lk", "bf16", "e4m3", [50, 129], [700, 129], 8, 2, False, True),
    ("f16q_f16k_reduce", "f16", "f16", [300, 200], [300, 260], 16, 2, True, True),
    ("f16q_f16k_perhead_noncausal", "f16", "f16", [200], [260], 6, 2, False, False),
    ("f16q_e4m3k_reduce_g32", "f16", "e4m3", [300], [300], 32, 1, True, True),
    ("f16q_e4m3k_mha", "f16", "e4m3", [400], [400], 2, 2, True, True),
    # 469 block columns: more than one pass over the KV groups per tile
    ("bf16q_e4m3k_long_context", "bf16", "e4m3", [40], [60000], 8, 2, True, True),
]


@pytest.mark.parametrize("case", FLAT_CASES, ids=[c[0] for c in FLAT_CASES])
def test_proxy_dtypes_flat(msa, case):
    name, qd, kd, lq, lk, hq, hkv, red, causal = case
    g = torch.Generator().manual_seed(len(name) + 500)
    q = torch.randn(sum(lq), hq, 128, generator=g).to(DT[qd])
    k = torch.randn(sum(lk), hkv, 128, generator=g).to(DT[kd])
    cu_q, cu_k = workloads.cu_from_lengths(lq), workloads.cu_from_lengths(lk)
    T = max((n + 127) // 128 for n in lk) + 1
    ref = oracle.proxy_score(q, k, cu_q, cu_k, causal=causal, max_k_tiles=T, reduce_heads=red)
    got = msa.msa_proxy_score(q.to(DEV), k.to(DEV), cu_q.to(DEV), cu_k.to(DEV), causal=causal,
                              max_k_tiles=T, reduce_heads=red)
    torch.cuda.synchronize()
    fault_clear(msa)
    check_proxy(got, ref, label=name)


PAGED_CASES = [
    # name, q dtype, seqused, query tokens per request (None: prefill), hq, hkv, reduce,
    # pass max_seqlen_q
    ("decode_sq1_reduce_e4m3", "bf16", [8192, 300, 129, 128, 3000], 1, 32, 2, True, True),
    ("decode_sq4_perhead_e4m3_f16q", "f16", [5000, 700], 4, 16, 2, False, True),
    ("decode_sq2_two_m_tiles_e4m3", "bf16", [3000, 900, 128], 2, 32, 2, True, False),
    ("prefill_reduce_e4m3_f16q", "f16", [300, 517], None, 16, 2, True, False),
]


@pytest.mark.parametrize("case", PAGED_CASES, ids=[c[0] for c in PAGED_CASES])
def test_proxy_dtypes_paged_e4m3(msa, case):
    """Paged E4M3 K pool (one page per block), with an unmapped page."""
    name, qd, seqused, sq, hq, hkv, red, pass_sq = case
    g = torch.Generator().manual_seed(len(name) + 700)
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
    k = torch.randn(npg, hkv, 128, 128, generator=g).to(torch.float8_e4m3fn)
    q = torch.randn(sum(lens_q), hq, 128, generator=g).to(DT[qd])
    su = torch.tensor(seqused, dtype=torch.int32)
    T = max(pages) + 1
    got = msa.msa_proxy_score(q.to(DEV), k.to(DEV), cu_q.to(DEV), None, causal=True,
                              max_k_tiles=T, reduce_heads=red, page_table=pt.to(DEV),
                              seqused_k=su.to(DEV), max_seqlen_q=max(lens_q) if pass_sq else None)
    torch.cuda.synchronize()
    fault_clear(msa)
    ref = oracle.proxy_score(q, k, cu_q, None, page_table=pt, seqused_k=su, causal=True,
                             max_k_tiles=T, reduce_heads=red)
    check_proxy(got, ref, label=name)


@pytest.mark.parametrize("sq", [1, None])
def test_proxy_f16_paged(msa, sq):
    """fp16 q with an fp16 paged K pool, decode-shaped (one query token per
    request, column slices) and prefill-shaped, with an unmapped page."""
    g = torch.Generator().manual_seed(900 + (sq or 0))
    seqused = [4000, 700, 129]
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
    pt[1, 1] = npg + 3
    k = torch.randn(npg, 2, 128, 128, generator=g).to(torch.float16)
    q = torch.randn(sum(lens_q), 16, 128, generator=g).to(torch.float16)
    su = torch.tensor(seqused, dtype=torch.int32)
    T = max(pages) + 1
    got = msa.msa_proxy_score(q.to(DEV), k.to(DEV), cu_q.to(DEV), None, causal=True,
                              max_k_tiles=T, reduce_heads=True, page_table=pt.to(DEV),
                              seqused_k=su.to(DEV), max_seqlen_q=sq)
    torch.cuda.synchronize()
    fault_clear(msa)
    ref = oracle.proxy_score(q, k, cu_q, None, page_table=pt, seqused_k=su, causal=True,
                             max_k_tiles=T, reduce_heads=True)
    check_proxy(got, ref, label=f"f16_paged_sq{sq}")


def test_proxy_e4m3_equals_bf16_copy(msa):
    """The in-kernel upconversion gives exactly the scores of the same K
    converted to bf16 beforehand (E4M3 is exact in bf16): bit-identical."""
    g = torch.Generator().manual_seed(77)
    lens = [700, 300]
    q = torch.randn(sum(lens), 16, 128, generator=g).to(torch.bfloat16).to(DEV)
    k8 = torch.randn(sum(lens), 2, 128, generator=g).to(torch.float8_e4m3fn).to(DEV)
    cu = workloads.cu_from_lengths(lens).to(DEV)
    for red in (False, True):
        a = msa.msa_proxy_score(q, k8, cu, cu, causal=True, max_k_tiles=7, reduce_heads=red)
        b = msa.msa_proxy_score(q, k8.to(torch.bfloat16), cu, cu, causal=True, max_k_tiles=7,
                                reduce_heads=red)
        torch.cuda.synchronize()
        fault_clear(msa)
        assert torch.equal(a, b)
