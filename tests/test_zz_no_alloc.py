"""The allocation-free paged decode entry point.

msa_sparse_decode_noalloc serves callers that cannot allocate device memory
(engines with a fixed memory plan, plugin interfaces without a workspace,
code where cudaMalloc may not be called): it keeps its scratch in a fixed
array inside the library instead of a workspace. These tests check, through
the C ABI, that it returns what the regular forward returns for the same
decode, on two calls in a row (the second call finds the first call's
leftovers in the shared array), and that problems too large for the array are
refused before anything runs. This file is collected last on purpose.
"""
import ctypes as C

import pytest
import torch

import workloads
from parity_util import fault_clear


@pytest.fixture(scope="module")
def msa():
    import block_sparse_top_msa_gb300 as m
    m.build()
    m.lib()
    return m


def _decode_inputs(seed, sq, seqused, hq, hkv, topk, device):
    g = torch.Generator().manual_seed(seed)
    B = len(seqused)
    cu_q = torch.arange(0, B * sq + 1, sq, dtype=torch.int32)
    pages = [(n + 127) // 128 for n in seqused]
    npg = sum(pages) + 2
    perm = torch.randperm(npg, generator=g).to(torch.int32)
    pt = torch.zeros(B, max(pages), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, :n] = perm[off:off + n]
        off += n
    k = torch.randn(npg, hkv, 128, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(npg, hkv, 128, 128, generator=g).to(torch.bfloat16)
    q = torch.randn(B * sq, hq, 128, generator=g).to(torch.bfloat16)
    q2k = workloads.select_blocks(workloads.query_positions(cu_q, seqused), hkv, topk, g)
    d = dict(q=q, k=k, v=v, q2k_indices=q2k, cu_seqlens_q=cu_q, page_table=pt,
             seqused_k=torch.tensor(seqused, dtype=torch.int32))
    return {n: t.to(device) for n, t in d.items()}


@pytest.mark.gpu
def test_noalloc_decode_matches_forward_twice(msa):
    dev = "cuda:0"
    cases = [(0, 4, [9000, 300, 2000, 130, 4000, 700], 32, 2, 16),
             (1, 1, [5000, 128, 70000, 260], 64, 4, 16)]
    for seed, sq, seqused, hq, hkv, topk in cases:  # the same kernels: the same bits
        inp = _decode_inputs(seed, sq, seqused, hq, hkv, topk, dev)
        ref_out, ref_lse = msa.msa_sparse_attention_fwd(
            inp["q"], inp["k"], inp["v"], inp["q2k_indices"], inp["cu_seqlens_q"], None,
            causal=True, page_table=inp["page_table"], seqused_k=inp["seqused_k"],
            max_seqlen_q=sq, return_softmax_lse=True)
        for _ in range(2):
            out = torch.full_like(inp["q"], float("nan"))
            lse = torch.full(inp["q"].shape[:2], float("nan"), dtype=torch.float32, device=dev)
            msa.msa_sparse_decode_noalloc(inp["q"], inp["k"], inp["v"], inp["q2k_indices"],
                                          inp["cu_seqlens_q"], inp["page_table"],
                                          inp["seqused_k"], max_seqlen_q=sq, causal=True,
                                          out=out, lse=lse)
            torch.cuda.synchronize()
            fault_clear(msa)
            assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_noalloc_refuses_problems_larger_than_its_scratch(msa):
    L = msa.lib()
    limit = L.msa_sparse_decode_noalloc_scratch_limit()
    assert limit == 16 << 20
    A = C.c_void_p(0x10000)  # never dereferenced: the size check comes first
    # 4096 requests of 4 tokens x 8 KV heads, topk 64: the forward's workspace
    # is far beyond 16 MiB.
    need = msa.msa_sparse_attention_workspace_size(4096, 4096 * 4, 128, 8, 128, 64, 4, True)
    assert need > limit
    st = L.msa_sparse_decode_noalloc(A, A, A, A, 64, A, A, 1024, 1024, A, 4096, 4096 * 4, 128,
                                     8, 128, 4, 1, 0.0, A, None, None)
    assert msa.status_string(st) == "MSA_WORKSPACE_TOO_SMALL"
    # Arguments the forward rejects get the forward's status, with no device call.
    st = L.msa_sparse_decode_noalloc(A, A, A, A, 16, A, A, 4, 4, A, 1, 8, 8, 1, 64, 8, 1, 0.0, A,
                                     None, None)
    assert msa.status_string(st) == "MSA_UNSUPPORTED"
    st = L.msa_sparse_decode_noalloc(A, A, A, A, 16, A, None, 4, 4, A, 1, 8, 8, 1, 128, 8, 1, 0.0,
                                     A, None, None)
    assert msa.status_string(st) == "MSA_INVALID_ARG"


@pytest.mark.gpu
def test_noalloc_empty_call_returns_ok(msa):
    """A call with no query rows (total_q = 0) is valid, as it is for the
    regular forward: MSA_OK, nothing launched, nothing written."""
    dev = "cuda:0"
    inp = _decode_inputs(3, 1, [500, 300], 16, 2, 4, dev)
    q = inp["q"][:0]
    out = torch.empty_like(q)
    L = msa.lib()
    st = L.msa_sparse_decode_noalloc(
        C.c_void_p(inp["q"].data_ptr()), C.c_void_p(inp["k"].data_ptr()),
        C.c_void_p(inp["v"].data_ptr()), C.c_void_p(inp["q2k_indices"].data_ptr()), 4,
        C.c_void_p(torch.zeros(3, dtype=torch.int32, device=dev).data_ptr()),
        C.c_void_p(inp["page_table"].data_ptr()), inp["page_table"].shape[1], inp["k"].shape[0],
        C.c_void_p(inp["seqused_k"].data_ptr()), 2, 0, 16, 2, 128, 1, 1, 0.0,
        C.c_void_p(inp["q"].data_ptr()), None, None)
    torch.cuda.synchronize()
    assert msa.status_string(st) == "MSA_OK"
    fault_clear(msa)
    del out
