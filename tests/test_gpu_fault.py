"""The bounded-wait path: a wait that can never be satisfied expires, the
fault is reported through the fault word, and the context stays usable."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import check_attention, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import block_sparse_top_msa_gb300 as m
    m.build()
    m.lib()
    return m


def test_expired_wait_is_reported_and_context_survives(msa):
    assert msa.msa_read_device_fault() == 0
    msa.msa_selftest_wait_timeout(2000)  # 2 ms on a barrier nothing arrives at
    torch.cuda.synchronize()
    assert msa.msa_read_device_fault() == 16
    assert msa.msa_read_device_fault() == 0  # reading clears it
    # The same process keeps computing correctly afterwards.
    g = torch.Generator().manual_seed(1)
    lens = [300]
    q = torch.randn(300, 8, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(300, 2, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(300, 2, 128, generator=g).to(torch.bfloat16)
    cu = workloads.cu_from_lengths(lens)
    q2k = workloads.select_blocks(workloads.query_positions(cu, lens), 2, 3, g)
    out, lse = msa.msa_sparse_attention_fwd(q.cuda(), k.cuda(), v.cuda(), q2k.cuda(), cu.cuda(),
                                            cu.cuda(), causal=True, return_softmax_lse=True)
    torch.cuda.synchronize()
    assert msa.msa_read_device_fault() == 0
    ref_out, ref_lse = oracle.sparse_attention(q, k, v, q2k, cu, cu, causal=True,
                                               softmax_scale=f32(128 ** -0.5))
    check_attention(out, lse, ref_out, ref_lse, label="after_timeout")


def test_selftest_rejects_bad_limits(msa):
    assert msa.lib().msa_selftest_wait_timeout(0, None) == msa.MSA_INVALID_ARG
    assert msa.lib().msa_selftest_wait_timeout(2000000, None) == msa.MSA_INVALID_ARG
