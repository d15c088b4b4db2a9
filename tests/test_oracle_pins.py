"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test ties one oracle function to something fixed independently: a library
routine the method reduces to in a special case (dense causal attention via
torch's scaled_dot_product_attention, torch's float8/bf16 casts, Python's
sort), a closed form, a hand-worked example under tests/golden/, or brute force
on tiny inputs. CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _all_visible(positions, n_kv, width):
    """q2k rows listing every causally visible block (ascending, -1 padded)."""
    n = positions.shape[0]
    out = torch.full((n_kv, n, width), -1, dtype=torch.int32)
    for r, p in enumerate(positions.tolist()):
        if p < 0:
            continue
        nb = p // 128 + 1
        out[:, r, :nb] = torch.arange(nb, dtype=torch.int32)
    return out


def _dense_sdpa(q, k, v, lens_q, lens_k, causal, scale):
    """Dense attention per sequence with torch SDPA in fp64 (right-aligned mask)."""
    outs = []
    cq = ck = 0
    Hq, Hkv = q.shape[1], k.shape[1]
    for lq, lk in zip(lens_q, lens_k):
        qq = q[cq:cq + lq].double().permute(1, 0, 2)
        kk = k[ck:ck + lk].double().permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        vv = v[ck:ck + lk].double().permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        if causal:
            qi = torch.arange(lq)[:, None] + (lk - lq)
            kj = torch.arange(lk)[None, :]
            mask = kj <= qi
        else:
            mask = torch.ones(lq, lk, dtype=torch.bool)
        o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask,
                                                             scale=scale)
        outs.append(o.permute(1, 0, 2))
        cq += lq
        ck += lk
    return torch.cat(outs).numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_dense_reduction_equals_sdpa_flat_varlen_gqa(causal):
    """topk covering every visible block reduces MSA to dense attention."""
    g = torch.Generator().manual_seed(11)
    lens_q = [300, 129, 517]
    lens_k = [300, 390, 517] if causal else [300, 129, 517]
    Hq, Hkv, d = 4, 2, 128
    q = torch.randn(sum(lens_q), Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(sum(lens_k), Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(sum(lens_k), Hkv, d, generator=g).to(torch.bfloat16)
    cu_q = workloads.cu_from_lengths(lens_q)
    cu_k = workloads.cu_from_lengths(lens_k)
    if causal:
        pos = workloads.query_positions(cu_q, lens_k)
    else:
        pos = torch.cat([torch.full((lq,), lk - 1) for lq, lk in zip(lens_q, lens_k)])
    q2k = _all_visible(pos, Hkv, 8)
    scale = 0.0883883461356163  # float32(1/sqrt(128))
    out, lse = oracle.sparse_attention(q, k, v, q2k, cu_q, cu_k, causal=causal,
                                       softmax_scale=scale)
    ref = _dense_sdpa(q, k, v, lens_q, lens_k, causal, scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # LSE against torch.logsumexp of the masked dense logits.
    cq = ck = 0
    for lq, lk in zip(lens_q, lens_k):
        qq = q[cq:cq + lq].double()
        kk = k[ck:ck + lk].double().repeat_interleave(Hq // Hkv, 1)
        logits = torch.einsum("ihc,jhc->hij", qq, kk) * scale
        if causal:
            m = torch.arange(lk)[None, :] <= (torch.arange(lq)[:, None] + lk - lq)
            logits = logits.masked_fill(~m[None], -math.inf)
        ref_lse = torch.logsumexp(logits, dim=-1).permute(1, 0).numpy()
        np.testing.assert_allclose(lse[cq:cq + lq], ref_lse, rtol=0, atol=1e-10)
        cq += lq
        ck += lk


def _to_paged(k, lens, Hkv, d, g):
    """Scatter flat keys into a 128-token page pool under a random page table."""
    pages = [(n + 127) // 128 for n in lens]
    npg = sum(pages) + 3  # a few unused pages
    perm = torch.randperm(npg, generator=g)
    pool = torch.randn(npg, Hkv, 128, d, generator=g).to(k.dtype)
    pt = torch.full((len(lens), max(pages) + 2), -1, dtype=torch.int32)
    c = off = 0
    for b, n in enumerate(lens):
        for t in range(pages[b]):
            p = int(perm[off])
            off += 1
            pt[b, t] = p
            seg = k[c + 128 * t:c + min(n, 128 * (t + 1))]
            pool[p, :, :seg.shape[0]] = seg.permute(1, 0, 2)
        c += n
    return pool, pt


def test_paged_layout_equals_flat():
    """Paged addressing (page_table + seqused_k) gives the flat result."""
    g = torch.Generator().manual_seed(5)
    lens_k = [333, 700]
    lens_q = [4, 1]
    Hq, Hkv, d = 8, 2, 128
    kf = torch.randn(sum(lens_k), Hkv, d, generator=g).to(torch.bfloat16)
    vf = torch.randn(sum(lens_k), Hkv, d, generator=g).to(torch.bfloat16)
    q = torch.randn(sum(lens_q), Hq, d, generator=g).to(torch.bfloat16)
    cu_q = workloads.cu_from_lengths(lens_q)
    cu_k = workloads.cu_from_lengths(lens_k)
    pos = workloads.query_positions(cu_q, lens_k)
    q2k = workloads.select_blocks(pos, Hkv, 3, g)
    out_f, lse_f = oracle.sparse_attention(q, kf, vf, q2k, cu_q, cu_k, causal=True)
    gp = torch.Generator().manual_seed(9)
    kp, pt = _to_paged(kf, lens_k, Hkv, d, gp)
    gp = torch.Generator().manual_seed(9)
    vp, pt2 = _to_paged(vf, lens_k, Hkv, d, gp)
    assert torch.equal(pt, pt2)
    out_p, lse_p = oracle.sparse_attention(q, kp, vp, q2k, cu_q, None, causal=True,
                                           page_table=pt,
                                           seqused_k=torch.tensor(lens_k, dtype=torch.int32))
    np.testing.assert_array_equal(out_p, out_f)
    np.testing.assert_array_equal(lse_p, lse_f)


def test_paged_proxy_equals_flat():
    """Paged addressing gives the flat proxy scores, per head and reduced."""
    g = torch.Generator().manual_seed(6)
    lens_k = [333, 700]
    lens_q = [1, 300]
    Hq, Hkv, d = 8, 2, 128
    kf = torch.randn(sum(lens_k), Hkv, d, generator=g).to(torch.bfloat16)
    q = torch.randn(sum(lens_q), Hq, d, generator=g).to(torch.bfloat16)
    cu_q = workloads.cu_from_lengths(lens_q)
    cu_k = workloads.cu_from_lengths(lens_k)
    kp, pt = _to_paged(kf, lens_k, Hkv, d, torch.Generator().manual_seed(9))
    su = torch.tensor(lens_k, dtype=torch.int32)
    for red in (False, True):
        flat = oracle.proxy_score(q, kf, cu_q, cu_k, causal=True, max_k_tiles=7, reduce_heads=red)
        paged = oracle.proxy_score(q, kp, cu_q, None, page_table=pt, seqused_k=su, causal=True,
                                   max_k_tiles=7, reduce_heads=red)
        np.testing.assert_array_equal(paged, flat)


def test_zero_query_closed_form():
    """q = 0: every visible logit is 0, so lse = ln|J| and out = mean of V over J.

    The key sets J below are written out by hand for each case.
    """
    g = torch.Generator().manual_seed(3)
    Lq, Lk = 40, 300  # right-aligned: query i sits at key position 260 + i
    d = 128
    q = torch.zeros(Lq, 2, d, dtype=torch.bfloat16)
    k = torch.randn(Lk, 1, d, generator=g).to(torch.bfloat16)
    v = torch.randn(Lk, 1, d, generator=g).to(torch.bfloat16)
    cu_q = workloads.cu_from_lengths([Lq])
    cu_k = workloads.cu_from_lengths([Lk])
    q2k = torch.full((1, Lq, 3), -1, dtype=torch.int32)
    cases = {
        0: ([0, 2], list(range(0, 128)) + list(range(256, 261))),   # pos 260
        10: ([2], list(range(256, 271))),                            # pos 270
        39: ([0, 1, 2], list(range(0, 300))),                        # pos 299 = last key
        20: ([1, 5], list(range(128, 256))),                         # block 5 beyond Lk
        21: ([3], []),                                               # block 3 beyond Lk
    }
    for row, (sel, _) in cases.items():
        q2k[0, row, :len(sel)] = torch.tensor(sel, dtype=torch.int32)
    out, lse = oracle.sparse_attention(q, k, v, q2k, cu_q, cu_k, causal=True, softmax_scale=0.5)
    vd = v[:, 0].double().numpy()
    for row, (_, J) in cases.items():
        for h in range(2):
            if J:
                assert lse[row, h] == pytest.approx(math.log(len(J)), abs=1e-12)
                np.testing.assert_allclose(out[row, h], vd[J].mean(axis=0), atol=1e-12)
            else:
                assert lse[row, h] == -math.inf
                assert np.all(out[row, h] == 0.0)


def test_two_block_hand_example():
    spec = json.load(open(os.path.join(GOLDEN, "two_block_example.json")))
    s = spec["setup"]
    L, d = s["seqlen"], s["head_dim"]
    q = torch.zeros(L, 1, d)
    q[:, 0, 0] = s["q_dim0"]
    k = torch.zeros(L, 1, d)
    v = torch.zeros(L, 1, d)
    for b in range(2):
        k[128 * b:128 * (b + 1), 0, 0] = s["block_key_dim0"][b]
        v[128 * b:128 * (b + 1), 0, :] = s["block_value"][b]
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    cu = workloads.cu_from_lengths([L])
    for case in spec["cases"]:
        q2k = torch.full((1, L, 2), -1, dtype=torch.int32)
        q2k[0, case["row"]] = torch.tensor(case["selection"], dtype=torch.int32)
        out, lse = oracle.sparse_attention(q, k, v, q2k, cu, cu, causal=case["causal"],
                                           softmax_scale=s["softmax_scale"], rows=[case["row"]])
        n = case["counts"]
        logits = [s["q_dim0"] * s["block_key_dim0"][b] * s["softmax_scale"] for b in range(2)]
        w = [n[b] * math.exp(logits[b]) for b in range(2)]
        if sum(n) == 0:
            assert lse[0, 0] == -math.inf and np.all(out[0, 0] == 0)
            continue
        assert lse[0, 0] == pytest.approx(math.log(sum(w)), abs=1e-12), case["why"]
        expect = sum(w[b] * s["block_value"][b] for b in range(2)) / sum(w)
        np.testing.assert_allclose(out[0, 0], expect, atol=1e-12, err_msg=case["why"])


def test_convexity_and_block_mass():
    """V column 0 = 1 gives out = 1; V column 1+t = [key in block t] gives the
    softmax mass on block t: exactly 0 off the selection, summing to 1; every
    output lies in the per-column hull of the selected, visible V rows."""
    g = torch.Generator().manual_seed(21)
    L, Hq, Hkv, d = 1000, 4, 2, 128
    nblk = (L + 127) // 128
    q = (3 * torch.randn(L, Hq, d, generator=g)).to(torch.bfloat16)
    k = torch.randn(L, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(L, Hkv, d, generator=g)
    v[:, :, 0] = 1.0
    for t in range(nblk):
        v[:, :, 1 + t] = 0.0
        v[128 * t:128 * (t + 1), :, 1 + t] = 1.0
    v = v.to(torch.bfloat16)
    cu = workloads.cu_from_lengths([L])
    pos = workloads.query_positions(cu, [L])
    q2k = workloads.select_blocks(pos, Hkv, 3, g)
    out, lse = oracle.sparse_attention(q, k, v, q2k, cu, cu, causal=True)
    np.testing.assert_allclose(out[:, :, 0], 1.0, atol=1e-12)
    mass = out[:, :, 1:1 + nblk]
    np.testing.assert_allclose(mass.sum(-1), 1.0, atol=1e-12)
    vv = v.double().numpy()
    for i in range(L):
        for h in range(Hq):
            sel = set(int(x) for x in q2k[h // 2, i].tolist() if x >= 0)
            for t in range(nblk):
                if t not in sel:
                    assert mass[i, h, t] == 0.0
            keys = [j for t in sel for j in range(128 * t, min(L, 128 * t + 128)) if j <= i]
            lo = vv[keys, h // 2].min(0)
            hi = vv[keys, h // 2].max(0)
            assert np.all(out[i, h] >= lo - 1e-12) and np.all(out[i, h] <= hi + 1e-12)


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # Hand-known codes: 1.0, max finite, smallest subnormal, smallest normal, -0.
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9
    assert got[0x08] == 2.0 ** -6 and got[0x80] == 0.0 and math.copysign(1, got[0x80]) < 0


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    got = oracle.bf16_decode(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_fp16_decode_all_codes():
    """All 65536 binary16 patterns against torch's float16 -> float64 cast, plus
    hand-known codes (subnormal scale 2^-24, smallest normal 2^-14, bias 15,
    largest finite 65504, infinities, -0 and the NaN patterns)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.fp16_decode(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    # NaN: exponent field 31 with a non-zero mantissa, either sign.
    exp_field, mant = (bits >> 10) & 31, bits & 1023
    assert np.array_equal(nan, (exp_field == 31) & (mant != 0))
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert got[0x0001] == 2.0 ** -24 and got[0x03FF] == 1023 * 2.0 ** -24
    assert got[0x0400] == 2.0 ** -14 and got[0x3C00] == 1.0 and got[0x3555] == 1365 / 4096
    assert got[0x7BFF] == 65504.0 and got[0xC000] == -2.0
    assert got[0x7C00] == math.inf and got[0xFC00] == -math.inf
    assert got[0x8000] == 0.0 and math.copysign(1, got[0x8000]) < 0


def test_fp16_attention_equals_bf16_on_shared_values():
    """fp16 q / K / V give bit-identical oracle results to bf16 inputs holding
    the same values (k/16 with |k| < 256: exact in both formats)."""
    g = torch.Generator().manual_seed(9)
    L, d = 300, 128

    def vals(*shape):
        return (torch.randint(-255, 256, shape, generator=g).double() / 16.0)

    q, k, v = vals(L, 4, d) * 0.25, vals(L, 2, d) * 0.25, vals(L, 2, d)
    cu = workloads.cu_from_lengths([L])
    q2k = workloads.select_blocks(workloads.query_positions(cu, [L]), 2, 2, g)
    for t in (q, k, v):
        assert torch.equal(t.to(torch.float16).double(), t)
        assert torch.equal(t.to(torch.bfloat16).double(), t)
    oh, lh = oracle.sparse_attention(q.half(), k.half(), v.half(), q2k, cu, cu, causal=True)
    ob, lb = oracle.sparse_attention(q.bfloat16(), k.bfloat16(), v.bfloat16(), q2k, cu, cu,
                                     causal=True)
    np.testing.assert_array_equal(oh, ob)
    np.testing.assert_array_equal(lh, lb)
    assert np.isfinite(lh).all()


def test_e4m3_attention_uses_decoded_values():
    """An E4M3 K/V run equals the bf16 run on the same (exactly representable) values."""
    g = torch.Generator().manual_seed(8)
    L, d = 260, 128
    q = torch.randn(L, 2, d, generator=g).to(torch.bfloat16)
    k8 = torch.randn(L, 1, d, generator=g).to(torch.float8_e4m3fn)
    v8 = torch.randn(L, 1, d, generator=g).to(torch.float8_e4m3fn)
    cu = workloads.cu_from_lengths([L])
    q2k = workloads.select_blocks(workloads.query_positions(cu, [L]), 1, 2, g)
    o8, l8 = oracle.sparse_attention(q, k8, v8, q2k, cu, cu, causal=True)
    ob, lb = oracle.sparse_attention(q, k8.to(torch.bfloat16), v8.to(torch.bfloat16), q2k, cu, cu,
                                     causal=True)
    np.testing.assert_array_equal(o8, ob)
    np.testing.assert_array_equal(l8, lb)


def test_e2m1_decode_all_codes():
    """The sixteen E2M1 codes (NVFP4 elements: sign, 2 exponent bits with bias
    1, 1 mantissa bit, subnormal at exponent 0) decode to the format's values."""
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    np.testing.assert_array_equal(got[:8], want)
    np.testing.assert_array_equal(got[8:], [-x for x in want])
    assert np.signbit(got[8])  # code 8 is -0
    # only the low nibble is a code
    np.testing.assert_array_equal(oracle.e2m1_decode(np.array([0x37, 0xF7], dtype=np.uint8)),
                                  [6.0, 6.0])


def _nvfp4_offsets(hkv, d=128):
    data, sc = hkv * 128 * d // 2, hkv * 128 * d // 16
    return 0, data, data + sc, 2 * data + sc  # K data, K scales, V data, V scales


def test_nvfp4_dequant_reads_nibbles_and_scales():
    """Hand-placed bytes of a two-head planar page land where the reading puts
    them: element 2i in the low nibble of byte i, K scales token-major, V
    scales in scale-index-major 4 x 4 tiles, global scales multiplied in."""
    hkv = 2
    stride = workloads.nvfp4_page_stride(hkv)
    kd, ks, vd, vs = _nvfp4_offsets(hkv)
    pool = np.zeros((2, stride), dtype=np.uint8)
    # K, page 1, head 1, token 5: byte 3 = 0x72 -> element 6 = code 2 (1.0), 7 = code 7 (6.0)
    pool[1, kd + (1 * 128 + 5) * 64 + 3] = 0x72
    pool[1, ks + (1 * 128 + 5) * 8 + 0] = 0x40          # E4M3 2.0 for elements 0..15
    # V, page 0, head 0: every code 2 (1.0); one scale: token 6, scale index 5
    pool[0, vd:vd + 128 * 64] = 0x22
    pool[0, vs + 32 * (6 // 4) + 16 * (5 // 4) + 4 * (5 % 4) + 6 % 4] = 0x48  # E4M3 4.0
    k, v = oracle.nvfp4_dequant(pool, hkv, 128, k_global_scale=0.5, v_global_scale=0.25)
    assert k.shape == (2, hkv, 128, 128)
    nz = np.argwhere(k != 0)
    assert [tuple(x) for x in nz] == [(1, 1, 5, 6), (1, 1, 5, 7)]
    assert k[1, 1, 5, 6] == 1.0 * 2.0 * 0.5 and k[1, 1, 5, 7] == 6.0 * 2.0 * 0.5
    nz = np.argwhere(v != 0)
    assert [tuple(x) for x in nz] == [(0, 0, 6, c) for c in range(80, 96)]
    assert np.all(v[0, 0, 6, 80:96] == 1.0 * 4.0 * 0.25)
    # the same scale byte read token-major would belong to token 6, scale 6
    assert 32 * 1 + 16 * 1 + 4 * 1 + 2 != 6 * 8 + 5


def test_nvfp4_attention_equals_attention_on_decoded_values():
    """The NVFP4 route is attention over the decoded K and V: the oracle on the
    fp64 decode equals the bf16 oracle on the same (exactly representable)
    values, and the K global scale acts as a softmax-scale factor."""
    g = torch.Generator().manual_seed(12)
    hkv, hq, seqused, sq = 2, 8, [700, 300], 2
    npg = sum((n + 127) // 128 for n in seqused) + 2
    pool = workloads.nvfp4_pool(npg, hkv, g, "cpu")
    perm = torch.randperm(npg, generator=g).to(torch.int32)
    pt = torch.zeros(2, 6, dtype=torch.int32)
    pt[0, :6], pt[1, :3] = perm[:6], perm[6:9]
    cu = torch.tensor([0, sq, 2 * sq], dtype=torch.int32)
    su = torch.tensor(seqused, dtype=torch.int32)
    q = torch.randn(2 * sq, hq, 128, generator=g).to(torch.bfloat16)
    q2k = workloads.select_blocks(workloads.query_positions(cu, seqused), hkv, 4, g)
    k, v = oracle.nvfp4_dequant(pool, hkv, 128, k_global_scale=0.5, v_global_scale=0.25)
    o4, l4 = oracle.sparse_attention(q, k, v, q2k, cu, page_table=pt, seqused_k=su, causal=True,
                                     softmax_scale=0.1)
    kb, vb = torch.from_numpy(k).to(torch.bfloat16), torch.from_numpy(v).to(torch.bfloat16)
    assert np.array_equal(kb.double().numpy(), k) and np.array_equal(vb.double().numpy(), v)
    ob, lb = oracle.sparse_attention(q, kb, vb, q2k, cu, page_table=pt, seqused_k=su, causal=True,
                                     softmax_scale=0.1)
    np.testing.assert_array_equal(o4, ob)
    np.testing.assert_array_equal(l4, lb)
    k1, _ = oracle.nvfp4_dequant(pool, hkv, 128, k_global_scale=1.0, v_global_scale=0.25)
    o1, l1 = oracle.sparse_attention(q, k1, v, q2k, cu, page_table=pt, seqused_k=su, causal=True,
                                     softmax_scale=0.05)
    np.testing.assert_allclose(o1, o4, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l4, rtol=0, atol=1e-12)


def test_proxy_closed_form():
    """q_h = (h+1) e0 and k_j[0] = j mod 128: the block max of (h+1)(j mod 128) is
    (h+1)*127 for a full visible block, (h+1)*(pos - 128 t) on the diagonal,
    (h+1)*(Lk-1-128t) on a ragged tail and -inf above the causal limit."""
    lens_q, lens_k = [5, 300], [700, 300]
    Hq, Hkv, d = 4, 2, 128
    q = torch.zeros(sum(lens_q), Hq, d)
    for h in range(Hq):
        q[:, h, 0] = h + 1
    k = torch.zeros(sum(lens_k), Hkv, d)
    c = 0
    for n in lens_k:
        k[c:c + n, :, 0] = (torch.arange(n) % 128).float()[:, None]
        c += n
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    cu_q, cu_k = workloads.cu_from_lengths(lens_q), workloads.cu_from_lengths(lens_k)
    T = 6
    per = oracle.proxy_score(q, k, cu_q, cu_k, causal=True, max_k_tiles=T)
    red = oracle.proxy_score(q, k, cu_q, cu_k, causal=True, max_k_tiles=T, reduce_heads=True)
    assert per.shape == (Hq, T, sum(lens_q)) and red.shape == (1, T, sum(lens_q))
    r = 0
    for lq, lk in zip(lens_q, lens_k):
        for i in range(lq):
            pos = lk - lq + i
            for t in range(T):
                if 128 * t > pos or 128 * t >= lk:
                    base = -math.inf
                else:
                    base = min(pos, lk - 1, 128 * t + 127) - 128 * t
                for h in range(Hq):
                    assert per[h, t, r] == (h + 1) * base
                assert red[0, t, r] == Hq * base
            r += 1


def test_proxy_matches_dense_logit_max():
    """Random inputs: proxy = blockwise max of the dense masked logit matrix (torch)."""
    g = torch.Generator().manual_seed(2)
    L, Hq, Hkv, d = 400, 4, 1, 128
    q = torch.randn(L, Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(L, Hkv, d, generator=g).to(torch.bfloat16)
    cu = workloads.cu_from_lengths([L])
    got = oracle.proxy_score(q, k, cu, cu, causal=True)
    logits = torch.einsum("ihc,jc->hij", q.double(), k[:, 0].double())
    mask = torch.arange(L)[None, :] <= torch.arange(L)[:, None]
    logits = logits.masked_fill(~mask[None], -math.inf)
    T = (L + 127) // 128
    pad = torch.full((Hq, L, T * 128), -math.inf, dtype=torch.float64)
    pad[:, :, :L] = logits
    ref = pad.view(Hq, L, T, 128).amax(-1).permute(0, 2, 1).numpy()
    np.testing.assert_array_equal(got, ref)


def test_topk_hand_cases():
    inf = math.inf
    s = np.array([[[1.0], [3.0], [3.0], [2.0], [-inf], [np.nan], [3.0], [0.5]]], dtype=np.float32)
    assert oracle.topk_select(s, 3, 1)[0, 0].tolist() == [1, 2, 6]
    assert oracle.topk_select(s, 2, 1)[0, 0].tolist() == [1, 2]          # tie -> lower ids
    assert oracle.topk_select(s, 4, 1)[0, 0].tolist() == [1, 2, 3, 6]
    assert oracle.topk_select(s, 8, 2)[1, 0].tolist() == [0, 1, 2, 3, 6, 7, -1, -1]
    allneg = np.full((1, 5, 1), -inf, dtype=np.float32)
    assert oracle.topk_select(allneg, 3, 1)[0, 0].tolist() == [-1, -1, -1]


def test_topk_brute_force_random_with_ties():
    rng = np.random.default_rng(4)
    for trial in range(20):
        Hs, T, n, k = (1, 2)[trial % 2], int(rng.integers(1, 40)), 7, int(rng.integers(1, 17))
        s = rng.integers(-3, 4, size=(Hs, T, n)).astype(np.float32)  # many ties
        s[rng.random(s.shape) < 0.2] = -np.inf
        got = oracle.topk_select(s, k, 2)
        for h in range(2):
            for r in range(n):
                col = s[0 if Hs == 1 else h, :, r]
                ok = [t for t in range(T) if col[t] != -np.inf]
                best = sorted(ok, key=lambda t: (-float(col[t]), t))[:k]
                exp = sorted(best) + [-1] * (k - len(best))
                assert got[h, r].tolist() == exp


def test_union_brute_force_and_invariants():
    g = torch.Generator().manual_seed(17)
    lens = [300, 45, 513]
    Hkv, topk, W = 2, 4, 8
    cu = workloads.cu_from_lengths(lens)
    pos = workloads.query_positions(cu, lens)
    q2k = workloads.select_blocks(pos, Hkv, topk, g)
    # Plant duplicates, out-of-range ids and ids above the causal limit.
    q2k[0, 3, 1] = q2k[0, 3, 0]
    q2k[1, 10, 2] = 99
    q2k[0, 350, 3] = 4  # seq 2 row 5: block 4 is above its causal limit
    ulen, ublk, mem = oracle.build_union(q2k, cu, cu, causal=True, tile_tokens=W)
    cap = W * topk
    tau = 0
    for b, L in enumerate(lens):
        s = int(cu[b])
        nblk = (L + 127) // 128
        for t0 in range(s, s + L, W):
            for h in range(Hkv):
                rowsets = []
                for w in range(W):
                    t = t0 + w
                    if t >= s + L:
                        rowsets.append(set())
                        continue
                    p = t - s
                    rowsets.append({int(x) for x in q2k[h, t].tolist()
                                    if 0 <= x < nblk and 128 * x <= p})
                union = sorted(set().union(*rowsets))
                assert ulen[h, tau] == len(union)
                assert ublk[h, tau].tolist() == union + [-1] * (cap - len(union))
                for w in range(W):
                    bits = [j for j in range(cap) if (int(mem[h, tau, w, j // 32]) >> (j % 32)) & 1]
                    assert [union[j] for j in bits] == sorted(rowsets[w])
            tau += 1
    assert tau == ulen.shape[1]


def test_proxy_e4m3_and_fp16_equal_bf16_on_shared_values():
    """The proxy with E4M3 index-K, or with fp16 q and K, gives bit-identical
    oracle scores to bf16 inputs holding the same values ("flashinfer.msa_ops.
    msa_proxy_score", Parameters q (bf16 or fp16) and k (E4M3 upconverted)):
    E4M3 K values are exact in bf16 and fp16, and k/16 with |k| < 256 is exact
    in both 16-bit formats. Flat and paged, per head and reduced over heads."""
    g = torch.Generator().manual_seed(21)
    lens_q, lens_k = [3, 260], [700, 260]
    Hq, Hkv, d = 8, 2, 128
    cu_q = workloads.cu_from_lengths(lens_q)
    cu_k = workloads.cu_from_lengths(lens_k)
    su = torch.tensor(lens_k, dtype=torch.int32)
    q = torch.randn(sum(lens_q), Hq, d, generator=g).to(torch.bfloat16)
    k8 = torch.randn(sum(lens_k), Hkv, d, generator=g).to(torch.float8_e4m3fn)
    k8p, pt = _to_paged(k8.view(torch.uint8), lens_k, Hkv, d, torch.Generator().manual_seed(4))
    k8p = k8p.view(torch.float8_e4m3fn)
    kbp = k8p.to(torch.bfloat16)
    qs = (torch.randint(-255, 256, (sum(lens_q), Hq, d), generator=g).double() / 16.0)
    ks = (torch.randint(-255, 256, (sum(lens_k), Hkv, d), generator=g).double() / 16.0)
    for red in (False, True):
        kw = dict(causal=True, max_k_tiles=6, reduce_heads=red)
        e8 = oracle.proxy_score(q, k8, cu_q, cu_k, **kw)
        eb = oracle.proxy_score(q, k8.to(torch.bfloat16), cu_q, cu_k, **kw)
        np.testing.assert_array_equal(e8, eb)
        p8 = oracle.proxy_score(q, k8p, cu_q, None, page_table=pt, seqused_k=su, **kw)
        pb = oracle.proxy_score(q, kbp, cu_q, None, page_table=pt, seqused_k=su, **kw)
        np.testing.assert_array_equal(p8, pb)
        np.testing.assert_array_equal(p8, e8)
        fh = oracle.proxy_score(qs.half(), ks.half(), cu_q, cu_k, **kw)
        fb = oracle.proxy_score(qs.bfloat16(), ks.bfloat16(), cu_q, cu_k, **kw)
        np.testing.assert_array_equal(fh, fb)
        h8 = oracle.proxy_score(q.half(), k8, cu_q, cu_k, **kw)
        hh = oracle.proxy_score(q.half(), k8.half(), cu_q, cu_k, **kw)
        np.testing.assert_array_equal(h8, hh)
        assert np.isfinite(e8[..., 3:]).any()
