"""The C-ABI library loads, exports every symbol include/msa.h declares, and
decides argument errors on the host before touching the GPU (CPU only: every
call here returns before its first CUDA runtime call)."""
import ctypes as C
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


@pytest.fixture(scope="module")
def L():
    import block_sparse_top_msa_gb300 as msa
    msa.build()
    return msa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("msa_sparse_attention_fwd", "msa_sparse_attention_workspace_size",
              "msa_proxy_score", "msa_topk_select", "msa_build_union", "msa_status_string",
              "msa_union_tile_tokens", "msa_read_device_fault"):
        assert f in names


def test_library_exports_every_declared_symbol(L):
    import block_sparse_top_msa_gb300 as msa
    out = subprocess.run(["nm", "-D", "--defined-only", msa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, missing
    for f in declared_functions():
        assert hasattr(L, f)


def test_status_strings(L):
    import block_sparse_top_msa_gb300 as msa
    assert msa.status_string(0) == "MSA_OK"
    assert msa.status_string(1) == "MSA_INVALID_ARG"
    assert msa.status_string(2) == "MSA_UNSUPPORTED"
    assert msa.status_string(3) == "MSA_WORKSPACE_TOO_SMALL"
    assert msa.status_string(4) == "MSA_CUDA_ERROR"
    assert msa.status_string(99) == "MSA_UNKNOWN_STATUS"


def test_tile_tokens_and_workspace_size(L):
    import block_sparse_top_msa_gb300 as msa
    assert msa.msa_union_tile_tokens(64, 8) == 16
    assert msa.msa_union_tile_tokens(4, 1) == 32
    assert msa.msa_union_tile_tokens(32, 32) == 128
    assert msa.msa_union_tile_tokens(256, 1) == 1
    assert msa.msa_union_tile_tokens(24, 2) == 10  # G = 12: floor(128 / 12)
    ws = msa.msa_sparse_attention_workspace_size(2, 65536, 64, 8, 128, 16, 32768, 0)
    # tile info + lengths + union lists + membership words, each 256-byte padded
    tiles = 65536 // 16 + 2
    assert ws >= tiles * 8 + 8 * tiles * 4 + 8 * tiles * 256 * 4 + 8 * tiles * 16 * 8 * 4
    assert msa.msa_sparse_attention_workspace_size(2, 100, 64, 8, 64, 16, 50, 0) == 0
    assert msa.msa_sparse_attention_workspace_size(2, 100, 64, 7, 128, 16, 50, 0) == 0
    assert msa.msa_sparse_attention_workspace_size(2, 100, 64, 8, 128, 65, 50, 0) == 0
    paged = msa.msa_sparse_attention_workspace_size(128, 512, 64, 4, 128, 16, 4, 1)
    flat = msa.msa_sparse_attention_workspace_size(128, 512, 64, 4, 128, 16, 4, 0)
    assert paged >= flat > 0


def test_workspace_size_with_kv_route(L):
    """The K/V-aware size adds two 256-byte-rounded bf16 copies of K and V
    exactly for flat E4M3 K/V on prefill-sized calls (query rows x query heads
    at least key rows x KV heads), and equals the plain size otherwise."""
    import block_sparse_top_msa_gb300 as msa
    BF16, FP16, E4M3 = 0, 1, 2
    args = (2, 65536, 32, 4, 128, 16, 32768)
    base = msa.msa_sparse_attention_workspace_size(*args, 0)
    copy = (65536 * 4 * 128 * 2 + 255) // 256 * 256
    assert msa.msa_sparse_attention_workspace_size_kv(*args, 0, E4M3, 65536) == base + 2 * copy
    assert msa.msa_sparse_attention_workspace_size_kv(*args, 0, BF16, 65536) == base
    assert msa.msa_sparse_attention_workspace_size_kv(*args, 0, FP16, 65536) == base
    # paged E4M3 and decode-sized flat E4M3 keep the in-kernel conversion
    assert (msa.msa_sparse_attention_workspace_size_kv(*args, 1, E4M3, 65536)
            == msa.msa_sparse_attention_workspace_size(*args, 1))
    dec = (128, 128, 32, 4, 128, 16, 1)
    assert (msa.msa_sparse_attention_workspace_size_kv(*dec, 0, E4M3, 128 * 8192)
            == msa.msa_sparse_attention_workspace_size(*dec, 0))
    # the boundary of the rule: total_q * Hq == total_k * Hkv takes the copy
    edge = (1, 1000, 32, 4, 128, 16, 1000)
    e_base = msa.msa_sparse_attention_workspace_size(*edge, 0)
    assert msa.msa_sparse_attention_workspace_size_kv(*edge, 0, E4M3, 8000) == e_base + 2 * (
        (8000 * 4 * 256 + 255) // 256 * 256)
    assert msa.msa_sparse_attention_workspace_size_kv(*edge, 0, E4M3, 8001) == e_base
    assert msa.msa_sparse_attention_workspace_size_kv(2, 100, 64, 8, 64, 16, 50, 0, E4M3, 100) == 0
    assert msa.msa_sparse_attention_workspace_size_kv(*args, 0, E4M3, -1) == 0
    # the torch-dtype spelling of the binding
    assert (msa.msa_sparse_attention_workspace_size_kv(*args, 0, torch.float8_e4m3fn, 65536)
            == base + 2 * copy)


def test_paged_copy_route_sizes(L):
    """Paged E4M3 (total_k carrying the page table width) and NVFP4 add a bf16
    page pool of batch x max_pages pages for K and V plus the renumbered table
    exactly on prefill-sized calls (query rows x query heads at least
    batch x max_pages x 128 x KV heads)."""
    import block_sparse_top_msa_gb300 as msa
    E4M3 = 2
    r256 = lambda x: (x + 255) // 256 * 256
    pool = lambda b, mp, hkv: 2 * r256(b * mp * hkv * 128 * 128 * 2) + r256(b * mp * 4)
    args = (2, 4096, 32, 4, 128, 16, 2048)
    base = msa.msa_sparse_attention_workspace_size(*args, 1)
    assert msa.msa_sparse_attention_workspace_size_kv(*args, 1, E4M3, 8) == base + pool(2, 8, 4)
    assert msa.msa_sparse_attention_nvfp4_workspace_size(*args, 8) == base + pool(2, 8, 4)
    # the boundary: 4096 x 32 = 2 x 128 x 128 x 4
    assert msa.msa_sparse_attention_nvfp4_workspace_size(*args, 128) == base + pool(2, 128, 4)
    assert msa.msa_sparse_attention_nvfp4_workspace_size(*args, 129) == base
    assert msa.msa_sparse_attention_workspace_size_kv(*args, 1, 0, 8) == base  # bf16: no copy
    # decode-shaped (G <= 16, at most 16 query tokens per request): the block
    # lists (units x topk of (page, keys)), one counter per unit, and the
    # (m, l) and O partials of up to 1024 CTAs x 2 segments x 16 rows
    dec = (128, 128, 64, 4, 128, 16, 1)
    units = 128 * 4
    lists = r256(units * 16 * 8) + r256(units * 4) + r256(1024 * 2 * 16 * 2 * 4) + r256(
        1024 * 2 * 16 * 128 * 4)
    assert (msa.msa_sparse_attention_nvfp4_workspace_size(*dec, 1024)
            == msa.msa_sparse_attention_workspace_size(*dec, 1) + lists)
    wide = (128, 128, 128 * 4, 4, 128, 16, 1)  # G = 128: no decode kernel
    assert (msa.msa_sparse_attention_nvfp4_workspace_size(*wide, 1024)
            == msa.msa_sparse_attention_workspace_size(*wide, 1))
    assert msa.msa_sparse_attention_nvfp4_workspace_size(*args, 0) == 0


A = 0x10000  # a 64 KiB-aligned fake device address; never dereferenced on these paths


def fwd(L, **kw):
    args = dict(q=A, qdt=0, k=A, v=A, kvdt=0, q2k=A, topk=16, cu_q=A, cu_k=A, pt=None,
                max_pages=0, num_pages=0, su=None, batch=1, total_q=128, total_k=128, hq=8, hkv=2,
                d=128, max_sq=128, causal=1, scale=0.0, out=A, lse=None, ws=A, ws_bytes=1 << 40,
                stream=None)
    args.update(kw)
    vp = lambda x: None if x is None else C.c_void_p(x)
    return L.msa_sparse_attention_fwd(
        vp(args["q"]), args["qdt"], vp(args["k"]), vp(args["v"]), args["kvdt"], vp(args["q2k"]),
        args["topk"], vp(args["cu_q"]), vp(args["cu_k"]), vp(args["pt"]), args["max_pages"],
        args["num_pages"], vp(args["su"]), args["batch"], args["total_q"], args["total_k"],
        args["hq"], args["hkv"], args["d"], args["max_sq"], args["causal"], args["scale"],
        vp(args["out"]), vp(args["lse"]), vp(args["ws"]), args["ws_bytes"], vp(args["stream"]))


def test_forward_argument_errors(L):
    # Two length sources (cu_seqlens_k and page_table): declined, not resolved.
    assert fwd(L, pt=A, su=A, max_pages=4, num_pages=4) == 1
    # No length source at all.
    assert fwd(L, cu_k=None) == 1
    # Paged without seqused_k.
    assert fwd(L, cu_k=None, pt=A, max_pages=4, num_pages=4) == 1
    assert fwd(L, hq=8, hkv=3) == 1                 # Hq % Hkv != 0
    assert fwd(L, q=A + 8) == 1                      # misaligned q
    assert fwd(L, ws=A + 64) == 1                    # misaligned workspace
    assert fwd(L, q=None) == 1
    assert fwd(L, total_k=0) == 1
    assert fwd(L, d=64) == 2                         # head_dim
    assert fwd(L, qdt=2) == 2                        # fp8 q
    assert fwd(L, qdt=1) == 2                        # fp16 q with bf16 K/V
    assert fwd(L, qdt=0, kvdt=1) == 2                # bf16 q with fp16 K/V
    assert fwd(L, qdt=1, kvdt=2) == 2                # fp16 q with E4M3 K/V
    assert fwd(L, qdt=1, kvdt=1, ws_bytes=16) == 3   # fp16 q and K/V: accepted
    assert fwd(L, topk=0) == 2 and fwd(L, topk=65) == 2
    assert fwd(L, hq=256, hkv=1) == 2                # G > 128
    assert fwd(L, ws_bytes=16) == 3                  # workspace too small
    assert fwd(L, total_q=0) == 0                    # nothing to do, no launch


def fp4(L, prepare=False, **kw):
    args = dict(q=A, qdt=0, k=A, ks=A, v=A, vs=A, stride=36864, kgs=0.5, vgs=2.0, q2k=A, topk=16,
                cu_q=A, pt=A, max_pages=4, num_pages=4, su=A, batch=1, total_q=4, hq=8, hkv=2,
                d=128, max_sq=4, scale=0.0, out=A, lse=None, ws=A, ws_bytes=1 << 40)
    args.update(kw)
    vp = lambda x: None if x is None else C.c_void_p(x)
    a = (vp(args["q"]), args["qdt"], vp(args["k"]), vp(args["ks"]), vp(args["v"]),
         vp(args["vs"]), args["stride"], args["kgs"], args["vgs"], vp(args["q2k"]), args["topk"],
         vp(args["cu_q"]), vp(args["pt"]), args["max_pages"], args["num_pages"], vp(args["su"]),
         args["batch"], args["total_q"], args["hq"], args["hkv"], args["d"], args["max_sq"],
         args["scale"], vp(args["out"]), vp(args["lse"]), vp(args["ws"]), args["ws_bytes"])
    if prepare:
        p = C.c_void_p(123)
        st = L.msa_sparse_attention_nvfp4_prepare(*a, C.byref(p))
        return st, p
    return L.msa_sparse_attention_nvfp4_paged(*a, None)


def test_nvfp4_argument_errors(L):
    """The packed-NVFP4 paged route decides its argument errors on the host."""
    assert fp4(L, ks=None) == 1 and fp4(L, vs=None) == 1 and fp4(L, k=None) == 1
    assert fp4(L, pt=None) == 1                       # the route is paged only
    assert fp4(L, su=None) == 1                       # paged length comes from seqused_k
    assert fp4(L, ks=A + 8) == 1                      # 16-byte alignment of every view
    assert fp4(L, stride=0) == 1 and fp4(L, stride=36872) == 1
    assert fp4(L, kgs=0.0) == 1 and fp4(L, vgs=-1.0) == 1
    assert fp4(L, kgs=float("inf")) == 1 and fp4(L, vgs=float("nan")) == 1
    assert fp4(L, qdt=1) == 2                         # fp16 q: bf16 only on this route
    assert fp4(L, d=64) == 2
    assert fp4(L, ws_bytes=16) == 3                   # the paged workspace is still required
    assert fp4(L, total_q=0) == 0                     # nothing to do, no launch
    st, p = fp4(L, prepare=True, kgs=-2.0)
    assert st == 1 and not p.value
    st, p = fp4(L, prepare=True, total_q=0)
    assert st == 0 and p.value
    assert L.msa_sparse_attention_run(p, None) == 0   # empty plan: no launch
    L.msa_sparse_attention_plan_free(p)


def test_prepared_forward_host_paths(L):
    """prepare applies the forward's checks (and leaves no plan on failure);
    an empty problem gives a plan whose run launches nothing."""
    vp = C.c_void_p

    def prepare(**kw):
        args = dict(q=A, qdt=0, k=A, v=A, kvdt=0, q2k=A, topk=16, cu_q=A, cu_k=A, pt=None,
                    max_pages=0, num_pages=0, su=None, batch=1, total_q=128, total_k=128, hq=8,
                    hkv=2, d=128, max_sq=128, causal=1, scale=0.0, out=A, lse=None, ws=A,
                    ws_bytes=1 << 40)
        args.update(kw)
        p = vp(123)
        v_ = lambda x: None if x is None else vp(x)
        st = L.msa_sparse_attention_prepare(
            v_(args["q"]), args["qdt"], v_(args["k"]), v_(args["v"]), args["kvdt"],
            v_(args["q2k"]), args["topk"], v_(args["cu_q"]), v_(args["cu_k"]), v_(args["pt"]),
            args["max_pages"], args["num_pages"], v_(args["su"]), args["batch"], args["total_q"],
            args["total_k"], args["hq"], args["hkv"], args["d"], args["max_sq"], args["causal"],
            args["scale"], v_(args["out"]), v_(args["lse"]), v_(args["ws"]), args["ws_bytes"],
            C.byref(p))
        return st, p

    st, p = prepare(hq=8, hkv=3)
    assert st == 1 and not p.value
    st, p = prepare(d=64)
    assert st == 2 and not p.value
    st, p = prepare(ws_bytes=16)
    assert st == 3 and not p.value
    st, p = prepare(total_q=0)
    assert st == 0 and p.value
    assert L.msa_sparse_attention_run(p, None) == 0  # nothing to launch
    L.msa_sparse_attention_plan_free(p)
    assert L.msa_sparse_attention_run(None, None) == 1
    L.msa_sparse_attention_plan_free(None)


def test_other_entry_point_errors(L):
    vp = C.c_void_p
    # proxy: paged with head_dim 64 -> unsupported; paged without seqused_k or
    # max_pages -> invalid; both length kinds -> invalid
    assert L.msa_proxy_score(vp(A), 0, vp(A), 0, vp(A), None, vp(A), 4, vp(A), 1, 128, 128, 8, 2,
                             64, 128, 1, 1, 1, vp(A), None) == 2
    assert L.msa_proxy_score(vp(A), 0, vp(A), 0, vp(A), None, vp(A), 4, None, 1, 128, 128, 8, 2,
                             128, 128, 1, 1, 1, vp(A), None) == 1
    assert L.msa_proxy_score(vp(A), 0, vp(A), 0, vp(A), None, vp(A), 0, vp(A), 1, 128, 128, 8, 2,
                             128, 128, 1, 1, 1, vp(A), None) == 1
    assert L.msa_proxy_score(vp(A), 0, vp(A), 0, vp(A), vp(A), vp(A), 4, vp(A), 1, 128, 128, 8, 2,
                             128, 128, 1, 1, 1, vp(A), None) == 1
    assert L.msa_proxy_score(vp(A), 0, vp(A), 0, vp(A), vp(A), None, 0, None, 1, 128, 128, 8, 2,
                             64, 128, 1, 1, 1, vp(A), None) == 2   # head_dim
    assert L.msa_proxy_score(vp(A), 0, vp(A), 0, vp(A), vp(A), None, 0, None, 1, 128, 128, 48, 1,
                             128, 128, 1, 1, 1, vp(A), None) == 2  # reduce_heads, G = 48
    assert L.msa_proxy_score(vp(A), 0, vp(A), 0, vp(A), vp(A), None, 0, None, 1, 128, 128, 8, 2,
                             128, 128, 0, 1, 1, vp(A), None) == 1  # max_k_tiles 0
    # proxy dtypes: q bf16 or fp16, K of q's type or E4M3; nothing else
    BF16, FP16, E4M3 = 0, 1, 2
    for qd, kd in ((BF16, FP16), (FP16, BF16), (E4M3, E4M3), (BF16, 9)):
        assert L.msa_proxy_score(vp(A), qd, vp(A), kd, vp(A), vp(A), None, 0, None, 1, 128, 128,
                                 8, 2, 128, 128, 1, 1, 1, vp(A), None) == 2, (qd, kd)
    # top-k
    assert L.msa_topk_select(vp(A), 3, 8, 16, 4, 2, vp(A), None) == 1   # heads 3 vs 2
    assert L.msa_topk_select(vp(A), 1, 8, 16, 65, 2, vp(A), None) == 2  # topk
    assert L.msa_topk_select(vp(A), 1, 8, 0, 4, 2, vp(A), None) == 0    # empty
    # union: exactly one length source
    assert L.msa_build_union(vp(A), 4, vp(A), vp(A), vp(A), 4, 1, 16, 1, 1, 16, 2, vp(A), vp(A),
                             vp(A), None, None) == 1
    assert L.msa_build_union(vp(A), 4, vp(A), vp(A), None, 0, 1, 16, 1, 1, 0, 2, vp(A), vp(A),
                             vp(A), None, None) == 1                     # tile_tokens 0
    assert L.msa_read_device_fault(None, None) == 1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import block_sparse_top_msa_gb300 as msa
    monkeypatch.setattr(msa, "_lib", None)
    monkeypatch.setattr(msa, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        msa.lib()


def test_nvfp4_views_follow_the_planar_page():
    """nvfp4_views exposes the four regions of each planar page as the strided
    (pages, Hkv, 128, bytes) views the NVFP4 entry point documents."""
    import block_sparse_top_msa_gb300 as msa
    import workloads
    hkv, npg = 3, 5
    stride = workloads.nvfp4_page_stride(hkv)
    assert stride == 2 * hkv * 128 * (64 + 8)
    pool = (torch.arange(npg * stride, dtype=torch.int64) % 251).to(torch.uint8).view(npg, stride)
    k, ks, v, vs = msa.nvfp4_views(pool, hkv)
    assert k.shape == v.shape == (npg, hkv, 128, 64)
    assert ks.shape == vs.shape == (npg, hkv, 128, 8)
    for t in (k, ks, v, vs):
        assert t.stride(0) == stride
    data, sc = hkv * 128 * 64, hkv * 128 * 8
    flat = pool.reshape(-1)
    p, h, r = 4, 2, 77
    assert int(k[p, h, r, 9]) == int(flat[p * stride + h * 8192 + r * 64 + 9])
    assert int(ks[p, h, r, 5]) == int(flat[p * stride + data + h * 1024 + r * 8 + 5])
    assert int(v[p, h, r, 63]) == int(flat[p * stride + data + sc + h * 8192 + r * 64 + 63])
    assert int(vs[p, h, r, 0]) == int(flat[p * stride + 2 * data + sc + h * 1024 + r * 8])
