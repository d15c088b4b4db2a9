"""Benchmark of the MSA forward on one GB300 (or N independent replicas).

Headline workload: flat varlen prefill, 2 sequences x 32768 tokens, 64 query /
8 KV heads, head_dim 128, bf16, causal, top-16 of 128-token blocks per query
(diagonal, first and previous block plus random visible blocks). One step is
one pass of the forward (union metadata + sparse attention) over that batch.

value       effective TFLOP/s = 4 * d * sum over (query, head) of the visible
            keys in its selected blocks, divided by the device time per step
e2e         the same metric through the public API with host buffers: pinned
            host -> device copies of the step's inputs, the call, and the
            device -> host copy of out and lse, all inside the timed region
roofline    the attention kernel alone (CUDA events the library records on the
            launching stream between its own launches) against the measured
            bf16 tensor peak
cpu_baseline  the fp64 CPU oracle on a bounded row sample of the same workload
decode / decode_nvfp4 / prefill_nvfp4 / two_stage / e4m3_prefill
            secondary measurements: the paged decode with bf16 and with packed
            NVFP4 K/V (KV GB/s vs HBM), the paged NVFP4 prefill and the flat
            E4M3 prefill on both of their routes (TFLOP/s), and the two-stage
            proxy -> top-k -> attention pipeline; each timed with L2 flushed
            between launches

``--impl reference`` times the oracle itself (host cores) on a bounded sample.
Under torchrun with N > 1 every rank runs the same workload on its own GPU
(replicas; no collective on the data path) and the step time is the max over
ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MSA fwd TFLOP/s (prefill) and KV GB/s (decode) vs GB300 roofline, 1 GPU"
D = 128


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    return units_per_rank * world / max_seconds


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- measurement helpers
# DRAM bytes per launch of the headline attention kernel, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum; see the profile named below).
# Reported only while the kernel sources' code still hashes to the fingerprint
# of the build that was captured; otherwise the roofline's "traffic" is null.
TRAFFIC_SOURCES = ("prefill.cu", "common.cuh", "tmem_wide.cuh", "internal.h", "tmap.h", "api.cu",
                   "union.cu", "tile_map.cuh")
TRAFFIC_MEASURED = {"fingerprint": "e319bba7fc4a81d7", "bytes_per_launch": 2.4285e9,
                    "profile": "profiles/prefill_kernel_flat_varlen_2x32768_traffic.md"}


def kernel_fingerprint():
    """Hash of the kernel sources' code: comments and blank lines are left
    out, so editing a comment keeps a capture valid and editing code does not."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "block_sparse_top_msa_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def measured_traffic():
    if kernel_fingerprint() == TRAFFIC_MEASURED["fingerprint"]:
        return TRAFFIC_MEASURED["bytes_per_launch"]
    return None

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        loaded = [x for x in sm if x >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def l2_flush_buffer(device):
    return torch.empty(256 << 20, dtype=torch.uint8, device=device)


def time_launch(fn, device, reps=5, flush=None):
    """Median device time (s) of fn() over reps launches, L2 flushed before each."""
    times = []
    for _ in range(reps):
        if flush is not None:
            flush.fill_(1)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize(device)
        times.append(s.elapsed_time(e) * 1e-3)
    return statistics.median(times)


# ---------------------------------------------------------------- work accounting
def visible_counts(q2k, cu_q, k_lens, causal=True):
    """Per (kv head, query): visible keys in its distinct selected blocks."""
    dev = q2k.device
    hkv, tq, topk = q2k.shape
    cu = cu_q.cpu().tolist()
    pos = workloads.query_positions(cu_q.cpu(), k_lens).to(dev)
    lk = torch.cat([torch.full((cu[b + 1] - cu[b],), int(k_lens[b]), dtype=torch.int64)
                    for b in range(len(cu) - 1)]).to(dev)
    ids = q2k.long()
    srt, _ = torch.sort(torch.where(ids >= 0, ids, torch.full_like(ids, 1 << 40)), dim=-1)
    dup = torch.zeros_like(srt, dtype=torch.bool)
    dup[..., 1:] = srt[..., 1:] == srt[..., :-1]
    lim = torch.minimum(lk, pos + 1) if causal else lk
    start = srt * 128
    n = torch.clamp(torch.minimum(lim[None, :, None] - start, torch.full_like(start, 128)), min=0)
    n = torch.where((srt < (1 << 40)) & ~dup, n, torch.zeros_like(n))
    return n.sum(-1)  # (hkv, tq)


# ---------------------------------------------------------------- headline: flat prefill
PROFILE_SPEC = workloads.PrefillSpec("flat_prefill_1x8192_h64kv8_top16", [8192], 64, 8, 16,
                                     first_prev=True)


def prefill_inputs(device, seed=0, small=False):
    spec = PROFILE_SPEC if small else workloads.FLAT_VARLEN
    inp = workloads.make_prefill(spec, seed, device=device)
    return spec, inp


def run_prefill(msa, inp, out, lse, ws, max_sq):
    return msa.msa_sparse_attention_fwd(
        inp["q"], inp["k"], inp["v"], inp["q2k_indices"], inp["cu_seqlens_q"],
        inp["cu_seqlens_k"], causal=True, softmax_scale=inp["softmax_scale"],
        max_seqlen_q=max_sq, out=out, lse=lse, workspace=ws)


def cpu_baseline_prefill(inp, rows_target=3072, threads=None):
    """fp64 oracle on a bounded row sample; returns (TFLOP/s, cores, sample, seconds)."""
    import oracle
    cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    tq = cpu["q"].shape[0]
    g = torch.Generator().manual_seed(1234)
    rows = torch.sort(torch.randperm(tq, generator=g)[:rows_target])[0].to(torch.int32)
    hkv = cpu["k"].shape[1]
    G = cpu["q"].shape[1] // hkv
    cnt = visible_counts(cpu["q2k_indices"], cpu["cu_seqlens_q"], cpu["lengths"])
    flops = 4.0 * D * G * float(cnt[:, rows.long()].sum())
    cores = threads or os.cpu_count() or 1
    scale = float(np.float32(inp["softmax_scale"]))
    oracle.sparse_attention(cpu["q"], cpu["k"], cpu["v"], cpu["q2k_indices"],
                            cpu["cu_seqlens_q"], cpu["cu_seqlens_k"], causal=True,
                            softmax_scale=scale, rows=rows[:8], threads=cores)  # warm
    t0 = time.perf_counter()
    oracle.sparse_attention(cpu["q"], cpu["k"], cpu["v"], cpu["q2k_indices"],
                            cpu["cu_seqlens_q"], cpu["cu_seqlens_k"], causal=True,
                            softmax_scale=scale, rows=rows, threads=cores)
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, cores, f"{len(rows)} of {tq} query rows x all {cpu['q'].shape[1]} heads", dt


def _oracle_attention_s(inp, rows, threads, paged=False):
    """Seconds of one oracle sparse_attention call over `rows` (all rows when None)."""
    import oracle
    kw = dict(causal=True, softmax_scale=float(np.float32(inp.get("softmax_scale", D ** -0.5))),
              rows=rows, threads=threads)
    if paged:
        kw.update(page_table=inp["page_table"], seqused_k=inp["seqused_k"])
    t0 = time.perf_counter()
    oracle.sparse_attention(inp["q"], inp["k"], inp["v"], inp["q2k_indices"],
                            inp["cu_seqlens_q"], inp.get("cu_seqlens_k"), **kw)
    return time.perf_counter() - t0


def _attn_flops(inp, rows, k_lens):
    hkv = inp["k"].shape[1]
    G = inp["q"].shape[1] // hkv
    cnt = visible_counts(inp["q2k_indices"], inp["cu_seqlens_q"], k_lens)
    return 4.0 * D * G * float(cnt.sum() if rows is None else cnt[:, rows.long()].sum())


def _row_sample(tq, n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.sort(torch.randperm(tq, generator=g)[:n])[0].to(torch.int32)


def cpu_baseline_suite(device, cores, inp2):
    """The oracle on the other workloads and on one thread: the tiny flat
    prefill and the paged decode in full; the mixed E4M3 prefill and the
    two-stage pipeline on row samples, with the full-workload time
    extrapolated by work (visible keys, or causal key counts for the proxy)
    and marked so; the flat varlen prefill on one thread (a row sample)."""
    import oracle
    res = {}
    # flat varlen prefill, one thread
    rows = _row_sample(inp2["q"].shape[0], 128, 11)
    dt = _oracle_attention_s(inp2, rows, 1)
    res["one_thread"] = {"workload": workloads.FLAT_VARLEN.name, "threads": 1,
                         "sample": "128 query rows x all heads",
                         "tflops": _attn_flops(inp2, rows, inp2["lengths"]) / dt / 1e12,
                         "seconds": round(dt, 3)}
    # tiny flat prefill, in full
    inp = workloads.make_prefill(workloads.TINY_FLAT, 0, device="cpu")
    dt = _oracle_attention_s(inp, None, cores)
    res["tiny_flat"] = {"workload": workloads.TINY_FLAT.name, "sample": "full",
                        "tflops": _attn_flops(inp, None, inp["lengths"]) / dt / 1e12,
                        "seconds": round(dt, 3)}
    # paged decode, in full (s_q 1 and 4)
    for sq in (1, 4):
        inp = workloads.make_decode(workloads.PAGED_DECODE, 0, device="cpu", seqlen_q=sq)
        su = inp["seqused_k"].tolist()
        dt = _oracle_attention_s(inp, None, cores, paged=True)
        res[f"paged_decode_sq{sq}"] = {
            "workload": workloads.PAGED_DECODE.name, "seqlen_q": sq, "sample": "full",
            "tflops": _attn_flops(inp, None, su) / dt / 1e12, "seconds": round(dt, 3)}
        del inp
    # mixed E4M3 prefill: row sample, extrapolated
    inp = workloads.make_prefill(workloads.MIXED_E4M3, 0, device=device)
    inp = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    tq = inp["q"].shape[0]
    rows = _row_sample(tq, 512, 12)
    dt = _oracle_attention_s(inp, rows, cores)
    f_s, f_all = _attn_flops(inp, rows, inp["lengths"]), _attn_flops(inp, None, inp["lengths"])
    res["mixed_e4m3"] = {"workload": workloads.MIXED_E4M3.name,
                         "sample": f"512 of {tq} query rows x all heads",
                         "tflops": f_s / dt / 1e12, "seconds": round(dt, 3),
                         "full_seconds_extrapolated": round(dt * f_all / f_s, 1),
                         "extrapolated": True}
    del inp
    # two-stage: proxy scores, top-k and attention for a row sample
    spec = workloads.TWO_STAGE
    inp = workloads.make_two_stage(spec, 0, device=device)
    inp = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    L = spec.seqlens[0]
    T = (L + 127) // 128
    rows = _row_sample(L, 64, 13)
    t0 = time.perf_counter()
    sc = oracle.proxy_score(inp["proxy_q"], inp["index_k"], inp["cu_seqlens_q"],
                            inp["cu_seqlens_k"], causal=True, max_k_tiles=T, reduce_heads=True,
                            rows=rows, threads=cores)
    t_proxy = time.perf_counter() - t0
    t0 = time.perf_counter()
    sel = oracle.topk_select(np.ascontiguousarray(sc.astype(np.float32)), spec.topk,
                             spec.num_kv_heads)
    t_topk = time.perf_counter() - t0
    q2k = torch.full((spec.num_kv_heads, L, spec.topk), -1, dtype=torch.int32)
    q2k[:, rows.long()] = torch.as_tensor(np.asarray(sel), dtype=torch.int32)
    inp["q2k_indices"] = q2k
    t_attn = _oracle_attention_s(inp, rows, cores)
    keys_s = float((rows.long() + 1).sum())  # causal keys of the sampled rows
    keys_all = L * (L + 1) / 2
    f_s = _attn_flops(inp, rows, [L])
    res["two_stage"] = {
        "workload": spec.name, "sample": f"64 of {L} query rows (proxy over all heads, top-k, "
        "attention)", "seconds": round(t_proxy + t_topk + t_attn, 3),
        "proxy_tflops": 2.0 * D * spec.proxy_heads * keys_s / t_proxy / 1e12,
        "attention_tflops": f_s / t_attn / 1e12,
        "full_seconds_extrapolated": round(t_proxy * keys_all / keys_s + t_attn * L / len(rows), 1),
        "extrapolated": True}
    return res


def bench_prefill(msa, args, device, world, rank):
    spec, inp = prefill_inputs(device, small=args.profile_small)
    tq, hq, _ = inp["q"].shape
    hkv = inp["k"].shape[1]
    G = hq // hkv
    max_sq = max(inp["lengths"])
    cnt = visible_counts(inp["q2k_indices"], inp["cu_seqlens_q"], inp["lengths"])
    flops = 4.0 * D * G * float(cnt.sum())
    blocks = (inp["q2k_indices"] >= 0).sum().item()
    flops_block = 4.0 * D * G * 128 * float(blocks)
    # Bytes the attention kernel must move at least once: q and K/V read, out written.
    alg_bytes = (inp["q"].numel() * inp["q"].element_size() * 2 +
                 (inp["k"].numel() + inp["v"].numel()) * inp["k"].element_size())
    out = torch.empty_like(inp["q"])
    lse = torch.empty((tq, hq), dtype=torch.float32, device=device)
    need = msa.msa_sparse_attention_workspace_size(len(inp["lengths"]), tq, hq, hkv, D, 16,
                                                   max_sq, False)
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    # Executed MMA work: union blocks per 128-row tile (same W as the forward).
    W = msa.msa_union_tile_tokens(hq, hkv)
    ulen = msa.msa_build_union(inp["q2k_indices"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                               causal=True, tile_tokens=W)[0]
    union_blocks = float(ulen.sum().item())
    flops_exec = union_blocks * 4.0 * D * 128 * 128

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for _ in range(args.warmup):
        run_prefill(msa, inp, out, lse, ws, max_sq)
    torch.cuda.synchronize(device)
    barrier(world)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize(device)
        barrier(world)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for i in range(args.steps):
            msa.msa_set_timing_events(evs[i])  # host-side only: which events to record
            run_prefill(msa, inp, out, lse, ws, max_sq)
        end.record()
        torch.cuda.synchronize(device)
        msa.msa_set_timing_events(None)
        barrier(world)
    wall = start.elapsed_time(end) * 1e-3
    meta_times = [e[0].elapsed_time(e[1]) * 1e-3 for e in evs]
    attn_times = [e[1].elapsed_time(e[2]) * 1e-3 for e in evs]
    step_s = max_over_ranks(wall / args.steps, world, device if world > 1 else None)
    attn_s = statistics.mean(attn_times)
    fault = msa.msa_read_device_fault()
    pk = peaks()
    achieved = flops / attn_s / 1e12
    res = dict(
        spec=spec, inp=inp, flops=flops, flops_block=flops_block, flops_exec=flops_exec,
        step_s=step_s, wall_s=wall, attn_s=attn_s, meta_s=statistics.mean(meta_times),
        value=aggregate_value(flops, world, step_s) / 1e12, clocks=clk.summary(), fault=fault,
        # The timed region is a fraction of a second of 18 ms launches: the
        # burst bf16 figure is the denominator (the sustained one is listed).
        roofline={"bound": "tensor", "achieved": round(achieved, 2),
                  "peak": pk["bf16"], "unit": "TFLOP/s",
                  "frac": round(achieved / pk["bf16"], 4),
                  "peak_sustained": pk["bf16_sus"],
                  "traffic": None if args.profile_small else measured_traffic(),
                  "traffic_source": TRAFFIC_MEASURED["profile"],
                  "algorithmic_bytes": int(alg_bytes),
                  "kernel": "prefill_kernel<bf16>",
                  "peak_kind": f"bf16_tflops, burst ({pk['source']})",
                  "achieved_is": "algorithmic FLOP per launch / mean launch time"},
        executed_tflops=flops_exec / attn_s / 1e12,
        work_efficiency=flops / flops_exec,
        union_blocks_per_tile=union_blocks / ulen.numel(),
    )
    if args.profile_small:
        res["e2e"] = None
        return res
    # End-to-end through the public API with host buffers: every step copies
    # its inputs from pinned host memory and reads out and lse back. Steps are
    # pipelined the way a caller streaming batches would run them: copy-in,
    # compute and copy-out on three streams with two device buffer sets, so
    # the copies of neighbouring steps overlap this step's kernels.
    host = {k: v.cpu().pin_memory() for k, v in inp.items()
            if torch.is_tensor(v) and k in ("q", "k", "v", "q2k_indices", "cu_seqlens_q",
                                            "cu_seqlens_k")}
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    lse_h = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    sets = [{k: torch.empty_like(v, device=device) for k, v in host.items()} for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    lses = [lse, torch.empty_like(lse)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_h[0].numel() * out_h[0].element_size() + lse_h[0].numel() * lse_h[0].element_size()
    s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):  # every buffer set starts free
        for ev in (ev_cmp[b], ev_out[b]):
            ev.record(s_out)

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_cmp[b])  # the step two back has read these inputs
            for k2, v2 in host.items():
                sets[b][k2].copy_(v2, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[b])
            s_cmp.wait_event(ev_out[b])  # and its results have been copied out
            d = dict(sets[b], softmax_scale=inp["softmax_scale"])
            run_prefill(msa, d, outs[b], lses[b], ws, max_sq)
            ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[b])
            out_h[b].copy_(outs[b], non_blocking=True)
            lse_h[b].copy_(lses[b], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(device)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The copies alone, once each, for reading the pipelined time against.
    s.record(s_in)
    with torch.cuda.stream(s_in):
        for k2, v2 in host.items():
            sets[0][k2].copy_(v2, non_blocking=True)
    e.record(s_in)
    torch.cuda.synchronize(device)
    h2d_ms = s.elapsed_time(e)
    s.record(s_out)
    with torch.cuda.stream(s_out):
        out_h[0].copy_(outs[0], non_blocking=True)
        lse_h[0].copy_(lses[0], non_blocking=True)
    e.record(s_out)
    torch.cuda.synchronize(device)
    d2h_ms = s.elapsed_time(e)
    # At least 10 steps: the pipeline's fill (first copy-in) and drain (last
    # copy-out) are paid once per timed run.
    n_e2e = max(10, args.steps)
    s.record(s_in)
    for i in range(n_e2e):
        e2e_step(i)
    e.record(s_out)
    torch.cuda.synchronize(device)
    e2e_s = s.elapsed_time(e) * 1e-3 / n_e2e
    e2e_s = max_over_ranks(e2e_s, world, device if world > 1 else None)
    res["e2e"] = {"value": round(aggregate_value(flops, world, e2e_s) / 1e12, 3),
                  "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                  "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_s * 1e3, 3),
                  "h2d_ms_alone": round(h2d_ms, 3), "d2h_ms_alone": round(d2h_ms, 3),
                  "pipelined": "copy-in, compute, copy-out on three streams, two buffer sets"}
    return res


# ---------------------------------------------------------------- secondary: paged decode
DECODE_PROFILE_SPEC = workloads.DecodeSpec("paged_decode_b64_U[8192,32768]_h64kv4_top16", 64,
                                           (8192, 32768), 64, 4, 16)


def bench_decode(msa, device, flush, seed=0, small=False, sqs=(1, 4), reps=7):
    spec = DECODE_PROFILE_SPEC if small else workloads.PAGED_DECODE
    out = {}
    pk = peaks()
    for sq in sqs:
        inp = workloads.make_decode(spec, seed, device=device, seqlen_q=sq)
        q2k, pt, su = inp["q2k_indices"], inp["page_table"], inp["seqused_k"]
        hkv = inp["k"].shape[1]
        G = inp["q"].shape[1] // hkv
        # Distinct valid K+V bytes of each (request, KV head)'s union of pages.
        B = pt.shape[0]
        ids = q2k.view(hkv, B, sq * q2k.shape[2]).long()
        lens = su.long()
        srt, _ = torch.sort(torch.where(ids >= 0, ids, torch.full_like(ids, 1 << 40)), dim=-1)
        first = torch.ones_like(srt, dtype=torch.bool)
        first[..., 1:] = srt[..., 1:] != srt[..., :-1]
        valid = torch.clamp(torch.minimum(lens[None, :, None] - srt * 128,
                                          torch.full_like(srt, 128)), min=0)
        valid = torch.where((srt < (1 << 40)) & first, valid, torch.zeros_like(valid))
        kv_bytes = float(valid.sum()) * D * 2 * 2
        meta = (inp["q"].numel() * 2 * 2 + inp["q"].shape[0] * inp["q"].shape[1] * 4 +
                q2k.numel() * 4 + pt.numel() * 4)
        o = torch.empty_like(inp["q"])
        lse = torch.empty(inp["q"].shape[:2], dtype=torch.float32, device=device)
        need = msa.msa_sparse_attention_workspace_size(B, inp["q"].shape[0], inp["q"].shape[1],
                                                       hkv, D, q2k.shape[2], sq, True)
        ws = torch.empty(need, dtype=torch.uint8, device=device)

        def call():
            msa.msa_sparse_attention_fwd(inp["q"], inp["k"], inp["v"], q2k, inp["cu_seqlens_q"],
                                         None, causal=True, page_table=pt, seqused_k=su,
                                         max_seqlen_q=sq, out=o, lse=lse, workspace=ws)

        for _ in range(3):
            call()
        # The whole call between events recorded around it (nothing between
        # its kernels, so the attention kernel's early start is kept), then
        # the attention launch alone from the library's own events.
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts, ta = [], []
        for _ in range(reps):
            flush.fill_(1)
            torch.cuda._sleep(200_000)  # keeps the GPU busy while the host enqueues the call
            e0.record()
            call()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for _ in range(reps):
            flush.fill_(1)
            msa.msa_set_timing_events(ev)
            call()
            ev[2].synchronize()
            ta.append(ev[1].elapsed_time(ev[2]) * 1e-3)
        msa.msa_set_timing_events(None)
        t, t_attn = statistics.median(ts), statistics.median(ta)
        gbs = (kv_bytes + meta) / t / 1e9
        gbs_attn = (kv_bytes + meta) / t_attn / 1e9
        out[f"seqlen_q_{sq}"] = {
            "value": round(gbs, 1), "unit": "GB/s", "us": round(t * 1e6, 2),
            "attention_us": round(t_attn * 1e6, 2),
            "kv_bytes": int(kv_bytes), "meta_bytes": int(meta),
            "roofline": {"bound": "hbm", "achieved": round(gbs_attn, 1), "peak": pk["hbm"],
                         "unit": "GB/s", "frac": round(gbs_attn / pk["hbm"], 4), "traffic": None,
                         "kernel": "prefill_kernel<bf16> (paged, split items)"}}
        if sq == 1:
            out["proxy_seqlen_q_1"] = bench_decode_proxy(msa, inp, flush, pk, reps)
        del inp
        torch.cuda.empty_cache()
    out["workload"] = spec.name
    return out


DECODE_NVFP4_PROFILE_SPEC = workloads.DecodeSpec(
    "nvfp4_paged_decode_b64_U[8192,32768]_h64kv4_top16", 64, (8192, 32768), 64, 4, 16,
    kv_dtype="nvfp4", k_global_scale=0.25, v_global_scale=0.125)


def bench_decode_nvfp4(msa, device, flush, seed=0, sqs=(1, 4), reps=7, small=False):
    """Paged decode with packed NVFP4 K/V (planar page pool, E4M3 block scales,
    global scales): the same batch, selection and metric as the bf16 decode;
    K/V bytes are 64 code + 8 scale bytes per token and side."""
    spec = DECODE_NVFP4_PROFILE_SPEC if small else workloads.PAGED_DECODE_NVFP4
    out = {}
    pk = peaks()
    for sq in sqs:
        inp = workloads.make_decode(spec, seed, device=device, seqlen_q=sq)
        q2k, pt, su = inp["q2k_indices"], inp["page_table"], inp["seqused_k"]
        hkv = q2k.shape[0]
        kk, ks, vv, vs = msa.nvfp4_views(inp["kv_pool"], hkv)
        B = pt.shape[0]
        ids = q2k.view(hkv, B, sq * q2k.shape[2]).long()
        srt, _ = torch.sort(torch.where(ids >= 0, ids, torch.full_like(ids, 1 << 40)), dim=-1)
        first = torch.ones_like(srt, dtype=torch.bool)
        first[..., 1:] = srt[..., 1:] != srt[..., :-1]
        valid = torch.clamp(torch.minimum(su.long()[None, :, None] - srt * 128,
                                          torch.full_like(srt, 128)), min=0)
        valid = torch.where((srt < (1 << 40)) & first, valid, torch.zeros_like(valid))
        kv_bytes = float(valid.sum()) * (D // 2 + D // 16) * 2
        meta = (inp["q"].numel() * 2 * 2 + inp["q"].shape[0] * inp["q"].shape[1] * 4 +
                q2k.numel() * 4 + pt.numel() * 4)
        o = torch.empty_like(inp["q"])
        lse = torch.empty(inp["q"].shape[:2], dtype=torch.float32, device=device)
        need = msa.msa_sparse_attention_nvfp4_workspace_size(
            B, inp["q"].shape[0], inp["q"].shape[1], hkv, D, q2k.shape[2], sq, pt.shape[1])
        ws = torch.empty(need, dtype=torch.uint8, device=device)

        def call():
            msa.msa_sparse_attention_nvfp4_paged(
                inp["q"], kk, ks, vv, vs, q2k, inp["cu_seqlens_q"], page_table=pt, seqused_k=su,
                k_global_scale=inp["k_global_scale"], v_global_scale=inp["v_global_scale"],
                max_seqlen_q=sq, out=o, lse=lse, workspace=ws)

        for _ in range(3):
            call()
        # The whole call between events recorded around it (nothing between
        # its kernels, so the attention kernel's early start is kept), then
        # the attention launch alone from the library's own events.
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts, ta = [], []
        for _ in range(reps):
            flush.fill_(1)
            torch.cuda._sleep(200_000)  # keeps the GPU busy while the host enqueues the call
            e0.record()
            call()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for _ in range(reps):
            flush.fill_(1)
            msa.msa_set_timing_events(ev)
            call()
            ev[2].synchronize()
            ta.append(ev[1].elapsed_time(ev[2]) * 1e-3)
        msa.msa_set_timing_events(None)
        t, t_attn = statistics.median(ts), statistics.median(ta)
        gbs, gbs_attn = (kv_bytes + meta) / t / 1e9, (kv_bytes + meta) / t_attn / 1e9
        out[f"seqlen_q_{sq}"] = {
            "value": round(gbs, 1), "unit": "GB/s", "us": round(t * 1e6, 2),
            "attention_us": round(t_attn * 1e6, 2), "kv_bytes": int(kv_bytes),
            "meta_bytes": int(meta),
            "roofline": {"bound": "hbm", "achieved": round(gbs_attn, 1), "peak": pk["hbm"],
                         "unit": "GB/s", "frac": round(gbs_attn / pk["hbm"], 4), "traffic": None,
                         "kernel": "fp4_list_kernel + fp4_decode_kernel (paged NVFP4 decode)"}}
        del inp
        torch.cuda.empty_cache()
    out["workload"] = spec.name
    return out


def bench_nvfp4_prefill(msa, device, flush, seed=0, reps=3):
    """Paged prefill over a planar NVFP4 pool, on both routes: the default one
    (bf16 page pool decoded once per call, then the bf16 attention kernel) and
    the in-kernel decode (paged workspace size only)."""
    spec = workloads.PAGED_PREFILL_NVFP4
    inp = workloads.make_paged_prefill_nvfp4(spec, seed, device=device)
    q, q2k, cu, pt = inp["q"], inp["q2k_indices"], inp["cu_seqlens_q"], inp["page_table"]
    tq, hq, _ = q.shape
    hkv = q2k.shape[0]
    G = hq // hkv
    max_sq = max(inp["lengths"])
    cnt = visible_counts(q2k, cu, inp["lengths"])
    flops = 4.0 * D * G * float(cnt.sum())
    kk, ks, vv, vs = msa.nvfp4_views(inp["kv_pool"], hkv)
    out = torch.empty_like(q)
    lse = torch.empty((tq, hq), dtype=torch.float32, device=device)
    pk = peaks()
    B = pt.shape[0]
    sizes = {
        "bf16_pool": msa.msa_sparse_attention_nvfp4_workspace_size(B, tq, hq, hkv, D, spec.topk,
                                                                   max_sq, pt.shape[1]),
        "in_kernel": msa.msa_sparse_attention_workspace_size(B, tq, hq, hkv, D, spec.topk, max_sq,
                                                             True)}
    res = {"workload": spec.name, "tokens": int(tq)}
    for route, need in sizes.items():
        ws = torch.empty(need, dtype=torch.uint8, device=device)

        def call():
            msa.msa_sparse_attention_nvfp4_paged(
                q, kk, ks, vv, vs, q2k, cu, page_table=pt, seqused_k=inp["seqused_k"],
                k_global_scale=inp["k_global_scale"], v_global_scale=inp["v_global_scale"],
                max_seqlen_q=max_sq, out=out, lse=lse, workspace=ws)

        for _ in range(2):
            call()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ts, ta = [], []
        for _ in range(reps):
            flush.fill_(1)
            msa.msa_set_timing_events(ev)
            call()
            ev[2].synchronize()
            ts.append(ev[0].elapsed_time(ev[2]) * 1e-3)
            ta.append(ev[1].elapsed_time(ev[2]) * 1e-3)
        msa.msa_set_timing_events(None)
        t, t_attn = statistics.median(ts), statistics.median(ta)
        res[route] = {
            "value": round(flops / t / 1e12, 2), "unit": "TFLOP/s", "ms": round(t * 1e3, 3),
            "attention_ms": round(t_attn * 1e3, 3),
            "roofline": {"bound": "tensor", "achieved": round(flops / t_attn / 1e12, 2),
                         "peak": pk["bf16"], "unit": "TFLOP/s",
                         "frac": round(flops / t_attn / 1e12 / pk["bf16"], 4)}}
        del ws
    res["value"], res["unit"] = res["bf16_pool"]["value"], "TFLOP/s"
    del inp
    torch.cuda.empty_cache()
    return res


def bench_decode_proxy(msa, inp, flush, pk, reps):
    """Paged proxy scores (reduce_heads) of the decode batch: every key of every
    request is visible to its one query token, so the kernel streams the whole
    K cache; HBM-bound."""
    q, k, pt, su = inp["q"], inp["k"], inp["page_table"], inp["seqused_k"]
    T = pt.shape[1]
    scores = torch.empty((1, T, q.shape[0]), dtype=torch.float32, device=q.device)

    def call():
        msa.msa_proxy_score(q, k, inp["cu_seqlens_q"], None, causal=True, max_k_tiles=T,
                            reduce_heads=True, output=scores, page_table=pt, seqused_k=su,
                            max_seqlen_q=1)

    call()
    t = time_launch(call, q.device, reps=reps, flush=flush)
    kbytes = float(su.long().sum()) * k.shape[1] * D * 2
    nbytes = kbytes + q.numel() * 2 + scores.numel() * 4 + pt.numel() * 4
    return {"value": round(nbytes / t / 1e9, 1), "unit": "GB/s", "us": round(t * 1e6, 2),
            "k_bytes": int(kbytes),
            "roofline": {"bound": "hbm", "achieved": round(nbytes / t / 1e9, 1), "peak": pk["hbm"],
                         "unit": "GB/s", "frac": round(nbytes / t / 1e9 / pk["hbm"], 4),
                         "kernel": "proxy_kernel (paged, column slices)"}}


# ---------------------------------------------------------------- secondary: two-stage
def bench_two_stage(msa, device, flush, seed=0):
    spec = workloads.TWO_STAGE
    inp = workloads.make_two_stage(spec, seed, device=device)
    L = spec.seqlens[0]
    T = (L + 127) // 128
    pk = peaks()
    scores = torch.empty((1, T, L), dtype=torch.float32, device=device)
    q2k = torch.empty((spec.num_kv_heads, L, spec.topk), dtype=torch.int32, device=device)
    res = {"workload": spec.name}

    def proxy():
        msa.msa_proxy_score(inp["proxy_q"], inp["index_k"], inp["cu_seqlens_q"],
                            inp["cu_seqlens_k"], causal=True, max_k_tiles=T, reduce_heads=True,
                            output=scores)

    def topk():
        msa.msa_topk_select(scores, spec.topk, spec.num_kv_heads, out=q2k)

    proxy()
    topk()
    t_proxy = time_launch(proxy, device, reps=3, flush=flush)
    t_topk = time_launch(topk, device, reps=5, flush=flush)
    pflops = 2.0 * D * spec.proxy_heads * L * (L + 1) / 2
    res["proxy"] = {"tflops": round(pflops / t_proxy / 1e12, 2), "ms": round(t_proxy * 1e3, 3),
                    "frac_of_bf16_peak": round(pflops / t_proxy / 1e12 / pk["bf16"], 4)}
    tk_bytes = scores.numel() * 4 + q2k.numel() * 4
    res["topk"] = {"gbs": round(tk_bytes / t_topk / 1e9, 1), "us": round(t_topk * 1e6, 2),
                   "frac_of_hbm": round(tk_bytes / t_topk / 1e9 / pk["hbm"], 4)}
    out = torch.empty_like(inp["q"])
    lse = torch.empty(inp["q"].shape[:2], dtype=torch.float32, device=device)
    need = msa.msa_sparse_attention_workspace_size(1, L, spec.num_qo_heads, spec.num_kv_heads, D,
                                                   spec.topk, L, False)
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def attn():
        msa.msa_sparse_attention_fwd(inp["q"], inp["k"], inp["v"], q2k, inp["cu_seqlens_q"],
                                     inp["cu_seqlens_k"], causal=True, max_seqlen_q=L, out=out,
                                     lse=lse, workspace=ws)

    attn()
    ts = []
    for _ in range(3):
        flush.fill_(1)
        msa.msa_set_timing_events(ev)
        attn()
        ev[2].synchronize()
        ts.append(ev[1].elapsed_time(ev[2]) * 1e-3)
    msa.msa_set_timing_events(None)
    t_attn = statistics.median(ts)
    G = spec.num_qo_heads // spec.num_kv_heads
    cnt = visible_counts(q2k, inp["cu_seqlens_q"], spec.seqlens)
    aflops = 4.0 * D * G * float(cnt.sum())
    W = msa.msa_union_tile_tokens(spec.num_qo_heads, spec.num_kv_heads)
    ulen = msa.msa_build_union(q2k, inp["cu_seqlens_q"], inp["cu_seqlens_k"], causal=True,
                               tile_tokens=W)[0]
    flops_exec = float(ulen.sum().item()) * 4.0 * D * 128 * 128
    res["attention"] = {"tflops": round(aflops / t_attn / 1e12, 2), "ms": round(t_attn * 1e3, 3),
                        "frac_of_bf16_peak": round(aflops / t_attn / 1e12 / pk["bf16"], 4),
                        "executed_mma_tflops": round(flops_exec / t_attn / 1e12, 2),
                        "work_efficiency": round(aflops / flops_exec, 4),
                        "union_blocks_per_tile": round(float(ulen[ulen > 0].float().mean().item()), 2)}
    res["pipeline_ms"] = round((t_proxy + t_topk + t_attn) * 1e3, 3)
    return res


# ---------------------------------------------------------------- secondary: tiny flat prefill
def bench_tiny(msa, device, flush, seed=0, reps=20):
    """The tiny flat prefill (1 x 1024 tokens, 4/1 heads, top-4): a
    latency-bound call (32 query tiles of 32 tokens for one KV head, far
    fewer work items than SMs); the whole call (union and attention kernels)
    by events around it, the L2 flushed before each."""
    spec = workloads.TINY_FLAT
    inp = workloads.make_prefill(spec, seed, device=device)
    tq, hq, _ = inp["q"].shape
    hkv = inp["k"].shape[1]
    flops = 4.0 * D * (hq // hkv) * float(
        visible_counts(inp["q2k_indices"], inp["cu_seqlens_q"], inp["lengths"]).sum())
    max_sq = max(inp["lengths"])
    need = msa.msa_sparse_attention_workspace_size(len(inp["lengths"]), tq, hq, hkv, D, spec.topk,
                                                   max_sq, False)
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    out = torch.empty_like(inp["q"])
    lse = torch.empty((tq, hq), dtype=torch.float32, device=device)

    def call():
        run_prefill(msa, inp, out, lse, ws, max_sq)

    for _ in range(3):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(reps):
        flush.fill_(1)
        torch.cuda._sleep(200_000)  # keeps the GPU busy while the host enqueues the call
        e0.record()
        call()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3)
    t = statistics.median(ts)
    return {"workload": spec.name, "tflops": round(flops / t / 1e12, 3), "us": round(t * 1e6, 2),
            "algorithmic_gflop": round(flops / 1e9, 3),
            "roofline": {"bound": "latency", "note": "32 work items on a 152-SM GPU"}}


# ---------------------------------------------------------------- secondary: E4M3 K/V prefill
def bench_e4m3(msa, device, flush, seed=0, reps=3):
    """Flat varlen prefill with E4M3 K/V, bf16 q, on both routes: the default
    one (workspace_size_kv bytes: K/V decoded to a bf16 copy by one HBM-bound
    pass, then the bf16 attention kernel) and the in-kernel conversion (plain
    workspace size). The line's value is the default route's whole call."""
    spec = workloads.MIXED_E4M3
    inp = workloads.make_prefill(spec, seed, device=device)
    tq, hq, _ = inp["q"].shape
    hkv = inp["k"].shape[1]
    tk = inp["k"].shape[0]
    G = hq // hkv
    max_sq = max(inp["lengths"])
    cnt = visible_counts(inp["q2k_indices"], inp["cu_seqlens_q"], inp["lengths"])
    flops = 4.0 * D * G * float(cnt.sum())
    out = torch.empty_like(inp["q"])
    lse = torch.empty((tq, hq), dtype=torch.float32, device=device)
    W = msa.msa_union_tile_tokens(hq, hkv)
    ulen = msa.msa_build_union(inp["q2k_indices"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                               causal=True, tile_tokens=W)[0]
    flops_exec = float(ulen.sum().item()) * 4.0 * D * 128 * 128
    pk = peaks()
    res = {"workload": spec.name, "tokens": int(tq)}
    sizes = {
        "bf16_copy": msa.msa_sparse_attention_workspace_size_kv(
            len(inp["lengths"]), tq, hq, hkv, D, spec.topk, max_sq, False, inp["k"].dtype, tk),
        "in_kernel": msa.msa_sparse_attention_workspace_size(
            len(inp["lengths"]), tq, hq, hkv, D, spec.topk, max_sq, False)}
    for route, need in sizes.items():
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        for _ in range(2):
            run_prefill(msa, inp, out, lse, ws, max_sq)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ts, ta = [], []
        for _ in range(reps):
            flush.fill_(1)
            msa.msa_set_timing_events(ev)
            run_prefill(msa, inp, out, lse, ws, max_sq)
            ev[2].synchronize()
            ts.append(ev[0].elapsed_time(ev[2]) * 1e-3)
            ta.append(ev[1].elapsed_time(ev[2]) * 1e-3)
        msa.msa_set_timing_events(None)
        t, t_attn = statistics.median(ts), statistics.median(ta)
        res[route] = {
            "value": round(flops / t / 1e12, 2), "unit": "TFLOP/s", "ms": round(t * 1e3, 3),
            "attention_ms": round(t_attn * 1e3, 3),
            "roofline": {"bound": "tensor", "achieved": round(flops / t_attn / 1e12, 2),
                         "peak": pk["bf16"], "unit": "TFLOP/s",
                         "frac": round(flops / t_attn / 1e12 / pk["bf16"], 4)},
            "executed_mma_tflops": round(flops_exec / t_attn / 1e12, 2)}
        del ws
    res["work_efficiency"] = round(flops / flops_exec, 4)
    res["value"], res["unit"] = res["bf16_copy"]["value"], "TFLOP/s"
    del inp
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- reference arm: the oracle
def reference_arm(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    spec = workloads.FLAT_VARLEN
    inp = workloads.make_prefill(spec, 0, device="cpu")
    tq = inp["q"].shape[0]
    hkv = inp["k"].shape[1]
    G = inp["q"].shape[1] // hkv
    cnt = visible_counts(inp["q2k_indices"], inp["cu_seqlens_q"], inp["lengths"])
    cores = os.cpu_count() or 1
    rows_per_step = 64
    g = torch.Generator().manual_seed(77)
    scale = float(np.float32(inp["softmax_scale"]))
    times, flops = [], []
    for step in range(args.warmup + args.steps):
        rows = torch.sort(torch.randperm(tq, generator=g)[:rows_per_step])[0].to(torch.int32)
        f = 4.0 * D * G * float(cnt[:, rows.long()].sum())
        t0 = time.perf_counter()
        oracle.sparse_attention(inp["q"], inp["k"], inp["v"], inp["q2k_indices"],
                                inp["cu_seqlens_q"], inp["cu_seqlens_k"], causal=True,
                                softmax_scale=scale, rows=rows, threads=cores)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            flops.append(f)
    v = sum(flops) / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec.name, "global_batch": 2, "seq_len": 32768,
                       "parallelism": "none (host cores)"},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"{rows_per_step} random query rows x all heads per step"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="msa", choices=["msa", "reference"])
    ap.add_argument("--no-secondary", action="store_true", help="skip decode / two-stage")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-small", action="store_true",
                    help="profiling case: prefill only, 1 x 8192 tokens, 64/8 heads, top-16")
    ap.add_argument("--profile-decode", type=int, default=0, metavar="SQ",
                    help="profiling case: paged decode only, 64 requests, seqlen_q SQ")
    ap.add_argument("--profile-decode-full", action="store_true",
                    help="profiling case: the full paged decode only (128 requests), s_q 1 and 4")
    ap.add_argument("--profile-e4m3", action="store_true",
                    help="profiling case: the E4M3 K/V varlen prefill only")
    ap.add_argument("--profile-nvfp4-small", action="store_true",
                    help="profiling case: the NVFP4 paged decode on 64 requests, s_q 1")
    ap.add_argument("--profile-nvfp4", action="store_true",
                    help="profiling case: the packed NVFP4 paged decode only")
    ap.add_argument("--profile-two-stage", action="store_true",
                    help="profiling case: proxy score, top-k and attention of the two-stage "
                         "workload only")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, world, rank)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import block_sparse_top_msa_gb300 as msa
    msa.build()
    if args.profile_decode:
        flush = l2_flush_buffer(device)
        r = bench_decode(msa, device, flush, small=True, sqs=(args.profile_decode,),
                         reps=args.steps)
        print(json.dumps({"profile_decode": r}))
        return 0
    if args.profile_decode_full:
        flush = l2_flush_buffer(device)
        print(json.dumps({"profile_decode_full": bench_decode(msa, device, flush,
                                                              reps=max(args.steps, 3))}))
        return 0
    if args.profile_nvfp4_small:
        flush = l2_flush_buffer(device)
        print(json.dumps({"profile_nvfp4_small": bench_decode_nvfp4(
            msa, device, flush, sqs=(1,), reps=args.steps, small=True)}))
        return 0
    if args.profile_nvfp4:
        flush = l2_flush_buffer(device)
        print(json.dumps({"profile_nvfp4": bench_decode_nvfp4(msa, device, flush,
                                                              reps=args.steps),
                          "profile_nvfp4_prefill": bench_nvfp4_prefill(msa, device, flush)}))
        return 0
    if args.profile_e4m3:
        flush = l2_flush_buffer(device)
        print(json.dumps({"profile_e4m3": bench_e4m3(msa, device, flush, reps=args.steps)}))
        return 0
    if args.profile_two_stage:
        flush = l2_flush_buffer(device)
        print(json.dumps({"profile_two_stage": bench_two_stage(msa, device, flush)}))
        return 0
    if args.profile_small:
        args.no_secondary = args.no_cpu_baseline = True
    res = bench_prefill(msa, args, device, world, rank)
    flush = l2_flush_buffer(device)
    secondary = {}
    if not args.no_secondary and rank == 0:
        inp_keep = res.pop("inp")
        del inp_keep
        torch.cuda.empty_cache()
        secondary["decode"] = bench_decode(msa, device, flush)
        torch.cuda.empty_cache()
        secondary["decode_nvfp4"] = bench_decode_nvfp4(msa, device, flush)
        torch.cuda.empty_cache()
        secondary["prefill_nvfp4"] = bench_nvfp4_prefill(msa, device, flush)
        torch.cuda.empty_cache()
        secondary["two_stage"] = bench_two_stage(msa, device, flush)
        torch.cuda.empty_cache()
        secondary["e4m3_prefill"] = bench_e4m3(msa, device, flush)
        torch.cuda.empty_cache()
        secondary["tiny_prefill"] = bench_tiny(msa, device, flush)
    else:
        res.pop("inp")
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        _, inp_cpu = prefill_inputs(device)
        v, cores, sample, dt = cpu_baseline_prefill(inp_cpu)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": sample, "seconds": round(dt, 2)}
        if not args.no_secondary:
            inp2 = {k: (t.cpu() if torch.is_tensor(t) else t) for k, t in inp_cpu.items()}
            del inp_cpu
            torch.cuda.empty_cache()
            cpu["other"] = cpu_baseline_suite(device, cpu["cores"], inp2)
    if rank == 0:
        spec = res["spec"]
        line = {
            "metric": METRIC, "value": round(res["value"], 3), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(res["step_s"] * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": spec.name, "global_batch": len(spec.seqlens) * world,
                       "seq_len": spec.seqlens[0],
                       "num_qo_heads": 64, "num_kv_heads": 8, "head_dim": 128, "topk": 16,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (q 1.07 GB, k+v 268 MB, out 1.07 GB per step)"},
            "roofline": res["roofline"],
            "cpu_baseline": cpu,
            "e2e": res["e2e"],
            "gpu_launches": 2 * args.steps,
            "clocks": res["clocks"],
            "work": {"algorithmic_tflop": round(res["flops"] / 1e12, 4),
                     "block_granular_tflop": round(res["flops_block"] / 1e12, 4),
                     "executed_mma_tflop": round(res["flops_exec"] / 1e12, 4),
                     "work_efficiency": round(res["work_efficiency"], 4),
                     "executed_mma_tflops": round(res["executed_tflops"], 2),
                     "union_blocks_per_tile": round(res["union_blocks_per_tile"], 2),
                     "attention_ms": round(res["attn_s"] * 1e3, 3),
                     "metadata_ms": round(res["meta_s"] * 1e3, 3)},
            "device_fault_word": res["fault"],
        }
        line.update(secondary)
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
