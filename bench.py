#!/usr/bin/env python3
"""Benchmark of the paged block-sparse attend on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extra]

Headline: the decode workload (64 requests, seq 16k-32k, 64/8 heads, head_dim 128, top-k 16
blocks of 128, bf16 paged KV). A step is one pass of the whole hot path over that batch: query
positions, sparse block table compaction, K/V gather, attend and scale folding, all inside one
C-ABI call (pbs_sparse_decode_attention). ``value`` is decode tokens/s with inputs resident in
HBM; ``e2e`` is the same metric with the per-step inputs (q, top-k, page table, seq_lens) copied
from pinned host buffers and the output copied back inside the timed region. The roofline is the
attend kernel's algorithmic bytes per launch over its CUDA-event duration against the measured
HBM copy bandwidth. Secondary numbers (prefill TFLOP/s, fp8 MTP decode, mixed NVFP4, table build)
go under ``extra``.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same workload (the
pages publish no implementation that runs here; the oracle is the reference arm).
Multi-GPU (torchrun, one rank per GPU): every rank runs its own replica of the workload
(independent requests: weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

# Every oracle worker process runs one numpy thread, so the reported core count is exact.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms: float, pg, device) -> float:
    """The slowest rank's step time (every rank gets it): the job is as fast as its slowest replica."""
    if pg is None:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: float, ms: float) -> float:
    """Whole-job throughput: every rank processed units_per_rank units in (at most) ms."""
    return world * units_per_rank / (ms * 1e-3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), \
            "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open(os.path.join("/tmp", f"pbs_clocks_{os.getpid()}.csv"), "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.out is not None:
            self.out.close()

    def summary(self):
        path = os.path.join("/tmp", f"pbs_clocks_{os.getpid()}.csv")
        if self.proc is None or not os.path.exists(path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.remove(path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": n}


def kernel_source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_block_sparse_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(profile_name: str, src_hash: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this kernel source."""
    p = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(p):
        return None
    rec = {}
    for line in open(p):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            v = v.strip()
            if v.startswith("`") and "`" in v[1:]:
                v = v[1:v.index("`", 1)]  # the backticked value; anything after it is a comment
            rec[k.strip()] = v
    if rec.get("kernel_source_sha256_16") != src_hash:
        return None
    try:
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------------------------
# timing helpers
# --------------------------------------------------------------------------------------------

class L2Flush:
    """Before every timed step: write a buffer larger than L2, then read a second one. The write
    evicts whatever the last step left in L2; the read makes those now-dirty flush lines get
    written back here, outside the timed region, so the step starts with a cold and clean L2
    instead of paying for the flush's own write-backs."""

    def __init__(self, nbytes: int = L2_FLUSH_BYTES):
        self.w = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
        self.r = torch.ones(nbytes // 4, dtype=torch.float32, device="cuda")
        self.s = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.add_(1)
        torch.sum(self.r, dim=0, out=self.s)


L2_NOTE = "flushed before every step (256 MiB write, then 256 MiB read: cold, clean L2)"


def time_steps(fn, steps: int, warmup: int, flush: L2Flush, stream: torch.cuda.Stream):
    """Per-step CUDA-event times (ms) on `stream`, L2 flushed before every step."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush()
            fn()
        stream.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for s, e in evs:
            flush()
            s.record(stream)
            fn()
            e.record(stream)
        stream.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


KV_ROW_BYTES = {"bf16": 2 * 128 * 2, "fp8_e4m3": 2 * 128, "nvfp4": 2 * 72}


def decode_bytes(b, ctx: torch.Tensor) -> float:
    """Algorithmic HBM bytes of one decode attend: every attended K/V row once per query row (the
    per-row sum), Q, O, top-k and the page-table entries of the selected blocks."""
    d = b.dec
    rows = d.q.shape[0]
    kv = float(ctx.to(torch.int64).sum().item()) * b.num_kv_heads * KV_ROW_BYTES[b.kv_dtype]
    qo = 2.0 * rows * b.num_heads * 128 * 2
    meta = rows * b.topk * 4 * 2 + rows * 4
    return kv + qo + meta


def decode_union_bytes(b) -> float:
    """decode_bytes with the K/V rows counted once per (request, kv head) over the request's
    decode_query_len right-aligned rows: the union of the keys the rows attend. Within a block a
    row attends a prefix (all 128 keys of a full block, keys up to its position of its own block),
    so the union over rows is, per selected block, the longest prefix any row attends."""
    d = b.dec
    tk = d.topk.reshape(-1, d.topk.shape[-1]).cpu().numpy()
    sl = d.seq_lens.cpu().numpy()
    dql = d.decode_query_len
    union = 0
    for req, L in enumerate(sl.tolist()):
        longest = {}
        for i in range(dql):
            pos = L - dql + i
            if pos < 0:
                continue
            own = pos // 128
            for blk in set(int(x) for x in tk[req * dql + i]):
                if 0 <= blk <= own:
                    n = 128 if blk < own else pos - 128 * own + 1
                    longest[blk] = max(longest.get(blk, 0), n)
        union += sum(longest.values())
    rows = d.q.shape[0]
    kv = float(union) * b.num_kv_heads * KV_ROW_BYTES[b.kv_dtype]
    return kv + 2.0 * rows * b.num_heads * 128 * 2 + rows * b.topk * 4 * 2 + rows * 4


def table_bytes(b, ctx: torch.Tensor) -> float:
    """Algorithmic bytes of one prefill table build: every top-k row read, one page-table entry per
    causally valid distinct block (ceil(ctx / 128) of them per row), the table rows and ctx
    written."""
    p = b.pre
    tk = p.topk.reshape(-1, p.topk.shape[-1])
    valid = int(((ctx.to(torch.int64) + 127) // 128).sum().item())
    return float(tk.numel() * 4 + valid * 4 + tk.shape[0] * b.topk * 8 * 4 + tk.shape[0] * 4)


def prefill_flops(ctx: torch.Tensor, num_heads: int) -> float:
    """Algorithmic FLOPs: QK^T and PV over the attended keys only, 4 * Hq * D per (token, key)."""
    return 4.0 * num_heads * 128 * float(ctx.to(torch.int64).sum().item())


# --------------------------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------------------------

def run_decode(pbs, b, steps, warmup, flush, stream, sparse_table=None, splits=None):
    d = b.dec
    out = torch.empty_like(d.q)

    def step():
        pbs.sparse_decode_attention(d.q, b.cache, b.kv_dtype, b.num_kv_heads, d.topk, d.page_table, d.seq_lens,
                                    d.decode_query_len, b.softmax_scale, b.k_scale, b.v_scale, b.block_page_stride,
                                    out=out, stream=stream, sparse_table=sparse_table, splits=splits)
    return time_steps(step, steps, warmup, flush, stream)


def run_prefill(pbs, b, steps, warmup, flush, stream, workspace="auto", kernel=None, sparse_table=None):
    p = b.pre
    out = torch.empty_like(p.q)

    def step():
        pbs.sparse_prefill_attention(p.q, b.cache, b.kv_dtype, b.num_kv_heads, p.topk, p.page_table,
                                     p.cu_seqlens_q, p.seq_lens, b.softmax_scale, b.k_scale, b.v_scale,
                                     b.block_page_stride, out=out, stream=stream, workspace=workspace, kernel=kernel,
                                     sparse_table=sparse_table)
    return time_steps(step, steps, warmup, flush, stream)


def gather_segments(pbs, b, ws_bytes):
    """Token segments the gathered-row kernel cuts a prefill call into on a workspace of ws_bytes
    (the largest multiple of 256 tokens whose workspace fits, or the whole call)."""
    p = b.pre
    T = p.q.shape[0]

    def need(tokens):
        return pbs.prefill_workspace_bytes(tokens, p.seq_lens.shape[0], b.num_heads, b.num_kv_heads,
                                           p.topk.shape[-1], p.page_table.shape[1])
    if need(T) <= ws_bytes:
        return 1
    lo, hi = 0, T // 256
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if need(mid * 256) <= ws_bytes:
            lo = mid
        else:
            hi = mid - 1
    return -(-T // (lo * 256)) if lo > 0 else 0


def decode_ctx(pbs, b):
    d = b.dec
    _, ctx = pbs.build_sparse_block_table_decode(d.topk, d.page_table, d.seq_lens, d.decode_query_len,
                                                 b.block_page_stride)
    return ctx


def prefill_ctx(pbs, b):
    p = b.pre
    _, ctx = pbs.build_sparse_block_table_prefill(p.topk, p.page_table, p.cu_seqlens_q, p.seq_lens,
                                                  b.block_page_stride)
    return ctx


def e2e_decode(pbs, b, steps, warmup, stream):
    """Same step through the public API with host inputs: pinned H2D copies of q, top-k, page
    table and seq_lens, the attend, and the D2H copy of the output, all inside the timed region."""
    d = b.dec
    host = {k: getattr(d, k).cpu().pin_memory() for k in ("q", "topk", "page_table", "seq_lens")}
    dev = {k: torch.empty_like(getattr(d, k)) for k in host}
    out = torch.empty_like(d.q)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()

    def step():
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        pbs.sparse_decode_attention(dev["q"], b.cache, b.kv_dtype, b.num_kv_heads, dev["topk"], dev["page_table"],
                                    dev["seq_lens"], d.decode_query_len, b.softmax_scale, b.k_scale, b.v_scale,
                                    b.block_page_stride, out=out, stream=stream)
        out_h.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
        stream.synchronize()
        t0 = time.perf_counter()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(steps):
            step()
        e.record(stream)
        stream.synchronize()
        wall = time.perf_counter() - t0
    ms = max(s.elapsed_time(e), wall * 1e3) / steps
    return ms, h2d, d2h


def extra_measurements(pbs, steps, warmup, flush, stream, hbm, bf16):
    res = {}
    # the decode workload fed its prebuilt table (built once per step, shared by every sparse
    # layer) next to the fused call that compacts each row itself
    b = workloads.decode(device="cuda")
    d = b.dec
    tbl = pbs.build_sparse_block_table_decode(d.topk, d.page_table, d.seq_lens, d.decode_query_len, 8)
    by = decode_bytes(b, tbl[1]) + tbl[0].numel() * 4 + tbl[1].numel() * 4
    t = statistics.median(run_decode(pbs, b, steps, warmup, flush, stream, sparse_table=tbl))
    tf = statistics.median(run_decode(pbs, b, steps, warmup, flush, stream))
    res["decode_b64_bf16_prebuilt_table"] = {"ms": t, "fused_ms": tf, "GB/s": by / (t * 1e-3) / 1e9,
                                             "frac_of_hbm_peak": by / (t * 1e-3) / 1e9 / hbm}
    del b, d, tbl
    torch.cuda.empty_cache()
    # decode table build alone (the standalone G1 kernel)
    b = workloads.prefill(device="cuda")
    p = b.pre
    sbt = torch.empty(p.q.shape[0], b.topk * 8, dtype=torch.int32, device="cuda")
    ctxb = torch.empty(p.q.shape[0], dtype=torch.int32, device="cuda")

    def tstep():
        pbs.build_sparse_block_table_prefill(p.topk, p.page_table, p.cu_seqlens_q, p.seq_lens, 8, sparse_bt=sbt,
                                             sparse_ctx=ctxb, stream=stream)
    t = statistics.median(time_steps(tstep, steps, warmup, flush, stream))
    ctx = prefill_ctx(pbs, b)
    tb = table_bytes(b, ctx)
    res["table_build_prefill_22528rows"] = {"ms": t, "GB/s": tb / (t * 1e-3) / 1e9,
                                            "frac_of_hbm_peak": tb / (t * 1e-3) / 1e9 / hbm, "algorithmic_bytes": tb}
    fl = prefill_flops(ctx, b.num_heads)
    ts = run_prefill(pbs, b, max(2, steps // 4), min(warmup, 3), flush, stream)
    t = statistics.median(ts)
    res["prefill_varlen_bf16"] = {"ms": t, "TFLOP/s": fl / (t * 1e-3) / 1e12,
                                  "frac_of_bf16_peak": fl / (t * 1e-3) / 1e12 / bf16, "algorithmic_tflop": fl / 1e12}
    # the same call without a workspace: the tile kernel applies bf16 P as hi + lo parts
    t = statistics.median(run_prefill(pbs, b, max(2, steps // 4), min(warmup, 3), flush, stream, workspace=None))
    res["prefill_varlen_bf16_no_workspace"] = {"ms": t, "TFLOP/s": fl / (t * 1e-3) / 1e12,
                                               "frac_of_bf16_peak": fl / (t * 1e-3) / 1e12 / bf16}
    # the same call on the gathered-row kernel (the binding's default workspace: its token segments)
    ws = pbs.prefill_workspace(p.q.shape[0], p.seq_lens.shape[0], b.num_heads, b.num_kv_heads, b.topk,
                               p.page_table.shape[1], "cuda", stream)
    t = statistics.median(run_prefill(pbs, b, max(2, steps // 4), min(warmup, 3), flush, stream, workspace=ws,
                                      kernel="gather"))
    res["prefill_varlen_bf16_gathered_rows"] = {"ms": t, "TFLOP/s": fl / (t * 1e-3) / 1e12,
                                                "frac_of_bf16_peak": fl / (t * 1e-3) / 1e12 / bf16,
                                                "workspace_bytes": ws.numel(),
                                                "segments": gather_segments(pbs, b, ws.numel())}
    del ws
    pbs._prefill_workspaces.clear()
    # the same call fed the prebuilt prefill table (built once, as every sparse layer would share it)
    tbl = pbs.build_sparse_block_table_prefill(p.topk, p.page_table, p.cu_seqlens_q, p.seq_lens, 8)
    t = statistics.median(run_prefill(pbs, b, max(2, steps // 4), min(warmup, 3), flush, stream, sparse_table=tbl))
    res["prefill_varlen_bf16_prebuilt_table"] = {"ms": t, "TFLOP/s": fl / (t * 1e-3) / 1e12,
                                                 "frac_of_bf16_peak": fl / (t * 1e-3) / 1e12 / bf16}
    del tbl
    del b, p, sbt, ctxb
    torch.cuda.empty_cache()
    # the same prompts with GQA 16 (tile = 8 tokens x 16 heads)
    b = workloads.prefill_g16(device="cuda")
    fl = prefill_flops(prefill_ctx(pbs, b), b.num_heads)
    t = statistics.median(run_prefill(pbs, b, max(2, steps // 4), min(warmup, 3), flush, stream))
    tg = statistics.median(run_prefill(pbs, b, max(2, steps // 4), min(warmup, 3), flush, stream, kernel="gather"))
    res["prefill_varlen_gqa16_bf16"] = {"ms": t, "TFLOP/s": fl / (t * 1e-3) / 1e12,
                                        "frac_of_bf16_peak": fl / (t * 1e-3) / 1e12 / bf16,
                                        "algorithmic_tflop": fl / 1e12, "gather_ms": tg,
                                        "gather_TFLOP/s": fl / (tg * 1e-3) / 1e12}
    pbs._prefill_workspaces.clear()
    del b
    torch.cuda.empty_cache()
    # the prefill prompts on fp8 and NVFP4 caches, on both tcgen05 kernels (K and V converted to
    # images first) and on the token-centric kernel
    for kv in ("fp8_e4m3", "nvfp4"):
        b = workloads.prefill(device="cuda", kv_dtype=kv)
        fl = prefill_flops(prefill_ctx(pbs, b), b.num_heads)
        r = {}
        for kern in ("tile", "gather", "token"):
            t = statistics.median(run_prefill(pbs, b, max(2, steps // 4), min(warmup, 3), flush, stream,
                                              kernel=kern))
            r[f"{kern}_ms"] = t
            r[f"{kern}_TFLOP/s"] = fl / (t * 1e-3) / 1e12
            r[f"{kern}_frac_of_bf16_peak"] = fl / (t * 1e-3) / 1e12 / bf16
        res[f"prefill_varlen_{kv}"] = r
        pbs._tile_workspaces.clear()
        pbs._prefill_workspaces.clear()
        del b
        torch.cuda.empty_cache()
    # fp8 MTP decode: algorithmic bytes = the union of each request's K/V rows over its two
    # right-aligned rows (each kernel CTA serves one row, so the per-row sum is what it reads)
    b = workloads.mtp_fp8(device="cuda")
    ctx = decode_ctx(pbs, b)
    by = decode_bytes(b, ctx)
    byu = decode_union_bytes(b)
    t = statistics.median(run_decode(pbs, b, steps, warmup, flush, stream))
    res["mtp_fp8_decode"] = {"ms": t, "tokens/s": b.dec.q.shape[0] / (t * 1e-3),
                             "union_bytes": byu, "per_row_sum_bytes": by,
                             "GB/s": byu / (t * 1e-3) / 1e9, "frac_of_hbm_peak": byu / (t * 1e-3) / 1e9 / hbm,
                             "per_row_sum_GB/s": by / (t * 1e-3) / 1e9,
                             "per_row_sum_frac_of_hbm_peak": by / (t * 1e-3) / 1e9 / hbm}
    del b
    torch.cuda.empty_cache()
    # the decode workload's shape on fp8 and NVFP4 caches
    for kv in ("fp8_e4m3", "nvfp4"):
        b = workloads.decode(device="cuda", kv_dtype=kv)
        by = decode_bytes(b, decode_ctx(pbs, b))
        t = statistics.median(run_decode(pbs, b, steps, warmup, flush, stream))
        res[f"decode_b64_{kv}"] = {"ms": t, "tokens/s": b.dec.q.shape[0] / (t * 1e-3), "GB/s": by / (t * 1e-3) / 1e9,
                                   "frac_of_hbm_peak": by / (t * 1e-3) / 1e9 / hbm, "algorithmic_bytes": by}
        del b
        torch.cuda.empty_cache()
    # mixed NVFP4: decode then prefill in one stream
    b = workloads.mixed_nvfp4(device="cuda")
    ctx = decode_ctx(pbs, b)
    by = decode_bytes(b, ctx)
    td = statistics.median(run_decode(pbs, b, steps, warmup, flush, stream))
    fl = prefill_flops(prefill_ctx(pbs, b), b.num_heads)
    tp = statistics.median(run_prefill(pbs, b, max(2, steps // 4), min(warmup, 3), flush, stream))
    # the same batch through the one-call mixed entry (decode rows then prefill tokens)
    d, p = b.dec, b.pre
    qm = torch.cat([d.q, p.q])
    tkm = torch.cat([d.topk[0], p.topk[0]])
    om = torch.empty_like(qm)

    def mstep():
        pbs.sparse_mixed_attention(qm, b.cache, b.kv_dtype, b.num_kv_heads, tkm, d.page_table, d.seq_lens,
                                   d.decode_query_len, p.page_table, p.cu_seqlens_q, p.seq_lens, b.softmax_scale,
                                   b.k_scale, b.v_scale, b.block_page_stride, out=om, stream=stream)
    tm = statistics.median(time_steps(mstep, max(2, steps // 4), min(warmup, 3), flush, stream))
    chosen = pbs.prefill_kernel_choice(p.q.shape[0], p.seq_lens.shape[0], b.kv_dtype, b.page_bytes, b.num_heads,
                                       b.num_kv_heads, p.topk.shape[-1], p.page_table.shape[1],
                                       workspace_bytes=1 << 62)
    res["mixed_nvfp4"] = {"decode_ms": td, "decode_GB/s": by / (td * 1e-3) / 1e9,
                          "decode_frac_of_hbm_peak": by / (td * 1e-3) / 1e9 / hbm,
                          "prefill_ms": tp, "prefill_TFLOP/s": fl / (tp * 1e-3) / 1e12,
                          "prefill_frac_of_bf16_peak": fl / (tp * 1e-3) / 1e12 / bf16, "prefill_kernel": chosen,
                          "total_ms": td + tp, "one_call_ms": tm}
    # the prefill part on each prefill kernel (tile and gathered rows: NVFP4 K / V converted to
    # images, then tcgen05)
    for kern in ("gather", "tile", "token"):
        t = statistics.median(run_prefill(pbs, b, max(2, steps // 4), min(warmup, 3), flush, stream, kernel=kern))
        res["mixed_nvfp4"][f"prefill_{kern}_ms"] = t
        res["mixed_nvfp4"][f"prefill_{kern}_TFLOP/s"] = fl / (t * 1e-3) / 1e12
    pbs._tile_workspaces.clear()
    pbs._prefill_workspaces.clear()
    del qm, tkm, om
    del b
    torch.cuda.empty_cache()
    return res


# --------------------------------------------------------------------------------------------
# oracle (cpu_baseline leg and the reference arm)
# --------------------------------------------------------------------------------------------

def oracle_row_pages(b):
    """Host copies of the cache pages each decode row reads (plumbing, before any timing)."""
    d = b.dec
    tk = d.topk.cpu().numpy()
    pt = d.page_table.cpu().numpy()
    out = []
    for r in range(d.q.shape[0]):
        req = r // d.decode_query_len
        blocks = sorted({int(x) for x in tk[0, r] if 0 <= x < pt.shape[1]})
        pages = np.array([int(pt[req, x]) * b.block_page_stride + j for x in blocks for j in range(8)], np.int64)
        host = {}
        if len(pages):
            data = b.cache.index_select(0, torch.from_numpy(pages).to(b.cache.device)).cpu().numpy()
            host = {int(pg): data[i] for i, pg in enumerate(pages)}
        out.append(host)
    return out


def oracle_pool(b):
    """The oracle on every host core: one spawn-started worker per core, each holding its share of
    the decode rows and their pages (see oracle/host_rows.py)."""
    from oracle.host_rows import DecodeRowPool, host_cores
    d = b.dec
    return DecodeRowPool(host_cores(), oracle_row_pages(b), q=d.q.cpu().to(torch.float64).numpy(),
                         kv_dtype=b.kv_dtype, num_kv_heads=b.num_kv_heads, topk=d.topk.cpu().numpy(),
                         page_table=d.page_table.cpu().numpy(), seq_lens=d.seq_lens.cpu().numpy(),
                         decode_query_len=d.decode_query_len, softmax_scale=b.softmax_scale, k_scale=b.k_scale,
                         v_scale=b.v_scale, block_page_stride=b.block_page_stride)


def reference_arm(args, world, rank):
    if rank != 0:
        return
    torch.cuda.set_device(0)
    b = workloads.decode(device="cuda")
    rates = []
    budget = max(2.0, 20.0 / max(args.steps, 1))
    with oracle_pool(b) as pool:
        for i in range(args.warmup + args.steps):
            rate, done, t = pool.run(budget)
            if i >= args.warmup:
                rates.append((rate, done, t))
        workers = pool.workers
    rate = statistics.median(r for r, _, _ in rates)
    ms = 1e3 * b.dec.q.shape[0] / rate
    line = {
        "impl": "reference", "metric": "decode tokens/s", "value": rate, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": b.name, "batch": 64, "heads": "64/8", "head_dim": 128, "topk_blocks": 16,
                   "kv": "bf16 paged, page 16", "l2": "oracle on host"},
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": workers, "kind": "oracle",
                         "sample": f"{rates[0][1]} decode rows per step ({budget:.1f} s on each of {workers} "
                                   f"worker processes, one numpy thread each, rows of the 64-row batch dealt "
                                   f"round-robin; pages copied to host before timing)"},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def secondary_line(pbs, args, world, rank, local, pg, stream, flush, hbm, bf16, peak_src):
    """One JSON line for a non-headline workload (prefill TFLOP/s, or decode GB/s for fp8/NVFP4)."""
    make = {"prefill": workloads.prefill, "mtp_fp8": workloads.mtp_fp8, "mixed_nvfp4": workloads.mixed_nvfp4,
            "prefill_g16": workloads.prefill_g16, "table_prefill": workloads.prefill,
            "decode_fp8": lambda device, seed: workloads.decode(device=device, seed=seed, kv_dtype="fp8_e4m3"),
            "decode_nvfp4": lambda device, seed: workloads.decode(device=device, seed=seed, kv_dtype="nvfp4")}
    b = make[args.workload](device="cuda", seed={"prefill": 1002, "mtp_fp8": 1003, "mixed_nvfp4": 1004,
                                                 "prefill_g16": 1005, "decode_fp8": 1001, "decode_nvfp4": 1001,
                                                 "table_prefill": 1002}[args.workload] + 17 * rank)
    if pg:
        pg.barrier()
    with ClockSampler(local) as clk:
        part = {"prefill": "prefill", "prefill_g16": "prefill", "table_prefill": "table"}.get(args.workload,
                                                                                              args.part)
        launches = 1  # per step
        kernel = None if args.prefill_kernel == "auto" else args.prefill_kernel
        if part == "table":
            # the standalone prefill table build: top-k rows, the page-table entries they name, the
            # table and ctx written
            p = b.pre
            sbt = torch.empty(p.q.shape[0], b.topk * 8, dtype=torch.int32, device="cuda")
            ctxb = torch.empty(p.q.shape[0], dtype=torch.int32, device="cuda")

            def tstep():
                pbs.build_sparse_block_table_prefill(p.topk, p.page_table, p.cu_seqlens_q, p.seq_lens, 8,
                                                     sparse_bt=sbt, sparse_ctx=ctxb, stream=stream)
            times = time_steps(tstep, args.steps, args.warmup, flush, stream)
            work = table_bytes(b, prefill_ctx(pbs, b))
            unit, bound, peak, metric = "GB/s", "hbm", hbm, "table build HBM GB/s"
        elif part == "prefill":
            work = prefill_flops(prefill_ctx(pbs, b), b.num_heads)
            ws = "auto"
            if args.prefill_segment_tokens > 0:
                # a workspace for segments of this many tokens (smaller device footprint, for profiling)
                p = b.pre
                ws = torch.empty(pbs.prefill_workspace_bytes(args.prefill_segment_tokens, p.seq_lens.shape[0],
                                                             b.num_heads, b.num_kv_heads, p.topk.shape[-1],
                                                             p.page_table.shape[1]), dtype=torch.uint8, device="cuda")
            times = run_prefill(pbs, b, args.steps, args.warmup, flush, stream, kernel=kernel, workspace=ws)
            unit, bound, peak, metric = "TFLOP/s", "tensor", bf16, "prefill TFLOP/s"
            p = b.pre
            # the binding's default call on the tile kernel: V conversion, then the attend; on the
            # gathered-row kernel: the conversion, then index, attend and merge per token segment
            chosen = pbs.prefill_kernel_choice(p.q.shape[0], p.seq_lens.shape[0], b.kv_dtype, b.page_bytes,
                                               b.num_heads, b.num_kv_heads, p.topk.shape[-1], p.page_table.shape[1],
                                               kernel=kernel, workspace_bytes=1 << 62)
            if chosen == "tile" and 0 < pbs.prefill_tile_workspace_bytes(
                    p.seq_lens.shape[0], b.num_kv_heads, p.page_table.shape[1], b.kv_dtype) <= pbs.TILE_WORKSPACE_CAP:
                launches = 2
            elif chosen == "gather":
                # the conversion kernel, then per token segment the index, attend and merge kernels
                wsb = ws.numel() if isinstance(ws, torch.Tensor) else pbs.prefill_workspace(
                    p.q.shape[0], p.seq_lens.shape[0], b.num_heads, b.num_kv_heads, p.topk.shape[-1],
                    p.page_table.shape[1], "cuda", stream).numel()
                # (and the tile kernel's attend over the requests' leading tiles, top-k <= 16)
                launches = 1 + (1 if p.topk.shape[-1] <= 16 else 0) + 3 * gather_segments(pbs, b, wsb)
        else:
            # rows of one request share their K/V rows: the union counts each once
            per_row = decode_bytes(b, decode_ctx(pbs, b))
            work = decode_union_bytes(b) if b.dec.decode_query_len > 1 else per_row
            times = run_decode(pbs, b, args.steps, args.warmup, flush, stream, splits=args.splits)
            unit, bound, peak, metric = "GB/s", "hbm", hbm, "decode HBM GB/s"
    ms = max_over_ranks(statistics.mean(times), pg, "cuda")
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    achieved = work / (statistics.mean(times) * 1e-3) / scale
    traffic = None
    if args.workload == "prefill" and part == "prefill":
        # DRAM bytes per launch of the step's dominant kernel, from its committed ncu summary
        if chosen == "gather":
            traffic = recorded_traffic("gather_attend_prefill_varlen.md",
                                       kernel_source_hash("attend_prefill_gather.cu", "tc_device.cuh",
                                                          "pbs_device.cuh"))
        elif chosen == "tile":
            traffic = recorded_traffic("prefill_tc_prefill_varlen_bf16.md",
                                       kernel_source_hash("attend_prefill_tc.cu", "tc_device.cuh", "pbs_device.cuh"))
    if rank == 0:
        print(json.dumps({
            "metric": metric, "value": job_rate(world, work, ms) / scale, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if b.kv_dtype == "bf16" else b.kv_dtype,
            "data": "synthetic", "config": {"workload": b.name, "part": part,
                                            "l2": L2_NOTE},
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                         "traffic": traffic, "peak_source": f"{peak_src} (burst, kernel timed alone)",
                         "algorithmic_work_per_launch": work,
                         **({"per_row_sum_bytes": per_row, "per_row_sum_frac": per_row / (statistics.mean(times) * 1e-3)
                             / scale / peak} if part == "decode" and b.dec.decode_query_len > 1 else {})},
            "gpu_launches": args.steps * launches, "clocks": clk.summary()}), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


# --------------------------------------------------------------------------------------------
# main
# --------------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=64,
                    help="decode requests (64 is the headline workload; smaller only for profiling)")
    ap.add_argument("--part", choices=["decode", "prefill"], default="decode",
                    help="which half of the mixed NVFP4 batch --workload mixed_nvfp4 times")
    ap.add_argument("--splits", type=int, choices=[1, 2, 4, 8], default=None,
                    help="force the decode attend's split count (profiling and tuning)")
    ap.add_argument("--prefill-kernel", choices=["auto", "token", "tile", "gather"], default="auto",
                    help="force the prefill kernel of --workload prefill / prefill_g16 / mixed_nvfp4 --part prefill")
    ap.add_argument("--prefill-segment-tokens", type=int, default=0,
                    help="gathered-row prefill: a workspace for segments of this many tokens (profiling)")
    ap.add_argument("--workload", choices=["decode", "prefill", "prefill_g16", "mtp_fp8", "mixed_nvfp4", "decode_fp8",
                                           "decode_nvfp4", "table_prefill"],
                    default="decode",
                    help="timed workload (the headline line is decode; the others for profiling and tuning)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, world, rank)

    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    from paged_block_sparse_gb300 import _build
    if rank == 0:
        _build.build()
    if pg:
        pg.barrier()
    import paged_block_sparse_gb300 as pbs
    hbm, bf16, bf16_sus, peak_src = peaks()

    stream = torch.cuda.Stream()
    flush = L2Flush()
    if args.workload != "decode":
        return secondary_line(pbs, args, world, rank, local, pg, stream, flush, hbm, bf16, peak_src)
    b = workloads.decode(device="cuda", seed=1001 + 17 * rank, batch=args.batch)
    ctx = decode_ctx(pbs, b)
    by = decode_bytes(b, ctx)
    rows = b.dec.q.shape[0]
    b_name = b.name if args.batch == 64 else f"decode_b{args.batch}_16k-32k_top16_bf16 (profiling size)"

    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        times = run_decode(pbs, b, args.steps, args.warmup, flush, stream, splits=args.splits)
    torch.cuda.synchronize()
    ms = max_over_ranks(statistics.mean(times), pg, "cuda")
    if pg:
        pg.barrier()
    value = job_rate(world, rows, ms)
    achieved = by / (statistics.mean(times) * 1e-3) / 1e9
    src_hash = kernel_source_hash("attend.cu", "pbs_device.cuh")
    traffic = recorded_traffic("attend_decode_b64_bf16.md", src_hash)

    e2e_ms, h2d, d2h = (float("nan"), 0, 0) if args.no_e2e else e2e_decode(pbs, b, max(3, args.steps // 2), 3,
                                                                             stream)
    e2e_ms = max_over_ranks(e2e_ms, pg, "cuda")
    extra = {}
    if not args.no_extra and rank == 0:
        del b
        torch.cuda.empty_cache()
        try:
            extra = extra_measurements(pbs, max(5, args.steps // 2), args.warmup, flush, stream, hbm, bf16)
        except Exception as e:  # secondary numbers must not hide the headline line
            extra = {"error": repr(e)[:300]}
        b = None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        bb = workloads.decode(device="cuda", seed=1001)
        with oracle_pool(bb) as pool:
            rate, done, t = pool.run(10.0)
            workers = pool.workers
        cpu = {"value": rate, "unit": "tokens/s", "cores": workers, "kind": "oracle",
               "sample": f"{done} decode rows of the 64-row batch ({t:.1f} s on each of {workers} worker "
                         f"processes, one fp64 numpy thread each; pages copied to host before timing)"}
        del bb

    if rank == 0:
        line = {
            "metric": "decode tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": b_name, "batch": rows, "decode_query_len": 1,
                       "seq_lens": "U[16384, 32768]", "heads": "64/8", "head_dim": 128, "topk_blocks": 16,
                       "kv": "bf16 paged LBHNC, page 16, K|V per row", "parallelism": f"replicas x{world}",
                       "l2": L2_NOTE},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": traffic, "peak_source": f"{peak_src} hbm_gbs (burst, kernel timed alone)",
                         "algorithmic_bytes_per_launch": by},
            "e2e": {"value": job_rate(world, rows, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "extra": extra,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
