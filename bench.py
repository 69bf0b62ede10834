"""Benchmark of the paged-KV hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step runs every operation of the path once, each on its own synthetic
workload resident in HBM (inputs larger than L2, so no flush is needed):

  index helpers + append  4096 requests, prefix U[0,256], append U[1,128],
                          32 kv heads, head_dim 128, page 16, fp16, NHD
  decode (long context)   batch 256, lognormal kv (median 4096, cap 32768),
                          page 64, 64/8 heads, window 4095, sinks, 4 query tokens
  decode (Llama-shaped)   batch 64, kv U[512,8192], page 16, 32/8 heads, bf16, HND
  prefill d128 / d192     batch 16, q U[128,2048], prefix U[0,2048], page 32,
                          32/8 heads, causal, LSE

Each operation is bracketed by CUDA events on the launching stream.  The
headline value is the Llama-shaped decode's algorithmic HBM bandwidth; the
JSON line also carries every part's throughput, the roofline of the kernel
that dominates the step, the oracle's CPU throughput on a bounded sample
(cpu_baseline), and an end-to-end number through the public API with the
query, block table and lengths copied from one pinned host staging buffer
and the output copied back.

With --impl reference the same metric is measured for the fp64 CPU oracle
on the host cores (bounded sample per step).
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = ("paged-KV attn: decode HBM GB/s, prefill TFLOP/s, append GB/s; "
          "% of GB300 roofline")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD = ("hot-path step: helpers+append (4096 req, 32 kv heads, fp16, NHD) + "
            "long-context decode (B=256, 64/8 heads, window 4095, sinks, Q=4, page 64) + "
            "Llama-3-8B-shaped decode (B=64, kv U[512,8192], 32/8 heads, d128, page 16, HND) + "
            "causal ragged prefill (B=16, 32/8 heads, page 32; d128 and d192/128); "
            "headline = Llama-shaped decode")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ---- algorithmic work per part ----------------------------------------------------------

def decode_bytes(c) -> int:
    """K and V rows each visible query row set needs (read once per kv head),
    query, output, the block-table entries used and the lengths."""
    S = c.pool.page_size
    cum = None if c.cum_seq_lens_q is None else c.cum_seq_lens_q.tolist()
    kv_tok = 0
    pages = 0
    for b, L in enumerate(c.pt.lengths):
        Q = c.q_len_per_req if cum is None else cum[b + 1] - cum[b]
        lo = max(0, L - Q - c.window_left) if c.window_left >= 0 else 0
        kv_tok += L - lo
        pages += (L + S - 1) // S - lo // S
    row = c.num_kv_heads * c.head_dim * c.pool.k.element_size()  # 1 byte per E4M3 element
    qo = 2 * c.query.numel() * 2
    return kv_tok * row * 2 + qo + pages * 4 + len(c.pt.lengths) * 4


def append_bytes(c) -> int:
    nnz, H, D = c.append_key.shape
    return nnz * (2 * 2 * H * D * c.append_key.element_size() + 8)


def prefill_flops(c) -> int:
    tot = 0
    for q, kv in zip(c.seq_lens_q.tolist(), c.seq_lens_kv.tolist()):
        pre = kv - q
        pairs = q * pre + q * (q + 1) // 2 if c.causal else q * kv
        tot += pairs
    return 2 * (c.d_qk + c.d_vo) * c.num_qo_heads * tot


# ---- clocks ---------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples (the JSON line carries their summary); PKV_BENCH_OUT
        # picks the directory
        out_dir = os.environ.get("PKV_BENCH_OUT", os.path.join(ROOT, "bench_out"))
        self.path = os.path.join(out_dir, f"clocks_gpu{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = sorted({n for _, _, fl in rows for n, f in zip(names, fl) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "samples": len(rows), "reasons": seen}


# ---- distributed plumbing -----------------------------------------------------------------------

def dist_setup(n_gpus: int):
    """Rank, world size and local rank from the launcher's environment; for
    more than one rank, a process group (NCCL with GPUs, else gloo) whose
    collectives fail after PKV_DIST_TIMEOUT_S seconds (default 600) instead of
    waiting for a rank that died."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import datetime
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        timeout = datetime.timedelta(seconds=float(os.environ.get("PKV_DIST_TIMEOUT_S", "600")))
        dist.init_process_group(backend, timeout=timeout)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x: float, ws: int, dev) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def allreduce_sum(x: float, ws: int, dev) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---- our arm ----------------------------------------------------------------------------------------

def tagged(name: str, fn):
    """fn wrapped in an NVTX range named after its workload, so that a
    profiler's launch list can be split by workload (`ncu --nvtx
    --print-nvtx-rename kernel`).  A push and a pop cost well under a
    microsecond of host time and nothing on the device."""
    nv = getattr(torch.cuda, "nvtx", None)
    try:
        nv.range_push(name)
        nv.range_pop()
    except Exception:  # a torch build without NVTX: untagged
        return fn

    def run():
        nv.range_push(name)
        try:
            fn()
        finally:
            nv.range_pop()
    return run


class Part:
    def __init__(self, name, fn, work, unit, bound, kernel):
        self.name, self.work, self.unit, self.bound = name, work, unit, bound
        self.fn = tagged(name, fn)
        self.kernel = kernel  # source file of the dominant kernel of this part
        self.ms = []


def rank_seed(rank: int) -> int:
    """Seed offset of a rank's workloads: every rank draws its own requests
    of the same shape (weak scaling, no shared data)."""
    return 1000 * rank


def aggregate_parts(stats, ws: int, dev, pk_peaks) -> dict:
    """Whole-job result per part from each rank's (name, mean ms, work,
    unit): work summed over ranks, divided by the slowest rank's time;
    roofline_frac is per GPU."""
    out = {}
    for name, mean_ms, work, unit in stats:
        mean_ms = allreduce_max(mean_ms, ws, dev)
        work = allreduce_sum(float(work), ws, dev)
        if unit == "GB/s":
            val = work / (mean_ms * 1e-3) / 1e9
            peak = pk_peaks["hbm_gbs"]
        else:
            val = work / (mean_ms * 1e-3) / 1e12
            peak = pk_peaks["bf16_tflops"]
        out[name] = {"value": round(val, 2), "unit": unit, "ms": round(mean_ms, 4),
                     "work": int(work), "roofline_frac": round(val / peak / ws, 4)}
    return out


def make_parts(rank: int, dev):
    import paged_kv_cache_316_gb300 as pk
    from paged_kv_cache_316_gb300 import workloads as wl
    parts = []
    seed_off = rank_seed(rank)

    # index helpers + append
    ap = wl.append_sweep(4096, seed=1 + seed_off, layout=wl.NHD, device=dev, fill="empty")
    ak, av = ap.append_key, ap.append_value
    kvi, kvp, last = (x.to(dev) for x in (ap.kv_indices, ap.kv_indptr, ap.kv_last_page_len))
    aind = ap.append_indptr.to(dev)
    nnz = ak.shape[0]
    seq = torch.empty(4096, dtype=torch.int32, device=dev)
    bi = torch.empty(nnz, dtype=torch.int32, device=dev)
    pos = torch.empty(nnz, dtype=torch.int32, device=dev)
    pool = ap.pool.storage[0]

    def run_helpers():
        pk.paged_seq_lens(kvp, last, 16, seq)
        pk.paged_batch_indices_positions(aind, seq, nnz, bi, pos)

    def run_append():
        pk.paged_append(ak, av, bi, pos, pool, kvi, kvp, last, kv_layout="NHD")

    run_helpers()
    parts.append(Part("index_helpers", run_helpers, 4096 * 12 + nnz * 8 + 4097 * 4, "GB/s",
                      "hbm", "append.cu"))
    parts.append(Part("append", run_append, append_bytes(ap), "GB/s", "hbm", "append.cu"))

    def decode_part(name, c):
        kv = c.pool.storage[0]
        B = len(c.pt.lengths)
        ws = torch.zeros(max(1, pk.paged_decode_workspace_size(
            B, c.q_len_per_req, c.num_qo_heads, c.num_kv_heads, 128, c.max_seq_len,
            c.pool.page_size, c.window_left)), dtype=torch.uint8, device=dev)
        bt, sl = c.block_tables.to(dev), c.seq_lens.to(dev)
        sinks = None if c.sinks is None else c.sinks.to(dev)
        out = torch.empty_like(c.query)

        def run():
            pk.paged_decode(c.query, kv, ws, bt, sl, c.max_seq_len, bmm1_scale=c.bmm1_scale,
                            bmm2_scale=c.bmm2_scale, window_left=c.window_left, sinks=sinks,
                            kv_layout="HND", q_len_per_req=c.q_len_per_req, out=out)
        p = Part(name, run, decode_bytes(c), "GB/s", "hbm", "decode.cu")
        p.case, p.ws, p.bt, p.sl, p.sinks = c, ws, bt, sl, sinks
        return p

    # the long-context decode (reads only) runs between the append and the
    # Llama-shaped decode, so that the headline part does not pay the
    # write-back of the append's dirty L2 lines
    parts.append(decode_part("decode_long", wl.long_decode(seed=0 + seed_off, device=dev)))
    llama = wl.llama_decode(seed=0 + seed_off, device=dev)
    parts.append(decode_part("decode_llama", llama))

    for dqk in (128, 192):
        c = wl.ragged_prefill(seed=0 + seed_off, d_qk=dqk, device=dev)
        ws = torch.zeros(pk.paged_prefill_workspace_size(16, 32, c.max_q, c.max_kv),
                         dtype=torch.uint8, device=dev)
        lq, lkv, bt = c.seq_lens_q.to(dev), c.seq_lens_kv.to(dev), c.block_tables.to(dev)
        out = torch.empty((c.q.shape[0], 32, 128), dtype=c.q.dtype, device=dev)
        lse = torch.empty((c.q.shape[0], 32), dtype=torch.float32, device=dev)

        def run(c=c, ws=ws, lq=lq, lkv=lkv, bt=bt, out=out, lse=lse):
            pk.paged_prefill(c.q, c.pool.k, c.pool.v, c.scale, ws, c.max_q, c.max_kv, lq, lkv,
                             bt, causal=True, out=out, lse=lse, kv_layout="HND")
        parts.append(Part(f"prefill_d{dqk}", run, prefill_flops(c), "TFLOP/s", "tensor",
                          "prefill.cu"))
    return parts


def make_next_parts(rank: int, dev):
    """Rows beyond the hot path's configurations, measured the same way but
    outside the step: variable-length multi-token decode and non-paged prefill."""
    import paged_kv_cache_316_gb300 as pk
    from paged_kv_cache_316_gb300 import workloads as wl
    c = wl.long_decode_varlen(seed=rank_seed(rank), device=dev)
    B = len(c.pt.lengths)
    ws = torch.zeros(max(1, pk.paged_decode_workspace_size(
        B, c.q_len_per_req, c.num_qo_heads, c.num_kv_heads, c.head_dim, c.max_seq_len,
        c.pool.page_size, c.window_left)), dtype=torch.uint8, device=dev)
    bt, sl, cum = c.block_tables.to(dev), c.seq_lens.to(dev), c.cum_seq_lens_q.to(dev)
    sinks = c.sinks.to(dev)
    kv = c.pool.storage[0]
    out = torch.empty_like(c.query)

    def run():
        pk.paged_decode(c.query, kv, ws, bt, sl, c.max_seq_len, bmm1_scale=c.bmm1_scale,
                        window_left=c.window_left, sinks=sinks, kv_layout=c.pool.layout,
                        cum_seq_lens_q=cum, max_q_len=c.q_len_per_req, out=out)
    parts = [Part("decode_varlen", run, decode_bytes(c), "GB/s", "hbm", "decode.cu")]

    # the ragged prefill with contiguous (non-paged) K/V, d_qk 128
    pc = wl.ragged_prefill(seed=rank_seed(rank), d_qk=128, device=dev)
    ks, vs = [], []
    for b in range(len(pc.pt.lengths)):
        k, v = wl.read_tokens(pc.pool, pc.pt, b)
        ks.append(k)
        vs.append(v)
    kc, vc = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
    pws = torch.zeros(pk.paged_prefill_workspace_size(16, 32, pc.max_q, pc.max_kv), dtype=torch.uint8,
                      device=dev)
    lq, lkv = pc.seq_lens_q.to(dev), pc.seq_lens_kv.to(dev)
    pout = torch.empty((pc.q.shape[0], 32, 128), dtype=pc.q.dtype, device=dev)
    plse = torch.empty((pc.q.shape[0], 32), dtype=torch.float32, device=dev)

    def run_prefill():
        pk.paged_prefill(pc.q, kc, vc, pc.scale, pws, pc.max_q, pc.max_kv, lq, lkv, None,
                         causal=True, out=pout, lse=plse)
    parts.append(Part("prefill_d128_contiguous", run_prefill, prefill_flops(pc), "TFLOP/s", "tensor",
                      "prefill.cu"))

    # the Llama-shaped decode over an E4M3 (FP8) cache
    c8 = wl.llama_decode(seed=rank_seed(rank), device=dev, kv_dtype=wl.E4M3)
    ws8 = torch.zeros(max(1, pk.paged_decode_workspace_size(
        64, 1, 32, 8, 128, c8.max_seq_len, 16, -1)), dtype=torch.uint8, device=dev)
    bt8, sl8 = c8.block_tables.to(dev), c8.seq_lens.to(dev)
    out8 = torch.empty_like(c8.query)

    def run_fp8():
        pk.paged_decode(c8.query, c8.pool.storage[0], ws8, bt8, sl8, c8.max_seq_len,
                        bmm1_scale=c8.bmm1_scale, kv_layout=c8.pool.layout, out=out8)
    parts.append(Part("decode_llama_e4m3", run_fp8, decode_bytes(c8), "GB/s", "hbm", "decode.cu"))

    # the append sweep point in E4M3
    a8 = wl.append_sweep(4096, seed=1 + rank_seed(rank), layout=wl.NHD, device=dev, fill="empty",
                         dtype=wl.E4M3)
    kvi8, kvp8, last8 = (x.to(dev) for x in (a8.kv_indices, a8.kv_indptr, a8.kv_last_page_len))
    seq8 = pk.paged_seq_lens(kvp8, last8, 16)
    bi8, pos8 = pk.paged_batch_indices_positions(a8.append_indptr.to(dev), seq8, a8.append_key.shape[0])
    pool8 = a8.pool.storage[0]

    def run_append8():
        pk.paged_append(a8.append_key, a8.append_value, bi8, pos8, pool8, kvi8, kvp8, last8, kv_layout="NHD")
    parts.append(Part("append_e4m3", run_append8, append_bytes(a8), "GB/s", "hbm", "append.cu"))

    # the ragged prefill (d_qk 128) over an E4M3 query and E4M3 caches, with
    # device scales: QK in E4M3 MMAs, V widened inside the attention kernel
    pf = wl.ragged_prefill(seed=rank_seed(rank), d_qk=128, device=dev, q_dtype=wl.E4M3,
                           kv_dtype=wl.E4M3)
    fws = torch.zeros(pk.paged_prefill_fp8_workspace_size(
        16, 32, 8, pf.max_q, pf.max_kv, pf.q.shape[0], 128, 128, pf.q.dtype, pf.pool.k.dtype),
        dtype=torch.uint8, device=dev)
    flq, flkv, fbt = pf.seq_lens_q.to(dev), pf.seq_lens_kv.to(dev), pf.block_tables.to(dev)
    fout = torch.empty((pf.q.shape[0], 32, 128), dtype=torch.bfloat16, device=dev)
    flse = torch.empty((pf.q.shape[0], 32), dtype=torch.float32, device=dev)
    qs, kscale, vscale = (torch.ones(1, device=dev) for _ in range(3))

    def run_prefill8():
        pk.paged_prefill(pf.q, pf.pool.k, pf.pool.v, pf.scale, fws, pf.max_q, pf.max_kv, flq, flkv,
                         fbt, causal=True, out=fout, lse=flse, kv_layout="HND", q_scale=qs,
                         k_scale=kscale, v_scale=vscale)
    parts.append(Part("prefill_d128_e4m3", run_prefill8, prefill_flops(pf), "TFLOP/s", "tensor",
                      "prefill.cu"))
    return parts


SWEEP_BATCHES = (4, 16, 64, 256, 1024, 4096)


def time_flushed(fn, iters: int, flush, st) -> float:
    """Median CUDA-event time (ms) of `iters` runs of fn, each preceded by a
    write of `flush` (twice the L2) outside the timed region, so that no run
    finds its inputs in L2."""
    ms = []
    for _ in range(iters):
        flush.zero_()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        z.record(st)
        ms.append((a, z))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(z) for a, z in ms)


def run_sweeps(rank: int, dev, iters: int, pk_peaks) -> dict:
    """Every other configuration of the workloads, each timed as the median
    of `iters` runs with L2 flushed before each: the append sweep (4 ..
    4096 requests appending U[1,128] tokens, and one token each), the append
    page's worked example (NHD / HND, 5-D / tuple cache), the 4-request
    decode of 45/8/25/22 keys (HND / NHD) and the Llama-shaped decode in NHD.
    Small ones are latency-bound: their microseconds are the figure to read."""
    import paged_kv_cache_316_gb300 as pk
    from paged_kv_cache_316_gb300 import workloads as wl
    st = torch.cuda.current_stream()
    flush = torch.empty(2 * 129 * 2 ** 20 // 4 * 4, dtype=torch.uint8, device=dev)
    hbm = pk_peaks["hbm_gbs"]
    out = {}

    def entry(ms, nbytes, **kw):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return dict(kw, us=round(ms * 1e3, 2), bytes=int(nbytes), value=round(gbs, 2), unit="GB/s",
                    roofline_frac=round(gbs / hbm, 4))

    def append_point(c, layout_name, tag):
        kvi, kvp, last = (x.to(dev) for x in (c.kv_indices, c.kv_indptr, c.kv_last_page_len))
        seq = pk.paged_seq_lens(kvp, last, c.pool.page_size)
        nnz = c.append_key.shape[0]
        bi, pos = pk.paged_batch_indices_positions(c.append_indptr.to(dev), seq, nnz)
        ak, av = c.append_key.to(dev), c.append_value.to(dev)
        kv = c.pool.storage[0] if len(c.pool.storage) == 1 else c.pool.storage

        run = tagged(tag, lambda: pk.paged_append(ak, av, bi, pos, kv, kvi, kvp, last,
                                                  kv_layout=layout_name))
        for _ in range(3):
            run()
        return time_flushed(run, iters, flush, st), append_bytes(c), nnz

    for one in (False, True):
        rows = []
        for B in SWEEP_BATCHES:
            c = wl.append_sweep(B, seed=1 + rank_seed(rank), layout=wl.NHD, one_token=one, device=dev,
                                fill="empty")
            ms, nb, nnz = append_point(c, "NHD", f"sweep_append{'_one' if one else ''}_{B}")
            rows.append(entry(ms, nb, batch=B, tokens=nnz))
            del c
        out["append_one_token" if one else "append"] = rows
    ex = {}
    for layout, lname in ((wl.NHD, "NHD"), (wl.HND, "HND")):
        for form in ("5d", "tuple"):
            c = wl.append_example(layout=layout, form=form, device=dev)
            ms, nb, nnz = append_point(c, lname, f"sweep_example_{lname}_{form}")
            ex[f"{lname}_{form}"] = entry(ms, nb, tokens=nnz)
    out["append_example"] = ex

    def decode_point(c, lname, tag):
        B = len(c.pt.lengths)
        ws = torch.zeros(max(1, pk.paged_decode_workspace_size(
            B, c.q_len_per_req, c.num_qo_heads, c.num_kv_heads, 128, c.max_seq_len, c.pool.page_size,
            c.window_left)), dtype=torch.uint8, device=dev)
        q, kv = c.query.to(dev), c.pool.storage[0].to(dev)
        bt, sl = c.block_tables.to(dev), c.seq_lens.to(dev)
        o = torch.empty_like(q)

        run = tagged(tag, lambda: pk.paged_decode(q, kv, ws, bt, sl, c.max_seq_len,
                                                  bmm1_scale=c.bmm1_scale, kv_layout=lname, out=o))
        for _ in range(3):
            run()
        return time_flushed(run, iters, flush, st), decode_bytes(c)

    pr = {}
    for layout, lname in ((wl.HND, "HND"), (wl.NHD, "NHD")):
        ms, nb = decode_point(wl.pr1_decode(seed=rank_seed(rank), layout=layout, device=dev), lname,
                              f"sweep_decode_pr1_{lname}")
        pr[lname] = entry(ms, nb)
    out["decode_pr1"] = pr
    ms, nb = decode_point(wl.llama_decode(seed=rank_seed(rank), layout=wl.NHD, device=dev), "NHD",
                          "sweep_decode_llama_nhd")
    out["decode_llama_nhd"] = entry(ms, nb)
    out["note"] = (f"median of {iters} runs, L2 flushed (a {flush.numel() >> 20} MB write) before each run; "
                   "bytes are the algorithmic bytes of the call")
    return out


def traffic_for(kernel_file: str, part: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel source as it is now."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        d = json.load(open(path))
        e = d[part]
        src = os.path.join(ROOT, "paged_kv_cache_316_gb300", "csrc", kernel_file)
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return e["dram_bytes_per_launch"] if e.get("src_sha") == sha else None
    except Exception:
        return None


def _repeat_for(budget_s, fn):
    """Run fn() (returning work units) until ~budget_s of wall time; at least
    once.  Returns (units, seconds, repetitions)."""
    units, reps, t0 = 0, 0, time.perf_counter()
    while True:
        units += fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            return units, el, reps


def cpu_baselines(llama_case, budget_s: float = 4.0):
    """The oracle, as it stands, on bounded samples of each operation's
    workload, timed on the host cores: single-threaded and with all the
    threads the oracle can use (OpenMP; its append is a serial loop).  Rates
    are work / time on the sample, in the unit of the GPU part."""
    import oracle
    from paged_kv_cache_316_gb300 import workloads as wl
    u16 = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    all_thr = oracle.max_threads()
    res = {}
    # decode: requests 0-3 of the Llama-shaped decode, all heads, full length
    c = llama_case
    subs = []
    for b in range(4):
        pages = c.pt.pages[b]
        idx = torch.tensor(pages, dtype=torch.long, device=c.pool.k.device)
        k = c.pool.k.index_select(0, idx).cpu().contiguous()
        v = c.pool.v.index_select(0, idx).cpu().contiguous()
        subs.append((c.query[b:b + 1].cpu().contiguous(), k, v, c.pt.lengths[b],
                     np.arange(len(pages), dtype=np.int32)[None, :]))

    def dec(thr):
        nb = 0
        for q, k, v, L, bt in subs:
            oracle.decode(u16(q), u16(k), u16(v), k[0].numel(), k.shape[0], bt, np.array([L], np.uint32),
                          L, c.bmm1_scale, 1.0, -1, None, 1, 32, 8, 128, 16, wl.HND, wl.BF16, threads=thr)
            nb += L * 8 * 128 * 2 * 2 + 2 * 32 * 128 * 2 + ((L + 15) // 16) * 4 + 4
        return nb
    for name, thr in (("single", 1), ("all", all_thr)):
        nb, el, reps = _repeat_for(budget_s, lambda: dec(thr))
        res.setdefault("decode_llama", {})[name] = {
            "value": round(nb / el / 1e9, 4), "unit": "GB/s", "cores": thr, "reps": reps, "s": round(el, 2)}
    res["decode_llama"]["sample"] = ("requests 0-3 of the Llama-shaped decode (all 32 heads, full kv "
                                     "length, kv lengths %s)" % [s_[3] for s_ in subs])
    # append: 64 requests of the append sweep's shape (fp16, 32 kv heads)
    a = wl.append_sweep(64, seed=1, layout=wl.NHD)
    sl = oracle.seq_lens(a.kv_indptr.numpy(), a.kv_last_page_len.numpy(), 16)
    bi, pos = oracle.batch_indices_positions(a.append_indptr.numpy(), sl, a.append_key.shape[0])
    pool = a.pool.storage[0]
    pk_, pv_ = u16(pool[:, 0]), u16(pool[:, 1])

    def app():
        oracle.append(u16(a.append_key), u16(a.append_value), bi, pos, pk_, pv_, a.pool.k_page_stride,
                      a.pool.num_pages, a.kv_indices.numpy(), a.kv_indptr.numpy(),
                      a.kv_last_page_len.numpy(), 32, 128, 16, wl.NHD)
        return append_bytes(a)
    nb, el, reps = _repeat_for(budget_s / 2, app)
    one = {"value": round(nb / el / 1e9, 4), "unit": "GB/s", "cores": 1, "reps": reps, "s": round(el, 2)}
    res["append"] = {"single": one, "all": dict(one, note="the oracle's append is a serial loop"),
                     "sample": f"64 requests of the append sweep's shape ({a.append_key.shape[0]} tokens, "
                               "fp16, 32 kv heads, d 128, page 16, NHD)"}
    # prefill: one request (q 1024, prefix 1024) of the ragged prefill's shape
    # with 4 qo heads over 1 kv head (the per-head work of the 32/8 config)
    pc = wl.prefill_case([1024], [2048], 32, 4, 1, 128, 128, wl.HND, wl.BF16, seed=5)
    fl = prefill_flops(pc)

    def pre(thr):
        oracle.prefill(u16(pc.q), u16(pc.pool.k), u16(pc.pool.v), pc.pool.k_page_stride,
                       pc.pool.v_page_stride, pc.pool.num_pages, pc.scale, pc.seq_lens_q.numpy(),
                       pc.seq_lens_kv.numpy(), pc.block_tables.numpy(), True, 4, 1, 128, 128, 32, wl.HND,
                       wl.BF16, threads=thr)
        return fl
    for name, thr in (("single", 1), ("all", all_thr)):
        f, el, reps = _repeat_for(budget_s, lambda: pre(thr))
        res.setdefault("prefill_d128", {})[name] = {
            "value": round(f / el / 1e12, 6), "unit": "TFLOP/s", "cores": thr, "reps": reps, "s": round(el, 2)}
    res["prefill_d128"]["sample"] = ("one causal request (q 1024 after a 1024-token prefix) of the ragged "
                                     "prefill's shape, 4 qo heads / 1 kv head, d 128")
    dl = res["decode_llama"]
    return {"value": dl["all"]["value"], "unit": "GB/s", "cores": all_thr, "kind": "oracle",
            "sample": "fp64 oracle decode of " + dl["sample"] + "; per_op holds every operation, "
                      "single-threaded and on all threads",
            "per_op": res}


def e2e_decode(part, steps: int, dev):
    """Decode through the public API with the step's inputs (query, block
    table, lengths) copied from one pinned host staging buffer into device
    memory and the output copied back to pinned host memory, every step."""
    import paged_kv_cache_316_gb300 as pk
    c = part.case
    inputs = [c.query.cpu(), c.block_tables.cpu(), c.seq_lens.cpu()]
    offs, total = [], 0
    for t in inputs:  # 256-byte aligned segments of one staging buffer
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(total, dtype=torch.uint8, device=dev)
    views_h, views_d = [], []
    for t, o in zip(inputs, offs):
        n = t.numel() * t.element_size()
        hv = hbuf[o:o + n].view(t.dtype).view(t.shape)
        hv.copy_(t)
        views_h.append(hv)
        views_d.append(dbuf[o:o + n].view(t.dtype).view(t.shape))
    dq, dbt, dsl = views_d
    hout = torch.empty(c.query.shape, dtype=c.query.dtype).pin_memory()
    kv = c.pool.storage[0]
    dout = torch.empty_like(c.query)

    @functools.partial(tagged, "e2e_decode")
    def step():
        dbuf.copy_(hbuf, non_blocking=True)
        pk.paged_decode(dq, kv, part.ws, dbt, dsl, c.max_seq_len, bmm1_scale=c.bmm1_scale,
                        kv_layout="HND", out=dout)
        hout.copy_(dout, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        step()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    assert torch.equal(hout, dout.cpu())
    h2d = sum(t.numel() * t.element_size() for t in inputs)
    return ms, h2d, hout.numel() * hout.element_size()


def run_ours(args):
    ws, rank, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from paged_kv_cache_316_gb300 import build as _build
    if rank == 0 or ws == 1:
        _build.build()
    barrier(ws)
    import paged_kv_cache_316_gb300 as pk

    parts = make_parts(rank, dev)
    st = torch.cuda.current_stream()
    for _ in range(args.warmup):
        for p in parts:
            p.fn()
    torch.cuda.synchronize()

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in parts] for _ in range(args.steps)]
    launches0 = pk.kernel_launches()
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(st)
        for s in range(args.steps):
            for i, p in enumerate(parts):
                ev[s][i][0].record(st)
                p.fn()
                ev[s][i][1].record(st)
        t1.record(st)
        torch.cuda.synchronize()
    barrier(ws)
    launches = pk.kernel_launches() - launches0
    total_ms = t0.elapsed_time(t1)
    for i, p in enumerate(parts):
        p.ms = [ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps)]
    total_ms = allreduce_max(total_ms, ws, dev)

    pk_peaks, peak_src = peaks()
    out_parts = aggregate_parts([(p.name, sum(p.ms) / len(p.ms), p.work, p.unit) for p in parts],
                                ws, dev, pk_peaks)
    step_ms = total_ms / args.steps
    dom = max(parts, key=lambda p: sum(p.ms))
    d = out_parts[dom.name]
    per_launch_work = dom.work
    ach = (per_launch_work / (d["ms"] * 1e-3)) / (1e9 if dom.unit == "GB/s" else 1e12)
    peak = pk_peaks["hbm_gbs"] if dom.unit == "GB/s" else pk_peaks["bf16_tflops"]
    roofline = {"kernel": dom.name, "bound": dom.bound, "achieved": round(ach, 2), "peak": peak,
                "unit": dom.unit, "frac": round(ach / peak, 4),
                "peak_source": f"{peak_src} ({'hbm_gbs' if dom.unit == 'GB/s' else 'bf16_tflops'})",
                "traffic": traffic_for(dom.kernel, dom.name)}

    # rows beyond the step's configurations: timed the same way, after the step
    nxt = make_next_parts(rank, dev)
    # each part: warm-up runs right before its timed runs, then `steps`
    # calls back to back between two events (consecutive calls, as a serving
    # loop issues them: one call's launch overlaps the previous call's tail)
    for p in nxt:
        for _ in range(args.warmup):
            p.fn()
        torch.cuda.synchronize()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(args.steps):
            p.fn()
        z.record(st)
        torch.cuda.synchronize()
        p.ms = [a.elapsed_time(z) / args.steps]
    next_rows = aggregate_parts([(p.name, sum(p.ms) / len(p.ms), p.work, p.unit) for p in nxt],
                                ws, dev, pk_peaks)

    sweeps = run_sweeps(rank, dev, 50, pk_peaks) if not args.no_sweeps else None

    llama = next(p for p in parts if p.name == "decode_llama")
    e2e_ms, h2d, d2h = e2e_decode(llama, max(10, args.steps // 4), dev)
    e2e_ms = allreduce_max(e2e_ms, ws, dev)
    value = out_parts["decode_llama"]["value"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{ws} (independent requests)",
                   "l2": "step parts: no flush, every part's inputs exceed the 129 MB L2; sweeps: "
                         "L2 flushed before every timed run",
                   "headline_part": "decode_llama"},
        "parts": out_parts, "roofline": roofline,
        "next_rows": dict(next_rows, note="outside the step and its ms_per_step: variable-length "
                                          "multi-token decode on the long-context shape (1..4 query "
                                          "tokens per request); the ragged prefill (d_qk 128) with "
                                          "contiguous, non-paged K/V; the Llama-shaped decode and the "
                                          "4096-request append over an E4M3 (FP8) cache; the ragged "
                                          "prefill (d_qk 128) over an E4M3 query and E4M3 caches"),
        "e2e": {"value": round(allreduce_sum(float(llama.work), ws, dev) / (e2e_ms * 1e-3) / 1e9, 2),
                "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "what": "paged_decode through the Python API; query, block table and lengths "
                        "copied from one pinned host staging buffer (one copy) and the output "
                        "copied back each step"},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    if sweeps is not None:
        line["sweeps"] = sweeps
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baselines(llama.case)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The oracle as it stands, timed on the host cores, on bounded samples of
    the Llama-shaped decode (2 requests, all heads, per step)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_316_gb300 import workloads as wl
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    c = wl.llama_decode(seed=0, device=dev)
    u16 = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    samples = []
    for b in range(len(c.pt.lengths)):
        pages = c.pt.pages[b]
        idx = torch.tensor(pages, dtype=torch.long, device=c.pool.k.device)
        k = c.pool.k.index_select(0, idx).cpu().contiguous()
        v = c.pool.v.index_select(0, idx).cpu().contiguous()
        samples.append((c.query[b:b + 1].cpu().contiguous(), k, v, c.pt.lengths[b]))

    def step(i):
        nb = 0
        for j in range(2):
            q, k, v, L = samples[(2 * i + j) % len(samples)]
            bt = np.arange(k.shape[0], dtype=np.int32)[None, :]
            oracle.decode(u16(q), u16(k), u16(v), k[0].numel(), k.shape[0], bt,
                          np.array([L], np.uint32), L, c.bmm1_scale, 1.0, -1, None, 1, 32, 8,
                          128, 16, wl.HND, wl.BF16)
            nb += L * 8 * 128 * 2 * 2 + 2 * 32 * 128 * 2 + ((L + 15) // 16) * 4 + 4
        return nb

    for i in range(args.warmup):
        step(i)
    tot_b, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        tot_b += step(args.warmup + i)
    el = time.perf_counter() - t0
    val = tot_b / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "headline_part": "decode_llama",
                       "reference": "fp64 CPU oracle (the pages ship no code to run)"},
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "kind": "oracle",
                             "cores": oracle.max_threads(),
                             "sample": "per step: 2 requests of the Llama-shaped decode "
                                       "(all 32 heads, full kv length), fp64 oracle"},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweeps", action="store_true",
                    help="skip the sweep / small-configuration measurements")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
