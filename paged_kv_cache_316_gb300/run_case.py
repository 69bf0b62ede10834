"""Run one operation of the library on its named synthetic workload.

    python -m paged_kv_cache_316_gb300.run_case --op prefill [--d-qk 128] [--iters 3] [--kv-dtype e4m3]
                                                [--contiguous]
    python -m paged_kv_cache_316_gb300.run_case --op decode_llama | decode_long | decode_varlen | append
                                                [--batch N] [--iters 3] [--kv-dtype e4m3]

Used to drive profilers (ncu) on one kernel at a size that keeps a capture
short; it prints the mean CUDA-event time per call, which is informational
only (the benchmark is bench.py).
"""
from __future__ import annotations

import argparse
import json

import torch

from . import binding as pk
from . import workloads as wl


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", required=True,
                    choices=["prefill", "decode_llama", "decode_long", "decode_varlen", "append"])
    ap.add_argument("--d-qk", type=int, default=128)
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--kv-dtype", choices=["same", "e4m3"], default="same",
                    help="the cache in the query's dtype, or E4M3 (FP8; prefill: query and caches)")
    ap.add_argument("--contiguous", action="store_true",
                    help="prefill: the same keys as contiguous (non-paged) K/V, no block table")
    a = ap.parse_args()
    dev = torch.device("cuda:0")
    from . import build
    build.build()

    if a.op == "prefill":
        e4 = a.kv_dtype == "e4m3"  # E4M3 query and caches, unit device scales
        kw = dict(q_dtype=wl.E4M3, kv_dtype=wl.E4M3) if e4 else {}
        c = wl.ragged_prefill(d_qk=a.d_qk, device=dev, **kw)
        B = c.seq_lens_q.shape[0]
        nbytes = (pk.paged_prefill_fp8_workspace_size(B, c.num_qo_heads, c.num_kv_heads, c.max_q, c.max_kv,
                                                      c.q.shape[0], c.d_qk, c.d_vo, c.q.dtype, c.pool.k.dtype)
                  if e4 else pk.paged_prefill_workspace_size(B, c.num_qo_heads, c.max_q, c.max_kv))
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        lq, lkv, bt = c.seq_lens_q.to(dev), c.seq_lens_kv.to(dev), c.block_tables.to(dev)
        scales = dict(q_scale=torch.ones(1, device=dev), k_scale=torch.ones(1, device=dev),
                      v_scale=torch.ones(1, device=dev)) if e4 else {}

        if a.contiguous:  # each request's keys gathered into [rows, Hkv, d] tensors
            ks, vs = zip(*(wl.read_tokens(c.pool, c.pt, b) for b in range(B)))
            kc, vc = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()

            def run():
                pk.paged_prefill(c.q, kc, vc, c.scale, ws, c.max_q, c.max_kv, lq, lkv, None, causal=True,
                                 **scales)
        else:
            def run():
                pk.paged_prefill(c.q, c.pool.k, c.pool.v, c.scale, ws, c.max_q, c.max_kv, lq, lkv,
                                 bt, causal=True, kv_layout="HND", **scales)
    elif a.op in ("decode_llama", "decode_long", "decode_varlen"):
        kvd = dict(kv_dtype=wl.E4M3) if a.kv_dtype == "e4m3" else {}
        if a.op == "decode_varlen":  # (batch: the first requests of the same draws)
            c = wl.long_decode_varlen(device=dev, batch=a.batch or 256, **kvd)
        elif not a.batch:
            c = (wl.llama_decode(device=dev, **kvd) if a.op == "decode_llama"
                 else wl.long_decode(device=dev, **kvd))
        elif a.op == "decode_llama":  # the first `batch` requests of the same length draw
            L = wl.uniform_lengths(wl.generator(0), 64, 512, 8192)[:a.batch]
            c = wl.decode_case(L, 16, 32, 8, 128, wl.HND, wl.BF16, device=dev, bt_width=512, **kvd)
        else:
            L = wl.lognormal_lengths(wl.generator(0), 256, 4096.0, 1.0, 4, 32768)[:a.batch]
            c = wl.decode_case(L, 64, 64, 8, 128, wl.HND, wl.BF16, q_len_per_req=4,
                               window_left=4095, with_sinks=True, device=dev, bt_width=512, **kvd)
        B = len(c.pt.lengths)
        ws = torch.zeros(max(1, pk.paged_decode_workspace_size(
            B, c.q_len_per_req, c.num_qo_heads, c.num_kv_heads, c.head_dim, c.max_seq_len,
            c.pool.page_size, c.window_left)), dtype=torch.uint8, device=dev)
        bt, sl = c.block_tables.to(dev), c.seq_lens.to(dev)
        sinks = None if c.sinks is None else c.sinks.to(dev)
        kv = c.pool.storage[0]

        cum = None if c.cum_seq_lens_q is None else c.cum_seq_lens_q.to(dev)
        vl = {} if cum is None else dict(cum_seq_lens_q=cum, max_q_len=c.q_len_per_req)

        def run():
            pk.paged_decode(c.query, kv, ws, bt, sl, c.max_seq_len, bmm1_scale=c.bmm1_scale,
                            window_left=c.window_left, sinks=sinks, kv_layout=c.pool.layout,
                            q_len_per_req=c.q_len_per_req, **vl)
    else:
        c = wl.append_sweep(a.batch or 4096, seed=1, layout=wl.NHD, device=dev, fill="empty",
                            **(dict(dtype=wl.E4M3) if a.kv_dtype == "e4m3" else {}))
        kvi, kvp, last = (x.to(dev) for x in (c.kv_indices, c.kv_indptr, c.kv_last_page_len))
        seq = pk.paged_seq_lens(kvp, last, 16)
        nnz = c.append_key.shape[0]
        bi, pos = pk.paged_batch_indices_positions(c.append_indptr.to(dev), seq, nnz)
        pool = c.pool.storage[0]

        def run():
            pk.paged_append(c.append_key, c.append_value, bi, pos, pool, kvi, kvp, last,
                            kv_layout="NHD")

    run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        run()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"op": a.op, "d_qk": a.d_qk, "batch": a.batch, "iters": a.iters,
                      "ms_per_call": e0.elapsed_time(e1) / max(1, a.iters)}))


if __name__ == "__main__":
    main()
