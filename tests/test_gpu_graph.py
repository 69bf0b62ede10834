"""The hot path under CUDA-graph capture: every call is asynchronous on the
caller's stream and allocates nothing, so append, decode (uniform and
variable-length) and prefill can be captured into one graph -- including the
programmatic-dependent launches inside decode and prefill -- and every
replay reproduces the eager results bit for bit; each replay's outputs are
also checked against the fp64 oracle (append bit-exact, attention within
|err| <= 2e-2 + 1e-2 |ref|, LSE within 1e-3)."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_316_gb300 as pk
from paged_kv_cache_316_gb300 import workloads as wl
from _gpu import DEV, assert_attn_close, assert_lse_close
from _util import oracle_append, oracle_decode, oracle_prefill

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype in (torch.bfloat16, torch.float16) else t


def test_graph_replay_matches_eager():
    # the cases are drawn on the CPU (the oracle reads them there) and copied
    # to the device
    # append into its own pool, zeroed before every run
    ap = wl.append_sweep(16, seed=3, layout=wl.NHD, fill="empty")
    ap.pool.storage[0].zero_()
    nnz = ap.append_key.shape[0]
    cpu_pool = ap.pool.storage[0].clone()
    sl_ref = oracle.seq_lens(ap.kv_indptr.numpy(), ap.kv_last_page_len.numpy(), 16)
    bi_ref, pos_ref = oracle.batch_indices_positions(ap.append_indptr.numpy(), sl_ref, nnz)
    assert oracle_append(ap, bi_ref, pos_ref) == 0  # (in place, on ap's CPU pool)
    pool_ref = ap.pool.storage[0]
    kvi, kvp, last = (x.to(DEV) for x in (ap.kv_indices, ap.kv_indptr, ap.kv_last_page_len))
    ak, av = ap.append_key.to(DEV), ap.append_value.to(DEV)
    seq = pk.paged_seq_lens(kvp, last, 16)
    bi, pos = pk.paged_batch_indices_positions(ap.append_indptr.to(DEV), seq, nnz)
    pool = cpu_pool.to(DEV)
    # decode, uniform and variable-length
    dc = wl.decode_case([900, 2500, 64, 4100], 16, 32, 8, 128, wl.HND, q_len_per_req=2,
                        window_left=1000, with_sinks=True, seed=31)
    vc = wl.decode_case([1300, 70, 3000], 32, 64, 8, 128, wl.HND, q_lens=[1, 4, 2],
                        with_sinks=True, seed=32)
    ws_d = torch.zeros(max(1, pk.paged_decode_workspace_size(4, 2, 32, 8, 128, dc.max_seq_len, 16, 1000)),
                       dtype=torch.uint8, device=DEV)
    ws_v = torch.zeros(max(1, pk.paged_decode_workspace_size(3, 4, 64, 8, 128, vc.max_seq_len, 32, -1)),
                       dtype=torch.uint8, device=DEV)
    d_q, d_kv = dc.query.to(DEV), dc.pool.storage[0].to(DEV)
    v_q, v_kv = vc.query.to(DEV), vc.pool.storage[0].to(DEV)
    d_args = [t.to(DEV) for t in (dc.block_tables, dc.seq_lens, dc.sinks)]
    v_args = [t.to(DEV) for t in (vc.block_tables, vc.seq_lens, vc.sinks, vc.cum_seq_lens_q)]
    d_out, d_lse = torch.empty_like(d_q), torch.empty(d_q.shape[:2], device=DEV)
    v_out, v_lse = torch.empty_like(v_q), torch.empty(v_q.shape[:2], device=DEV)
    # prefill
    pc = wl.prefill_case([130, 64, 300], [200, 64, 900], 32, 32, 8, 128, 128, wl.HND, wl.BF16,
                         seed=33)
    ws_p = torch.zeros(pk.paged_prefill_workspace_size(3, 32, pc.max_q, pc.max_kv), dtype=torch.uint8,
                       device=DEV)
    p_q, p_k, p_v = pc.q.to(DEV), pc.pool.k.to(DEV), pc.pool.v.to(DEV)
    p_args = [t.to(DEV) for t in (pc.seq_lens_q, pc.seq_lens_kv, pc.block_tables)]
    p_out = torch.empty((pc.q.shape[0], 32, 128), dtype=pc.q.dtype, device=DEV)
    p_lse = torch.empty((pc.q.shape[0], 32), dtype=torch.float32, device=DEV)

    def step():
        pk.paged_append(ak, av, bi, pos, pool, kvi, kvp, last, kv_layout="NHD")
        pk.paged_decode(d_q, d_kv, ws_d, d_args[0], d_args[1], dc.max_seq_len,
                        bmm1_scale=dc.bmm1_scale, window_left=1000, sinks=d_args[2],
                        q_len_per_req=2, out=d_out, lse=d_lse)
        pk.paged_decode(v_q, v_kv, ws_v, v_args[0], v_args[1], vc.max_seq_len,
                        bmm1_scale=vc.bmm1_scale, sinks=v_args[2], cum_seq_lens_q=v_args[3],
                        max_q_len=4, out=v_out, lse=v_lse)
        pk.paged_prefill(p_q, p_k, p_v, pc.scale, ws_p, pc.max_q, pc.max_kv,
                         p_args[0], p_args[1], p_args[2], causal=True, out=p_out, lse=p_lse,
                         kv_layout="HND")

    d_ref, v_ref, p_ref = oracle_decode(dc), oracle_decode(vc), oracle_prefill(pc)

    def check_against_oracle(tag):
        assert torch.equal(pool.cpu().view(torch.int16), pool_ref.view(torch.int16)), f"{tag}: append"
        assert_attn_close(d_out, d_ref[0], f"{tag}: decode out")
        assert_lse_close(d_lse, d_ref[1], f"{tag}: decode lse")
        assert_attn_close(v_out, v_ref[0], f"{tag}: varlen out")
        assert_lse_close(v_lse, v_ref[1], f"{tag}: varlen lse")
        assert_attn_close(p_out, p_ref[0], f"{tag}: prefill out")
        assert_lse_close(p_lse, p_ref[1], f"{tag}: prefill lse")

    outs = (pool, d_out, d_lse, v_out, v_lse, p_out, p_lse)
    pool.zero_()
    step()
    torch.cuda.synchronize()
    check_against_oracle("eager")
    eager = [t.clone() for t in outs]
    for t in outs[1:]:
        t.fill_(0)
    pool.zero_()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    for rep in range(2):
        for t in outs[1:]:
            t.fill_(0)
        pool.zero_()
        g.replay()
        torch.cuda.synchronize()
        names = ("append pool", "decode out", "decode lse", "varlen out", "varlen lse", "prefill out",
                 "prefill lse")
        bad = [n for n, e, t in zip(names, eager, outs) if not torch.equal(_bits(e), _bits(t))]
        assert not bad, f"replay differs from eager: {bad}"
        check_against_oracle(f"replay {rep}")


def test_graph_follows_device_scale_tensors():
    # a decode captured once with device-tensor scales (and the programmatic
    # dependent launch) picks up new scale values written between replays
    c = wl.decode_case([2100, 90, 4000], 16, 32, 8, 128, wl.HND, q_len_per_req=2,
                       with_sinks=True, seed=42)
    kv, bt, sl, sk = (t.to(DEV) for t in (c.pool.storage[0], c.block_tables, c.seq_lens, c.sinks))
    q = c.query.to(DEV)
    ws = torch.zeros(max(1, pk.paged_decode_workspace_size(3, 2, 32, 8, 128, c.max_seq_len, 16)),
                     dtype=torch.uint8, device=DEV)
    s1 = torch.tensor([0.09], device=DEV)
    s2 = torch.tensor([1.0], device=DEV)
    out, lse = torch.empty_like(q), torch.empty(q.shape[:2], device=DEV)

    def step():
        pk.paged_decode(q, kv, ws, bt, sl, c.max_seq_len, bmm1_scale=s1, bmm2_scale=s2,
                        sinks=sk, q_len_per_req=2, out=out, lse=lse, enable_pdl=True)

    def eager(a, b):
        o = pk.paged_decode(q, kv, ws, bt, sl, c.max_seq_len, bmm1_scale=a, bmm2_scale=b,
                            sinks=sk, q_len_per_req=2, lse=(l := torch.empty_like(lse)))
        torch.cuda.synchronize()
        return o, l

    step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    for a, b in ((0.09, 1.0), (0.03, 0.5), (0.12, 2.0)):
        s1.fill_(a)
        s2.fill_(b)
        out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        ro, rl = eager(a, b)
        assert torch.equal(_bits(out), _bits(ro)), (a, b)
        assert torch.equal(lse, rl), (a, b)
        # the replay's values themselves, against the oracle at those scales
        # (the device tensors hold fp32 values: the oracle gets the same ones)
        fa, fb = float(np.float32(a)), float(np.float32(b))
        oo, ol, _ = oracle_decode(dataclasses.replace(c, bmm1_scale=fa, bmm2_scale=fb))
        assert_attn_close(out, oo, f"replay out {a, b}")
        assert_lse_close(lse, ol, f"replay lse {a, b}")


def test_graph_follows_fp8_prefill_scales():
    # an E4M3 prefill captured once reads q/k/v scales written between replays
    c = wl.prefill_case([130, 64, 300], [200, 64, 900], 32, 32, 8, 128, 128, wl.HND, wl.BF16, seed=43,
                        q_dtype=wl.E4M3, kv_dtype=wl.E4M3)
    B = 3
    ws = torch.zeros(pk.paged_prefill_fp8_workspace_size(B, 32, 8, c.max_q, c.max_kv, c.q.shape[0], 128, 128,
                                                         c.q.dtype, c.pool.k.dtype),
                     dtype=torch.uint8, device=DEV)
    lq, lkv, bt = (t.to(DEV) for t in (c.seq_lens_q, c.seq_lens_kv, c.block_tables))
    gq, gk, gv = c.q.to(DEV), c.pool.k.to(DEV), c.pool.v.to(DEV)
    sc = [torch.ones(1, device=DEV) for _ in range(3)]
    out = torch.empty((c.q.shape[0], 32, 128), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((c.q.shape[0], 32), dtype=torch.float32, device=DEV)

    def call(o, l, scales):
        pk.paged_prefill(gq, gk, gv, c.scale, ws, c.max_q, c.max_kv, lq, lkv, bt, causal=True,
                         out=o, lse=l, kv_layout="HND", q_scale=scales[0], k_scale=scales[1], v_scale=scales[2])

    call(out, lse, sc)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            call(out, lse, sc)
    torch.cuda.current_stream().wait_stream(side)
    for vals in ((1.0, 1.0, 1.0), (0.5, 1.5, 0.25), (2.0, 0.75, 3.0)):
        for t, v in zip(sc, vals):
            t.fill_(v)
        out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        ro, rl = torch.empty_like(out), torch.empty_like(lse)
        call(ro, rl, [torch.tensor([v], device=DEV) for v in vals])
        torch.cuda.synchronize()
        assert torch.equal(_bits(out), _bits(ro)), vals
        assert torch.equal(lse, rl), vals
        oo, ol, _ = oracle_prefill(dataclasses.replace(c, q_scale=vals[0], k_scale=vals[1], v_scale=vals[2]))
        assert_attn_close(out, oo, f"replay out {vals}")
        assert_lse_close(lse, ol, f"replay lse {vals}")
