"""GPU-test helpers: move workload cases to the device, call the library
through its binding, compare with the oracle at the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_316_gb300 as pk
from paged_kv_cache_316_gb300 import workloads as wl

# attention output: |err| <= 2e-2 + 1e-2 |ref|; LSE: |err| <= 1e-3
ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3
DEV = torch.device("cuda:0")


def assert_attn_close(got, ref, what="out"):
    g = got.float().cpu().double().numpy() if torch.is_tensor(got) else np.asarray(got)
    r = np.asarray(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - r)
    bad = err > ATOL + RTOL * np.abs(r)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")


def assert_lse_close(got, ref, what="lse"):
    g = got.cpu().double().numpy() if torch.is_tensor(got) else np.asarray(got)
    r = np.asarray(ref)
    assert g.shape == r.shape
    ninf = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), ninf), f"{what}: -inf pattern differs"
    err = np.abs(g[~ninf] - r[~ninf])
    assert err.size == 0 or err.max() <= LSE_TOL, f"{what}: max err {err.max():.3e}"


def _scale(v, as_tensor):
    return torch.tensor([v], dtype=torch.float32, device=DEV) if as_tensor else v


def decode_on_gpu(c: wl.DecodeCase, with_lse=True, err_word=None, layout=None, ws=None,
                  tensor_scales=False, enable_pdl=None):
    pool = c.pool
    kv = pool.storage[0].to(DEV) if len(pool.storage) == 1 else tuple(t.to(DEV) for t in pool.storage)
    B = c.seq_lens.shape[0]
    ws_bytes = pk.paged_decode_workspace_size(B, c.q_len_per_req, c.num_qo_heads, c.num_kv_heads,
                                              c.head_dim, c.max_seq_len, pool.page_size,
                                              c.window_left)
    if ws is None:
        ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device=DEV)
    assert ws.numel() >= ws_bytes
    lse = torch.empty((c.query.shape[0], c.num_qo_heads), dtype=torch.float32,
                      device=DEV) if with_lse else None
    out = pk.paged_decode(c.query.to(DEV), kv, ws, c.block_tables.to(DEV), c.seq_lens.to(DEV),
                          c.max_seq_len, bmm1_scale=_scale(c.bmm1_scale, tensor_scales),
                          bmm2_scale=_scale(c.bmm2_scale, tensor_scales), window_left=c.window_left,
                          enable_pdl=enable_pdl,
                          sinks=None if c.sinks is None else c.sinks.to(DEV),
                          kv_layout=pool.layout if layout is None else layout,
                          q_len_per_req=c.q_len_per_req, lse=lse, err_word=err_word,
                          **({} if c.cum_seq_lens_q is None else
                             dict(cum_seq_lens_q=c.cum_seq_lens_q.to(DEV), max_q_len=c.q_len_per_req)))
    torch.cuda.synchronize()
    return out, lse


def prefill_on_gpu(c: wl.PrefillCase, err_word=None):
    B = c.seq_lens_q.shape[0]
    fp8 = c.q_dtype == wl.E4M3 or c.kv_dtype == wl.E4M3
    if fp8:
        nbytes = pk.paged_prefill_fp8_workspace_size(
            B, c.num_qo_heads, c.num_kv_heads, c.max_q, c.max_kv, c.q.shape[0], c.d_qk, c.d_vo,
            c.q.dtype, c.pool.k.dtype)
    else:
        nbytes = pk.paged_prefill_workspace_size(B, c.num_qo_heads, c.max_q, c.max_kv)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    kw = {}
    if fp8:
        def dev_scale(x):
            return torch.tensor([x], dtype=torch.float32, device=DEV)
        kw = dict(q_scale=dev_scale(c.q_scale), k_scale=dev_scale(c.k_scale),
                  v_scale=dev_scale(c.v_scale), o_data_type=wl.torch_dtype(c.dtype))
    out, lse = pk.paged_prefill(c.q.to(DEV), c.pool.k.to(DEV), c.pool.v.to(DEV), c.scale, ws,
                                c.max_q, c.max_kv, c.seq_lens_q.to(DEV), c.seq_lens_kv.to(DEV),
                                c.block_tables.to(DEV), causal=c.causal,
                                kv_layout=c.pool.layout, err_word=err_word, **kw)
    torch.cuda.synchronize()
    return out, lse


def err_word():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def compact_request(pool: wl.Pool, pt: wl.PageTable, b: int, kv_len: int | None = None):
    """CPU pool holding only request b's pages (logical order) and its block
    table row -- for checking sampled requests of a full-size case."""
    pages = pt.pages[b]
    idx = torch.tensor(pages, dtype=torch.long, device=pool.k.device)

    def pick(t):  # (through a byte view for 8-bit floats)
        if t.element_size() == 1:
            return t.view(torch.uint8).index_select(0, idx).cpu().contiguous().view(t.dtype)
        return t.index_select(0, idx).cpu().contiguous()
    k, v = pick(pool.k), pick(pool.v)
    sub = wl.Pool((k, v), k, v, pool.layout, len(pages), pool.num_heads, pool.page_size,
                  pool.d_k, pool.d_v, k[0].numel(), v[0].numel())
    L = pt.lengths[b] if kv_len is None else kv_len
    spt = wl.PageTable([L], pool.page_size, len(pages), [list(range(len(pages)))])
    return sub, spt
