"""Test helpers: run the oracle on workload cases, library reference formulas."""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_316_gb300 import workloads as wl


def u16(t: torch.Tensor) -> np.ndarray:
    """uint16 numpy view of a 16-bit torch tensor on the CPU (shares memory);
    uint8 for an 8-bit (e4m3) tensor."""
    assert t.device.type == "cpu"
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    assert t.element_size() == 2
    return t.view(torch.int16).numpy().view(np.uint16)


def oracle_decode(c: wl.DecodeCase, threads=None):
    p = c.pool
    return oracle.decode(
        u16(c.query), u16(p.k), u16(p.v), p.k_page_stride, p.num_pages,
        c.block_tables.numpy(), c.seq_lens.numpy().astype(np.uint32),
        c.max_seq_len, c.bmm1_scale, c.bmm2_scale, c.window_left,
        None if c.sinks is None else c.sinks.numpy(), c.q_len_per_req,
        c.num_qo_heads, c.num_kv_heads, c.head_dim, p.page_size, p.layout,
        c.dtype, threads=threads,
        cum_seq_lens_q=None if c.cum_seq_lens_q is None else c.cum_seq_lens_q.numpy(),
        kv_dtype=c.kv_dtype)


def oracle_prefill(c: wl.PrefillCase, threads=None):
    p = c.pool
    return oracle.prefill(
        u16(c.q), u16(p.k), u16(p.v), p.k_page_stride, p.v_page_stride,
        p.num_pages, c.scale, c.seq_lens_q.numpy(), c.seq_lens_kv.numpy(),
        c.block_tables.numpy(), c.causal, c.num_qo_heads, c.num_kv_heads,
        c.d_qk, c.d_vo, p.page_size, p.layout, c.dtype, threads=threads,
        q_dtype=c.q_dtype, kv_dtype=c.kv_dtype, q_scale=c.q_scale, k_scale=c.k_scale,
        v_scale=c.v_scale)


def oracle_append(c: wl.AppendCase, batch_indices, positions, layout=None):
    p = c.pool
    return oracle.append(
        u16(c.append_key), u16(c.append_value), np.asarray(batch_indices),
        np.asarray(positions), u16(p.k), u16(p.v), p.k_page_stride, p.num_pages,
        c.kv_indices.numpy(), c.kv_indptr.numpy(), c.kv_last_page_len.numpy(),
        c.num_kv_heads, c.head_dim, p.page_size, p.layout if layout is None else layout)


def sdpa64(q, k, v, scale, causal=False):
    """Library attention in float64: q [n_q, H, d], k [n_k, H, d], v [n_k, H, dv]
    (heads already matched) -> [n_q, H, dv]."""
    qq = q.double().permute(1, 0, 2).unsqueeze(0)
    kk = k.double().permute(1, 0, 2).unsqueeze(0)
    vv = v.double().permute(1, 0, 2).unsqueeze(0)
    o = F.scaled_dot_product_attention(qq, kk, vv, scale=scale, is_causal=causal)
    return o.squeeze(0).permute(1, 0, 2)


def logsumexp64(q, k, scale):
    """torch.logsumexp of the scaled logits: q [n_q, H, d], k [n_k, H, d] -> [n_q, H]."""
    s = torch.einsum("qhd,khd->hqk", q.double(), k.double()) * scale
    return torch.logsumexp(s, dim=-1).permute(1, 0)


def expand_heads(x, group):
    """Repeat each kv head ``group`` times along dim 1 (consecutive grouping)."""
    return x.repeat_interleave(group, dim=1)
