"""The three operations chained on one pool, as a serving step uses them:
the append page's worked example (4 requests appending 45/8/25/22 tokens
into 8 reserved pages of a 1000-page pool, page_size 16, 32 kv heads,
head_dim 128) goes through paged_seq_lens -> paged_batch_indices_positions
-> paged_append; then paged_decode (1 and 4 query tokens per request) and
paged_prefill (the appended tokens as causal queries) read that same pool
through a block table built from the same kv_indptr / kv_indices.  The fp64
oracle runs the same chain on a CPU copy: the pool after the append must be
bit-identical, decode and prefill within |err| <= 2e-2 + 1e-2 |ref| and LSE
within 1e-3.  The append page notes that the page table already covers the
appended tokens, which is what lets the attention calls read them at once."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_316_gb300 as pk
from paged_kv_cache_316_gb300 import workloads as wl
from _gpu import DEV, assert_attn_close, assert_lse_close, err_word
from _util import u16

pytestmark = pytest.mark.gpu


def _block_table(kv_indptr, kv_indices, width):
    """Row b holds request b's pages kv_indices[kv_indptr[b] .. kv_indptr[b+1]),
    the rest poison (never read)."""
    B = kv_indptr.shape[0] - 1
    bt = np.full((B, width), wl.POISON, np.int32)
    for b in range(B):
        pg = kv_indices[kv_indptr[b]:kv_indptr[b + 1]]
        bt[b, :len(pg)] = pg
    return bt


@pytest.mark.parametrize("layout,form", [(wl.HND, "5d"), (wl.NHD, "tuple")], ids=["HND-5d", "NHD-tuple"])
def test_append_then_decode_and_prefill_on_the_same_pool(layout, form):
    ex = wl.APPEND_EXAMPLE
    c = wl.append_case(ex["lengths"], [0, 0, 0, 0], ex["page_size"], ex["num_kv_heads"], ex["head_dim"],
                       layout, wl.BF16, seed=71, pool_pages=ex["max_num_pages"], page_ids=ex["pages"],
                       form=form)
    H, D, S, B, nnz = 32, 128, 16, 4, 100
    ind, ptr, last = c.kv_indices.numpy(), c.kv_indptr.numpy(), c.kv_last_page_len.numpy()
    # ---- the oracle's chain, on a CPU copy of the pool
    ref_storage = tuple(t.clone() for t in c.pool.storage)
    if form == "5d":
        rk, rv = ref_storage[0][:, 0], ref_storage[0][:, 1]
    else:
        rk, rv = ref_storage
    sl_ref = oracle.seq_lens(ptr, last, S)
    bi_ref, pos_ref = oracle.batch_indices_positions(c.append_indptr.numpy(), sl_ref, nnz)
    assert oracle.append(u16(c.append_key), u16(c.append_value), bi_ref, pos_ref, u16(rk), u16(rv),
                         c.pool.k_page_stride, ex["max_num_pages"], ind, ptr, last, H, D, S, layout) == 0
    assert sl_ref.tolist() == ex["lengths"]
    # ---- the library's chain
    storage = tuple(t.to(DEV) for t in c.pool.storage)
    kv = storage[0] if form == "5d" else storage
    gk, gv = (storage[0][:, 0], storage[0][:, 1]) if form == "5d" else storage
    dptr, dind, dlast = (x.to(DEV) for x in (c.kv_indptr, c.kv_indices, c.kv_last_page_len))
    err = err_word()
    seq = pk.paged_seq_lens(dptr, dlast, S)
    bi, pos = pk.paged_batch_indices_positions(c.append_indptr.to(DEV), seq, nnz)
    pk.paged_append(c.append_key.to(DEV), c.append_value.to(DEV), bi, pos, kv, dind, dptr, dlast,
                    kv_layout="HND" if layout == wl.HND else "NHD", err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert seq.cpu().tolist() == sl_ref.tolist()
    assert bi.cpu().tolist() == bi_ref.tolist() and pos.cpu().tolist() == pos_ref.tolist()
    for g, r in zip(storage, ref_storage):
        assert torch.equal(g.cpu().view(torch.int16), r.view(torch.int16)), "pool after append"

    bt = _block_table(ptr, ind, 4)
    dbt = torch.from_numpy(bt).to(DEV)
    lens = np.asarray(sl_ref, np.uint32)
    kv_layout = "HND" if layout == wl.HND else "NHD"
    g = torch.Generator().manual_seed(72)
    # ---- decode: 1 and 4 query tokens per request (the last tokens of each
    # sequence), 64 qo heads over the 32 kv heads, with and without sinks
    for Q, sinks in ((1, None), (4, torch.randn(64, generator=g))):
        q = torch.randn((B * Q, 64, D), generator=g).to(torch.bfloat16)
        scale = 1.0 / np.sqrt(D)
        ws = torch.zeros(max(1, pk.paged_decode_workspace_size(B, Q, 64, H, D, 45, S, -1)),
                         dtype=torch.uint8, device=DEV)
        lse = torch.empty((B * Q, 64), dtype=torch.float32, device=DEV)
        out = pk.paged_decode(q.to(DEV), kv, ws, dbt, seq, 45, bmm1_scale=scale,
                              sinks=None if sinks is None else sinks.to(DEV), kv_layout=kv_layout,
                              q_len_per_req=Q, lse=lse)
        torch.cuda.synchronize()
        ro, rl, oerr = oracle.decode(u16(q), u16(rk), u16(rv), c.pool.k_page_stride, ex["max_num_pages"],
                                     bt, lens, 45, scale, 1.0, -1,
                                     None if sinks is None else sinks.numpy(), Q, 64, H, D, S, layout,
                                     wl.BF16)
        assert oerr == 0
        assert_attn_close(out, ro, f"decode Q={Q}")
        assert_lse_close(lse, rl, f"decode Q={Q} lse")
    # ---- prefill: the appended tokens as causal queries over the same keys
    lq = torch.tensor(ex["lengths"], dtype=torch.int32)
    qp = torch.randn((nnz, 64, D), generator=g).to(torch.bfloat16)
    scale = 1.0 / np.sqrt(D)
    ws = torch.zeros(pk.paged_prefill_workspace_size(B, 64, 45, 45), dtype=torch.uint8, device=DEV)
    out, lse = pk.paged_prefill(qp.to(DEV), gk, gv, scale, ws, 45, 45, lq.to(DEV), seq, dbt,
                                causal=True, kv_layout=kv_layout)
    torch.cuda.synchronize()
    ro, rl, oerr = oracle.prefill(u16(qp), u16(rk), u16(rv), c.pool.k_page_stride, c.pool.v_page_stride,
                                  ex["max_num_pages"], scale, lq.numpy(), sl_ref, bt, True, 64, H, D, D,
                                  S, layout, wl.BF16)
    assert oerr == 0
    assert_attn_close(out, ro, "prefill")
    assert_lse_close(lse, rl, "prefill lse")
