"""GPU parity for the index helpers and the append scatter: bit-exact against
the oracle (whole pool compared), in NHD/HND and 5-D/tuple forms, plus the
full-size sweep point checked through properties that hold at any size."""
from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_316_gb300 as pk
from paged_kv_cache_316_gb300 import workloads as wl
from _gpu import DEV, err_word
from _util import oracle_append, u16

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "append_example.json")


def _bits(t):
    return t.view(torch.int16)


def _gpu_helpers(c):
    S = c.pool.page_size
    seq = pk.paged_seq_lens(c.kv_indptr.to(DEV), c.kv_last_page_len.to(DEV), S)
    bi, pos = pk.paged_batch_indices_positions(c.append_indptr.to(DEV), seq,
                                               c.append_key.shape[0])
    torch.cuda.synchronize()
    return seq, bi, pos


def _run_append(c, bi, pos, err=None):
    storage = [t.to(DEV) for t in c.pool.storage]
    cache = storage[0] if len(storage) == 1 else tuple(storage)
    pk.paged_append(c.append_key.to(DEV), c.append_value.to(DEV), bi, pos, cache,
                    c.kv_indices.to(DEV), c.kv_indptr.to(DEV), c.kv_last_page_len.to(DEV),
                    kv_layout=c.pool.layout, err_word=err)
    torch.cuda.synchronize()
    return [t.cpu() for t in storage]


def test_example_helpers_match_printed_output():
    ex = json.load(open(GOLDEN))
    c = wl.append_example()
    seq, bi, pos = _gpu_helpers(c)
    assert seq.cpu().tolist() == ex["seq_lens"]
    assert bi.cpu().tolist() == ex["batch_indices"]
    assert pos.cpu().tolist() == ex["positions"]


@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
@pytest.mark.parametrize("form", ["5d", "tuple"])
def test_example_append_bit_exact(layout, form):
    c = wl.append_example(layout=layout, form=form)
    _, bi, pos = _gpu_helpers(c)
    got = _run_append(c, bi, pos)
    sl = oracle.seq_lens(c.kv_indptr.numpy(), c.kv_last_page_len.numpy(), 16)
    obi, opos = oracle.batch_indices_positions(c.append_indptr.numpy(), sl, 100)
    assert oracle_append(c, obi, opos) == 0  # in place on the CPU pool
    for g, r in zip(got, c.pool.storage):
        assert torch.equal(_bits(g), _bits(r)), "pool differs from the oracle"


@pytest.mark.parametrize("batch,one_token,layout,seed",
                         [(4, False, wl.NHD, 1), (16, False, wl.HND, 2), (64, True, wl.NHD, 3),
                          (256, False, wl.HND, 4), (37, False, wl.NHD, 5)])
def test_sweep_append_bit_exact(batch, one_token, layout, seed):
    c = wl.append_sweep(batch, seed=seed, layout=layout, one_token=one_token)
    seq, bi, pos = _gpu_helpers(c)
    sl = oracle.seq_lens(c.kv_indptr.numpy(), c.kv_last_page_len.numpy(), 16)
    obi, opos = oracle.batch_indices_positions(c.append_indptr.numpy(), sl,
                                               c.append_key.shape[0])
    assert np.array_equal(seq.cpu().numpy(), sl)
    assert np.array_equal(bi.cpu().numpy(), obi) and np.array_equal(pos.cpu().numpy(), opos)
    got = _run_append(c, bi, pos)
    assert oracle_append(c, obi, opos) == 0
    for g, r in zip(got, c.pool.storage):
        assert torch.equal(_bits(g), _bits(r))


def test_helpers_with_empty_requests_and_tail():
    # requests 1 and 3 append nothing; entries past the last request get -1
    indptr = torch.tensor([0, 3, 3, 7, 7], dtype=torch.int32)
    seq = torch.tensor([5, 2, 9, 4], dtype=torch.int32)
    bi, pos = pk.paged_batch_indices_positions(indptr.to(DEV), seq.to(DEV), 9)
    obi, opos = oracle.batch_indices_positions(indptr.numpy(), seq.numpy(), 9)
    assert bi.cpu().numpy().tolist() == obi.tolist()
    assert pos.cpu().numpy().tolist() == opos.tolist()


@pytest.mark.parametrize("field,bit", [("batch", 4), ("pos", 2), ("page", 1)])
def test_append_errors_skip_and_flag(field, bit):
    c = wl.append_sweep(3, seed=5)
    _, bi, pos = _gpu_helpers(c)
    b2, p2 = bi.clone(), pos.clone()
    if field == "batch":
        b2[0] = 7
    elif field == "pos":
        p2[0] = c.pt.lengths[int(bi[0])]
    else:
        c.kv_indices[int(c.kv_indptr[int(bi[0])]) + int(pos[0]) // 16] = c.pool.num_pages + 3
    err = err_word()
    got = _run_append(c, b2, p2, err)
    assert int(err.item()) == bit
    # the bad entry is skipped; every other entry lands where the oracle puts it
    assert oracle_append(c, b2.cpu().numpy(), p2.cpu().numpy()) == bit
    assert torch.equal(_bits(got[0]), _bits(c.pool.storage[0]))


def test_full_size_sweep_properties():
    """4096 requests, prefix U[0,256], append U[1,128], 32 heads, d 128: every
    appended token reads back bit-exactly through the page table and no other
    slot of the pool changes."""
    c = wl.append_sweep(4096, seed=1, layout=wl.NHD, device=DEV, fill="randn")
    S, H, D = 16, 32, 128
    kvi, kvp, last = (x.to(DEV) for x in (c.kv_indices, c.kv_indptr, c.kv_last_page_len))
    seq = pk.paged_seq_lens(kvp, last, S)
    nnz = c.append_key.shape[0]
    bi, pos = pk.paged_batch_indices_positions(c.append_indptr.to(DEV), seq, nnz)
    pool = c.pool.storage[0]
    before = pool.clone()
    err = err_word()
    pk.paged_append(c.append_key, c.append_value, bi, pos, pool, kvi, kvp, last,
                    kv_layout="NHD", err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # helper outputs against the oracle (index work: exact)
    sl = oracle.seq_lens(c.kv_indptr.numpy(), c.kv_last_page_len.numpy(), S)
    obi, opos = oracle.batch_indices_positions(c.append_indptr.numpy(), sl, nnz)
    assert np.array_equal(bi.cpu().numpy(), obi) and np.array_equal(pos.cpu().numpy(), opos)
    # gather every appended token back through the page table (plain indexing)
    b64, p64 = torch.from_numpy(obi).long().to(DEV), torch.from_numpy(opos).long().to(DEV)
    page = kvi.long()[kvp.long()[b64] + p64 // S]
    slot = p64 % S
    assert torch.equal(_bits(pool[page, 0, slot]), _bits(c.append_key))
    assert torch.equal(_bits(pool[page, 1, slot]), _bits(c.append_value))
    # nothing else moved
    changed = (_bits(pool) != _bits(before)).any(dim=-1).any(dim=-1)  # [P, 2, S]
    expect = torch.zeros_like(changed)
    expect[page, :, slot] = True
    assert torch.equal(changed, expect)


@pytest.mark.parametrize("heads,page,layout,dtype,seed",
                         [(64, 32, wl.HND, wl.BF16, 11),   # 16 KB rows: two 8 KB pieces each
                          (48, 16, wl.NHD, wl.F16, 12),    # 12 KB rows: pieces of 32 and 16 heads
                          (4, 8, wl.HND, wl.BF16, 13),     # 1 KB rows, 8-slot pages
                          (48, 64, wl.HND, wl.E4M3, 14)],  # 6 KB E4M3 rows, 64-slot pages
                         ids=["h64", "h48", "h4", "h48-e4m3"])
def test_append_head_counts_and_pages(heads, page, layout, dtype, seed):
    # rows cut into several whole-head pieces, an uneven last piece, small
    # rows and other page sizes: the pool after the append bit-exact against
    # the oracle (untouched slots and pages included)
    g = np.random.default_rng(seed)
    n = [int(x) for x in g.integers(1, 90, size=23)]
    prefix = [int(x) for x in g.integers(0, 200, size=23)]
    c = wl.append_case(n, prefix, page, heads, 128, layout, dtype, seed=seed, slack=0.2)
    seq, bi, pos = _gpu_helpers(c)
    got = _run_append(c, bi, pos)
    sl = oracle.seq_lens(c.kv_indptr.numpy(), c.kv_last_page_len.numpy(), page)
    obi, opos = oracle.batch_indices_positions(c.append_indptr.numpy(), sl, c.append_key.shape[0])
    assert np.array_equal(bi.cpu().numpy(), obi) and np.array_equal(pos.cpu().numpy(), opos)
    assert oracle_append(c, obi, opos) == 0
    for gt, r in zip(got, c.pool.storage):
        assert torch.equal(gt.view(torch.uint8), r.view(torch.uint8))


@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
def test_fp8_append_bit_exact(layout):
    # 8-bit (E4M3) cache elements are copied byte for byte
    c = wl.append_sweep(64, seed=8, layout=layout)
    c8 = wl.append_case([int(x) for x in (c.append_indptr[1:] - c.append_indptr[:-1])],
                        [0] * 64, 16, 32, 128, layout, wl.E4M3, seed=8, slack=0.1)
    seq, bi, pos = _gpu_helpers(c8)
    got = _run_append(c8, bi, pos)
    sl = oracle.seq_lens(c8.kv_indptr.numpy(), c8.kv_last_page_len.numpy(), 16)
    obi, opos = oracle.batch_indices_positions(c8.append_indptr.numpy(), sl, c8.append_key.shape[0])
    assert oracle_append(c8, obi, opos) == 0
    for g, r in zip(got, c8.pool.storage):
        assert torch.equal(g.view(torch.uint8), r.view(torch.uint8))
