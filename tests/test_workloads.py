"""The seeded synthetic inputs are reproducible: the same seed gives the same
tensors, lengths and page assignment; another seed gives other ones of the
same shape; pages are reserved without overlap between requests."""
from __future__ import annotations

import torch

from paged_kv_cache_316_gb300 import workloads as wl


def _same(a, b):
    return torch.equal(a.view(torch.uint8) if a.element_size() == 1 else a, b.view(torch.uint8)
                       if b.element_size() == 1 else b)


def test_decode_case_is_reproducible():
    kw = dict(q_len_per_req=2, window_left=100, with_sinks=True)
    a = wl.decode_case([300, 45, 900], 16, 32, 8, 128, wl.HND, seed=5, **kw)
    b = wl.decode_case([300, 45, 900], 16, 32, 8, 128, wl.HND, seed=5, **kw)
    c = wl.decode_case([300, 45, 900], 16, 32, 8, 128, wl.HND, seed=6, **kw)
    assert _same(a.query, b.query) and _same(a.pool.storage[0], b.pool.storage[0])
    assert a.pt.pages == b.pt.pages and torch.equal(a.sinks, b.sinks)
    assert not _same(a.query, c.query) and a.query.shape == c.query.shape


def test_prefill_and_fp8_cases_are_reproducible():
    a = wl.prefill_case([30, 7], [60, 7], 16, 8, 2, 128, 128, seed=7, q_dtype=wl.E4M3, kv_dtype=wl.E4M3)
    b = wl.prefill_case([30, 7], [60, 7], 16, 8, 2, 128, 128, seed=7, q_dtype=wl.E4M3, kv_dtype=wl.E4M3)
    assert _same(a.q, b.q) and _same(a.pool.k, b.pool.k) and _same(a.pool.v, b.pool.v)
    assert a.q.dtype == torch.float8_e4m3fn and a.pool.k.dtype == torch.float8_e4m3fn


def test_pages_are_disjoint_between_requests():
    pt = wl.reserve_pages([45, 8, 25, 22, 300], 16, wl.generator(3), slack=0.2)
    flat = [p for pages in pt.pages for p in pages]
    assert len(flat) == len(set(flat))
    assert all(len(pages) == (L + 15) // 16 for pages, L in zip(pt.pages, pt.lengths))
    assert max(flat) < pt.num_pages
