"""GPU parity for causal ragged paged prefill against the fp64 oracle:
outputs within |err| <= 2e-2 + 1e-2 |ref|, LSE within 1e-3."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_316_gb300 import workloads as wl
from _gpu import (DEV, assert_attn_close, assert_lse_close, compact_request, err_word,
                  prefill_on_gpu)
from _util import oracle_prefill

pytestmark = pytest.mark.gpu


def _check(c, **kw):
    out, lse = prefill_on_gpu(c, **kw)
    ro, rl, _ = oracle_prefill(c)
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)
    return out, lse


CASES = [
    # q lens, kv lens, page, Hqo, Hkv, d_qk, causal, dtype, layout, seed
    ([130, 7, 64], [200, 7, 300], 32, 32, 8, 128, True, wl.BF16, wl.HND, 1),
    ([1, 255, 129], [1, 255, 700], 32, 32, 8, 192, True, wl.BF16, wl.HND, 2),
    ([300, 50], [300, 333], 16, 8, 8, 128, False, wl.F16, wl.NHD, 3),
    ([64, 200], [500, 200], 64, 16, 2, 192, False, wl.BF16, wl.NHD, 4),
    ([513], [1100], 8, 4, 1, 128, True, wl.F16, wl.HND, 5),
    ([77, 300], [500, 300], 16, 16, 4, 192, True, wl.BF16, wl.HND, 6),    # 96-key tiles, 16-slot pages
    ([130, 45], [900, 45], 256, 8, 2, 192, True, wl.F16, wl.NHD, 7),     # tiles inside 256-slot pages
    ([200], [333], 8, 6, 2, 192, False, wl.BF16, wl.HND, 8),             # odd group: block B absent
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_small_shapes(case):
    lq, lkv, S, hq, hk, dqk, causal, dt, lay, seed = case
    c = wl.prefill_case(lq, lkv, S, hq, hk, dqk, 128, lay, dt, causal=causal, seed=seed,
                        slack=0.2)
    _check(c)


def test_page_permutation_bit_identical():
    lq, lkv = [200, 90], [400, 90]
    a = wl.prefill_case(lq, lkv, 32, 8, 2, 128, 128, seed=3, slack=0.5)
    b = wl.prefill_case(lq, lkv, 32, 8, 2, 128, 128, seed=4, slack=0.5)
    b.q.copy_(a.q)
    for r in range(2):
        k, v = wl.read_tokens(a.pool, a.pt, r)
        wl.write_tokens(b.pool, b.pt, r, k, v)
    assert a.pt.pages != b.pt.pages
    oa, la = prefill_on_gpu(a)
    ob, lb = prefill_on_gpu(b)
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(la, lb)


def test_never_reads_padding_or_unused_slots():
    lq, lkv = [40, 100], [70, 100]
    c = wl.prefill_case(lq, lkv, 32, 8, 2, 128, 128, seed=5, fill="nan", bt_width=9)
    for b, n in enumerate(lkv):
        k = wl.randn((n, 2, 128), torch.bfloat16, wl.generator(10 + b))
        v = wl.randn((n, 2, 128), torch.bfloat16, wl.generator(20 + b))
        wl.write_tokens(c.pool, c.pt, b, k, v)
    assert int(c.block_tables[0, 5]) == wl.POISON
    err = err_word()
    _check(c, err_word=err)
    assert int(err.item()) == 0


def test_short_kv_flagged():
    c = wl.prefill_case([100, 20], [60, 20], 16, 8, 8, 128, 128, seed=6)
    err = err_word()
    out, lse = prefill_on_gpu(c, err_word=err)
    ro, rl, oerr = oracle_prefill(c)
    assert int(err.item()) & oracle.E_QLEN and oerr & oracle.E_QLEN
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("d_qk", [128, 192])
def test_ragged_config_full_size_sampled(d_qk):
    """Full-size config on the GPU; a few (request, head) pairs checked
    against the oracle on compact copies of those requests' pages."""
    c = wl.ragged_prefill(d_qk=d_qk, device=DEV)
    out, lse = prefill_on_gpu(c)
    lq = c.seq_lens_q.tolist()
    cu = np.concatenate([[0], np.cumsum(lq)])
    for b in sorted({0, int(np.argmax(lq)), len(lq) - 1}):
        pool, pt = compact_request(c.pool, c.pt, b)
        sub = dataclasses.replace(
            c, q=c.q[cu[b]:cu[b + 1]].cpu(), pool=pool, pt=pt, block_tables=pt.block_tables(),
            seq_lens_q=c.seq_lens_q[b:b + 1], seq_lens_kv=c.seq_lens_kv[b:b + 1])
        ro, rl, _ = oracle_prefill(sub)
        assert_attn_close(out[cu[b]:cu[b + 1]], ro, f"request {b}")
        assert_lse_close(lse[cu[b]:cu[b + 1]], rl, f"request {b} lse")
