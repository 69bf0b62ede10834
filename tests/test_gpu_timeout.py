"""Failure detection of the bounded pipeline waits, without faulting the GPU:
with a wait limit that no wait can meet (pkv_set_wait_limit_ns), a wait of
the prefill's warp-specialised pipeline (or of the append's bulk-copy ring)
runs out, the call's error word gets PKV_DEV_ERR_TIMEOUT, the kernel waits
for the copies and MMAs it had issued, frees its tensor memory and returns;
the call completes, and the next call on the same stream, with the default
limit, is right (checked against the fp64 oracle)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_316_gb300 as pk
from paged_kv_cache_316_gb300 import workloads as wl
from _gpu import DEV, assert_attn_close, assert_lse_close, err_word, prefill_on_gpu
from _util import oracle_append, oracle_prefill

pytestmark = pytest.mark.gpu

TIMEOUT = 16  # PKV_DEV_ERR_TIMEOUT
TINY_NS = 1   # no wait for copied data or another warp completes this fast


@pytest.fixture(autouse=True)
def _default_limit_afterwards():
    yield
    pk.set_wait_limit_ns(0)


@pytest.mark.parametrize("d_qk,e4m3", [(128, False), (192, False), (128, True)])
def test_prefill_wait_runs_out_then_next_call_is_right(d_qk, e4m3):
    # (E4M3 query and caches at d_qk 128: the kernel with the V widening warp)
    c = wl.prefill_case([300, 130, 700], [500, 130, 1400], 32, 32, 8, d_qk, 128, wl.HND, wl.BF16,
                        seed=81, **(dict(q_dtype=wl.E4M3, kv_dtype=wl.E4M3, k_scale=1.5) if e4m3 else {}))
    prev = pk.set_wait_limit_ns(TINY_NS)
    assert prev == 10 ** 9
    err = err_word()
    prefill_on_gpu(c, err_word=err)  # synchronises: the call ended
    assert int(err.item()) & TIMEOUT
    pk.set_wait_limit_ns(0)
    err = err_word()
    out, lse = prefill_on_gpu(c, err_word=err)
    assert int(err.item()) == 0
    ro, rl, _ = oracle_prefill(c)
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)


def test_append_wait_runs_out_then_next_call_is_right():
    c = wl.append_sweep(64, seed=82, layout=wl.NHD, fill="empty")
    c.pool.storage[0].zero_()
    nnz = c.append_key.shape[0]
    sl = oracle.seq_lens(c.kv_indptr.numpy(), c.kv_last_page_len.numpy(), 16)
    bi, pos = oracle.batch_indices_positions(c.append_indptr.numpy(), sl, nnz)
    ref = c.pool.storage[0].clone()
    kvi, kvp, last = (x.to(DEV) for x in (c.kv_indices, c.kv_indptr, c.kv_last_page_len))
    ak, av = c.append_key.to(DEV), c.append_value.to(DEV)
    gbi, gpos = torch.from_numpy(np.asarray(bi)).to(DEV), torch.from_numpy(np.asarray(pos)).to(DEV)
    pool = ref.to(DEV)
    assert oracle_append(c, bi, pos) == 0  # into c's CPU pool
    pk.set_wait_limit_ns(TINY_NS)
    err = err_word()
    pk.paged_append(ak, av, gbi, gpos, pool, kvi, kvp, last, kv_layout="NHD", err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & TIMEOUT
    pk.set_wait_limit_ns(0)
    pool.zero_()
    err = err_word()
    pk.paged_append(ak, av, gbi, gpos, pool, kvi, kvp, last, kv_layout="NHD", err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(pool.cpu().view(torch.int16), c.pool.storage[0].view(torch.int16))
