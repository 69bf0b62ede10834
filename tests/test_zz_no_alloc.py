"""paged_decode_noalloc -- decode for callers that cannot allocate device
memory at the call (a plugin inside another runtime's execution step, a
latency-critical loop, a process that reserved all device memory up front).
It must give what paged_decode gives with a caller workspace, call after
call, although every call reuses the same library-owned scratch array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import paged_kv_cache_316_gb300 as pk
from paged_kv_cache_316_gb300 import build, workloads as wl
from _gpu import DEV, assert_attn_close, assert_lse_close, decode_on_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    pk.load_library()


def _noalloc(c):
    kv = c.pool.storage[0].to(DEV)
    B = c.seq_lens.shape[0]
    lse = torch.empty((B * c.q_len_per_req, c.num_qo_heads), dtype=torch.float32, device=DEV)
    out = pk.paged_decode_noalloc(
        c.query.to(DEV), kv, c.block_tables.to(DEV), c.seq_lens.to(DEV), c.max_seq_len,
        bmm1_scale=c.bmm1_scale, bmm2_scale=c.bmm2_scale, window_left=c.window_left,
        sinks=None if c.sinks is None else c.sinks.to(DEV), kv_layout=c.pool.layout,
        q_len_per_req=c.q_len_per_req, lse=lse)
    torch.cuda.synchronize()
    return out, lse


def test_noalloc_matches_workspace_decode_on_consecutive_calls():
    # two different multi-split cases back to back: the second call must not
    # see anything the first one left in the shared scratch array
    a = wl.decode_case([3000, 700, 5000, 129], 16, 32, 8, 128, wl.HND, seed=41)
    b = wl.decode_case([2100, 4400, 35, 1800, 900], 64, 64, 8, 128, wl.NHD, q_len_per_req=4,
                       window_left=1500, with_sinks=True, seed=42)
    assert pk.paged_decode_workspace_size(4, 1, 32, 8, 128, a.max_seq_len, 16, -1) > 0
    for case in (a, b, a):
        ref_out, ref_lse = decode_on_gpu(case)
        out, lse = _noalloc(case)
        assert_attn_close(out, ref_out.float().cpu().double().numpy())
        assert_lse_close(lse, ref_lse.cpu().double().numpy())


def test_noalloc_rejects_sizes_beyond_its_array():
    # the long-context decode shape without its window (8 splits of 4096 keys
    # per request) needs more partial storage than the fixed array holds:
    # refused on the host, before any launch (pointers unused)
    need = pk.paged_decode_workspace_size(256, 4, 64, 8, 128, 32768, 64, -1)
    limit = 32 << 20
    assert need > limit
    lib = pk.load_library()
    fake = ctypes.c_void_p(0x1000)
    rc = lib.paged_decode_noalloc(fake, fake, fake, 2 * 8 * 64 * 128, 100000, fake, 512, fake,
                                  256, 32768, 0.088, 1.0, -1, None, 4, 64, 8, 128, 64, 1, 1,
                                  fake, None, None, None)
    assert rc == 4  # PKV_ERR_WORKSPACE
