"""paged_decode_noalloc -- decode for callers that cannot allocate device
memory at the call (a plugin inside another runtime's execution step, a
latency-critical loop, a process that reserved all device memory up front).
It runs the same kernels as paged_decode with a caller workspace, so it must
give bit for bit what paged_decode gives, call after call, although every
call reuses the same library-owned scratch array; and both must match the
fp64 oracle.

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
from _util import oracle_decode

pytestmark = pytest.mark.gpu

LIMIT = 32 << 20  # PKV_NOALLOC_SCRATCH_BYTES
PKV_ERR_WORKSPACE = 4


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    pk.load_library()


def _noalloc(c, dev_case=None):
    d = dev_case or {}
    kv = d.get("kv", c.pool.storage[0].to(DEV))
    rows = c.query.shape[0]
    lse = torch.empty((rows, c.num_qo_heads), dtype=torch.float32, device=DEV)
    out = pk.paged_decode_noalloc(
        d.get("q", c.query.to(DEV)), kv, d.get("bt", c.block_tables.to(DEV)),
        d.get("sl", c.seq_lens.to(DEV)), c.max_seq_len,
        bmm1_scale=c.bmm1_scale, bmm2_scale=c.bmm2_scale, window_left=c.window_left,
        sinks=None if c.sinks is None else c.sinks.to(DEV), kv_layout=c.pool.layout,
        q_len_per_req=c.q_len_per_req, lse=lse)
    torch.cuda.synchronize()
    return out, lse


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t


def test_noalloc_bit_identical_to_workspace_decode_and_matches_oracle():
    # different multi-split cases back to back, and the same case twice in a
    # row: no call may see anything an earlier one left in the shared array
    a = wl.decode_case([3000, 700, 5000, 129], 16, 32, 8, 128, wl.HND, seed=41)
    b = wl.decode_case([2100, 4400, 35, 1800, 900], 64, 64, 8, 128, wl.NHD, q_len_per_req=4,
                       window_left=1500, with_sinks=True, seed=42)
    assert pk.paged_decode_workspace_size(4, 1, 32, 8, 128, a.max_seq_len, 16, -1) > 0
    assert pk.paged_decode_workspace_size(5, 4, 64, 8, 128, b.max_seq_len, 64, 1500) > 0
    refs = {}
    for c in (a, b):
        ro, rl, _ = oracle_decode(c)
        refs[id(c)] = (ro, rl)
    for c in (a, b, b, a, a):
        ws_out, ws_lse = decode_on_gpu(c)
        out, lse = _noalloc(c)
        assert torch.equal(_bits(out), _bits(ws_out)), "differs from paged_decode"
        assert torch.equal(lse, ws_lse), "lse differs from paged_decode"
        ro, rl = refs[id(c)]
        assert_attn_close(out, ro)
        assert_lse_close(lse, rl)


def test_noalloc_allocates_nothing():
    # once the library's module is loaded on this device (the first call),
    # a call changes the device's free memory by nothing
    c = wl.decode_case([2500, 900, 4100], 16, 32, 8, 128, wl.HND, with_sinks=True, seed=43)
    d = dict(kv=c.pool.storage[0].to(DEV), q=c.query.to(DEV), bt=c.block_tables.to(DEV),
             sl=c.seq_lens.to(DEV))
    sinks = c.sinks.to(DEV)
    first, _ = _noalloc(c, d)
    out = torch.empty_like(first)
    lse = torch.empty((c.query.shape[0], 32), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        pk.paged_decode_noalloc(d["q"], d["kv"], d["bt"], d["sl"], c.max_seq_len,
                                bmm1_scale=c.bmm1_scale, sinks=sinks, kv_layout="HND",
                                out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.equal(_bits(out), _bits(first))


def _limit_boundary():
    """Largest batch whose workspace (1 query token, 32/8 heads, 2048 keys
    at most, page 16) fits the array, found with the size query."""
    def need(B):
        return pk.paged_decode_workspace_size(B, 1, 32, 8, 128, 2048, 16, -1)
    lo, hi = 1, 65535
    assert need(lo) <= LIMIT < need(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if need(mid) <= LIMIT:
            lo = mid
        else:
            hi = mid
    return lo, need(lo), need(lo + 1)


def test_noalloc_limit_boundary():
    B, fits, above = _limit_boundary()
    assert fits <= LIMIT < above
    # one batch more: refused on the host before any launch (the pointers
    # are never used)
    lib = pk.load_library()
    fake = ctypes.c_void_p(0x1000)
    rc = lib.paged_decode_noalloc(fake, fake, fake, 2 * 8 * 16 * 128, 100000, fake, 128, fake,
                                  B + 1, 2048, 0.088, 1.0, -1, None, 1, 32, 8, 128, 16, 1, 1,
                                  fake, None, None, None)
    assert rc == PKV_ERR_WORKSPACE
    # exactly the largest batch that fits: accepted, and the last request
    # (whose split partials sit at the far end of the array) is right
    lengths = [1] * (B - 1) + [2048]
    c = wl.decode_case(lengths, 16, 32, 8, 128, wl.HND, seed=44, bt_width=128)
    assert c.max_seq_len == 2048
    out, lse = _noalloc(c)
    ws_out, ws_lse = decode_on_gpu(c)
    assert torch.equal(_bits(out), _bits(ws_out))
    assert torch.equal(lse, ws_lse)


def test_noalloc_rejects_sizes_beyond_its_array():
    # the long-context decode shape without its window (8 splits of 4096 keys
    # per request) needs far more partial storage than the fixed array holds
    need = pk.paged_decode_workspace_size(256, 4, 64, 8, 128, 32768, 64, -1)
    assert need > LIMIT
    lib = pk.load_library()
    fake = ctypes.c_void_p(0x1000)
    rc = lib.paged_decode_noalloc(fake, fake, fake, 2 * 8 * 64 * 128, 100000, fake, 512, fake,
                                  256, 32768, 0.088, 1.0, -1, None, 4, 64, 8, 128, 64, 1, 1,
                                  fake, None, None, None)
    assert rc == PKV_ERR_WORKSPACE
