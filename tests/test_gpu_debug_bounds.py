"""The range-checking debug build of the library (libpagedkv_debug.so,
compiled with -DPKV_DEBUG_BOUNDS=1) on the GPU.

Every offset its kernels derive -- cache rows, query and output rows,
workspace partials, block-table entries, tensor-map coordinates, the shared
page lists -- is checked before the access.  Over shapes that take every
kernel variant (decode row tiles 16/32/64, the E4M3 swapped-operand and
plain paths, one and several splits with the merge, variable-length
queries; prefill d_qk 128/192, both layouts, pages 8..256, the E4M3
kind::f8f6f4 and widening paths, contiguous K/V; append with whole-row and
per-head pieces) no check may fire: the error word stays 0 and the results
match the oracle as in the release build's tests; nor over the benchmark's
workloads at full size.  One input the release
build tolerates silently -- output rows placed past the end of `out`, which
are documented as not written -- is reported by the debug build.

The module switches the binding to the debug library and back afterwards.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_316_gb300 as pk
from paged_kv_cache_316_gb300 import binding
from paged_kv_cache_316_gb300 import build as pk_build
from paged_kv_cache_316_gb300 import workloads as wl
from _gpu import (DEV, assert_attn_close, assert_lse_close, decode_on_gpu, err_word,
                  prefill_on_gpu)
from _util import oracle_append, oracle_decode, oracle_prefill

pytestmark = pytest.mark.gpu
BOUNDS = 64  # PKV_DEV_ERR_BOUNDS


@pytest.fixture(scope="module", autouse=True)
def debug_library():
    binding.load_library(pk_build.build(debug_bounds=True))
    assert binding.debug_bounds()
    yield
    binding.load_library(binding.library_path())
    assert not binding.debug_bounds()


DECODE = [
    # lengths, page, Hqo, Hkv, Q, window, sinks, dtype, kv dtype, layout, seed
    ([1, 63, 64, 65, 700], 16, 32, 8, 1, -1, False, wl.BF16, None, wl.HND, 1),     # 4 rows, MT 1
    ([1500, 3, 1029, 511], 16, 32, 8, 1, -1, True, wl.F16, None, wl.NHD, 2),
    ([2100, 777, 40], 64, 64, 8, 4, 300, True, wl.BF16, None, wl.HND, 3),          # 32 rows, window
    ([257, 1025, 64], 16, 32, 4, 8, 100, False, wl.F16, None, wl.NHD, 6),          # 64 rows
    ([5000, 10, 2049], 128, 8, 1, 3, 1000, True, wl.BF16, None, wl.HND, 7),        # splits + merge
    ([700, 45, 1500], 16, 32, 8, 1, -1, False, wl.BF16, wl.E4M3, wl.HND, 8),       # swapped operands
    ([2500, 7, 900], 8, 32, 8, 4, -1, True, wl.F16, wl.E4M3, wl.NHD, 9),           # E4M3, 16 rows
    ([3000, 129], 256, 16, 2, 2, 2000, False, wl.BF16, wl.E4M3, wl.HND, 10),       # 16 rows, page 256
]


@pytest.mark.parametrize("case", DECODE, ids=[f"d{i}" for i in range(len(DECODE))])
def test_decode_no_check_fires(case):
    L, S, hq, hk, Q, w, sk, dt, kvd, lay, seed = case
    c = wl.decode_case(L, S, hq, hk, 128, lay, dt, q_len_per_req=Q, window_left=w, with_sinks=sk,
                       seed=seed, bmm2_scale=0.8, slack=0.3, kv_dtype=kvd)
    err = err_word()
    out, lse = decode_on_gpu(c, err_word=err)
    assert int(err.item()) == 0
    ro, rl, _ = oracle_decode(c)
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)


def test_decode_varlen_no_check_fires():
    c = wl.decode_case([1300, 70, 3000, 5], 16, 32, 8, 128, wl.HND, q_len_per_req=4,
                       q_lens=[1, 4, 2, 3], with_sinks=True, seed=17, slack=0.2)
    err = err_word()
    out, lse = decode_on_gpu(c, err_word=err)
    assert int(err.item()) == 0
    ro, rl, _ = oracle_decode(c)
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)


PREFILL = [
    # q lens, kv lens, page, Hqo, Hkv, d_qk, causal, dtype, layout, E4M3 query, E4M3 caches, seed
    ([130, 7, 300, 1], [400, 7, 300, 2049], 16, 32, 8, 128, True, wl.BF16, wl.HND, False, False, 1),
    ([200, 129], [900, 129], 8, 16, 2, 192, True, wl.F16, wl.NHD, False, False, 2),
    ([0, 300, 0, 17], [40, 1000, 0, 17], 128, 8, 2, 128, False, wl.BF16, wl.HND, False, False, 3),
    ([129, 1], [2049, 1], 256, 16, 4, 128, False, wl.F16, wl.HND, False, False, 4),
    ([257, 33], [600, 33], 16, 16, 4, 128, True, wl.F16, wl.NHD, True, True, 5),    # kind::f8f6f4
    ([1, 255, 129], [1, 255, 700], 32, 32, 8, 192, True, wl.BF16, wl.HND, False, True, 6),  # widening
    ([1, 700, 64], [1, 1300, 64], 256, 6, 2, 128, True, wl.BF16, wl.NHD, True, True, 7),   # odd group
]


@pytest.mark.parametrize("case", PREFILL, ids=[f"p{i}" for i in range(len(PREFILL))])
def test_prefill_no_check_fires(case):
    ql, kvl, S, hq, hk, dqk, causal, dt, lay, q8, kv8, seed = case
    c = wl.prefill_case(ql, kvl, S, hq, hk, dqk, 128, lay, dt, causal=causal, seed=seed, slack=0.2,
                        q_dtype=wl.E4M3 if q8 else None, kv_dtype=wl.E4M3 if kv8 else None,
                        **(dict(q_scale=0.37, k_scale=1.9, v_scale=0.61) if (q8 or kv8) else {}))
    err = err_word()
    out, lse = prefill_on_gpu(c, err_word=err)
    assert int(err.item()) == 0
    ro, rl, _ = oracle_prefill(c)
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)


def _contiguous(c):
    ks, vs = zip(*(wl.read_tokens(c.pool, c.pt, b) for b in range(len(c.pt.lengths))))
    return torch.cat(ks).contiguous(), torch.cat(vs).contiguous()


def test_prefill_contiguous_no_check_fires():
    c = wl.prefill_case([130, 7, 300, 64], [400, 7, 300, 900], 32, 32, 8, 128, 128, wl.HND, wl.BF16,
                        seed=41, slack=0.2)
    k, v = _contiguous(c)
    B = len(c.pt.lengths)
    ws = torch.zeros(pk.paged_prefill_workspace_size(B, 32, c.max_q, c.max_kv), dtype=torch.uint8, device=DEV)
    err = err_word()
    out, lse = pk.paged_prefill(c.q.to(DEV), k.to(DEV), v.to(DEV), c.scale, ws, c.max_q, c.max_kv,
                                c.seq_lens_q.to(DEV), c.seq_lens_kv.to(DEV), None, causal=True, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ro, rl, _ = oracle_prefill(c)
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)


def test_output_rows_past_the_end_are_reported():
    # request 1's output rows placed so that its last 5 rows fall past the end
    # of `out`: both builds leave those rows unwritten (as documented) and
    # write the rest; the debug build also reports the placement
    ql, kvl = [40, 30], [100, 60]
    c = wl.prefill_case(ql, kvl, 16, 8, 2, 128, 128, wl.HND, wl.BF16, seed=43, slack=0.2)
    n_rows = sum(ql)
    ws = torch.zeros(pk.paged_prefill_workspace_size(2, 8, c.max_q, c.max_kv), dtype=torch.uint8, device=DEV)
    out = torch.full((n_rows, 8, 128), 3.0, dtype=c.q.dtype, device=DEV)
    lse = torch.full((n_rows, 8), 3.0, dtype=torch.float32, device=DEV)
    off_o = torch.tensor([0, n_rows - 25], dtype=torch.int32, device=DEV)
    err = err_word()
    pk.paged_prefill(c.q.to(DEV), c.pool.k.to(DEV), c.pool.v.to(DEV), c.scale, ws, c.max_q, c.max_kv,
                     c.seq_lens_q.to(DEV), c.seq_lens_kv.to(DEV), c.block_tables.to(DEV), causal=True,
                     kv_layout=c.pool.layout, out=out, lse=lse, batch_offsets_o=off_o, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == BOUNDS
    ro, rl, _ = oracle_prefill(c)
    assert_attn_close(out[:40], ro[:40])                  # request 0, rows 0..39
    assert_lse_close(lse[:40], rl[:40])
    assert_attn_close(out[45:], ro[40:65])                # request 1's first 25 rows
    assert_lse_close(lse[45:], rl[40:65])
    assert torch.all(out[40:45].float() == 3.0) and torch.all(lse[40:45] == 3.0)


APPEND = [
    # form, layout, dtype, heads, page, seed
    ("example", wl.NHD, wl.F16, 32, 16, 0),
    ("example", wl.HND, wl.F16, 32, 16, 0),
    ("case", wl.HND, wl.BF16, 64, 32, 11),   # two 8 KB pieces per row
    ("case", wl.NHD, wl.F16, 48, 16, 12),    # pieces of 32 and 16 heads
    ("case", wl.HND, wl.E4M3, 48, 64, 14),
]


@pytest.mark.parametrize("case", APPEND, ids=[f"a{i}" for i in range(len(APPEND))])
def test_append_no_check_fires(case):
    form, layout, dtype, heads, page, seed = case
    if form == "example":
        c = wl.append_example(layout=layout, form="tuple")
    else:
        g = np.random.default_rng(seed)
        n = [int(x) for x in g.integers(1, 90, size=23)]
        prefix = [int(x) for x in g.integers(0, 200, size=23)]
        c = wl.append_case(n, prefix, page, heads, 128, layout, dtype, seed=seed, slack=0.2)
    S = c.pool.page_size
    seq = pk.paged_seq_lens(c.kv_indptr.to(DEV), c.kv_last_page_len.to(DEV), S)
    bi, pos = pk.paged_batch_indices_positions(c.append_indptr.to(DEV), seq, c.append_key.shape[0])
    storage = [t.to(DEV) for t in c.pool.storage]
    cache = storage[0] if len(storage) == 1 else tuple(storage)
    err = err_word()
    pk.paged_append(c.append_key.to(DEV), c.append_value.to(DEV), bi, pos, cache,
                    c.kv_indices.to(DEV), c.kv_indptr.to(DEV), c.kv_last_page_len.to(DEV),
                    kv_layout=layout, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    sl = oracle.seq_lens(c.kv_indptr.numpy(), c.kv_last_page_len.numpy(), S)
    obi, opos = oracle.batch_indices_positions(c.append_indptr.numpy(), sl, c.append_key.shape[0])
    assert oracle_append(c, obi, opos) == 0
    for g_, r in zip(storage, c.pool.storage):
        assert torch.equal(g_.cpu().view(torch.uint8), r.view(torch.uint8))


FULL = ["decode_llama", "decode_llama_e4m3", "decode_long", "decode_varlen", "prefill_d128",
        "prefill_d192", "prefill_d128_e4m3", "append_4096", "append_4096_e4m3"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads_no_check_fires(name):
    # the benchmark's workloads at full size (the largest offsets: a 4096-
    # request append pool of several GB, 256-request long-context decode,
    # the ragged prefill): no derived offset leaves its buffer.  Their
    # results are checked against the oracle on sampled requests elsewhere.
    err = err_word()
    if name.startswith("decode"):
        kv8 = dict(kv_dtype=wl.E4M3) if name.endswith("e4m3") else {}
        c = {"decode_llama": wl.llama_decode, "decode_llama_e4m3": wl.llama_decode,
             "decode_long": wl.long_decode, "decode_varlen": wl.long_decode_varlen}[name](device=DEV, **kv8)
        decode_on_gpu(c, err_word=err)
    elif name.startswith("prefill"):
        kw = dict(q_dtype=wl.E4M3, kv_dtype=wl.E4M3) if name.endswith("e4m3") else {}
        c = wl.ragged_prefill(d_qk=192 if "192" in name else 128, device=DEV, **kw)
        prefill_on_gpu(c, err_word=err)
    else:
        c = wl.append_sweep(4096, seed=1, layout=wl.NHD, device=DEV, fill="empty",
                            **(dict(dtype=wl.E4M3) if name.endswith("e4m3") else {}))
        kvi, kvp, last = (x.to(DEV) for x in (c.kv_indices, c.kv_indptr, c.kv_last_page_len))
        seq = pk.paged_seq_lens(kvp, last, 16)
        bi, pos = pk.paged_batch_indices_positions(c.append_indptr.to(DEV), seq, c.append_key.shape[0])
        pk.paged_append(c.append_key, c.append_value, bi, pos, c.pool.storage[0], kvi, kvp, last,
                        kv_layout="NHD", err_word=err)
        torch.cuda.synchronize()
    assert int(err.item()) == 0
