"""GPU parity for paged GQA decode against the fp64 oracle: every output
element within |err| <= 2e-2 + 1e-2 |ref| and LSE within 1e-3, over small
shapes that span several tiles, splits and ragged tails, the configurations
at full size (sampled requests), guards and edge cases."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_316_gb300 import workloads as wl
import paged_kv_cache_316_gb300 as pk
from _gpu import (DEV, assert_attn_close, assert_lse_close, compact_request, decode_on_gpu,
                  err_word)
from _util import oracle_decode

pytestmark = pytest.mark.gpu


def _check(c, **kw):
    out, lse = decode_on_gpu(c, **kw)
    ro, rl, _ = oracle_decode(c)
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)
    return out, lse


@pytest.mark.parametrize("layout", [wl.HND, wl.NHD])
def test_pr1_config(layout):
    _check(wl.pr1_decode(layout=layout))


CASES = [
    # lengths, page, Hqo, Hkv, Q, window, sinks, dtype, layout, seed
    ([1, 63, 64, 65, 700], 16, 32, 8, 1, -1, False, wl.BF16, wl.HND, 1),
    ([1500, 3, 1029, 511], 16, 32, 8, 1, -1, True, wl.BF16, wl.NHD, 2),
    ([2100, 777, 40], 64, 64, 8, 4, 300, True, wl.BF16, wl.HND, 3),
    ([900, 4, 130], 8, 16, 16, 1, -1, False, wl.F16, wl.HND, 4),      # MHA, group 1
    ([333, 1200], 32, 32, 2, 2, -1, False, wl.BF16, wl.NHD, 5),       # group 16, 32 rows
    ([257, 1025, 64], 16, 32, 4, 8, 100, False, wl.F16, wl.NHD, 6),   # 64 rows
    ([5000, 10, 2049], 128, 8, 1, 3, 1000, True, wl.BF16, wl.HND, 7),
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_small_shapes(case):
    L, S, hq, hk, Q, w, sk, dt, lay, seed = case
    c = wl.decode_case(L, S, hq, hk, 128, lay, dt, q_len_per_req=Q, window_left=w,
                       with_sinks=sk, seed=seed, bmm2_scale=0.8, slack=0.3)
    _check(c)


def test_bmm_scales_and_window_zero():
    c = wl.decode_case([300, 45], 16, 32, 8, 128, wl.HND, q_len_per_req=1, window_left=0,
                       seed=9, bmm1_scale=0.05, bmm2_scale=2.5)
    _check(c)


@pytest.mark.parametrize("bmm1", [-0.06, 0.0], ids=["negative", "zero"])
def test_non_positive_logit_scale(bmm1):
    # a negative bmm1_scale favours the keys least aligned with q; zero makes
    # every visible key equally likely (out = bmm2 * mean of V, lse = log n,
    # plus the sink): both against the oracle, one and several splits, an
    # E4M3 cache on the swapped-operand path
    c = wl.decode_case([2500, 7, 900], 16, 32, 8, 128, wl.HND, seed=15, with_sinks=True,
                       bmm1_scale=bmm1, bmm2_scale=1.3, slack=0.2)
    _check(c)
    c8 = wl.decode_case([2500, 7, 900], 16, 32, 8, 128, wl.NHD, seed=16, kv_dtype=wl.E4M3,
                        bmm1_scale=bmm1, bmm2_scale=0.7, slack=0.2)
    _check(c8)


SCALE_CASES = [
    # uniform queries, split and single-split requests, sinks, window
    dict(L=[1500, 3, 1029, 5000], Q=2, w=700, sinks=True, q_lens=None),
    # variable-length queries
    dict(L=[1300, 70, 3000], Q=4, w=-1, sinks=False, q_lens=[1, 4, 2]),
]


@pytest.mark.parametrize("k", SCALE_CASES, ids=["uniform", "varlen"])
def test_device_scales_and_pdl_bit_identical(k):
    # bmm1/bmm2 given as device tensors, and the programmatic dependent
    # launch, give bit for bit what the host scalars and a plain launch give
    c = wl.decode_case(k["L"], 16, 32, 8, 128, wl.HND, q_len_per_req=k["Q"],
                       q_lens=k["q_lens"], window_left=k["w"], with_sinks=k["sinks"], seed=40,
                       bmm1_scale=0.07, bmm2_scale=1.7)
    ref_o, ref_l = _check(c)
    for ts, pdl in ((True, None), (False, True), (True, True)):
        o, l = decode_on_gpu(c, tensor_scales=ts, enable_pdl=pdl)
        assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16)), (ts, pdl)
        assert torch.equal(l, ref_l), (ts, pdl)


def test_tensor_scale_must_be_one_float32_on_device():
    c = wl.decode_case([100], 16, 32, 8, 128, wl.HND, seed=41)
    for bad in (torch.tensor([0.1], dtype=torch.float64, device=DEV),
                torch.tensor([0.1, 0.2], device=DEV), torch.tensor([0.1])):
        with pytest.raises(pk.PagedKVError):
            pk.paged_decode(c.query.to(DEV), c.pool.storage[0].to(DEV),
                            torch.zeros(1 << 20, dtype=torch.uint8, device=DEV),
                            c.block_tables.to(DEV), c.seq_lens.to(DEV), c.max_seq_len,
                            bmm1_scale=bad)


def test_page_permutation_bit_identical():
    a = wl.decode_case([700, 1300], 16, 32, 8, 128, wl.HND, seed=3, pool_pages=200)
    b = wl.decode_case([700, 1300], 16, 32, 8, 128, wl.HND, seed=4, pool_pages=200)
    b.query.copy_(a.query)
    for r in range(2):
        k, v = wl.read_tokens(a.pool, a.pt, r)
        wl.write_tokens(b.pool, b.pt, r, k, v)
    assert a.pt.pages != b.pt.pages
    oa, la = decode_on_gpu(a)
    ob, lb = decode_on_gpu(b)
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(la, lb)


def test_never_reads_padding_or_unused_slots():
    # block-table padding holds a huge page id and every slot outside the
    # sequences holds NaN: neither may reach the output
    L = [45, 8, 25, 22]
    c = wl.decode_case(L, 16, 32, 8, 128, wl.HND, seed=5, pool_pages=64, fill="nan",
                       bt_width=12)
    for b, n in enumerate(L):
        kv = wl.randn((n, 8, 128), torch.bfloat16, wl.generator(100 + b))
        vv = wl.randn((n, 8, 128), torch.bfloat16, wl.generator(200 + b))
        wl.write_tokens(c.pool, c.pt, b, kv, vv)
    assert int(c.block_tables[1, 5]) == wl.POISON
    err = err_word()
    _check(c, err_word=err)
    assert int(err.item()) == 0


def test_empty_and_short_requests():
    c = wl.decode_case([0, 1, 2, 600], 16, 32, 8, 128, wl.HND, q_len_per_req=2,
                       with_sinks=True, seed=6)
    err = err_word()
    out, lse = decode_on_gpu(c, err_word=err)
    ro, rl, oerr = oracle_decode(c)
    assert int(err.item()) == oerr == oracle.E_QLEN
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)
    c2 = dataclasses.replace(c, sinks=None)
    out, lse = decode_on_gpu(c2)
    ro, rl, _ = oracle_decode(c2)
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)


def test_bad_page_flagged_and_treated_as_absent():
    c = wl.decode_case([100, 50], 16, 32, 8, 128, wl.HND, seed=8, slack=0.5)
    c.block_tables[0, 2] = c.pool.num_pages + 10
    err = err_word()
    out, lse = decode_on_gpu(c, err_word=err)
    ro, rl, oerr = oracle_decode(c)
    assert int(err.item()) & oracle.E_PAGE and oerr & oracle.E_PAGE
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)


def test_workspace_reused_across_sizes():
    # one workspace serves calls of different sizes and split counts in
    # turn, the split partials of a larger call staying behind: each result
    # is within tolerance of the oracle and bit for bit the result with a
    # freshly zeroed workspace.
    big = wl.decode_case([3000, 2500, 4100, 900, 5000, 1800], 16, 32, 8, 128, wl.HND, seed=11,
                         window_left=-1, slack=0.2)
    small = wl.decode_case([2100, 4000], 32, 64, 8, 128, wl.HND, seed=12, q_len_per_req=2,
                           with_sinks=True, slack=0.2)
    fp8 = wl.decode_case([6000, 70, 2900], 16, 32, 8, 128, wl.HND, seed=14, kv_dtype=wl.E4M3,
                         bmm1_scale=0.07, bmm2_scale=0.6, slack=0.2)
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=DEV)
    for c in (big, small, fp8, big, fp8, small):
        out, lse = _check(c, ws=ws)
        fresh_out, fresh_lse = decode_on_gpu(c)
        assert torch.equal(out.view(torch.int16), fresh_out.view(torch.int16))
        assert torch.equal(lse, fresh_lse)


def test_hundreds_of_splits():
    # one long request on one kv head: the keys are cut into ~780 splits
    c = wl.decode_case([200000], 256, 64, 1, 128, wl.HND, seed=13, with_sinks=True)
    _check(c)


VARLEN = [
    # lengths, q_lens, page, Hqo, Hkv, window, sinks, layout, seed
    ([700, 40, 1500, 3, 2100], [3, 0, 1, 2, 4], 16, 64, 8, 300, True, wl.HND, 21),   # 32 rows
    ([900, 4000, 77], [4, 1, 2], 32, 16, 4, -1, False, wl.NHD, 22),                  # 16 rows
    ([1200, 650], [8, 5], 64, 64, 8, 511, True, wl.HND, 23),                          # 64 rows
]


@pytest.mark.parametrize("case", VARLEN, ids=[f"v{i}" for i in range(len(VARLEN))])
def test_variable_length_queries(case):
    L, ql, S, hq, hk, w, sk, lay, seed = case
    c = wl.decode_case(L, S, hq, hk, 128, lay, q_lens=ql, window_left=w, with_sinks=sk,
                       seed=seed, slack=0.2, bmm2_scale=1.3)
    err = err_word()
    out, lse = decode_on_gpu(c, err_word=err)
    ro, rl, oerr = oracle_decode(c)
    assert int(err.item()) == oerr == 0
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)


def test_variable_length_bad_entry_flagged_and_skipped():
    # request 1 claims more tokens than max_q_len: flagged, its rows untouched;
    # the others are computed as usual
    c = wl.decode_case([500, 800, 300], 16, 32, 8, 128, wl.HND, q_lens=[2, 3, 1], seed=24)
    B = 3
    ws = torch.zeros(max(1, pk.paged_decode_workspace_size(B, 2, 32, 8, 128, c.max_seq_len, 16)),
                     dtype=torch.uint8, device=DEV)
    out = torch.full((6, 32, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    err = err_word()
    pk.paged_decode(c.query.to(DEV), c.pool.storage[0].to(DEV), ws, c.block_tables.to(DEV),
                    c.seq_lens.to(DEV), c.max_seq_len, bmm1_scale=c.bmm1_scale,
                    cum_seq_lens_q=c.cum_seq_lens_q.to(DEV), max_q_len=2, out=out, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & oracle.E_QLEN
    ro, _, _ = oracle_decode(c)
    rows_ok = [0, 1, 5]  # requests 0 and 2
    assert_attn_close(out[rows_ok], ro[rows_ok])
    assert torch.all(out[2:5].float() == 7.0)


def test_without_lse_output():
    c = wl.decode_case([500, 20], 16, 32, 8, 128, wl.NHD, seed=10)
    out, _ = decode_on_gpu(c, with_lse=False)
    assert_attn_close(out, oracle_decode(c)[0])


def _sampled_full_size(c, requests):
    """Run the full case on the GPU; check the sampled requests' rows against
    the oracle run on a compact copy of just those requests' pages."""
    out, lse = decode_on_gpu(c)
    Q = c.q_len_per_req
    for b in requests:
        pool, pt = compact_request(c.pool, c.pt, b)
        sub = dataclasses.replace(
            c, query=c.query[b * Q:(b + 1) * Q].cpu(), pool=pool, pt=pt,
            block_tables=pt.block_tables(), seq_lens=torch.tensor([pt.lengths[0]], dtype=torch.int32),
            max_seq_len=pt.lengths[0],
            sinks=None if c.sinks is None else c.sinks.cpu())
        ro, rl, _ = oracle_decode(sub)
        assert_attn_close(out[b * Q:(b + 1) * Q], ro, f"request {b}")
        assert_lse_close(lse[b * Q:(b + 1) * Q], rl, f"request {b} lse")


def test_llama_config_full_size_sampled():
    c = wl.llama_decode(device=DEV)
    lengths = np.array(c.pt.lengths)
    pick = sorted({int(lengths.argmin()), int(lengths.argmax()), 0, 17, 63})
    _sampled_full_size(c, pick)


def test_long_context_config_full_size_sampled():
    c = wl.long_decode(device=DEV)
    lengths = np.array(c.pt.lengths)
    pick = sorted({int(lengths.argmin()), int(lengths.argmax()), 1, 100, 255})
    _sampled_full_size(c, pick)


def test_long_context_varlen_full_size_sampled():
    c = wl.long_decode_varlen(device=DEV)
    out, lse = decode_on_gpu(c)
    cum = c.cum_seq_lens_q.tolist()
    lengths = np.array(c.pt.lengths)
    for b in sorted({int(lengths.argmin()), int(lengths.argmax()), 3, 130, 255}):
        pool, pt = compact_request(c.pool, c.pt, b)
        Q = cum[b + 1] - cum[b]
        sub = dataclasses.replace(
            c, query=c.query[cum[b]:cum[b + 1]].cpu(), pool=pool, pt=pt,
            block_tables=pt.block_tables(), seq_lens=torch.tensor([pt.lengths[0]], dtype=torch.int32),
            max_seq_len=pt.lengths[0], sinks=c.sinks.cpu(), q_len_per_req=Q, cum_seq_lens_q=None)
        ro, rl, _ = oracle_decode(sub)
        assert_attn_close(out[cum[b]:cum[b + 1]], ro, f"request {b}")
        assert_lse_close(lse[cum[b]:cum[b + 1]], rl, f"request {b} lse")


FP8 = [
    # lengths, page, Hqo, Hkv, Q, window, sinks, query dtype, layout, seed
    ([700, 45, 1500], 16, 32, 8, 1, -1, False, wl.BF16, wl.HND, 51),     # 4 rows
    ([2100, 777, 40], 64, 64, 8, 4, 300, True, wl.BF16, wl.NHD, 52),     # 32 rows
    ([900, 130], 32, 16, 16, 1, -1, True, wl.F16, wl.HND, 53),           # MHA, fp16 query
    ([1025, 64], 16, 32, 4, 8, 100, False, wl.BF16, wl.HND, 54),         # 64 rows
    # at most 8 query rows take the swapped-operand MMAs: 8, 6 and 2 rows,
    # padding rows, windows, sinks, both layouts
    ([900, 130, 2500], 16, 32, 4, 1, 200, True, wl.BF16, wl.NHD, 55),    # 8 rows
    ([700, 3000], 32, 24, 8, 2, -1, True, wl.F16, wl.HND, 56),           # group 3 x 2 tokens
    ([513, 77, 4100], 64, 8, 8, 2, 100, False, wl.BF16, wl.HND, 57),     # 2 rows
]


@pytest.mark.parametrize("case", FP8, ids=[f"f{i}" for i in range(len(FP8))])
def test_fp8_cache(case):
    # E4M3 K/V cache with 16-bit query and output; bmm scales fold the cache scales
    L, S, hq, hk, Q, w, sk, dt, lay, seed = case
    c = wl.decode_case(L, S, hq, hk, 128, lay, dt, q_len_per_req=Q, window_left=w, with_sinks=sk,
                       seed=seed, kv_dtype=wl.E4M3, bmm1_scale=0.07, bmm2_scale=0.6, slack=0.2)
    err = err_word()
    _check(c, err_word=err)
    assert int(err.item()) == 0


def test_fp8_cache_full_size_sampled():
    # the Llama-shaped decode over an E4M3 cache
    c = wl.llama_decode(device=DEV, kv_dtype=wl.E4M3)
    lengths = np.array(c.pt.lengths)
    _sampled_full_size(c, sorted({int(lengths.argmin()), int(lengths.argmax()), 9, 40}))


def _key_factor(j: int) -> float:
    """Scale of key j: steps up at keys 100, 600 and 2500, so that each
    row's running max (base 2) rises by more than 2^8 several times after
    its first tile, in the first split and in later ones."""
    return 1.0 if j < 100 else 4.0 if j < 600 else 12.0 if j < 2500 else 24.0


def _rising_keys(c):
    """Multiply the keys of every request by _key_factor(position) (CPU pool,
    in place); returns the largest rise of a row's base-2 max over its first
    64-key tile, for checking that the case does what it is for."""
    rise = 0.0
    Q = c.q_len_per_req
    group = c.num_qo_heads // c.num_kv_heads
    for b, L in enumerate(c.pt.lengths):
        k, v = wl.read_tokens(c.pool, c.pt, b)
        f = torch.tensor([_key_factor(j) for j in range(L)], dtype=torch.float32).view(-1, 1, 1)
        k = (k.float() * f).to(k.dtype)
        wl.write_tokens(c.pool, c.pt, b, k, v)
        q = c.query[b * Q:(b + 1) * Q].double()                        # [Q, Hqo, D]
        kk = k.double().repeat_interleave(group, dim=1)                # [L, Hqo, D]
        s = torch.einsum("qhd,khd->qhk", q, kk) * c.bmm1_scale * 1.4426950408889634
        if L > 64:
            rise = max(rise, float((s[..., 64:].amax(-1) - s[..., :64].amax(-1)).max()))
    return rise


RISING = [
    # lengths, page, Hqo, Hkv, Q, window, sinks, layout, kv dtype, seed
    ([3000, 700, 5000, 129], 16, 32, 8, 1, -1, False, wl.HND, None, 61),     # 4 rows, 1..5 splits
    ([900, 2600], 64, 64, 8, 4, -1, True, wl.NHD, None, 62),                 # 32 rows
    ([1100, 4000], 32, 32, 4, 8, 3000, True, wl.HND, None, 63),              # 64 rows, window
    ([3000, 700, 129], 16, 32, 8, 1, -1, True, wl.NHD, wl.E4M3, 64),         # E4M3, 4 rows
    ([2600, 900], 64, 64, 8, 4, 2000, False, wl.HND, wl.E4M3, 65),           # E4M3, 32 rows
]


@pytest.mark.parametrize("case", RISING, ids=[f"r{i}" for i in range(len(RISING))])
def test_running_max_rises_far_after_first_tile(case):
    # the decode raises its running max only when a tile's exceeds it by more
    # than 2^8 and rescales O only then; these keys make that happen many
    # times (the rescale of O, and the (m, l) update across tiles and splits)
    L, S, hq, hk, Q, w, sk, lay, kvd, seed = case
    c = wl.decode_case(L, S, hq, hk, 128, lay, q_len_per_req=Q, window_left=w, with_sinks=sk,
                       seed=seed, slack=0.2, kv_dtype=kvd)
    assert _rising_keys(c) > 16.0
    err = err_word()
    _check(c, err_word=err)
    assert int(err.item()) == 0


def test_binding_refuses_shapes_the_abi_cannot_check():
    # the uniform decode's C entry points take no row count: the binding
    # checks query rows, out and lse against the requests before the call
    c = wl.decode_case([100, 50], 16, 32, 8, 128, wl.HND, q_len_per_req=2, seed=66)
    kv, bt, sl = c.pool.storage[0].to(DEV), c.block_tables.to(DEV), c.seq_lens.to(DEV)
    q = c.query.to(DEV)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    bad = [
        dict(query=q[:3]),                                                    # 3 rows for 2 x 2
        dict(out=torch.empty((3, 32, 128), dtype=q.dtype, device=DEV)),
        dict(out=torch.empty_like(q, dtype=torch.float16)),
        dict(lse=torch.empty((4, 32), dtype=torch.float64, device=DEV)),
        dict(lse=torch.empty((4, 31), dtype=torch.float32, device=DEV)),
        dict(block_tables=bt[:1]),
    ]
    for kw in bad:
        args = dict(query=q, block_tables=bt)
        args.update(kw)
        with pytest.raises(pk.PagedKVError):
            pk.paged_decode(args.pop("query"), kv, ws, args.pop("block_tables"), sl, c.max_seq_len,
                            q_len_per_req=2, **args)
        with pytest.raises(pk.PagedKVError):
            a2 = dict(query=q, block_tables=bt)
            a2.update(kw)
            pk.paged_decode_noalloc(a2.pop("query"), kv, a2.pop("block_tables"), sl, c.max_seq_len,
                                    q_len_per_req=2, **a2)
