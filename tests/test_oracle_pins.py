"""Pins for the fp64 oracle: each test checks it against something other than
itself -- the append page's printed example, closed forms, invariants, the
library attention routine (torch SDPA in float64) on special cases, and brute
force on tiny shapes.  CPU only."""
from __future__ import annotations

import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_316_gb300 import workloads as wl
from _util import (expand_heads, logsumexp64, oracle_append, oracle_decode,
                   oracle_prefill, sdpa64, u16)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "append_example.json")


@pytest.fixture(scope="module")
def example():
    with open(GOLDEN) as f:
        return json.load(f)


# ---- 16-bit widening ------------------------------------------------------------

@pytest.mark.parametrize("code,tdt", [(wl.F16, torch.float16), (wl.BF16, torch.bfloat16)])
def test_widen16_all_patterns(code, tdt):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.widen16(bits, code)
    ref = torch.from_numpy(bits.view(np.int16)).view(tdt).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---- append page example: helpers ---------------------------------------------------

def test_example_seq_lens(example):
    got = oracle.seq_lens(example["kv_page_indptr"], example["kv_last_page_len"],
                          example["page_size"])
    assert got.tolist() == example["seq_lens"]


def test_example_batch_indices_positions(example):
    sl = oracle.seq_lens(example["kv_page_indptr"], example["kv_last_page_len"],
                         example["page_size"])
    bi, pos = oracle.batch_indices_positions(example["kv_append_indptr"], sl,
                                             example["nnz_kv"])
    assert bi.tolist() == example["batch_indices"]
    assert pos.tolist() == example["positions"]


def test_positions_after_prefix():
    # 2 requests with 5 and 0 cached tokens append 3 and 2: the new tokens are
    # the last ones of each sequence (page table already counts them)
    bi, pos = oracle.batch_indices_positions([0, 3, 5], [8, 2], 5)
    assert bi.tolist() == [0, 0, 0, 1, 1]
    assert pos.tolist() == [5, 6, 7, 0, 1]
    # entries beyond the last request are marked -1
    bi, pos = oracle.batch_indices_positions([0, 1], [4], 3)
    assert bi.tolist() == [0, -1, -1] and pos.tolist() == [3, -1, -1]


# ---- append page example: scatter ----------------------------------------------------

def _example_positions(case):
    sl = oracle.seq_lens(case.kv_indptr.numpy(), case.kv_last_page_len.numpy(),
                         case.pool.page_size)
    return oracle.batch_indices_positions(case.append_indptr.numpy(), sl,
                                          case.append_key.shape[0])


@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
@pytest.mark.parametrize("form", ["5d", "tuple"])
def test_example_append(example, layout, form):
    c = wl.append_example(layout=layout, form=form)
    assert c.kv_indptr.tolist() == example["kv_page_indptr"]
    assert c.kv_indices.tolist() == example["kv_page_indices"]
    assert c.kv_last_page_len.tolist() == example["kv_last_page_len"]
    before = [t.clone() for t in c.pool.storage]
    bi, pos = _example_positions(c)
    assert oracle_append(c, bi, pos) == 0
    pool = c.pool
    # every appended token reads back bit-exactly through the page table
    off = 0
    for b, n in enumerate(example["kv_append_length"]):
        k, v = wl.read_tokens(pool, c.pt, b)
        assert torch.equal(k.view(torch.int16), c.append_key[off:off + n].view(torch.int16))
        assert torch.equal(v.view(torch.int16), c.append_value[off:off + n].view(torch.int16))
        off += n

    def at(t, page, slot):
        return t[page, slot] if layout == wl.NHD else t[page, :, slot]

    # request 0 token 44 -> page 2, slot 12; request 3 token 21 -> page 7, slot 5
    assert torch.equal(at(pool.k, 2, 12).view(torch.int16), c.append_key[44].view(torch.int16))
    assert torch.equal(at(pool.v, 7, 5).view(torch.int16), c.append_value[99].view(torch.int16))
    # pages 8..999 and the unwritten slots of pages 0..7 keep their old bits
    kb, vb = (before[0][:, 0], before[0][:, 1]) if form == "5d" else before
    assert torch.equal(pool.k[8:].view(torch.int16), kb[8:].view(torch.int16))
    assert torch.equal(pool.v[8:].view(torch.int16), vb[8:].view(torch.int16))
    for page, first_free in [(2, 13), (3, 8), (5, 9), (7, 6)]:
        for slot in range(first_free, 16):
            assert torch.equal(at(pool.k, page, slot).view(torch.int16),
                               at(kb, page, slot).view(torch.int16))
            assert torch.equal(at(pool.v, page, slot).view(torch.int16),
                               at(vb, page, slot).view(torch.int16))


def test_append_layouts_same_logical_content():
    cn = wl.append_sweep(6, seed=3, layout=wl.NHD)
    ch = wl.append_sweep(6, seed=3, layout=wl.HND)
    for c in (cn, ch):
        bi, pos = _example_positions(c)
        assert oracle_append(c, bi, pos) == 0
    for b in range(6):
        n = int(cn.append_indptr[b + 1] - cn.append_indptr[b])
        kn, vn = wl.read_tokens(cn.pool, cn.pt, b)
        kh, vh = wl.read_tokens(ch.pool, ch.pt, b)
        # the appended tokens (the last n) agree bit for bit across layouts
        assert torch.equal(kn[-n:].view(torch.int16), kh[-n:].view(torch.int16))
        assert torch.equal(vn[-n:].view(torch.int16), vh[-n:].view(torch.int16))
        off = int(cn.append_indptr[b])
        assert torch.equal(kn[-n:].view(torch.int16),
                           cn.append_key[off:off + n].view(torch.int16))


def test_append_errors_skip_and_flag():
    c = wl.append_sweep(3, seed=5)
    bi, pos = _example_positions(c)
    before = c.pool.storage[0].clone()
    bad_b = bi.copy(); bad_b[0] = 3
    assert oracle_append(c, bad_b[:1], pos[:1]) == oracle.E_BATCH
    bad_p = pos.copy(); bad_p[0] = c.pt.lengths[bi[0]]
    assert oracle_append(c, bi[:1], bad_p[:1]) == oracle.E_POS
    c.kv_indices[c.kv_indptr[bi[0]] + pos[0] // 16] = c.pool.num_pages
    assert oracle_append(c, bi[:1], pos[:1]) == oracle.E_PAGE
    assert torch.equal(c.pool.storage[0].view(torch.int16), before.view(torch.int16))


# ---- decode ---------------------------------------------------------------------------

def _small_decode(lengths, **kw):
    args = dict(page_size=4, num_qo_heads=4, num_kv_heads=2, head_dim=16,
                layout=wl.HND, seed=11)
    args.update(kw)
    return wl.decode_case(lengths, **args)


def _dense_kv(c, b):
    k, v = wl.read_tokens(c.pool, c.pt, b)
    g = c.num_qo_heads // c.num_kv_heads
    return expand_heads(k, g), expand_heads(v, g)


@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16])
def test_decode_matches_library_attention(layout, dtype):
    c = _small_decode([13, 1, 7, 20], layout=layout, dtype=dtype, bmm2_scale=0.75)
    out, lse, err = oracle_decode(c)
    assert err == 0
    for b in range(4):
        k, v = _dense_kv(c, b)
        q = c.query[b:b + 1]
        ref = sdpa64(q, k, v, c.bmm1_scale) * c.bmm2_scale
        np.testing.assert_allclose(out[b], ref[0].numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b], logsumexp64(q, k, c.bmm1_scale)[0].numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_decode_single_key_returns_v():
    c = _small_decode([1, 9], window_left=0)
    out, lse, err = oracle_decode(c)
    for b, L in enumerate([1, 9]):
        k, v = _dense_kv(c, b)
        np.testing.assert_allclose(out[b], v[L - 1].double().numpy(), rtol=0, atol=1e-15)
        s = (c.query[b].double() * k[L - 1].double()).sum(-1) * c.bmm1_scale
        np.testing.assert_allclose(lse[b], s.numpy(), rtol=1e-13, atol=1e-13)


def test_decode_uniform_keys_give_mean():
    c = _small_decode([11])
    k0, _ = wl.read_tokens(c.pool, c.pt, 0, 1)
    _, v = wl.read_tokens(c.pool, c.pt, 0)
    wl.write_tokens(c.pool, c.pt, 0, k0.expand(11, -1, -1).clone(), v)
    out, lse, _ = oracle_decode(c)
    g = c.num_qo_heads // c.num_kv_heads
    vm = expand_heads(v, g).double().mean(0)
    np.testing.assert_allclose(out[0], vm.numpy(), rtol=1e-13, atol=1e-14)
    s = (c.query[0].double() * expand_heads(k0, g)[0].double()).sum(-1) * c.bmm1_scale
    np.testing.assert_allclose(lse[0], (s + math.log(11)).numpy(), rtol=1e-13, atol=1e-13)


def test_decode_sink_closed_form():
    c = _small_decode([6, 17, 3], with_sinks=True)
    out_s, lse_s, _ = oracle_decode(c)
    sinks = c.sinks.double().numpy()
    c.sinks = None
    out, lse, _ = oracle_decode(c)
    w = np.exp(lse) / (np.exp(lse) + np.exp(sinks)[None, :])
    np.testing.assert_allclose(out_s, out * w[..., None], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse_s, np.logaddexp(lse, sinks[None, :]), rtol=1e-12)
    # V == 1 gives bmm2 * sum e^s / (sum e^s + e^sink)
    for t in c.pool.storage:
        t[:, 1].fill_(1.0)
    c.sinks = torch.tensor(sinks, dtype=torch.float32)
    out1, _, _ = oracle_decode(c)
    np.testing.assert_allclose(out1, np.broadcast_to(w[..., None], out1.shape), rtol=1e-12)
    # a sink at -1e30 is no sink
    c.sinks = torch.full_like(c.sinks, -1e30)
    for t in c.pool.storage:
        t[:, 1].normal_()
    c.sinks, base = None, oracle_decode(c)[0]
    c.sinks = torch.full((c.num_qo_heads,), -1e30)
    np.testing.assert_array_equal(oracle_decode(c)[0], base)


def test_decode_page_permutation_invariance():
    a = _small_decode([10, 15], seed=3, pool_pages=40)
    b = _small_decode([10, 15], seed=4, pool_pages=40)
    b.query.copy_(a.query)
    for r in range(2):
        k, v = wl.read_tokens(a.pool, a.pt, r)
        wl.write_tokens(b.pool, b.pt, r, k, v)
    assert a.pt.pages != b.pt.pages
    oa, la, _ = oracle_decode(a)
    ob, lb, _ = oracle_decode(b)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(la, lb)


def test_decode_gqa_equals_replicated_heads():
    c = _small_decode([9, 14], num_qo_heads=8, num_kv_heads=2)
    r = _small_decode([9, 14], num_qo_heads=8, num_kv_heads=8, seed=12)
    r.query.copy_(c.query)
    for b in range(2):
        k, v = wl.read_tokens(c.pool, c.pt, b)
        wl.write_tokens(r.pool, r.pt, b, expand_heads(k, 4), expand_heads(v, 4))
    oc, lc, _ = oracle_decode(c)
    orr, lr, _ = oracle_decode(r)
    np.testing.assert_array_equal(oc, orr)
    np.testing.assert_array_equal(lc, lr)


def test_decode_window_equals_truncated_sequence():
    L, w = 23, 6
    c = _small_decode([L], window_left=w)
    out, lse, _ = oracle_decode(c)
    t = _small_decode([w + 1], seed=13)
    t.query.copy_(c.query)
    k, v = wl.read_tokens(c.pool, c.pt, 0)
    wl.write_tokens(t.pool, t.pt, 0, k[L - w - 1:], v[L - w - 1:])
    ot, lt, _ = oracle_decode(t)
    np.testing.assert_array_equal(out, ot)
    np.testing.assert_array_equal(lse, lt)
    # a window covering everything equals no window
    for wl_ in (L - 1, L + 5):
        c.window_left = wl_
        np.testing.assert_array_equal(oracle_decode(c)[0], oracle_decode(
            _replace(c, window_left=-1))[0])


def _replace(c, **kw):
    import dataclasses
    return dataclasses.replace(c, **kw)


def test_decode_multi_token_matches_prefill_and_single_tokens():
    Q, lengths = 3, [9, 14]
    c = _small_decode(lengths, q_len_per_req=Q)
    out, lse, err = oracle_decode(c)
    assert err == 0
    # causal prefill with q_len = Q over the same pages
    p = wl.PrefillCase(c.query, c.pool, c.pt, c.block_tables,
                       torch.tensor([Q] * 2, dtype=torch.int32), c.seq_lens,
                       Q, max(lengths), c.bmm1_scale, True, c.num_qo_heads,
                       c.num_kv_heads, c.head_dim, c.head_dim, c.dtype)
    po, pl, _ = oracle_prefill(p)
    np.testing.assert_allclose(out, po, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, pl, rtol=0, atol=1e-14)
    # token t alone sees the first L - Q + t + 1 keys
    for b, L in enumerate(lengths):
        for t in range(Q):
            s = _replace(c, query=c.query[b * Q + t:b * Q + t + 1], q_len_per_req=1,
                         seq_lens=torch.tensor([L - Q + t + 1], dtype=torch.int32),
                         block_tables=c.block_tables[b:b + 1])
            so, sl, _ = oracle_decode(s)
            np.testing.assert_array_equal(so[0], out[b * Q + t])
            np.testing.assert_array_equal(sl[0], lse[b * Q + t])


def test_decode_varlen_with_equal_lengths_is_uniform():
    # cum_seq_lens_q with every request at Q tokens is the uniform layout
    fixed = _small_decode([9, 14, 6], q_len_per_req=2)
    var = _replace(fixed, cum_seq_lens_q=torch.tensor([0, 2, 4, 6], dtype=torch.int32))
    a, b = oracle_decode(fixed), oracle_decode(var)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_decode_varlen_rows_follow_their_request():
    # request b's rows are its Q_b last tokens, exactly as a lone request
    # with q_len_per_req = Q_b would give them; an empty request has no rows
    q_lens, lengths = [3, 0, 1, 2], [9, 5, 14, 7]
    c = _small_decode(lengths, q_lens=q_lens, window_left=4, with_sinks=True)
    out, lse, err = oracle_decode(c)
    assert err == 0 and out.shape[0] == sum(q_lens)
    cum = c.cum_seq_lens_q.tolist()
    for b, (Q, L) in enumerate(zip(q_lens, lengths)):
        if Q == 0:
            continue
        s = _replace(c, query=c.query[cum[b]:cum[b + 1]], q_len_per_req=Q, cum_seq_lens_q=None,
                     seq_lens=torch.tensor([L], dtype=torch.int32),
                     block_tables=c.block_tables[b:b + 1])
        so, sl, _ = oracle_decode(s)
        np.testing.assert_array_equal(so, out[cum[b]:cum[b + 1]])
        np.testing.assert_array_equal(sl, lse[cum[b]:cum[b + 1]])


def test_decode_varlen_matches_prefill():
    # without window and sinks, variable-length decode is causal prefill
    # with q_b = Q_b over the same pages
    q_lens, lengths = [2, 4, 1], [9, 14, 5]
    c = _small_decode(lengths, q_lens=q_lens)
    out, lse, err = oracle_decode(c)
    assert err == 0
    p = wl.PrefillCase(c.query, c.pool, c.pt, c.block_tables,
                       torch.tensor(q_lens, dtype=torch.int32), c.seq_lens,
                       max(q_lens), max(lengths), c.bmm1_scale, True, c.num_qo_heads,
                       c.num_kv_heads, c.head_dim, c.head_dim, c.dtype)
    po, pl, _ = oracle_prefill(p)
    np.testing.assert_allclose(out, po, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, pl, rtol=0, atol=1e-14)


def test_e4m3_codes_match_torch():
    # every 8-bit pattern decodes to torch's float8_e4m3fn value (NaN codes too)
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.widen16(codes, oracle.E4M3)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert got[0x7e] == 448.0 and got[0x01] == 2.0 ** -9  # largest normal, smallest subnormal


def test_decode_fp8_cache_equals_widened_cache():
    # every e4m3 value is a bf16 value: decode over an e4m3 cache equals decode
    # over the same values stored as bf16 (fp64 math on identical numbers)
    c8 = _small_decode([9, 14, 5], kv_dtype=wl.E4M3, with_sinks=True, window_left=6)
    wide = tuple(t.to(torch.bfloat16) for t in c8.pool.storage)
    p16 = dataclasses.replace(c8.pool, storage=wide, k=wide[0][:, 0], v=wide[0][:, 1])
    c16 = _replace(c8, pool=p16, kv_dtype=None)
    a, b = oracle_decode(c8), oracle_decode(c16)
    assert a[2] == 0
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_append_fp8_places_bytes():
    # 8-bit elements: every appended byte lands at its page slot, nothing else moves
    c = wl.append_case([3, 5], [2, 7], 4, 2, 16, wl.NHD, wl.E4M3, seed=7, slack=0.5)
    before = c.pool.storage[0].clone()
    sl = oracle.seq_lens(c.kv_indptr.numpy(), c.kv_last_page_len.numpy(), 4)
    bi, pos = oracle.batch_indices_positions(c.append_indptr.numpy(), sl, c.append_key.shape[0])
    assert oracle_append(c, bi, pos) == 0
    for i in range(len(bi)):
        b, p = int(bi[i]), int(pos[i])
        page = int(c.kv_indices[int(c.kv_indptr[b]) + p // 4])
        assert torch.equal(c.pool.k[page, p % 4].view(torch.uint8), c.append_key[i].view(torch.uint8))
        assert torch.equal(c.pool.v[page, p % 4].view(torch.uint8), c.append_value[i].view(torch.uint8))
    changed = (c.pool.storage[0].view(torch.uint8) != before.view(torch.uint8)).any(-1).any(-1)
    assert int(changed.sum()) <= 2 * len(bi)


def test_decode_split_merge_recombines():
    L = 24  # 6 pages of 4
    c = _small_decode([L])
    out, lse, _ = oracle_decode(c)
    k, v = wl.read_tokens(c.pool, c.pt, 0)
    parts = [(0, 8), (8, 12), (12, 24)]
    po, pl = [], []
    for lo, hi in parts:
        t = _small_decode([hi - lo], seed=14)
        t.query.copy_(c.query)
        wl.write_tokens(t.pool, t.pt, 0, k[lo:hi], v[lo:hi])
        o_, l_, _ = oracle_decode(t)
        po.append(o_[0]); pl.append(l_[0])
    for h in range(c.num_qo_heads):
        mo, ml = oracle.merge(np.stack([x[h] for x in po]), np.array([x[h] for x in pl]))
        np.testing.assert_allclose(mo, out[0, h], rtol=1e-12, atol=1e-14)
        assert abs(ml - lse[0, h]) < 1e-12
    # an empty part carries no weight
    mo, ml = oracle.merge(np.stack([po[0][0], np.zeros_like(po[0][0])]),
                          np.array([pl[0][0], -np.inf]))
    np.testing.assert_array_equal(mo, po[0][0]); assert ml == pl[0][0]


def test_decode_bmm2_linear():
    c = _small_decode([12, 5], bmm2_scale=1.0)
    o1, l1, _ = oracle_decode(c)
    c.bmm2_scale = 2.5
    o2, l2, _ = oracle_decode(c)
    np.testing.assert_allclose(o2, 2.5 * o1, rtol=1e-15, atol=0)
    np.testing.assert_array_equal(l1, l2)


def test_decode_empty_and_short():
    c = _small_decode([0, 5], with_sinks=True, q_len_per_req=2)
    out, lse, err = oracle_decode(c)
    assert err & oracle.E_QLEN  # request 0 holds fewer keys than query tokens
    assert np.all(out[0:2] == 0)
    np.testing.assert_array_equal(lse[0:2], np.broadcast_to(c.sinks.double().numpy(), (2, 4)))
    c.sinks = None
    out, lse, _ = oracle_decode(c)
    assert np.all(out[0:2] == 0) and np.all(np.isneginf(lse[0:2]))
    assert np.all(np.isfinite(out[2:]))


def test_decode_bad_page_flagged():
    c = _small_decode([10])
    c.block_tables[0, 1] = c.pool.num_pages
    assert oracle_decode(c)[2] & oracle.E_PAGE


def test_decode_never_reads_past_length():
    c = _small_decode([6, 3], fill="nan", bt_width=8)
    for b, L in enumerate([6, 3]):
        kv = wl.randn((L, 2, 16), torch.bfloat16, wl.generator(b))
        wl.write_tokens(c.pool, c.pt, b, kv, kv)
    out, lse, err = oracle_decode(c)
    assert err == 0 and np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


# ---- prefill ---------------------------------------------------------------------------

def _small_prefill(q_lens, kv_lens, **kw):
    args = dict(page_size=4, num_qo_heads=4, num_kv_heads=2, d_qk=16, d_vo=16,
                layout=wl.HND, seed=21)
    args.update(kw)
    return wl.prefill_case(q_lens, kv_lens, **args)


def _dense_prefill_kv(c, b):
    k, v = wl.read_tokens(c.pool, c.pt, b)
    g = c.num_qo_heads // c.num_kv_heads
    return expand_heads(k, g), expand_heads(v, g)


@pytest.mark.parametrize("d_qk,d_vo", [(16, 16), (24, 16)])
def test_prefill_square_causal_matches_library(d_qk, d_vo):
    lens = [7, 1, 12]
    c = _small_prefill(lens, lens, d_qk=d_qk, d_vo=d_vo)
    out, lse, err = oracle_prefill(c)
    assert err == 0
    off = 0
    for b, n in enumerate(lens):
        k, v = _dense_prefill_kv(c, b)
        q = c.q[off:off + n]
        ref = sdpa64(q, k, v, c.scale, causal=True)
        np.testing.assert_allclose(out[off:off + n], ref.numpy(), rtol=1e-12, atol=1e-13)
        # row i: logsumexp over keys 0..i
        for i in range(n):
            np.testing.assert_allclose(lse[off + i], logsumexp64(q[i:i + 1], k[:i + 1],
                                       c.scale)[0].numpy(), rtol=1e-12, atol=1e-13)
        off += n


def test_prefill_with_prefix_is_bottom_right_causal():
    q_lens, kv_lens = [3, 5], [10, 5]
    c = _small_prefill(q_lens, kv_lens)
    out, lse, _ = oracle_prefill(c)
    off = 0
    for b, (nq, nk) in enumerate(zip(q_lens, kv_lens)):
        k, v = _dense_prefill_kv(c, b)
        for i in range(nq):
            vis = nk - nq + i + 1
            ref = sdpa64(c.q[off + i:off + i + 1], k[:vis], v[:vis], c.scale)
            np.testing.assert_allclose(out[off + i], ref[0].numpy(), rtol=1e-12, atol=1e-13)
        off += nq


def test_prefill_noncausal_matches_library():
    q_lens, kv_lens = [4, 6], [9, 6]
    c = _small_prefill(q_lens, kv_lens, causal=False)
    out, lse, _ = oracle_prefill(c)
    off = 0
    for b, n in enumerate(q_lens):
        k, v = _dense_prefill_kv(c, b)
        ref = sdpa64(c.q[off:off + n], k, v, c.scale)
        np.testing.assert_allclose(out[off:off + n], ref.numpy(), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[off:off + n], logsumexp64(c.q[off:off + n], k,
                                   c.scale).numpy(), rtol=1e-12, atol=1e-13)
        off += n


FP8_PREFILL = [
    # (q stored as, caches stored as)
    (wl.E4M3, wl.E4M3),
    (None, wl.E4M3),
    (wl.E4M3, None),
]


@pytest.mark.parametrize("qd,kvd", FP8_PREFILL, ids=["q8_kv8", "q16_kv8", "q8_kv16"])
def test_prefill_fp8_equals_rescaled_16bit(qd, kvd):
    # Powers of two keep (stored value x scale) an exact bf16 value, so the
    # FP8 prefill must equal the 16-bit prefill over the rescaled tensors,
    # decoded by torch's float8 type (not the oracle's decoder)
    qs, ks, vs = 2.0, 0.25, 0.5
    c8 = _small_prefill([7, 3], [9, 3], q_dtype=qd, kv_dtype=kvd, q_scale=qs if qd else 1.0,
                        k_scale=ks if kvd else 1.0, v_scale=vs if kvd else 1.0)

    def rescale(t, f):
        return (t.to(torch.float64) * f).to(torch.bfloat16)

    q16 = rescale(c8.q, c8.q_scale)
    k16, v16 = rescale(c8.pool.k, c8.k_scale), rescale(c8.pool.v, c8.v_scale)
    assert torch.equal(q16.double(), c8.q.double() * c8.q_scale)  # exact
    p16 = dataclasses.replace(c8.pool, storage=(k16, v16), k=k16, v=v16)
    c16 = dataclasses.replace(c8, q=q16, pool=p16, q_dtype=None, kv_dtype=None, q_scale=1.0,
                              k_scale=1.0, v_scale=1.0)
    a, b = oracle_prefill(c8), oracle_prefill(c16)
    assert a[2] == b[2] == 0
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("d_qk,d_vo", [(16, 16), (24, 16)])
def test_prefill_fp8_scales_match_library(d_qk, d_vo):
    # arbitrary scales: q_scale and k_scale multiply the logits, v_scale the
    # output; against library attention on torch-dequantised tensors
    q_lens, kv_lens = [5, 4], [8, 4]
    c = _small_prefill(q_lens, kv_lens, q_dtype=wl.E4M3, kv_dtype=wl.E4M3, q_scale=0.37,
                       k_scale=1.9, v_scale=0.61, d_qk=d_qk, d_vo=d_vo)
    out, lse, err = oracle_prefill(c)
    assert err == 0
    off = 0
    for b, (nq, nk) in enumerate(zip(q_lens, kv_lens)):
        k, v = wl.read_tokens(c.pool, c.pt, b)
        g = c.num_qo_heads // c.num_kv_heads
        q = c.q[off:off + nq].double() * c.q_scale
        k = expand_heads(k.double() * c.k_scale, g)
        v = expand_heads(v.double() * c.v_scale, g)
        for i in range(nq):
            vis = nk - nq + i + 1
            ref = sdpa64(q[i:i + 1], k[:vis], v[:vis], c.scale)
            np.testing.assert_allclose(out[off + i], ref[0].numpy(), rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse[off + i], logsumexp64(q[i:i + 1], k[:vis], c.scale)[0].numpy(),
                                       rtol=1e-12, atol=1e-13)
        off += nq


def test_prefill_causal_ignores_later_keys():
    c = _small_prefill([6], [6])
    out, lse, _ = oracle_prefill(c)
    k, v = wl.read_tokens(c.pool, c.pt, 0)
    k2, v2 = k.clone(), v.clone()
    k2[4:] = -k2[4:] * 3
    v2[4:] = v2[4:] + 5
    wl.write_tokens(c.pool, c.pt, 0, k2, v2)
    out2, lse2, _ = oracle_prefill(c)
    np.testing.assert_array_equal(out[:4], out2[:4])
    np.testing.assert_array_equal(lse[:4], lse2[:4])
    assert not np.allclose(out[4:], out2[4:])


def test_prefill_first_row_single_key_and_uniform():
    c = _small_prefill([5], [5])
    out, lse, _ = oracle_prefill(c)
    k, v = _dense_prefill_kv(c, 0)
    np.testing.assert_allclose(out[0], v[0].double().numpy(), rtol=0, atol=1e-15)
    s = (c.q[0].double() * k[0].double()).sum(-1) * c.scale
    np.testing.assert_allclose(lse[0], s.numpy(), rtol=1e-13, atol=1e-13)
    c.q.zero_()  # q = 0: uniform weights over the visible keys
    out, lse, _ = oracle_prefill(c)
    for i in range(5):
        np.testing.assert_allclose(out[i], v[:i + 1].double().mean(0).numpy(), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[i], math.log(i + 1), rtol=0, atol=1e-14)


def test_prefill_gqa_and_page_permutation():
    c = _small_prefill([5, 8], [9, 8], num_qo_heads=8, num_kv_heads=2)
    r = _small_prefill([5, 8], [9, 8], num_qo_heads=8, num_kv_heads=8, seed=33)
    r.q.copy_(c.q)
    for b in range(2):
        k, v = wl.read_tokens(c.pool, c.pt, b)
        wl.write_tokens(r.pool, r.pt, b, expand_heads(k, 4), expand_heads(v, 4))
    assert c.pt.pages != r.pt.pages
    oc, lc, _ = oracle_prefill(c)
    orr, lr, _ = oracle_prefill(r)
    np.testing.assert_array_equal(oc, orr)
    np.testing.assert_array_equal(lc, lr)


def test_prefill_short_kv_flagged():
    c = _small_prefill([4], [2])
    out, lse, err = oracle_prefill(c)
    assert err & oracle.E_QLEN
    assert np.all(out[:2] == 0) and np.all(np.isneginf(lse[:2]))
