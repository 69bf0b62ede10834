"""GPU parity for causal ragged paged prefill against the fp64 oracle:
outputs within |err| <= 2e-2 + 1e-2 |ref|, LSE within 1e-3."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_316_gb300 as pk
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
    ([0, 300, 0, 17], [40, 1000, 0, 17], 128, 8, 2, 128, True, wl.BF16, wl.NHD, 9),   # requests without queries
    ([129, 1], [2049, 1], 256, 16, 4, 128, False, wl.F16, wl.HND, 10),  # 256-slot pages, one-key request
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


def _contiguous_kv(c):
    """The case's keys and values packed request after request: [sum kv, Hkv, d]."""
    ks, vs = [], []
    for b in range(len(c.pt.lengths)):
        k, v = wl.read_tokens(c.pool, c.pt, b)
        ks.append(k)
        vs.append(v)
    return torch.cat(ks).contiguous(), torch.cat(vs).contiguous()


@pytest.mark.parametrize("dqk", [128, 192])
def test_contiguous_kv_matches_paged(dqk):
    # block_tables = None: the same logical keys and values, packed
    c = wl.prefill_case([130, 7, 300, 64], [400, 7, 300, 900], 32, 32, 8, dqk, 128, wl.HND, wl.BF16,
                        seed=41, slack=0.2)
    k, v = _contiguous_kv(c)
    B = len(c.pt.lengths)
    ws = torch.zeros(pk.paged_prefill_workspace_size(B, 32, c.max_q, c.max_kv), dtype=torch.uint8, device=DEV)
    out, lse = pk.paged_prefill(c.q.to(DEV), k.to(DEV), v.to(DEV), c.scale, ws, c.max_q, c.max_kv,
                                c.seq_lens_q.to(DEV), c.seq_lens_kv.to(DEV), None, causal=True)
    torch.cuda.synchronize()
    ro, rl, _ = oracle_prefill(c)
    assert_attn_close(out, ro)
    assert_lse_close(lse, rl)


def test_batch_offsets_place_rows():
    # every request's queries, outputs, keys and values at shuffled row
    # offsets with gaps between them (contiguous K/V)
    ql, kvl = [130, 7, 300], [400, 7, 900]
    c = wl.prefill_case(ql, kvl, 32, 16, 4, 128, 128, wl.HND, wl.BF16, seed=42, slack=0.2, causal=True)
    k, v = _contiguous_kv(c)
    g = torch.Generator().manual_seed(5)
    B, H, Hk = 3, 16, 4

    def scatter(lens, gap):
        order = torch.randperm(B, generator=g).tolist()
        offs, at = [0] * B, gap
        for b in order:
            offs[b] = at
            at += lens[b] + gap
        return offs, at

    oq, nq = scatter(ql, 5)
    oo, no = scatter(ql, 3)
    ok_, nk = scatter(kvl, 17)
    ov, nv = scatter(kvl, 2)
    n_rows = max(nq, no)
    cu_q = [0] + list(np.cumsum(ql))
    cu_kv = [0] + list(np.cumsum(kvl))
    qx = torch.zeros((n_rows, H, 128), dtype=c.q.dtype)
    kx = torch.full((nk, Hk, 128), float("nan"), dtype=k.dtype)
    vx = torch.full((nv, Hk, 128), float("nan"), dtype=v.dtype)
    for b in range(B):
        qx[oq[b]:oq[b] + ql[b]] = c.q[cu_q[b]:cu_q[b + 1]]
        kx[ok_[b]:ok_[b] + kvl[b]] = k[cu_kv[b]:cu_kv[b + 1]]
        vx[ov[b]:ov[b] + kvl[b]] = v[cu_kv[b]:cu_kv[b + 1]]
    ws = torch.zeros(pk.paged_prefill_workspace_size(B, H, c.max_q, c.max_kv), dtype=torch.uint8, device=DEV)
    out = torch.full((n_rows, H, 128), 3.0, dtype=c.q.dtype, device=DEV)
    lse = torch.full((n_rows, H), 3.0, dtype=torch.float32, device=DEV)
    offs = [torch.tensor(o, dtype=torch.int32, device=DEV) for o in (oq, oo, ok_, ov)]
    pk.paged_prefill(qx.to(DEV), kx.to(DEV), vx.to(DEV), c.scale, ws, c.max_q, c.max_kv,
                     c.seq_lens_q.to(DEV), c.seq_lens_kv.to(DEV), None, causal=True, out=out, lse=lse,
                     batch_offsets_q=offs[0], batch_offsets_o=offs[1], batch_offsets_k=offs[2],
                     batch_offsets_v=offs[3])
    torch.cuda.synchronize()
    ro, rl, _ = oracle_prefill(c)
    written = torch.zeros(n_rows, dtype=torch.bool)
    for b in range(B):
        rows = slice(oo[b], oo[b] + ql[b])
        assert_attn_close(out[rows], ro[cu_q[b]:cu_q[b + 1]], f"request {b}")
        assert_lse_close(lse[rows], rl[cu_q[b]:cu_q[b + 1]], f"request {b} lse")
        written[rows] = True
    assert torch.all(out[~written.to(DEV)].float() == 3.0) and torch.all(lse[~written.to(DEV)] == 3.0)


FP8_CASES = [
    # q lens, kv lens, page, Hqo, Hkv, d_qk, causal, out dtype, layout, E4M3 query, E4M3 caches, seed
    ([130, 7, 64], [200, 7, 300], 32, 32, 8, 128, True, wl.BF16, wl.HND, True, True, 11),
    ([1, 255, 129], [1, 255, 700], 32, 32, 8, 192, True, wl.BF16, wl.HND, False, True, 12),
    ([300, 50], [300, 333], 16, 8, 8, 128, False, wl.F16, wl.NHD, True, False, 13),
    ([64, 200], [500, 200], 64, 16, 2, 192, False, wl.BF16, wl.NHD, True, True, 14),
    ([77, 300], [500, 300], 16, 16, 4, 192, True, wl.F16, wl.HND, True, True, 15),
    ([200], [333], 8, 6, 2, 128, True, wl.BF16, wl.HND, False, True, 16),
    # E4M3 query and caches at d_qk 128 take the kind::f8f6f4 kernel
    ([257, 33], [600, 33], 16, 16, 4, 128, True, wl.F16, wl.NHD, True, True, 20),
    ([129], [129], 64, 8, 2, 128, False, wl.BF16, wl.HND, True, True, 21),
    ([1, 700, 64], [1, 1300, 64], 256, 6, 2, 128, True, wl.BF16, wl.NHD, True, True, 22),   # odd group
]


@pytest.mark.parametrize("case", FP8_CASES, ids=[f"f{i}" for i in range(len(FP8_CASES))])
def test_fp8_small_shapes(case):
    lq, lkv, S, hq, hk, dqk, causal, dt, lay, q8, kv8, seed = case
    c = wl.prefill_case(lq, lkv, S, hq, hk, dqk, 128, lay, dt, causal=causal, seed=seed, slack=0.2,
                        q_dtype=wl.E4M3 if q8 else None, kv_dtype=wl.E4M3 if kv8 else None,
                        q_scale=0.37 if q8 else 1.0, k_scale=1.9 if kv8 else 1.0,
                        v_scale=0.61 if kv8 else 1.0)
    _check(c)


@pytest.mark.parametrize("scale", [-0.07, 0.0], ids=["negative", "zero"])
@pytest.mark.parametrize("dqk", [128, 192])
def test_non_positive_logit_scale(scale, dqk):
    # the softmax takes the row max after scaling when the scale is not
    # positive (a positive one is applied after the max of the raw scores);
    # zero gives every visible key the same weight
    c = wl.prefill_case([300, 90], [700, 90], 32, 16, 4, dqk, 128, wl.HND, wl.BF16, causal=True,
                        seed=31 + dqk, scale=scale, slack=0.2)
    _check(c)
    if dqk == 128:  # and on the E4M3 kernel
        c8 = wl.prefill_case([300, 90], [700, 90], 32, 16, 4, 128, 128, wl.NHD, wl.BF16, causal=True,
                             seed=33, scale=scale, slack=0.2, q_dtype=wl.E4M3, kv_dtype=wl.E4M3,
                             k_scale=1.5)
        _check(c8)


def test_fp8_with_unit_scales_equals_16bit_on_widened_values():
    # every E4M3 value is a bf16 value: where the E4M3 inputs are widened to
    # 16 bits first (d_qk 192), the E4M3 prefill with unit scales gives bit
    # for bit the 16-bit prefill over the same values
    c8 = wl.prefill_case([130, 7, 300], [400, 7, 300], 32, 32, 8, 192, 128, wl.HND, wl.BF16, seed=17,
                         slack=0.2, q_dtype=wl.E4M3, kv_dtype=wl.E4M3)
    o8, l8 = prefill_on_gpu(c8)
    k16, v16 = c8.pool.k.to(torch.bfloat16), c8.pool.v.to(torch.bfloat16)
    c16 = dataclasses.replace(c8, q=c8.q.to(torch.bfloat16), q_dtype=None, kv_dtype=None,
                              pool=dataclasses.replace(c8.pool, storage=(k16, v16), k=k16, v=v16))
    o16, l16 = prefill_on_gpu(c16)
    assert torch.equal(o8.view(torch.int16), o16.view(torch.int16))
    assert torch.equal(l8, l16)


def test_fp8_bad_page_flagged():
    c = wl.prefill_case([40], [100], 16, 8, 2, 128, 128, wl.HND, wl.BF16, seed=18, slack=0.5,
                        q_dtype=wl.E4M3, kv_dtype=wl.E4M3)
    c.block_tables[0, 2] = c.pool.num_pages + 5
    err = err_word()
    prefill_on_gpu(c, err_word=err)
    assert int(err.item()) & oracle.E_PAGE


def test_fp8_ragged_config_full_size_sampled():
    c = wl.ragged_prefill(d_qk=128, device=DEV, q_dtype=wl.E4M3, kv_dtype=wl.E4M3, q_scale=0.5,
                          k_scale=1.25, v_scale=0.8)
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



@pytest.mark.parametrize("d_qk", [128, 192])
def test_max_jumps_within_a_tile(d_qk):
    # keys 64..127 of every 128 (and 48..95 of every 96) score ~8x higher:
    # the running max jumps by far more than 2^8 inside a tile, which
    # exercises the late raise of the max (and the rescale of P already
    # written for the tile's first columns)
    c = wl.prefill_case([200, 130], [450, 300], 32, 8, 2, d_qk, 128, wl.HND, wl.BF16, seed=19, slack=0.1)
    for b in range(2):
        k, v = wl.read_tokens(c.pool, c.pt, b)
        j = torch.arange(k.shape[0])
        tile = 128 if d_qk == 128 else 96
        f = torch.where((j % tile) >= tile // 2, 8.0, 1.0).to(torch.float32)
        k2 = (k.float() * f[:, None, None]).to(k.dtype)
        wl.write_tokens(c.pool, c.pt, b, k2, v)
    _check(c)
