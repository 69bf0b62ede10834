"""The algorithmic work behind every roofline fraction the benchmark
reports, checked against counts made directly from the definitions:
keys visible to some query row (decode), unmasked (query, key) pairs
(prefill), bytes moved per appended token (append)."""
from __future__ import annotations

import bench
from paged_kv_cache_316_gb300 import workloads as wl


def _visible_keys(L, Q, window_left):
    """Keys some query token of the request attends to, by brute force."""
    seen = set()
    for t in range(Q):
        p = L - Q + t
        lo = 0 if window_left < 0 else max(0, p - window_left)
        seen.update(range(lo, p + 1))
    return seen


def test_decode_bytes_count_visible_keys_once():
    for window in (-1, 3, 0):
        c = wl.decode_case([10, 3, 17], 4, 4, 2, 128, wl.HND, q_len_per_req=2, window_left=window, seed=1)
        keys = [_visible_keys(L, 2, window) for L in c.pt.lengths]
        kv_tok = sum(len(k) for k in keys)
        pages = sum(len({j // 4 for j in k}) for k in keys)
        row = 2 * 128 * 2                      # kv heads x head_dim x 2 bytes
        q_and_out = 2 * (3 * 2 * 4 * 128) * 2  # query rows read + output rows written
        expect = kv_tok * row * 2 + q_and_out + pages * 4 + 3 * 4
        assert bench.decode_bytes(c) == expect, window


def test_decode_bytes_of_an_e4m3_cache_count_one_byte_per_element():
    a = wl.decode_case([40, 9], 8, 8, 2, 128, wl.HND, seed=2)
    b = wl.decode_case([40, 9], 8, 8, 2, 128, wl.HND, seed=2, kv_dtype=wl.E4M3)
    kv = (40 + 9) * 2 * 128 * 2  # K and V bytes at 1 byte per element
    assert bench.decode_bytes(a) - bench.decode_bytes(b) == kv


def test_append_bytes():
    c = wl.append_case([3, 5], [2, 0], 16, 4, 128, wl.NHD, seed=3)
    nnz = 8
    # K and V rows read from the inputs and written to the pages, plus
    # batch index and position of every entry
    assert bench.append_bytes(c) == nnz * (2 * 2 * 4 * 128 * 2 + 8)


def test_prefill_flops_count_unmasked_pairs():
    for causal in (True, False):
        c = wl.prefill_case([5, 3, 1], [9, 3, 4], 4, 8, 2, 192, 128, wl.HND, causal=causal, seed=4)
        pairs = 0
        for q, kv in zip([5, 3, 1], [9, 3, 4]):
            for i in range(q):
                last = kv - q + i if causal else kv - 1
                pairs += sum(1 for j in range(kv) if j <= last)
        # QK^T and PV: 2 FLOP per multiply-add, d_qk + d_vo of them per pair and head
        assert bench.prefill_flops(c) == 2 * (192 + 128) * 8 * pairs, causal
