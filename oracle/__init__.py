"""fp64 CPU oracle for paged-KV attention -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never touches it, and this package never touches the product:
the C source next to this file has its own decoders, enums and address
arithmetic, written from the three FlashInfer API pages
(``flashinfer.page.append_paged_kv_cache``,
``flashinfer.decode.trtllm_batch_decode_with_kv_cache``,
``flashinfer.prefill.cudnn_batch_prefill_with_kv_cache``).

The wrappers below only marshal numpy arrays into the C functions; every
step of the arithmetic is in ``pagedkv_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

NHD, HND = 0, 1
FP16, BF16, E4M3 = 0, 1, 2  # E4M3: 8-bit cache elements (OCP FP8)
E_PAGE, E_POS, E_BATCH, E_QLEN = 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when the compiler has it)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB lets the mutation test load a deliberately broken build
        _lib = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
        _lib.orc_has_openmp.restype = ctypes.c_int
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def _u16(a) -> np.ndarray:
    """16-bit float payload as a contiguous uint16 array (bits unchanged)."""
    a = np.ascontiguousarray(a)
    assert a.dtype.itemsize == 2, a.dtype
    return a.view(np.uint16)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _check_pool(arr, page_stride: int, num_pages: int):
    """The C code addresses page p at p * page_stride elements from the
    array's first element: refuse views whose layout says otherwise."""
    assert arr.dtype in (np.uint16, np.uint8), "pass uint16 (or, for e4m3, uint8) views of the pool"
    assert arr.ndim >= 2 and arr.shape[0] >= num_pages, (arr.shape, num_pages)
    assert arr.strides[0] == arr.dtype.itemsize * page_stride, (arr.strides, page_stride)
    assert arr[0].size <= page_stride and arr[0].flags.c_contiguous, "pages must be contiguous"


def max_threads() -> int:
    """OpenMP threads the oracle can use (1 when built without OpenMP)."""
    return max(1, _load().orc_has_openmp())


def seq_lens(kv_indptr, kv_last_page_len, page_size: int) -> np.ndarray:
    kv_indptr, last = _i32(kv_indptr), _i32(kv_last_page_len)
    B = last.shape[0]
    out = np.zeros(B, np.int32)
    _load().orc_seq_lens(_p(kv_indptr), _p(last), ctypes.c_int(B),
                         ctypes.c_int(page_size), _p(out))
    return out


def batch_indices_positions(append_indptr, seq_lens_, nnz: int):
    ind, sl = _i32(append_indptr), _i32(seq_lens_)
    B = sl.shape[0]
    bi = np.zeros(nnz, np.int32)
    pos = np.zeros(nnz, np.int32)
    _load().orc_batch_indices_positions(_p(ind), _p(sl), ctypes.c_int(B),
                                        ctypes.c_int64(nnz), _p(bi), _p(pos))
    return bi, pos


def append(append_key, append_value, batch_indices, positions, k_cache, v_cache,
           page_stride: int, max_num_pages: int, kv_indices, kv_indptr,
           kv_last_page_len, num_kv_heads: int, head_dim: int, page_size: int,
           layout: int) -> int:
    """Scatter in place into ``k_cache``/``v_cache`` (uint16 views of the
    pool, or uint8 for 8-bit elements; for the 5-D pool these are two views
    into one buffer).  Returns the error mask."""
    eb = k_cache.dtype.itemsize
    if eb == 1:
        ak = np.ascontiguousarray(append_key).view(np.uint8)
        av = np.ascontiguousarray(append_value).view(np.uint8)
    else:
        ak, av = _u16(append_key), _u16(append_value)
    bi, pos = _i32(batch_indices), _i32(positions)
    ind, ptr, last = _i32(kv_indices), _i32(kv_indptr), _i32(kv_last_page_len)
    for c in (k_cache, v_cache):
        _check_pool(c, page_stride, max_num_pages)
    return int(_load().orc_append(
        _p(ak), _p(av), ctypes.c_int64(bi.shape[0]), _p(bi), _p(pos),
        ctypes.c_void_p(k_cache.ctypes.data), ctypes.c_void_p(v_cache.ctypes.data),
        ctypes.c_int64(page_stride), ctypes.c_int64(max_num_pages), _p(ind),
        _p(ptr), _p(last), ctypes.c_int(last.shape[0]), ctypes.c_int(num_kv_heads),
        ctypes.c_int(head_dim), ctypes.c_int(page_size), ctypes.c_int(layout),
        ctypes.c_int(eb)))


def decode(query, k_cache, v_cache, page_stride: int, max_num_pages: int,
           block_tables, seq_lens_, max_seq_len: int, bmm1_scale: float,
           bmm2_scale: float, window_left: int, sinks, q_len_per_req: int,
           num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
           layout: int, dtype: int, threads: int | None = None, cum_seq_lens_q=None,
           kv_dtype: int | None = None):
    """Returns (out [rows, Hqo, D] float64, lse [rows, Hqo] float64, err) with
    rows = B*Q, or cum_seq_lens_q[B] for variable-length queries (request b
    then has rows cum[b] .. cum[b+1]-1 and q_len_per_req is unused)."""
    q = _u16(query)
    kc, vc = k_cache, v_cache
    _check_pool(kc, page_stride, max_num_pages)
    _check_pool(vc, page_stride, max_num_pages)
    bt = _i32(block_tables)
    sl = np.ascontiguousarray(np.asarray(seq_lens_), dtype=np.uint32)
    B = sl.shape[0]
    cq = None if cum_seq_lens_q is None else _i32(cum_seq_lens_q)
    if cq is not None:
        assert cq.shape == (B + 1,) and cq[0] == 0 and np.all(np.diff(cq) >= 0)
    rows = B * q_len_per_req if cq is None else int(cq[-1])
    kvd = dtype if kv_dtype is None else kv_dtype  # E4M3: uint8 views of the caches
    out = np.zeros((rows, num_qo_heads, head_dim), np.float64)
    lse = np.zeros((rows, num_qo_heads), np.float64)
    sk = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float32)
    nthr = threads or max_threads()
    # scratch holds one logit per key of a row; size it from the real lengths
    max_seq_len = max(int(max_seq_len), int(sl.max()) if B else 0)
    scratch = np.zeros(nthr * (max_seq_len + 1), np.float64)
    err = _load().orc_decode(
        _p(q), ctypes.c_void_p(kc.ctypes.data), ctypes.c_void_p(vc.ctypes.data),
        ctypes.c_int64(page_stride), ctypes.c_int64(max_num_pages), _p(bt),
        ctypes.c_int(bt.shape[1]), _p(sl), ctypes.c_int(B), ctypes.c_int(max_seq_len),
        ctypes.c_double(bmm1_scale), ctypes.c_double(bmm2_scale),
        ctypes.c_int(window_left), _p(sk), ctypes.c_int(q_len_per_req), _p(cq),
        ctypes.c_int(num_qo_heads), ctypes.c_int(num_kv_heads),
        ctypes.c_int(head_dim), ctypes.c_int(page_size), ctypes.c_int(layout),
        ctypes.c_int(dtype), ctypes.c_int(kvd), _p(out), _p(lse), _p(scratch), ctypes.c_int(nthr),
        ctypes.c_int(nthr))
    return out, lse, int(err)


def prefill(q, k_cache, v_cache, k_page_stride: int, v_page_stride: int,
            max_num_pages: int, scale: float, seq_lens_q, seq_lens_kv,
            block_tables, causal: bool, num_qo_heads: int, num_kv_heads: int,
            d_qk: int, d_vo: int, page_size: int, layout: int, dtype: int,
            threads: int | None = None, q_dtype: int | None = None,
            kv_dtype: int | None = None, q_scale: float = 1.0, k_scale: float = 1.0,
            v_scale: float = 1.0):
    """Returns (out [total_q, Hqo, d_vo], lse [total_q, Hqo], err), float64.
    q_dtype / kv_dtype (default `dtype`) may be E4M3, with uint8 arrays;
    q_scale, k_scale, v_scale dequantise the stored elements."""
    qd = dtype if q_dtype is None else q_dtype
    kvd = dtype if kv_dtype is None else kv_dtype
    qq = np.ascontiguousarray(q).view(np.uint8) if qd == E4M3 else _u16(q)
    lq, lkv = _i32(seq_lens_q), _i32(seq_lens_kv)
    _check_pool(k_cache, k_page_stride, max_num_pages)
    _check_pool(v_cache, v_page_stride, max_num_pages)
    bt = _i32(block_tables)
    B = lq.shape[0]
    total_q = int(lq.sum())
    out = np.zeros((total_q, num_qo_heads, d_vo), np.float64)
    lse = np.zeros((total_q, num_qo_heads), np.float64)
    nthr = threads or max_threads()
    slen = int(lkv.max()) + 1 if B else 1
    scratch = np.zeros(nthr * slen, np.float64)
    err = _load().orc_prefill(
        _p(qq), ctypes.c_void_p(k_cache.ctypes.data),
        ctypes.c_void_p(v_cache.ctypes.data), ctypes.c_int64(k_page_stride),
        ctypes.c_int64(v_page_stride), ctypes.c_int64(max_num_pages),
        ctypes.c_double(scale), _p(lq), _p(lkv), _p(bt), ctypes.c_int(bt.shape[1]),
        ctypes.c_int(B), ctypes.c_int(int(causal)), ctypes.c_int(num_qo_heads),
        ctypes.c_int(num_kv_heads), ctypes.c_int(d_qk), ctypes.c_int(d_vo),
        ctypes.c_int(page_size), ctypes.c_int(layout), ctypes.c_int(qd), ctypes.c_int(kvd),
        ctypes.c_double(q_scale), ctypes.c_double(k_scale), ctypes.c_double(v_scale),
        _p(out), _p(lse), _p(scratch), ctypes.c_int(slen), ctypes.c_int(nthr),
        ctypes.c_int(nthr))
    return out, lse, int(err)


def widen16(bits, dtype: int) -> np.ndarray:
    """Exact float64 value of each 16-bit pattern (fp16 or bf16), or of each
    8-bit pattern for E4M3."""
    b = np.ascontiguousarray(bits, dtype=np.uint8 if dtype == E4M3 else np.uint16)
    out = np.zeros(b.shape, np.float64)
    _load().orc_widen16(_p(b), ctypes.c_int64(b.size), ctypes.c_int(dtype), _p(out))
    return out


def merge(o_parts, lse_parts):
    """Combine partial (o_i, lse_i) over disjoint key sets."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, dim = o_parts.shape
    o = np.zeros(dim, np.float64)
    lse = np.zeros(1, np.float64)
    _load().orc_merge(_p(o_parts), _p(lse_parts), ctypes.c_int(n),
                      ctypes.c_int(dim), _p(o), _p(lse))
    return o, float(lse[0])
