"""Thin Python binding of libpagedkv.so (``include/pagedkv.h``).

Argument marshalling only: every function derives sizes and strides from
torch tensor shapes, passes device pointers and the current CUDA stream to
the C entry point of the same name, and raises on a non-zero status.  No
step of the computation happens here, and there is no CPU fallback: when the
library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

NHD, HND = 0, 1
F16, BF16, E4M3, F16_E4M3, BF16_E4M3 = 0, 1, 2, 3, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libpagedkv.so"
_lib = None

_c_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

_SIGNATURES = {
    "pkv_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "pkv_kernel_launches": ([], ctypes.c_ulonglong),
    "pkv_debug_bounds": ([], ctypes.c_int),
    "pkv_set_wait_limit_ns": ([ctypes.c_ulonglong], ctypes.c_ulonglong),
    "paged_seq_lens": ([_c_p, _c_p, _i32, _i32, _c_p, _c_p], ctypes.c_int),
    "paged_batch_indices_positions": ([_c_p, _c_p, _i32, _i64, _c_p, _c_p, _c_p],
                                      ctypes.c_int),
    "paged_append": ([_c_p, _c_p, _i64, _c_p, _c_p, _c_p, _c_p, _i64, _i64, _c_p,
                      _c_p, _c_p, _i32, _i32, _i32, _i32, _i32, _i32, _c_p, _c_p],
                     ctypes.c_int),
    "paged_decode_workspace_size": ([_i32] * 8, _sz),
    "paged_decode": ([_c_p, _c_p, _c_p, _i64, _i64, _c_p, _sz, _c_p, _i32, _c_p,
                      _i32, _i32, _f32, _f32, _i32, _c_p, _i32, _i32, _i32, _i32,
                      _i32, _i32, _i32, _c_p, _c_p, _c_p, _c_p], ctypes.c_int),
    "paged_decode_varlen": ([_c_p, _i64, _c_p, _c_p, _i64, _i64, _c_p, _sz, _c_p, _i32, _c_p,
                             _i32, _i32, _f32, _f32, _i32, _c_p, _i32, _c_p, _i32, _i32, _i32,
                             _i32, _i32, _i32, _c_p, _c_p, _c_p, _c_p], ctypes.c_int),
    "paged_decode_ex": ([_c_p, _i64, _c_p, _c_p, _i64, _i64, _c_p, _sz, _c_p, _i32, _c_p,
                         _i32, _i32, _f32, _f32, _c_p, _c_p, _i32, _c_p, _i32, _c_p, _i32, _i32,
                         _i32, _i32, _i32, _i32, _i32, _c_p, _c_p, _c_p, _c_p], ctypes.c_int),
    "paged_decode_noalloc": ([_c_p, _c_p, _c_p, _i64, _i64, _c_p, _i32, _c_p, _i32, _i32,
                              _f32, _f32, _i32, _c_p, _i32, _i32, _i32, _i32, _i32, _i32,
                              _i32, _c_p, _c_p, _c_p, _c_p], ctypes.c_int),
    "paged_prefill_workspace_size": ([_i32] * 4, _sz),
    "paged_prefill": ([_c_p, _i64, _c_p, _c_p, _i64, _i64, _i64, _f32, _c_p, _sz, _i32,
                       _i32, _c_p, _c_p, _c_p, _i32, _i32, _i32, _i32, _i32, _i32,
                       _i32, _i32, _i32, _i32, _c_p, _c_p, _c_p, _c_p], ctypes.c_int),
    "paged_prefill_ex": ([_c_p, _i64, _c_p, _c_p, _i64, _i64, _i64, _f32, _c_p, _sz, _i32,
                          _i32, _c_p, _c_p, _c_p, _i32, _i32, _i32, _i32, _i32, _i32,
                          _i32, _i32, _i32, _i32, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                          _c_p], ctypes.c_int),
    "paged_prefill_fp8_workspace_size": ([_i32] * 5 + [_i64] + [_i32] * 4, _sz),
    "paged_prefill_fp8": ([_c_p, _i64, _c_p, _c_p, _i64, _i64, _i64, _f32, _c_p, _c_p, _c_p, _c_p,
                           _sz, _i32, _i32, _c_p, _c_p, _c_p, _i32, _i32, _i32, _i32, _i32, _i32,
                           _i32, _i32, _i32, _i32, _i32, _i32, _c_p, _c_p, _c_p, _c_p], ctypes.c_int),
}


class PagedKVError(RuntimeError):
    pass


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def load_library(path: str | None = None):
    """Load libpagedkv.so from the package directory (raises if missing).
    With `path`, load that build of the library instead and route every later
    call to it (e.g. the range-checking libpagedkv_debug.so; passing
    library_path() switches back)."""
    global _lib
    if _lib is None or path is not None:
        path = path or library_path()
        if not os.path.exists(path):
            raise PagedKVError(
                f"{path} is not built: run `python -m paged_kv_cache_316_gb300.build` "
                "(nvcc, sm_103a) first; there is no fallback implementation")
        lib = ctypes.CDLL(path)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def debug_bounds() -> bool:
    """True when the loaded library is the range-checking debug build."""
    return bool(load_library().pkv_debug_bounds())


def kernel_launches() -> int:
    return int(load_library().pkv_kernel_launches())


def set_wait_limit_ns(ns: int) -> int:
    """Limit of the bounded pipeline waits of later append / prefill
    launches (0: the default, one second); returns the previous limit."""
    return int(load_library().pkv_set_wait_limit_ns(int(ns)))


def _check(status: int):
    if status != 0:
        msg = load_library().pkv_status_string(status).decode()
        raise PagedKVError(f"libpagedkv status {status}: {msg}")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise PagedKVError("tensor arguments must live on a CUDA device")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float8_e4m3fn:
        return E4M3
    raise PagedKVError(f"unsupported element type {t.dtype}")


def _decode_dtype(query: torch.Tensor, cache: torch.Tensor) -> int:
    """Decode's dtype code: the query/output type, with an E4M3 cache when
    the cache holds 8-bit floats."""
    q = _dtype_code(query)
    if q not in (F16, BF16):
        raise PagedKVError(f"query must be fp16 or bf16, not {query.dtype}")
    if cache.dtype == torch.float8_e4m3fn:
        return F16_E4M3 if q == F16 else BF16_E4M3
    if cache.dtype != query.dtype:
        raise PagedKVError("the cache holds the query's type or e4m3")
    return q


def _layout_code(kv_layout) -> int:
    if kv_layout in (NHD, "NHD"):
        return NHD
    if kv_layout in (HND, "HND"):
        return HND
    raise PagedKVError(f"kv_layout must be NHD or HND, got {kv_layout!r}")


def split_cache(kv_cache, layout: int):
    """(k_ptr, v_ptr, page_stride, num_pages, num_heads, page_size, head_dim)
    for a 5-D [P, 2, ...] tensor or a (k, v) tuple of 4-D tensors."""
    if isinstance(kv_cache, (tuple, list)):
        k, v = kv_cache
        if k.shape != v.shape or k.stride(0) != v.stride(0):
            raise PagedKVError("K and V caches must have the same shape and page stride")
        base = k
        kp, vp = k.data_ptr(), v.data_ptr()
        for t in (k, v):
            if not t[0].is_contiguous():
                raise PagedKVError("each page must be contiguous")
        shape = k.shape[1:]
    else:
        if kv_cache.dim() != 5 or kv_cache.shape[1] != 2:
            raise PagedKVError("a single kv_cache tensor must be [pages, 2, ...]")
        if not kv_cache[0].is_contiguous():
            raise PagedKVError("each page must be contiguous")
        base = kv_cache
        kp = kv_cache.data_ptr()
        vp = kv_cache[:, 1].data_ptr()
        shape = kv_cache.shape[2:]
    _ptr(base)
    if layout == HND:
        H, S, D = shape
    else:
        S, H, D = shape
    return kp, vp, base.stride(0), base.shape[0], H, S, D, base


def base_dtype(kv_cache) -> torch.dtype:
    return (kv_cache[0] if isinstance(kv_cache, (tuple, list)) else kv_cache).dtype


# ---- index helpers ------------------------------------------------------------------

def paged_seq_lens(kv_indptr, kv_last_page_len, page_size: int, seq_lens=None,
                   stream=None):
    B = kv_last_page_len.shape[0]
    if seq_lens is None:
        seq_lens = torch.empty(B, dtype=torch.int32, device=kv_indptr.device)
    _check(load_library().paged_seq_lens(_ptr(kv_indptr), _ptr(kv_last_page_len), B,
                                         page_size, _ptr(seq_lens), _stream(stream)))
    return seq_lens


def paged_batch_indices_positions(append_indptr, seq_lens, nnz: int,
                                  batch_indices=None, positions=None, stream=None):
    B = seq_lens.shape[0]
    dev = append_indptr.device
    if batch_indices is None:
        batch_indices = torch.empty(nnz, dtype=torch.int32, device=dev)
    if positions is None:
        positions = torch.empty(nnz, dtype=torch.int32, device=dev)
    _check(load_library().paged_batch_indices_positions(
        _ptr(append_indptr), _ptr(seq_lens), B, nnz, _ptr(batch_indices),
        _ptr(positions), _stream(stream)))
    return batch_indices, positions


# ---- append -----------------------------------------------------------------------------

def paged_append(append_key, append_value, batch_indices, positions, paged_kv_cache,
                 kv_indices, kv_indptr, kv_last_page_len, kv_layout="NHD",
                 err_word=None, stream=None) -> None:
    layout = _layout_code(kv_layout)
    kp, vp, stride, P, H, S, D, _ = split_cache(paged_kv_cache, layout)
    nnz = append_key.shape[0]
    if not (append_key.is_contiguous() and append_value.is_contiguous()):
        raise PagedKVError("append_key/append_value must be contiguous")
    if append_value.shape != append_key.shape or tuple(append_key.shape[1:]) != (H, D):
        raise PagedKVError(f"append_key/append_value must both be [nnz, {H}, {D}]")
    if append_key.dtype != base_dtype(paged_kv_cache) or append_value.dtype != append_key.dtype:
        raise PagedKVError("append_key/append_value hold the cache's element type")
    for t in (batch_indices, positions):
        if t.dtype != torch.int32 or t.numel() < nnz:
            raise PagedKVError(f"batch_indices/positions must be int32 with >= {nnz} entries")
    _check(load_library().paged_append(
        _ptr(append_key), _ptr(append_value), nnz, _ptr(batch_indices),
        _ptr(positions), kp, vp, stride, P, _ptr(kv_indices), _ptr(kv_indptr),
        _ptr(kv_last_page_len), kv_last_page_len.shape[0], H, D, S, layout,
        _dtype_code(append_key), _ptr(err_word), _stream(stream)))


# ---- decode -------------------------------------------------------------------------------

def _scale_arg(scale, device):
    """A host float -> (value, NULL); a one-element float32 tensor on the
    query's device -> (1.0, its address)."""
    if isinstance(scale, torch.Tensor):
        if scale.dtype != torch.float32 or scale.numel() != 1 or scale.device != device:
            raise PagedKVError("a tensor scale is one float32 value on the query's device")
        return 1.0, _ptr(scale)
    return float(scale), None


def paged_decode_workspace_size(batch_size, q_len_per_req, num_qo_heads, num_kv_heads,
                                head_dim, max_seq_len, page_size, window_left=-1) -> int:
    return int(load_library().paged_decode_workspace_size(
        batch_size, q_len_per_req, num_qo_heads, num_kv_heads, head_dim,
        max_seq_len, page_size, window_left))


def _check_decode_args(query, out, lse, block_tables, seq_lens, rows_needed: int):
    """The C ABI of the uniform decode takes no row count: the shapes it
    trusts are checked here, so that no kernel reads or writes past the end
    of query, out or lse."""
    rows, Hqo, _ = query.shape
    if not query.is_contiguous():
        raise PagedKVError("query must be contiguous [rows, num_qo_heads, head_dim]")
    if rows < rows_needed:
        raise PagedKVError(f"query has {rows} rows; the requests need {rows_needed}")
    if out.shape != query.shape or out.dtype != query.dtype or not out.is_contiguous():
        raise PagedKVError("out must be a contiguous tensor of the query's shape and dtype")
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (rows, Hqo)
                            or not lse.is_contiguous()):
        raise PagedKVError(f"lse must be a contiguous float32 [{rows}, {Hqo}] tensor")
    B = seq_lens.shape[0]
    if seq_lens.dim() != 1 or seq_lens.element_size() != 4:
        raise PagedKVError("seq_lens must be a 1-D tensor of 32-bit lengths")
    if block_tables.dim() != 2 or block_tables.shape[0] < B or block_tables.dtype != torch.int32 \
            or block_tables.stride(1) != 1:
        raise PagedKVError("block_tables must be int32 [>= batch_size, pages] with unit column stride")


def paged_decode(query, kv_cache, workspace, block_tables, seq_lens, max_seq_len: int,
                 bmm1_scale: float = 1.0, bmm2_scale: float = 1.0, window_left: int = -1,
                 sinks=None, kv_layout="HND", q_len_per_req: int = 1, out=None,
                 lse=None, err_word=None, stream=None, max_q_len=None, cum_seq_lens_q=None,
                 enable_pdl=None):
    """seq_lens: int32 (or uint32) tensor holding the unsigned kv lengths.
    With cum_seq_lens_q ([B+1] int32 on the device) and max_q_len, request b
    has the query rows cum[b] .. cum[b+1]-1 (variable-length queries) and
    q_len_per_req is ignored.  bmm1_scale / bmm2_scale may be one-element
    float32 device tensors, read when the kernels run; enable_pdl launches
    the call's first kernel as a programmatic dependent of the stream's
    previous kernel (None / False: an ordinary launch)."""
    layout = _layout_code(kv_layout)
    kp, vp, stride, P, Hkv, S, D, base = split_cache(kv_cache, layout)
    rows, Hqo, Dq = query.shape
    if Dq != D:
        raise PagedKVError("query head_dim differs from the cache's")
    B = seq_lens.shape[0]
    if out is None:
        out = torch.empty_like(query)
    if (cum_seq_lens_q is None) != (max_q_len is None):
        raise PagedKVError("cum_seq_lens_q and max_q_len go together")
    if cum_seq_lens_q is not None:
        if cum_seq_lens_q.dtype != torch.int32 or tuple(cum_seq_lens_q.shape) != (B + 1,):
            raise PagedKVError(f"cum_seq_lens_q must be int32 [{B + 1}]")
        _check_decode_args(query, out, lse, block_tables, seq_lens, 0)
    else:
        _check_decode_args(query, out, lse, block_tables, seq_lens, B * q_len_per_req)
    s1, s1_dev = _scale_arg(bmm1_scale, query.device)
    s2, s2_dev = _scale_arg(bmm2_scale, query.device)
    if s1_dev or s2_dev or enable_pdl:
        mq = int(max_q_len) if cum_seq_lens_q is not None else q_len_per_req
        _check(load_library().paged_decode_ex(
            _ptr(query), rows, kp, vp, stride, P, _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(block_tables),
            block_tables.stride(0), _ptr(seq_lens), B, max_seq_len, s1, s2, s1_dev, s2_dev,
            window_left, _ptr(sinks), mq, _ptr(cum_seq_lens_q), Hqo, Hkv, D, S, layout,
            _decode_dtype(query, base), 1 if enable_pdl else 0, _ptr(out), _ptr(lse),
            _ptr(err_word), _stream(stream)))
        return out
    if cum_seq_lens_q is not None:
        _check(load_library().paged_decode_varlen(
            _ptr(query), rows, kp, vp, stride, P, _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(block_tables),
            block_tables.stride(0), _ptr(seq_lens), B, max_seq_len, bmm1_scale,
            bmm2_scale, window_left, _ptr(sinks), int(max_q_len), _ptr(cum_seq_lens_q), Hqo,
            Hkv, D, S, layout, _decode_dtype(query, base), _ptr(out), _ptr(lse), _ptr(err_word),
            _stream(stream)))
        return out
    _check(load_library().paged_decode(
        _ptr(query), kp, vp, stride, P, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(block_tables),
        block_tables.stride(0), _ptr(seq_lens), B, max_seq_len, bmm1_scale,
        bmm2_scale, window_left, _ptr(sinks), q_len_per_req, Hqo, Hkv, D, S,
        layout, _decode_dtype(query, base), _ptr(out), _ptr(lse), _ptr(err_word),
        _stream(stream)))
    return out


def paged_decode_noalloc(query, kv_cache, block_tables, seq_lens, max_seq_len: int,
                         bmm1_scale: float = 1.0, bmm2_scale: float = 1.0,
                         window_left: int = -1, sinks=None, kv_layout="HND",
                         q_len_per_req: int = 1, out=None, lse=None, err_word=None,
                         stream=None):
    """paged_decode for callers that cannot allocate device memory at the
    call: the split partials use the library's fixed device scratch array
    (PKV_NOALLOC_SCRATCH_BYTES) instead of a workspace tensor.  Calls that
    overlap on the GPU share that array and race."""
    layout = _layout_code(kv_layout)
    kp, vp, stride, P, Hkv, S, D, base = split_cache(kv_cache, layout)
    rows, Hqo, Dq = query.shape
    if Dq != D:
        raise PagedKVError("query head_dim differs from the cache's")
    B = seq_lens.shape[0]
    if out is None:
        out = torch.empty_like(query)
    _check_decode_args(query, out, lse, block_tables, seq_lens, B * q_len_per_req)
    _check(load_library().paged_decode_noalloc(
        _ptr(query), kp, vp, stride, P, _ptr(block_tables), block_tables.stride(0),
        _ptr(seq_lens), B, max_seq_len, bmm1_scale, bmm2_scale, window_left, _ptr(sinks),
        q_len_per_req, Hqo, Hkv, D, S, layout, _decode_dtype(query, base), _ptr(out), _ptr(lse),
        _ptr(err_word), _stream(stream)))
    return out


# ---- prefill ---------------------------------------------------------------------------------

def paged_prefill_workspace_size(batch_size, num_qo_heads, max_token_per_sequence,
                                 max_sequence_kv) -> int:
    return int(load_library().paged_prefill_workspace_size(
        batch_size, num_qo_heads, max_token_per_sequence, max_sequence_kv))


def paged_prefill_fp8_workspace_size(batch_size, num_qo_heads, num_kv_heads,
                                     max_token_per_sequence, max_sequence_kv, total_q, d_qk, d_vo,
                                     q_dtype, kv_dtype) -> int:
    """Workspace of paged_prefill with an E4M3 query and/or caches (dtypes
    as torch dtypes)."""
    return int(load_library().paged_prefill_fp8_workspace_size(
        batch_size, num_qo_heads, num_kv_heads, max_token_per_sequence, max_sequence_kv, total_q,
        d_qk, d_vo, E4M3 if q_dtype == torch.float8_e4m3fn else BF16,
        E4M3 if kv_dtype == torch.float8_e4m3fn else BF16))


def _scale_ptr(t, device):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.numel() != 1 or t.device != device:
        raise PagedKVError("q_scale / k_scale / v_scale: one float32 value on the query's device")
    return _ptr(t)


def paged_prefill(q, k_cache, v_cache, scale: float, workspace,
                  max_token_per_sequence: int, max_sequence_kv: int,
                  actual_seq_lens_q, actual_seq_lens_kv, block_tables,
                  causal: bool = True, out=None, lse=None, kv_layout="HND",
                  err_word=None, stream=None, batch_offsets_q=None, batch_offsets_o=None,
                  batch_offsets_k=None, batch_offsets_v=None, q_scale=None, k_scale=None,
                  v_scale=None, o_data_type=None):
    """block_tables=None: k_cache / v_cache are contiguous [rows, Hkv, d]
    tensors (the page's non-paged case; kv_layout is then NHD).  The
    batch_offsets_* tensors ([B] int32 on the device, token rows) place each
    request's queries, outputs / LSEs and (contiguous K/V) keys / values.
    q and/or the (paged) caches may be float8_e4m3fn: q_scale, k_scale and
    v_scale (one float32 each on the device, or None for 1) dequantise them,
    and the output is o_data_type (bf16 when q is E4M3 and none is given);
    the workspace then needs paged_prefill_fp8_workspace_size bytes."""
    if block_tables is None:
        kv_layout = "NHD"
    layout = _layout_code(kv_layout)
    total_q, Hqo, d_qk = q.shape
    if block_tables is None:
        P, Hkv, dk = k_cache.shape
        S, dv = 1, v_cache.shape[2]
    elif layout == HND:
        P, Hkv, S, dk = k_cache.shape
        dv = v_cache.shape[3]
    else:
        P, S, Hkv, dk = k_cache.shape
        dv = v_cache.shape[3]
    if dk != d_qk:
        raise PagedKVError("q head_dim differs from the key cache's")
    e4 = torch.float8_e4m3fn
    fp8 = q.dtype == e4 or k_cache.dtype == e4 or any(x is not None for x in (q_scale, k_scale, v_scale))
    odt = o_data_type or (torch.bfloat16 if q.dtype == e4 else q.dtype)
    if out is None:
        out = torch.empty((total_q, Hqo, dv), dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty((total_q, Hqo), dtype=torch.float32, device=q.device)
    if tuple(out.shape) != (total_q, Hqo, dv) or out.dtype != odt or not out.is_contiguous():
        raise PagedKVError(f"out must be a contiguous {odt} [{total_q}, {Hqo}, {dv}] tensor")
    if tuple(lse.shape) != (total_q, Hqo) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise PagedKVError(f"lse must be a contiguous float32 [{total_q}, {Hqo}] tensor")
    if not q.is_contiguous():
        raise PagedKVError("q must be contiguous [total_q, num_qo_heads, d_qk]")
    B = actual_seq_lens_q.shape[0]
    bt_stride = 0 if block_tables is None else block_tables.stride(0)
    offsets = (batch_offsets_q, batch_offsets_o, batch_offsets_k, batch_offsets_v)
    if fp8:
        if block_tables is None or any(o is not None for o in offsets):
            raise PagedKVError("the E4M3 prefill takes paged caches and packed rows")
        if v_cache.dtype != k_cache.dtype:
            raise PagedKVError("k_cache and v_cache hold the same element type")
        _check(load_library().paged_prefill_fp8(
            _ptr(q), total_q, _ptr(k_cache), _ptr(v_cache), k_cache.stride(0), v_cache.stride(0),
            P, scale, _scale_ptr(q_scale, q.device), _scale_ptr(k_scale, q.device),
            _scale_ptr(v_scale, q.device), _ptr(workspace), workspace.numel() * workspace.element_size(),
            max_token_per_sequence, max_sequence_kv, _ptr(actual_seq_lens_q),
            _ptr(actual_seq_lens_kv), _ptr(block_tables), bt_stride, B, int(causal), Hqo, Hkv, d_qk,
            dv, S, layout, _dtype_code(q), _dtype_code(k_cache), _dtype_code(out), _ptr(out),
            _ptr(lse), _ptr(err_word), _stream(stream)))
    elif all(o is None for o in offsets):
        _check(load_library().paged_prefill(
            _ptr(q), total_q, _ptr(k_cache), _ptr(v_cache), k_cache.stride(0), v_cache.stride(0),
            P, scale, _ptr(workspace), workspace.numel() * workspace.element_size(),
            max_token_per_sequence, max_sequence_kv, _ptr(actual_seq_lens_q),
            _ptr(actual_seq_lens_kv), _ptr(block_tables), bt_stride, B,
            int(causal), Hqo, Hkv, d_qk, dv, S, layout, _dtype_code(q), _ptr(out),
            _ptr(lse), _ptr(err_word), _stream(stream)))
    else:
        _check(load_library().paged_prefill_ex(
            _ptr(q), total_q, _ptr(k_cache), _ptr(v_cache), k_cache.stride(0), v_cache.stride(0),
            P, scale, _ptr(workspace), workspace.numel() * workspace.element_size(),
            max_token_per_sequence, max_sequence_kv, _ptr(actual_seq_lens_q),
            _ptr(actual_seq_lens_kv), _ptr(block_tables), bt_stride, B,
            int(causal), Hqo, Hkv, d_qk, dv, S, layout, _dtype_code(q), _ptr(out),
            _ptr(lse), *(_ptr(o) for o in offsets), _ptr(err_word), _stream(stream)))
    return out, lse
