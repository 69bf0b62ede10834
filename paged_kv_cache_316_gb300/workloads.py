"""Seeded synthetic inputs for paged-KV attention.

Shared by the tests and the benchmark.  This module holds no step of the
attention, append or index arithmetic: it draws sequence lengths, reserves
physical pages for them the way a page allocator does before any call (the
append page notes that the page table already covers the appended tokens),
and fills tensors with N(0, 1) values.  Random draws come from
``torch.Generator`` objects seeded explicitly, on the CPU unless a device is
given.

Workload shapes follow the problem statements of the three FlashInfer API
pages (append_paged_kv_cache, trtllm_batch_decode_with_kv_cache,
cudnn_batch_prefill_with_kv_cache) and the benchmark configurations built on
them (see ``CONFIGS``).
"""
from __future__ import annotations

import itertools
import math
from dataclasses import dataclass, field

import torch

NHD, HND = 0, 1
F16, BF16, E4M3 = 0, 1, 2  # E4M3: 8-bit float cache elements
POISON = 0x7FFFFFFF  # block-table padding that must never be read

_TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, E4M3: torch.float8_e4m3fn}


def torch_dtype(code: int) -> torch.dtype:
    return _TORCH_DTYPE[code]


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, dtype: torch.dtype, g: torch.Generator, device="cpu"):
    """N(0,1) drawn in fp32, then rounded to ``dtype``."""
    return torch.randn(shape, generator=g, dtype=torch.float32,
                       device=device).to(dtype)


# ---- sequence lengths ---------------------------------------------------------

def uniform_lengths(g: torch.Generator, n: int, lo: int, hi: int) -> list[int]:
    """Integers uniform in [lo, hi] (inclusive)."""
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def lognormal_lengths(g: torch.Generator, n: int, median: float, sigma: float,
                      lo: int, cap: int) -> list[int]:
    z = torch.randn(n, generator=g, dtype=torch.float64)
    L = torch.exp(math.log(median) + sigma * z).round().clamp(lo, cap)
    return [int(x) for x in L.tolist()]


# ---- page reservation -----------------------------------------------------------

@dataclass
class PageTable:
    """Physical pages reserved for each request, in logical order."""
    lengths: list[int]
    page_size: int
    num_pages: int                      # pool size (max_num_pages)
    pages: list[list[int]] = field(default_factory=list)

    @property
    def batch(self) -> int:
        return len(self.lengths)

    def max_pages(self) -> int:
        return max((len(p) for p in self.pages), default=0)

    def block_tables(self, width: int | None = None, poison: int = POISON):
        """int32 [B, width]; entries past a request's pages hold ``poison``."""
        width = max(1, width or self.max_pages())
        bt = torch.full((self.batch, width), poison, dtype=torch.int32)
        for b, pg in enumerate(self.pages):
            if pg:
                bt[b, :len(pg)] = torch.tensor(pg, dtype=torch.int32)
        return bt

    def csr(self):
        """(kv_indptr [B+1], kv_indices [nnz_pages], kv_last_page_len [B])."""
        counts = [len(p) for p in self.pages]
        indptr = torch.zeros(self.batch + 1, dtype=torch.int32)
        if counts:
            indptr[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0).to(torch.int32)
        flat = [x for p in self.pages for x in p]
        indices = torch.tensor(flat, dtype=torch.int32) if flat else torch.zeros(0, dtype=torch.int32)
        last = torch.tensor([L - (len(p) - 1) * self.page_size if p else 0
                             for L, p in zip(self.lengths, self.pages)], dtype=torch.int32)
        return indptr, indices, last


def reserve_pages(lengths, page_size: int, g: torch.Generator | None,
                  slack: float = 0.0, extra: int = 0,
                  pool_pages: int | None = None) -> PageTable:
    """Reserve ceil(L / page_size) pages per request from a pool whose
    physical order is a random permutation (``g`` None: identity order)."""
    need = [-(-int(L) // page_size) for L in lengths]
    total = sum(need)
    pool = pool_pages if pool_pages is not None else total + math.ceil(slack * total) + extra
    assert pool >= total, (pool, total)
    order = torch.randperm(pool, generator=g).tolist() if g is not None else list(range(pool))
    pages, k = [], 0
    for n in need:
        pages.append(order[k:k + n])
        k += n
    return PageTable([int(L) for L in lengths], page_size, pool, pages)


# ---- the cache pool ---------------------------------------------------------------

@dataclass
class Pool:
    """Paged K/V storage.  ``k``/``v`` are views; ``page_stride`` is the
    distance in elements between consecutive pages of either view."""
    storage: tuple
    k: torch.Tensor
    v: torch.Tensor
    layout: int
    num_pages: int
    num_heads: int
    page_size: int
    d_k: int
    d_v: int
    k_page_stride: int
    v_page_stride: int


def make_pool(num_pages: int, num_heads: int, page_size: int, d_k: int,
              d_v: int | None, layout: int, dtype: torch.dtype,
              g: torch.Generator | None, form: str = "5d", device="cpu",
              fill: str = "randn") -> Pool:
    """``form`` '5d': one [P, 2, ...] tensor (K at [:, 0], V at [:, 1]);
    'tuple': separate K and V tensors.  ``fill``: 'randn', 'nan' or 'empty'."""
    d_v = d_k if d_v is None else d_v

    def page_shape(d):
        return (page_size, num_heads, d) if layout == NHD else (num_heads, page_size, d)

    def alloc(shape):
        if fill == "randn":
            return randn(shape, dtype, g, device)
        t = torch.empty(shape, dtype=dtype, device=device)
        if fill == "nan":
            t.fill_(float("nan"))
        return t

    if form == "5d":
        assert d_k == d_v
        st = alloc((num_pages, 2) + page_shape(d_k))
        stride = 2 * num_heads * page_size * d_k
        return Pool((st,), st[:, 0], st[:, 1], layout, num_pages, num_heads,
                    page_size, d_k, d_v, stride, stride)
    k = alloc((num_pages,) + page_shape(d_k))
    v = alloc((num_pages,) + page_shape(d_v))
    return Pool((k, v), k, v, layout, num_pages, num_heads, page_size, d_k, d_v,
                num_heads * page_size * d_k, num_heads * page_size * d_v)


def write_tokens(pool: Pool, pt: PageTable, b: int, keys: torch.Tensor,
                 values: torch.Tensor, start: int = 0) -> None:
    """Place logical tokens [start, start+n) of request b by plain indexing
    (test set-up of a pool's logical content; not the append kernel)."""
    S = pool.page_size
    for i in range(keys.shape[0]):
        j = start + i
        page, slot = pt.pages[b][j // S], j % S
        if pool.layout == NHD:
            pool.k[page, slot] = keys[i]
            pool.v[page, slot] = values[i]
        else:
            pool.k[page, :, slot] = keys[i]
            pool.v[page, :, slot] = values[i]


def read_tokens(pool: Pool, pt: PageTable, b: int, n: int | None = None):
    """Gather the logical K/V of request b ([L, H, d]) by plain indexing."""
    S = pool.page_size
    L = pt.lengths[b] if n is None else n
    ks, vs = [], []
    for j in range(L):
        page, slot = pt.pages[b][j // S], j % S
        if pool.layout == NHD:
            ks.append(pool.k[page, slot])
            vs.append(pool.v[page, slot])
        else:
            ks.append(pool.k[page, :, slot])
            vs.append(pool.v[page, :, slot])
    if not ks:
        return (pool.k.new_zeros((0, pool.num_heads, pool.d_k)),
                pool.v.new_zeros((0, pool.num_heads, pool.d_v)))
    return torch.stack(ks), torch.stack(vs)


# ---- named workloads ---------------------------------------------------------------

@dataclass
class DecodeCase:
    query: torch.Tensor          # [B*Q, Hqo, D] (or [sum q_lens, Hqo, D])
    pool: Pool
    pt: PageTable
    block_tables: torch.Tensor   # [B, width] int32 (poison padded)
    seq_lens: torch.Tensor       # [B] int32 holding the uint32 lengths
    max_seq_len: int
    bmm1_scale: float
    bmm2_scale: float
    window_left: int
    sinks: torch.Tensor | None   # [Hqo] fp32
    q_len_per_req: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: int
    # variable-length queries: request b owns query rows cum[b] .. cum[b+1]-1
    # and q_len_per_req holds the largest length (max_q_len)
    cum_seq_lens_q: torch.Tensor | None = None
    kv_dtype: int | None = None  # cache element type when it differs from dtype (E4M3)


def decode_case(lengths, page_size: int, num_qo_heads: int, num_kv_heads: int,
                head_dim: int, layout: int, dtype: int = BF16, q_len_per_req: int = 1,
                window_left: int = -1, with_sinks: bool = False, seed: int = 0,
                bmm1_scale: float | None = None, bmm2_scale: float = 1.0,
                pool_pages: int | None = None, slack: float = 0.0, form: str = "5d",
                device="cpu", bt_width: int | None = None, fill: str = "randn",
                shuffle: bool = True, q_lens=None, kv_dtype: int | None = None) -> DecodeCase:
    """Decode problem over freshly reserved pages.  q_lens (one entry per
    request) gives variable query lengths instead of q_len_per_req."""
    g = generator(seed)
    gd = g if str(device) == "cpu" else generator(seed + 7919, device)
    pt = reserve_pages(lengths, page_size, g if shuffle else None, slack=slack,
                       pool_pages=pool_pages)
    B = len(lengths)
    tdt = torch_dtype(dtype)
    kdt = torch_dtype(dtype if kv_dtype is None else kv_dtype)
    pool = make_pool(pt.num_pages, num_kv_heads, page_size, head_dim, head_dim,
                     layout, kdt, gd, form=form, device=device, fill=fill)
    cum = None
    if q_lens is not None:
        assert len(q_lens) == B
        cum = torch.tensor([0] + list(itertools.accumulate(q_lens)), dtype=torch.int32)
        q_len_per_req = max(q_lens) if B else 1
    rows = B * q_len_per_req if cum is None else int(cum[-1])
    query = randn((rows, num_qo_heads, head_dim), tdt, gd, device)
    sinks = randn((num_qo_heads,), torch.float32, g) if with_sinks else None
    if bmm1_scale is None:
        bmm1_scale = 1.0 / math.sqrt(head_dim)
    width = bt_width or max(1, pt.max_pages())
    return DecodeCase(query, pool, pt, pt.block_tables(width),
                      torch.tensor(pt.lengths, dtype=torch.int32),
                      max(pt.lengths) if B else 0, bmm1_scale, bmm2_scale,
                      window_left, sinks, q_len_per_req, num_qo_heads,
                      num_kv_heads, head_dim, dtype, cum, kv_dtype)


@dataclass
class PrefillCase:
    q: torch.Tensor              # [total_q, Hqo, d_qk]
    pool: Pool
    pt: PageTable
    block_tables: torch.Tensor
    seq_lens_q: torch.Tensor     # [B] int32
    seq_lens_kv: torch.Tensor    # [B] int32
    max_q: int
    max_kv: int
    scale: float
    causal: bool
    num_qo_heads: int
    num_kv_heads: int
    d_qk: int
    d_vo: int
    dtype: int
    # E4M3 (FP8) storage: the query and/or the caches hold 1-byte elements
    # whose values are the stored ones times q_scale / k_scale / v_scale
    q_dtype: int | None = None
    kv_dtype: int | None = None
    q_scale: float = 1.0
    k_scale: float = 1.0
    v_scale: float = 1.0


def prefill_case(q_lens, kv_lens, page_size: int, num_qo_heads: int,
                 num_kv_heads: int, d_qk: int, d_vo: int, layout: int = HND,
                 dtype: int = BF16, causal: bool = True, seed: int = 0,
                 scale: float | None = None, slack: float = 0.0, device="cpu",
                 bt_width: int | None = None, fill: str = "randn",
                 shuffle: bool = True, q_dtype: int | None = None,
                 kv_dtype: int | None = None, q_scale: float = 1.0, k_scale: float = 1.0,
                 v_scale: float = 1.0) -> PrefillCase:
    """q_dtype / kv_dtype = E4M3 store the query / caches as FP8 (N(0,1)
    draws rounded to E4M3); the scales dequantise them."""
    g = generator(seed)
    gd = g if str(device) == "cpu" else generator(seed + 7919, device)
    pt = reserve_pages(kv_lens, page_size, g if shuffle else None, slack=slack)
    tdt = torch_dtype(dtype)
    pool = make_pool(pt.num_pages, num_kv_heads, page_size, d_qk, d_vo, layout,
                     torch_dtype(dtype if kv_dtype is None else kv_dtype), gd, form="tuple",
                     device=device, fill=fill)
    total_q = int(sum(q_lens))
    q = randn((total_q, num_qo_heads, d_qk), torch_dtype(dtype if q_dtype is None else q_dtype),
              gd, device)
    if scale is None:
        scale = 1.0 / math.sqrt(d_qk)
    width = bt_width or max(1, pt.max_pages())
    return PrefillCase(q, pool, pt, pt.block_tables(width),
                       torch.tensor([int(x) for x in q_lens], dtype=torch.int32),
                       torch.tensor([int(x) for x in kv_lens], dtype=torch.int32),
                       max(q_lens) if len(q_lens) else 0,
                       max(kv_lens) if len(kv_lens) else 0, scale, causal,
                       num_qo_heads, num_kv_heads, d_qk, d_vo, dtype, q_dtype, kv_dtype,
                       q_scale, k_scale, v_scale)


@dataclass
class AppendCase:
    append_key: torch.Tensor     # [nnz, H, D]
    append_value: torch.Tensor
    append_indptr: torch.Tensor  # [B+1] int32
    pool: Pool
    pt: PageTable
    kv_indptr: torch.Tensor
    kv_indices: torch.Tensor
    kv_last_page_len: torch.Tensor
    num_kv_heads: int
    head_dim: int
    dtype: int


def append_case(append_lens, prefix_lens, page_size: int, num_kv_heads: int,
                head_dim: int, layout: int, dtype: int = F16, seed: int = 0,
                slack: float = 0.1, pool_pages: int | None = None,
                page_ids: list[int] | None = None, form: str = "5d",
                device="cpu", fill: str = "randn") -> AppendCase:
    """Requests with ``prefix_lens`` tokens already cached append
    ``append_lens`` more; pages are reserved for prefix + appended tokens."""
    g = generator(seed)
    gd = g if str(device) == "cpu" else generator(seed + 7919, device)
    tdt = torch_dtype(dtype)
    lengths = [int(a) + int(p) for a, p in zip(append_lens, prefix_lens)]
    if page_ids is not None:  # explicit physical pages, handed out in order
        need = [-(-L // page_size) for L in lengths]
        pt, k = PageTable(lengths, page_size, pool_pages, []), 0
        for n in need:
            pt.pages.append(page_ids[k:k + n])
            k += n
    else:
        pt = reserve_pages(lengths, page_size, g, slack=slack, pool_pages=pool_pages)
    pool = make_pool(pt.num_pages, num_kv_heads, page_size, head_dim, head_dim,
                     layout, tdt, gd, form=form, device=device, fill=fill)
    nnz = int(sum(int(a) for a in append_lens))
    ak = randn((nnz, num_kv_heads, head_dim), tdt, gd, device)
    av = randn((nnz, num_kv_heads, head_dim), tdt, gd, device)
    indptr = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(torch.tensor([int(a) for a in append_lens],
                                           dtype=torch.int64), 0).to(torch.int32)
    kv_indptr, kv_indices, last = pt.csr()
    return AppendCase(ak, av, indptr, pool, pt, kv_indptr, kv_indices, last,
                      num_kv_heads, head_dim, dtype)


# ---- the configurations the benchmark and the full-size tests use -------------------

def pr1_decode(seed: int = 0, layout: int = HND, device="cpu", **kw) -> DecodeCase:
    """bf16 GQA decode: 4 requests of 45/8/25/22 keys, page_size 16, 32 qo /
    8 kv heads, head_dim 128, a 64-page pool in random physical order."""
    return decode_case([45, 8, 25, 22], 16, 32, 8, 128, layout, BF16, seed=seed,
                       pool_pages=64, device=device, **kw)


def llama_decode(seed: int = 0, layout: int = HND, device="cpu", **kw) -> DecodeCase:
    """Llama-3-8B-shaped decode: 64 requests, kv lengths uniform in
    [512, 8192], page_size 16, 32/8 heads, head_dim 128, shuffled pages."""
    L = uniform_lengths(generator(seed), 64, 512, 8192)
    return decode_case(L, 16, 32, 8, 128, layout, BF16, seed=seed,
                       device=device, bt_width=8192 // 16, **kw)


def long_decode(seed: int = 0, layout: int = HND, device="cpu", **kw) -> DecodeCase:
    """Long-context decode: 256 requests, lognormal kv lengths (median 4096,
    sigma 1.0, clamped to [4, 32768]), page_size 64, 64/8 heads, window_left
    4095, per-head sinks, 4 query tokens per request (causal among them)."""
    L = lognormal_lengths(generator(seed), 256, 4096.0, 1.0, 4, 32768)
    return decode_case(L, 64, 64, 8, 128, layout, BF16, q_len_per_req=4,
                       window_left=4095, with_sinks=True, seed=seed,
                       device=device, bt_width=32768 // 64, **kw)


def long_decode_varlen(seed: int = 0, layout: int = HND, device="cpu", batch: int = 256,
                       **kw) -> DecodeCase:
    """The long-context decode with variable-length queries: each of the 256
    requests has 1 to 4 query tokens (uniform), max_q_len 4.  `batch` keeps
    the first requests of the same draws (a smaller case of the same shape)."""
    L = lognormal_lengths(generator(seed), 256, 4096.0, 1.0, 4, 32768)[:batch]
    ql = uniform_lengths(generator(seed + 101), 256, 1, 4)[:batch]
    return decode_case(L, 64, 64, 8, 128, layout, BF16, q_lens=ql, window_left=4095,
                       with_sinks=True, seed=seed, device=device, bt_width=32768 // 64, **kw)


def ragged_prefill(seed: int = 0, d_qk: int = 128, device="cpu", **kw) -> PrefillCase:
    """Causal ragged prefill: 16 requests, q lengths uniform in [128, 2048],
    kv = q + prefix with prefix uniform in [0, 2048], page_size 32, 32/8
    heads, HND, head_dim 128 (or d_qk 192 / d_vo 128)."""
    g = generator(seed)
    q = uniform_lengths(g, 16, 128, 2048)
    pre = uniform_lengths(g, 16, 0, 2048)
    kv = [a + b for a, b in zip(q, pre)]
    return prefill_case(q, kv, 32, 32, 8, d_qk, 128, HND, BF16, causal=True,
                        seed=seed, device=device, bt_width=4096 // 32, **kw)


APPEND_EXAMPLE = dict(lengths=[45, 8, 25, 22], page_size=16, num_kv_heads=32,
                      head_dim=128, max_num_pages=1000, pages=list(range(8)))


def append_example(layout: int = NHD, form: str = "5d", seed: int = 0,
                   device="cpu") -> AppendCase:
    """The append page's worked example: fp16, 100 new tokens split 45/8/25/22
    over 4 empty requests, page_size 16, 32 kv heads, head_dim 128, a
    1000-page pool pre-filled with N(0,1), requests on pages 0..7."""
    ex = APPEND_EXAMPLE
    return append_case(ex["lengths"], [0, 0, 0, 0], ex["page_size"],
                       ex["num_kv_heads"], ex["head_dim"], layout, F16, seed=seed,
                       pool_pages=ex["max_num_pages"], page_ids=ex["pages"],
                       form=form, device=device)


def append_sweep(batch: int, seed: int = 1, layout: int = NHD, one_token: bool = False,
                 device="cpu", dtype: int = F16, **kw) -> AppendCase:
    """Seeded append sweep point: ``batch`` requests with a cached prefix
    uniform in [0, 256] appending uniform [1, 128] tokens (or exactly one),
    32 kv heads, head_dim 128, page_size 16, fp16, pool = pages + 10%."""
    g = generator(seed)
    prefix = uniform_lengths(g, batch, 0, 256)
    app = [1] * batch if one_token else uniform_lengths(g, batch, 1, 128)
    return append_case(app, prefix, 16, 32, 128, layout, dtype, seed=seed,
                       slack=0.1, device=device, **kw)


CONFIGS = {
    "pr1_decode": "bf16 paged GQA decode, batch 4, kv lens [45,8,25,22], page 16, "
                  "32/8 heads, d 128, HND, 64-page permuted pool",
    "append_example": "fp16 append of 45/8/25/22 tokens, 32 kv heads, d 128, page 16, "
                      "1000-page pool, pages 0..7 (NHD and HND)",
    "append_sweep_4096": "fp16 append sweep point: 4096 requests, prefix U[0,256], "
                         "append U[1,128], 32 kv heads, d 128, page 16, NHD",
    "llama_decode": "bf16 decode, batch 64, kv U[512,8192], page 16, 32/8 heads, d 128, HND",
    "long_decode": "bf16 decode, batch 256, lognormal kv (median 4096, cap 32768), page 64, "
                   "64/8 heads, window 4095, sinks, q_len_per_req 4",
    "long_decode_varlen": "the long-context decode with 1..4 query tokens per request "
                          "(cum_seq_lens_q, max_q_len 4)",
    "ragged_prefill": "bf16 causal ragged prefill, batch 16, q U[128,2048], prefix "
                      "U[0,2048], page 32, 32/8 heads, d 128 (and 192/128)",
}
