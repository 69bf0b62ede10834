"""Paged-KV attention for GB300 (sm_103a): append scatter, split-KV GQA
decode and causal ragged prefill over a paged KV cache, as hand-written CUDA
behind a C ABI (``include/pagedkv.h``).

The Python layer only marshals torch tensors into that ABI; see ``binding``.
"""
from .binding import (  # noqa: F401
    NHD, HND, F16, BF16,
    PagedKVError,
    library_path,
    load_library,
    paged_seq_lens,
    paged_batch_indices_positions,
    paged_append,
    paged_decode_workspace_size,
    paged_decode,
    paged_decode_noalloc,
    paged_prefill_workspace_size,
    paged_prefill_fp8_workspace_size,
    paged_prefill,
    kernel_launches,
    set_wait_limit_ns,
    debug_bounds,
)
