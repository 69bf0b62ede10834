"""The C ABI on a machine without a GPU: the library builds for sm_103a,
loads, exports every entry point the header declares, and rejects bad
arguments on the host before any launch.  Every call below is rejected by
host validation (or has nothing to do), so the fake pointers it carries are
never dereferenced and no kernel is launched, on any machine."""
from __future__ import annotations

import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_316_gb300 import build, binding
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*?[\s\*]+(\w+)\s*\(",
                                 text, flags=re.M)) - {"if", "defined"})


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ["paged_seq_lens", "paged_batch_indices_positions", "paged_append",
              "paged_decode_workspace_size", "paged_decode", "paged_prefill_workspace_size",
              "paged_prefill", "pkv_status_string", "pkv_kernel_launches"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libpagedkv.so does not export {name}"


def test_debug_build_exports_the_same_abi(lib):
    # the range-checking variant (-DPKV_DEBUG_BOUNDS=1) builds for sm_103a,
    # exports every declared entry point and says which build it is
    from paged_kv_cache_316_gb300 import build
    dbg = ctypes.CDLL(build.build(debug_bounds=True))
    for name in declared_functions():
        assert hasattr(dbg, name), f"libpagedkv_debug.so does not export {name}"
    assert dbg.pkv_debug_bounds() == 1
    assert lib.pkv_debug_bounds() == 0


def test_wait_limit_is_set_and_restored(lib):
    # host state only: the limit later launches pass to their kernels
    lib.pkv_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.pkv_set_wait_limit_ns.restype = ctypes.c_ulonglong
    assert lib.pkv_set_wait_limit_ns(5000) == 1000000000  # the default: one second
    assert lib.pkv_set_wait_limit_ns(0) == 5000           # 0 restores the default
    assert lib.pkv_set_wait_limit_ns(0) == 1000000000


def test_status_strings(lib):
    assert lib.pkv_status_string(0) == b"ok"
    assert b"workspace" in lib.pkv_status_string(4)


def _append(lib, **over):
    good = 0x1000  # any 16-byte aligned non-null value: these calls fail before use
    args = dict(append_key=good, append_value=good, nnz=4, batch_indices=good, positions=good,
                k_cache=good, v_cache=good, page_stride=2 * 8 * 16 * 128, max_num_pages=10,
                kv_indices=good, kv_indptr=good, kv_last_page_len=good, batch_size=2,
                num_kv_heads=8, head_dim=128, page_size=16, layout=0, dtype=0,
                err_word=None, stream=None)
    args.update(over)
    return lib.paged_append(*args.values())


def test_append_rejects_bad_arguments(lib):
    assert _append(lib, layout=2) == 2
    assert _append(lib, dtype=5) == 2
    assert _append(lib, head_dim=12) == 2
    assert _append(lib, page_stride=100) == 2
    assert _append(lib, append_key=None) == 1
    assert _append(lib, k_cache=0x1004) == 2      # misaligned
    assert _append(lib, nnz=0, append_key=None) == 0  # nothing to do


def test_decode_rejects_bad_arguments(lib):
    good = 0x1000

    def call(**over):
        a = dict(query=good, k=good, v=good, stride=2 * 8 * 16 * 128, pages=64, ws=good,
                 ws_bytes=1 << 30, bt=good, bt_stride=10000, seq=good, B=4, max_len=100, s1=0.1,
                 s2=1.0, win=-1, sinks=None, Q=1, hqo=32, hkv=8, D=128, S=16, layout=1,
                 dtype=1, out=good, lse=None, err=None, stream=None)
        a.update(over)
        return lib.paged_decode(*a.values())

    assert call(layout=3) == 2
    assert call(hqo=30) == 2          # 30 % 8 != 0
    assert call(D=64) == 3            # head_dim 128 only
    assert call(S=24) == 3            # page size must be a power of two
    assert call(Q=9, hqo=64) == 3     # group 8 x 9 tokens = 72 rows > 64
    assert call(query=None) == 1
    assert call(ws_bytes=16, max_len=100000) == 4
    assert call(bt_stride=2) == 2     # block-table row narrower than max_seq_len
    assert call(B=0) == 0


def test_decode_varlen_rejects_bad_arguments(lib):
    good = 0x1000

    def call(**over):
        a = dict(query=good, ntok=10, k=good, v=good, stride=2 * 8 * 16 * 128, pages=64, ws=good,
                 ws_bytes=1 << 30, bt=good, bt_stride=10000, seq=good, B=4, max_len=100, s1=0.1,
                 s2=1.0, win=-1, sinks=None, maxq=4, cum=good, hqo=32, hkv=8, D=128, S=16,
                 layout=1, dtype=1, out=good, lse=None, err=None, stream=None)
        a.update(over)
        return lib.paged_decode_varlen(*a.values())

    assert call(cum=None) == 1          # cum_seq_lens_q required
    assert call(ntok=-1) == 2
    assert call(maxq=9, hqo=64) == 3    # group 8 x 9 tokens > 64 rows
    assert call(ntok=0) == 0            # no query rows: nothing to do


def test_decode_workspace_size_grows_with_length(lib):
    f = lib.paged_decode_workspace_size
    small = f(64, 1, 32, 8, 128, 512, 16, -1)
    big = f(64, 1, 32, 8, 128, 8192, 16, -1)
    assert 0 <= small <= big and big > 0
    # a window bounds the work per request, so the workspace stops growing
    assert f(256, 4, 64, 8, 128, 32768, 64, 4095) == f(256, 4, 64, 8, 128, 65536, 64, 4095)
    assert f(4, 1, 30, 8, 128, 100, 16, -1) == 0  # invalid sizes


def test_decode_window_slightly_longer_than_a_chunk_takes_one_split(lib):
    # the long-context shape: 32 rows per kv head give 4096-key splits, and
    # its window of 4095 + 4 keys (plus up to 63 for tile alignment) takes one
    # split of its own length -- no partials, no merge
    f = lib.paged_decode_workspace_size
    assert f(256, 4, 64, 8, 128, 32768, 64, 4095) == 0
    # a window well beyond the chunk still splits
    assert f(256, 4, 64, 8, 128, 32768, 64, 8191) > 0
    # without a window the same shape needs partials for up to 8 splits of
    # 4096 keys: B * Hkv * splits * rows * (128 + 1) floats
    need = f(256, 4, 64, 8, 128, 32768, 64, -1)
    assert need >= 256 * 8 * 8 * 32 * 129 * 4


def test_prefill_fp8_rejects_bad_arguments(lib):
    good = 0x1000
    E4M3, BF16, F16 = 2, 1, 0

    def call(**over):
        a = dict(q=good, total_q=150, k=good, v=good, ks=8 * 32 * 128, vs=8 * 32 * 128, pages=100,
                 scale=0.08, qs=None, kscale=None, vscale=None, ws=good, ws_bytes=1 << 30, maxq=100,
                 maxkv=200, lq=good, lkv=good, bt=good, bt_stride=8, B=2, causal=1, hqo=32, hkv=8, dqk=128,
                 dvo=128, S=32, layout=1, qd=E4M3, kvd=E4M3, od=BF16, out=good, lse=good, err=None,
                 stream=None)
        a.update(over)
        return lib.paged_prefill_fp8(*a.values())

    assert call(od=E4M3) == 2          # the output is 16-bit
    assert call(qd=F16) == 2           # a 16-bit query must match the output type
    assert call(bt=None) == 2          # E4M3 caches are paged
    assert call(ks=8 * 32 * 128 + 8) == 2  # E4M3 page strides: multiples of 16 bytes
    assert call(ws_bytes=4096, kvd=BF16) == 4  # too small for the widened query rows
    assert call(ws_bytes=4096, dqk=192, ks=8 * 32 * 192) == 4  # d_qk 192: everything widened
    assert call(dqk=64) == 3
    assert call(total_q=0) == 0
    size = lib.paged_prefill_fp8_workspace_size
    q8 = size(2, 32, 8, 100, 200, 150, 128, 128, E4M3, BF16)
    kv8 = size(2, 32, 8, 100, 200, 150, 128, 128, BF16, E4M3)
    both = size(2, 32, 8, 100, 200, 150, 128, 128, E4M3, E4M3)
    both192 = size(2, 32, 8, 100, 200, 150, 192, 128, E4M3, E4M3)
    base = lib.paged_prefill_workspace_size(2, 32, 100, 200)
    assert q8 - base >= 150 * 32 * 128 * 2                   # the widened query rows
    assert kv8 - base >= 2 * 200 * 8 * (128 + 128) * 2       # widened K and V
    assert both == base  # E4M3 query and caches at d_qk 128 are read as they are
    assert both192 - base >= 150 * 32 * 192 * 2 + 2 * 200 * 8 * (192 + 128) * 2


def test_prefill_rejects_bad_arguments(lib):
    good = 0x1000

    def call(**over):
        a = dict(q=good, total_q=150, k=good, v=good, ks=8 * 32 * 128, vs=8 * 32 * 128, pages=100,
                 scale=0.08, ws=good, ws_bytes=4096, maxq=100, maxkv=200, lq=good, lkv=good,
                 bt=good, bt_stride=8, B=2, causal=1, hqo=32, hkv=8, dqk=128, dvo=128, S=32,
                 layout=1, dtype=1, out=good, lse=good, err=None, stream=None)
        a.update(over)
        return lib.paged_prefill(*a.values())

    assert call(dqk=64) == 3
    assert call(dvo=192) == 3
    assert call(hkv=5) == 2
    assert call(lse=None) == 1        # the LSE output is required
    assert call(ws_bytes=8) == 4
    assert call(bt_stride=3) == 2     # 3 pages of 32 < max_sequence_kv 200
    assert call(S=4) == 3             # TMA boxes need pages of >= 8 slots
    assert call(bt=None, layout=1) == 2  # contiguous K/V is token-major: NHD only
    assert call(total_q=0) == 0       # no query rows: nothing to do
    assert call(B=0) == 0
