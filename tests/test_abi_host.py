"""The C-ABI library builds, loads and exports every symbol include/pa.h declares, and
rejects bad arguments on the host before touching the GPU.  CPU only: no call here
reaches a kernel launch or any CUDA runtime call."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED = 0, 1, 2


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    import paged_kv_cache_09_gb300 as pa
    pa.build()
    return pa.load()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("pa_slot_mapping", "pa_reshape_and_cache", "pa_decode", "pa_decode_append",
              "pa_prefill_chunk",
              "pa_decode_workspace_size", "pa_get_device_errors", "pa_status_string",
              "pa_build_info"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n
    nm = shutil.which("nm")
    if nm:
        import paged_kv_cache_09_gb300 as pa
        out = subprocess.run([nm, "-D", "--defined-only", pa.LIB_PATH], capture_output=True,
                             text=True).stdout
        exported = set(re.findall(r"\bT (pa_\w+)", out))
        assert set(_declared()) <= exported


def test_status_strings_and_build_info(lib):
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(1) == b"PA_ERR_INVALID_ARG"
    assert lib.pa_status_string(2) == b"PA_ERR_UNSUPPORTED"
    assert lib.pa_status_string(3) == b"PA_ERR_CUDA"
    assert lib.pa_status_string(4) == b"PA_ERR_TIMEOUT"
    assert b"sm_103a" in lib.pa_build_info()


def test_test_hooks_live_only_in_the_test_library(lib):
    # The product library has no failure-injection entry point; the failure-path test
    # library (same sources, PA_TEST_HOOKS) has it beside every declared symbol.
    from paged_kv_cache_09_gb300 import _build
    assert not hasattr(lib, "pa_test_hook")
    test_lib = ctypes.CDLL(_build.build_test())
    assert hasattr(test_lib, "pa_test_hook")
    for n in _declared():
        assert hasattr(test_lib, n), n


FAKE = 0x10000  # an aligned, non-null address that is never dereferenced on the host


def _decode(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, page_stride=832 * 4 * 256, num_pages=64, bt=FAKE,
             bt_stride=16, seq_lens=FAKE, num_seqs=1, max_seq_len=8192, hq=24, hkv=4, d=256,
             bs=832, scale=0.0625, out=FAKE, ws=FAKE, ws_bytes=1 << 20, nk=None, nv=None,
             ns=None)
    a.update(kw)
    return lib.pa_decode(a["q"], a["k"], a["v"], a["page_stride"], a["num_pages"], a["bt"],
                         a["bt_stride"], a["seq_lens"], a["num_seqs"], a["max_seq_len"], a["hq"],
                         a["hkv"], a["d"], a["bs"], a["scale"], a["out"], a["ws"],
                         a["ws_bytes"], a["nk"], a["nv"], a["ns"], None)


def _prefill(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, page_stride=832 * 4 * 256, num_pages=64, bt=FAKE,
             q_len=4096, q_start=4096, causal=1, hq=24, hkv=4, d=256, bs=832, scale=0.0625,
             out=FAKE, ws=None, ws_bytes=0)
    a.update(kw)
    return lib.pa_prefill_chunk(a["q"], a["k"], a["v"], a["page_stride"], a["num_pages"],
                                a["bt"], a["q_len"], a["q_start"], a["causal"], a["hq"],
                                a["hkv"], a["d"], a["bs"], a["scale"], a["out"], a["ws"],
                                a["ws_bytes"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), PA_ERR_INVALID_ARG),
    (dict(out=None), PA_ERR_INVALID_ARG),
    (dict(ws=None), PA_ERR_INVALID_ARG),
    (dict(num_seqs=0), PA_ERR_INVALID_ARG),
    (dict(max_seq_len=0), PA_ERR_INVALID_ARG),
    (dict(hq=25), PA_ERR_INVALID_ARG),
    (dict(bs=0), PA_ERR_INVALID_ARG),
    (dict(page_stride=100), PA_ERR_INVALID_ARG),
    (dict(bt_stride=9), PA_ERR_INVALID_ARG),          # 8192 / 832 needs 10 entries
    (dict(q=FAKE + 2), PA_ERR_INVALID_ARG),           # misaligned
    (dict(ws=FAKE + 16), PA_ERR_INVALID_ARG),         # workspace must be 256-byte aligned
    (dict(scale=float("nan")), PA_ERR_INVALID_ARG),
    (dict(nk=FAKE), PA_ERR_INVALID_ARG),              # fused write needs all three
    (dict(d=128, page_stride=832 * 4 * 128), PA_ERR_UNSUPPORTED),
    (dict(hq=40, hkv=4), PA_ERR_UNSUPPORTED),         # group of 10 > 8
])
def test_decode_rejects_bad_arguments(lib, kw, want):
    assert _decode(lib, **kw) == want


def _append(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, page_stride=832 * 4 * 256, num_pages=64, bt=FAKE,
             bt_stride=16, seq_lens=FAKE, num_seqs=1, max_seq_len=8192, hq=24, hkv=4, d=256,
             bs=832, scale=0.0625, out=FAKE, ws=FAKE, ws_bytes=1 << 20, nk=FAKE, nv=FAKE,
             slots=FAKE)
    a.update(kw)
    return lib.pa_decode_append(a["q"], a["k"], a["v"], a["page_stride"], a["num_pages"],
                                a["bt"], a["bt_stride"], a["seq_lens"], a["num_seqs"],
                                a["max_seq_len"], a["hq"], a["hkv"], a["d"], a["bs"], a["scale"],
                                a["out"], a["ws"], a["ws_bytes"], a["nk"], a["nv"], a["slots"],
                                None)


@pytest.mark.parametrize("kw,want", [
    (dict(nk=None), PA_ERR_INVALID_ARG),              # the appended token is required
    (dict(nv=None), PA_ERR_INVALID_ARG),
    (dict(nk=FAKE + 8), PA_ERR_INVALID_ARG),          # misaligned new K
    (dict(slots=FAKE + 4), PA_ERR_INVALID_ARG),       # int64 output must be 8-byte aligned
    (dict(q=None), PA_ERR_INVALID_ARG),               # and every pa_decode check
    (dict(bt_stride=9), PA_ERR_INVALID_ARG),
    (dict(hq=40, hkv=4), PA_ERR_UNSUPPORTED),
])
def test_decode_append_rejects_bad_arguments(lib, kw, want):
    assert _append(lib, **kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), PA_ERR_INVALID_ARG),
    (dict(bt=None), PA_ERR_INVALID_ARG),
    (dict(q_len=0), PA_ERR_INVALID_ARG),
    (dict(q_start=-1), PA_ERR_INVALID_ARG),
    (dict(q_start=2**31 - 100, q_len=200), PA_ERR_INVALID_ARG),
    (dict(hkv=5), PA_ERR_INVALID_ARG),
    (dict(k=FAKE + 8), PA_ERR_INVALID_ARG),
    (dict(ws=FAKE + 16, ws_bytes=1 << 20), PA_ERR_INVALID_ARG),  # workspace 256-byte aligned
    (dict(d=64, page_stride=832 * 4 * 64), PA_ERR_UNSUPPORTED),
])
def test_prefill_rejects_bad_arguments(lib, kw, want):
    assert _prefill(lib, **kw) == want


def test_cache_calls_reject_bad_arguments(lib):
    # num_tokens == 0 is a no-op even with null pointers; negative counts are errors.
    assert lib.pa_slot_mapping(None, None, None, 1, 4, 4, 0, 16, None, None) == PA_OK
    assert lib.pa_slot_mapping(FAKE, None, FAKE, 1, 4, 4, -1, 16, FAKE, None) == PA_ERR_INVALID_ARG
    assert lib.pa_slot_mapping(None, None, FAKE, 1, 4, 4, 3, 16, FAKE, None) == PA_ERR_INVALID_ARG
    assert lib.pa_slot_mapping(FAKE, None, FAKE, 1, 2, 4, 3, 16, FAKE, None) == PA_ERR_INVALID_ARG
    assert lib.pa_reshape_and_cache(None, None, None, None, 4096, 8, None, 0, 4, 256, 4,
                                    None) == PA_OK
    assert lib.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, 4096, 8, FAKE, 2, 4, 3, 4,
                                    None) == PA_ERR_INVALID_ARG   # row of 12 elements
    assert lib.pa_reshape_and_cache(FAKE + 4, FAKE, FAKE, FAKE, 4096, 8, FAKE, 2, 4, 256, 4,
                                    None) == PA_ERR_INVALID_ARG   # misaligned key
    assert lib.pa_get_device_errors(None, 0, None) == PA_ERR_INVALID_ARG


def test_workspace_size_is_zero_for_invalid_sizes(lib):
    assert lib.pa_decode_workspace_size(0, 24, 4, 256, 832, 8192) == 0
    assert lib.pa_decode_workspace_size(1, 24, 5, 256, 832, 8192) == 0
    assert lib.pa_decode_workspace_size(1, 24, 4, 128, 832, 8192) == 0


def _prep(lib, num_seqs=4, num_groups=2, tables=(FAKE, FAKE), strides=(16, 16), mbs=(10, 10),
          bss=(832, 16), slots=(FAKE, FAKE), positions=FAKE, sampled=None, ids=None):
    import ctypes
    G = len(tables)
    arr = lambda t, v: (t * G)(*v)
    return lib.pa_decode_input_prep(positions, sampled, ids, FAKE, FAKE, num_seqs, num_groups,
                                    arr(ctypes.c_void_p, tables), arr(ctypes.c_int64, strides),
                                    arr(ctypes.c_int, mbs), arr(ctypes.c_int, bss),
                                    arr(ctypes.c_void_p, slots), None)


@pytest.mark.parametrize("kw,want", [
    (dict(num_groups=0), PA_ERR_INVALID_ARG),
    (dict(num_groups=9, tables=(FAKE,) * 9, strides=(16,) * 9, mbs=(10,) * 9, bss=(16,) * 9,
          slots=(FAKE,) * 9), PA_ERR_INVALID_ARG),
    (dict(tables=(FAKE, None)), PA_ERR_INVALID_ARG),
    (dict(slots=(None, FAKE)), PA_ERR_INVALID_ARG),
    (dict(strides=(16, 9)), PA_ERR_INVALID_ARG),     # stride below max_blocks
    (dict(bss=(832, 0)), PA_ERR_INVALID_ARG),
    (dict(mbs=(0, 10)), PA_ERR_INVALID_ARG),
    (dict(sampled=FAKE), PA_ERR_INVALID_ARG),        # sampled ids without input_ids
    (dict(positions=None), PA_ERR_INVALID_ARG),
    (dict(num_seqs=-1), PA_ERR_INVALID_ARG),
])
def test_decode_input_prep_rejects_bad_arguments(lib, kw, want):
    assert _prep(lib, **kw) == want


def test_decode_input_prep_with_no_sequences_is_a_no_op(lib):
    assert _prep(lib, num_seqs=0, positions=None) == 0


def _varlen(lib, cu=(0, 10, 30), k_lens=(10, 40), bt_stride=1, num_seqs=None, **kw):
    import ctypes
    B = len(k_lens) if num_seqs is None else num_seqs
    cua = (ctypes.c_int32 * len(cu))(*cu)
    ska = (ctypes.c_int32 * max(1, len(k_lens)))(*k_lens)
    a = dict(q=FAKE, k=FAKE, v=FAKE, page_stride=832 * 4 * 256, num_pages=64, bt=FAKE,
             hq=24, hkv=4, d=256, bs=832, scale=0.0625, out=FAKE)
    a.update(kw)
    return lib.pa_prefill_varlen(a["q"], a["k"], a["v"], a["page_stride"], a["num_pages"],
                                 a["bt"], bt_stride, cua, ska, B, 1, a["hq"], a["hkv"], a["d"],
                                 a["bs"], a["scale"], a["out"], None, 0, None)


@pytest.mark.parametrize("kw,want", [
    (dict(cu=(1, 10, 30)), PA_ERR_INVALID_ARG),          # must start at 0
    (dict(cu=(0, 10, 5)), PA_ERR_INVALID_ARG),           # decreasing
    (dict(k_lens=(5, 40)), PA_ERR_INVALID_ARG),          # 10 rows over 5 keys
    (dict(k_lens=(10, 900)), PA_ERR_INVALID_ARG),        # 900 keys need 2 table entries
    (dict(q=None), PA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), PA_ERR_INVALID_ARG),
    (dict(d=128, page_stride=832 * 4 * 128), PA_ERR_UNSUPPORTED),
])
def test_prefill_varlen_rejects_bad_arguments(lib, kw, want):
    assert _varlen(lib, **kw) == want


def test_prefill_varlen_without_rows_is_a_no_op(lib):
    assert _varlen(lib, cu=(0, 0, 0), k_lens=(5, 7)) == 0
    assert _varlen(lib, cu=(0,), k_lens=(), num_seqs=0) == 0


@pytest.mark.parametrize("dst,src,nbytes", [
    (None, FAKE, 64),            # NULL destination
    (FAKE, None, 64),            # NULL source
    (FAKE + 8, FAKE + 4096, 64),  # misaligned destination
    (FAKE, FAKE + 4096 + 4, 64),  # misaligned source
    (FAKE, FAKE + 4096, 40),     # not a multiple of 16 bytes
])
def test_copy_rejects_bad_arguments(lib, dst, src, nbytes):
    assert lib.pa_copy(dst, src, nbytes, None) == PA_ERR_INVALID_ARG


def test_copy_of_nothing_is_a_no_op(lib):
    assert lib.pa_copy(None, None, 0, None) == PA_OK
