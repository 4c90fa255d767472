"""Failure path of the bounded waits, on the GPU, without faulting it; and a timing the
test build can force (consumers that start late).

The test library (libpa_test.so: the same sources built with PA_TEST_HOOKS and a 20 ms
limit on every bounded wait) can leave out the TMA loads of one ring stage (decode) or
one K/V ring unit (prefill) of every CTA.  The consumer waiting for them then runs into
its limit: the kernel sets PA_DEVERR_TIMEOUT, every other role of the CTA gives up, every
load that was issued lands, TMEM is freed, and the kernel returns.  The tests check
that pa_get_device_errors reports PA_ERR_TIMEOUT, that the outputs stay finite, and
that the same context then computes the right result once the hook is off.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import assert_attention_close
from workloads import bits

pytestmark = pytest.mark.gpu

PA_OK, PA_ERR_TIMEOUT = 0, 4
DEVERR_TIMEOUT = 8


@pytest.fixture(scope="module")
def test_lib(cuda_lib):
    from paged_kv_cache_09_gb300 import _build
    lib = ctypes.CDLL(_build.build_test())
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    lib.pa_test_hook.argtypes = [i32, i32, i32]
    lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.pa_decode_workspace_size.restype = sz
    lib.pa_decode.argtypes = [P, P, P, i64, i64, P, i64, P, i32, i32, i32, i32, i32, i32, f32,
                              P, P, sz, P, P, P, P]
    lib.pa_prefill_chunk.argtypes = [P, P, P, i64, i64, P, i32, i32, i32, i32, i32, i32, i32,
                                     f32, P, P, sz, P]
    lib.pa_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.pa_prefill_workspace_size.restype = sz
    lib.pa_get_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint), i32, P]
    assert lib.pa_test_hook(-1, -1, 0) == PA_OK
    yield lib
    lib.pa_test_hook(-1, -1, 0)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _errors(lib):
    bits_ = ctypes.c_uint(0)
    rc = lib.pa_get_device_errors(ctypes.byref(bits_), 1, _stream())
    return rc, int(bits_.value)


def _decode(lib, case, max_seq_len):
    S, hq, d = case.q.shape
    hkv, bs = case.k_cache.shape[2], case.block_size
    out = torch.empty_like(case.q)
    nbytes = lib.pa_decode_workspace_size(S, hq, hkv, d, bs, max_seq_len)
    ws = torch.empty(max(256, nbytes), dtype=torch.uint8, device="cuda")
    rc = lib.pa_decode(case.q.data_ptr(), case.k_cache.data_ptr(), case.v_cache.data_ptr(),
                       case.k_cache.stride(0), case.k_cache.shape[0],
                       case.block_table.data_ptr(), case.block_table.stride(0),
                       case.seq_lens.data_ptr(), S, max_seq_len, hq, hkv, d, bs, case.scale,
                       out.data_ptr(), ws.data_ptr(), ws.numel(), None, None, None, _stream())
    assert rc == PA_OK
    return out


def _prefill(lib, case, ws=None):
    q_len, hq, d = case.q.shape
    out = torch.empty_like(case.q)
    rc = lib.pa_prefill_chunk(case.q.data_ptr(), case.k_cache.data_ptr(),
                              case.v_cache.data_ptr(), case.k_cache.stride(0),
                              case.k_cache.shape[0], case.block_table[0].data_ptr(), q_len,
                              case.q_start, 1, hq, case.k_cache.shape[2], d, case.block_size,
                              case.scale, out.data_ptr(),
                              None if ws is None else ws.data_ptr(),
                              0 if ws is None else ws.numel(), _stream())
    assert rc == PA_OK
    return out


def test_decode_wait_that_runs_out_is_reported_and_the_context_stays_usable(test_lib,
                                                                           cuda_lib):
    lib = test_lib
    case = workloads.decode_8k(device="cuda")
    assert _errors(lib) == (PA_OK, 0)
    assert lib.pa_test_hook(1, -1, 0) == PA_OK  # every CTA loses its ring stage 1
    bad = _decode(lib, case, 8192)
    rc, errs = _errors(lib)
    assert rc == PA_ERR_TIMEOUT and errs & DEVERR_TIMEOUT, (rc, errs)
    assert torch.isfinite(bad.float()).all()
    assert lib.pa_test_hook(-1, -1, 0) == PA_OK
    for _ in range(2):
        good = _decode(lib, case, 8192)
        assert _errors(lib) == (PA_OK, 0)
        assert torch.equal(good, cuda_lib.decode(case.q, case.k_cache, case.v_cache,
                                                 case.block_table, case.seq_lens, case.scale,
                                                 8192))
    ref = oracle.decode(bits(case.q), bits(case.k_cache), bits(case.v_cache),
                        case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(), case.scale)
    assert_attention_close(good, ref, "decode after a timed-out call")
    assert cuda_lib.device_errors() == 0


def test_prefill_wait_that_runs_out_is_reported_and_the_context_stays_usable(test_lib,
                                                                            cuda_lib):
    lib = test_lib
    q_len, q_start, bs = 300, 700, 784
    case = workloads.paged_case(377, [q_start + q_len], bs, 5, q_rows=q_len, q_start=q_start,
                                device="cuda")
    slots = cuda_lib.slot_mapping(case.positions, case.block_table, bs, seq_idx=case.seq_idx)
    cuda_lib.reshape_and_cache(case.new_k, case.new_v, case.k_cache, case.v_cache, slots)
    torch.cuda.synchronize()
    assert _errors(lib) == (PA_OK, 0)
    assert lib.pa_test_hook(-1, 3, 0) == PA_OK  # every CTA loses its K/V ring unit 3
    _prefill(lib, case)
    rc, errs = _errors(lib)
    assert rc == PA_ERR_TIMEOUT and errs & DEVERR_TIMEOUT, (rc, errs)
    assert lib.pa_test_hook(-1, -1, 0) == PA_OK
    good = _prefill(lib, case)
    assert _errors(lib) == (PA_OK, 0)
    want = cuda_lib.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0],
                                  q_start, True, case.scale)
    assert torch.equal(good, want)
    ref = oracle.prefill(bits(case.q), bits(case.k_cache), bits(case.v_cache),
                         case.block_table[0].cpu().numpy(), q_start, True, case.scale)
    assert_attention_close(good, ref, "prefill after a timed-out call")
    assert cuda_lib.device_errors() == 0


@pytest.mark.parametrize("seq_len", [1537, 1553, 1665, 1696])
def test_decode_late_consumers_with_a_reloaded_stage(test_lib, cuda_lib, seq_len):
    # A split whose only stage holds the token being decoded loads that stage twice (the
    # second time after the token's K/V are written).  Consumer warps that start only
    # after both loads have landed must still take the second load: it completes on a
    # barrier of its own, since an mbarrier wait tells only two phases apart.  The test
    # build holds the consumers back 30 us; with both loads on one barrier they waited
    # for a phase that had already passed, until their wait ran out.
    lib = test_lib
    bs = 832
    case = workloads.paged_case(73, [seq_len], bs, 8, new_tokens=1, device="cuda")
    k_ref, v_ref = bits(case.k_cache).copy(), bits(case.v_cache).copy()
    slots_h = oracle.slot_mapping(case.positions.cpu().numpy(), case.block_table.cpu().numpy(),
                                  bs, case.seq_idx.cpu().numpy())
    oracle.reshape_and_cache(bits(case.new_k), bits(case.new_v), k_ref, v_ref, slots_h, bs)
    slots = cuda_lib.slot_mapping(case.positions, case.block_table, bs, seq_idx=case.seq_idx)
    torch.cuda.synchronize()
    assert lib.pa_test_hook(-1, -1, 30000) == PA_OK
    S, hq, d = case.q.shape
    out = torch.empty_like(case.q)
    ws = torch.empty(max(256, lib.pa_decode_workspace_size(S, hq, 4, d, bs, seq_len)),
                     dtype=torch.uint8, device="cuda")
    rc = lib.pa_decode(case.q.data_ptr(), case.k_cache.data_ptr(), case.v_cache.data_ptr(),
                       case.k_cache.stride(0), case.k_cache.shape[0],
                       case.block_table.data_ptr(), case.block_table.stride(0),
                       case.seq_lens.data_ptr(), S, seq_len, hq, 4, d, bs, case.scale,
                       out.data_ptr(), ws.data_ptr(), ws.numel(), case.new_k.data_ptr(),
                       case.new_v.data_ptr(), slots.data_ptr(), _stream())
    assert rc == PA_OK
    assert _errors(lib) == (PA_OK, 0)
    assert lib.pa_test_hook(-1, -1, 0) == PA_OK
    assert np.array_equal(bits(case.k_cache), k_ref) and np.array_equal(bits(case.v_cache), v_ref)
    ref = oracle.decode(bits(case.q), k_ref, v_ref, case.block_table.cpu().numpy(),
                        case.seq_lens.cpu().numpy(), case.scale)
    assert_attention_close(out, ref, f"late consumers, reloaded stage, L={seq_len}")


def test_prefill_split_and_packed_wait_that_runs_out(test_lib, cuda_lib):
    # The extended prefill kernel (items split into pieces, a packed last tile) on the
    # same failure path: one row over 8000 prior keys runs as 4 packed items cut into
    # pieces, and every CTA loses its K/V ring unit 1.  The merge kernel then combines
    # whatever the pieces left; the test checks the error and the next call.
    lib = test_lib
    q_len, q_start, bs = 1, 8000, 832
    case = workloads.paged_case(378, [q_start + q_len], bs, 12, q_rows=q_len, q_start=q_start,
                                device="cuda")
    slots = cuda_lib.slot_mapping(case.positions, case.block_table, bs, seq_idx=case.seq_idx)
    cuda_lib.reshape_and_cache(case.new_k, case.new_v, case.k_cache, case.v_cache, slots)
    torch.cuda.synchronize()
    need = lib.pa_prefill_workspace_size(q_len, q_start, 1, 24, 4, 256, bs)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert _errors(lib) == (PA_OK, 0)
    assert lib.pa_test_hook(-1, 1, 0) == PA_OK
    _prefill(lib, case, ws)
    rc, errs = _errors(lib)
    assert rc == PA_ERR_TIMEOUT and errs & DEVERR_TIMEOUT, (rc, errs)
    assert lib.pa_test_hook(-1, -1, 0) == PA_OK
    good = _prefill(lib, case, ws)
    assert _errors(lib) == (PA_OK, 0)
    ref = oracle.prefill(bits(case.q), bits(case.k_cache), bits(case.v_cache),
                         case.block_table[0].cpu().numpy(), q_start, True, case.scale)
    assert_attention_close(good, ref, "split, packed prefill after a timed-out call")
    assert cuda_lib.device_errors() == 0
