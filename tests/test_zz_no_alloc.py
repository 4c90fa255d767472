"""pa_decode_noalloc: decode for callers that cannot allocate device memory (for example a
runtime that hands nearly all device memory to its KV-cache pool at start-up).  It takes
its scratch from a fixed array inside the library instead of a caller workspace.

Called here straight through the C ABI and compared with pa_decode (the entry point with
a caller workspace) on the same inputs, twice in a row, within the attention tolerance
the other tests use; also checked against the oracle, and for the refusal of problems
whose partials exceed the fixed array.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import assert_attention_close, attention_errors
from workloads import bits

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 << 20
PA_ERR_UNSUPPORTED = 2


def _noalloc_fn(pa):
    lib = pa.load()
    fn = lib.pa_decode_noalloc
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    fn.argtypes = [P, P, P, i64, i64, P, i64, P, i32, i32, i32, i32, i32, i32, ctypes.c_float,
                   P, P]
    fn.restype = i32
    return fn


def _call_noalloc(pa, case, out, max_seq_len, num_seqs=None):
    fn = _noalloc_fn(pa)
    S, hq, d = case.q.shape
    _, bs, hkv, _ = case.k_cache.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctypes.c_void_p(case.q.data_ptr()), ctypes.c_void_p(case.k_cache.data_ptr()),
              ctypes.c_void_p(case.v_cache.data_ptr()), case.k_cache.stride(0), case.num_pages,
              ctypes.c_void_p(case.block_table.data_ptr()), case.block_table.stride(0),
              ctypes.c_void_p(case.seq_lens.data_ptr()), S if num_seqs is None else num_seqs,
              max_seq_len, hq, hkv, d, bs, case.scale, ctypes.c_void_p(out.data_ptr()), stream)


@pytest.mark.parametrize("make", ["decode_8k", "batched_decode"])
def test_noalloc_matches_pa_decode_twice(cuda_lib, make):
    pa = cuda_lib
    case = getattr(workloads, make)(device="cuda")
    msl = int(case.seq_lens.max())
    assert pa.decode_workspace_size(case.q.shape[0], 24, 4, 256, case.block_size,
                                    msl) <= SCRATCH_BYTES
    ref = pa.decode(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                    case.scale, msl)
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(case.q, float("nan"))
        assert _call_noalloc(pa, case, out, msl) == 0
        torch.cuda.synchronize()
        e = attention_errors(out, ref.double().cpu().numpy())
        assert e["finite"] and e["max_abs"] <= 1e-2 and e["max_rel"] <= 2e-2, e
    assert pa.device_errors() == 0


def test_noalloc_matches_oracle_after_a_different_problem(cuda_lib):
    # The shared array keeps the last call's contents; a call on another problem size must
    # not be affected by them.
    pa = cuda_lib
    big = workloads.decode_8k(784, device="cuda")
    out_big = torch.empty_like(big.q)
    assert _call_noalloc(pa, big, out_big, 8192) == 0
    case = workloads.paged_case(61, [300, 2000, 1], 832, 8, device="cuda")
    out = torch.empty_like(case.q)
    assert _call_noalloc(pa, case, out, 2000) == 0
    torch.cuda.synchronize()
    ref = oracle.decode(bits(case.q), bits(case.k_cache), bits(case.v_cache),
                        case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(), case.scale)
    assert_attention_close(out, ref, "noalloc vs oracle")


def test_noalloc_refuses_problems_beyond_the_fixed_scratch(cuda_lib):
    pa = cuda_lib
    case = workloads.decode_8k(832, device="cuda")
    out = torch.zeros_like(case.q)
    # 400 sequences of 24 heads need more partial space than the fixed array holds; the
    # call must refuse before touching any pointer (only sizes are looked at).
    assert pa.decode_workspace_size(400, 24, 4, 256, 832, 8192) > SCRATCH_BYTES
    assert _call_noalloc(pa, case, out, 8192, num_seqs=400) == PA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert not out.float().abs().sum().item()
