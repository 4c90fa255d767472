"""Slot mapping and KV write on the GPU vs the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import bits

pytestmark = pytest.mark.gpu


def _host(case):
    return dict(k=bits(case.k_cache), v=bits(case.v_cache), bt=case.block_table.cpu().numpy(),
                sl=case.seq_lens.cpu().numpy())


def test_slot_mapping_tiny_matches_oracle_and_hand_value(cuda_lib):
    pa = cuda_lib
    case = workloads.tiny_decode("cuda")
    got = pa.slot_mapping(case.positions, case.block_table, 832, seq_idx=case.seq_idx)
    bt = case.block_table.cpu().numpy()
    want = oracle.slot_mapping(case.positions.cpu().numpy(), bt, 832,
                               seq_idx=case.seq_idx.cpu().numpy())
    assert got.dtype == torch.int64
    assert np.array_equal(got.cpu().numpy(), want)
    # Token 1700 with 832-token pages: logical page 2, offset 36.
    assert int(got[0]) == int(bt[0, 2]) * 832 + 36
    assert pa.device_errors() == 0


@pytest.mark.parametrize("make", ["prefill_chunk", "batched_decode"])
def test_slot_mapping_matches_oracle(cuda_lib, make):
    pa = cuda_lib
    case = getattr(workloads, make)("cuda")
    got = pa.slot_mapping(case.positions, case.block_table, case.block_size,
                          seq_idx=case.seq_idx)
    want = oracle.slot_mapping(case.positions.cpu().numpy(), case.block_table.cpu().numpy(),
                               case.block_size, seq_idx=case.seq_idx.cpu().numpy())
    assert np.array_equal(got.cpu().numpy(), want)
    assert pa.device_errors() == 0


@pytest.mark.parametrize("bs", [784, 832, 64, 16, 1])
def test_slot_mapping_random_positions(cuda_lib, bs):
    pa = cuda_lib
    g = torch.Generator().manual_seed(bs)
    S, mb = 5, 12
    bt = torch.randperm(S * mb, generator=g).to(torch.int32).view(S, mb)
    n = 3000
    seq = torch.randint(0, S, (n,), generator=g, dtype=torch.int32)
    pos = torch.randint(0, mb * bs, (n,), generator=g, dtype=torch.int32)
    got = pa.slot_mapping(pos.cuda(), bt.cuda(), bs, seq_idx=seq.cuda())
    want = oracle.slot_mapping(pos.numpy(), bt.numpy(), bs, seq_idx=seq.numpy())
    assert np.array_equal(got.cpu().numpy(), want)
    assert pa.device_errors() == 0


def test_slot_mapping_padding_and_out_of_range(cuda_lib):
    pa = cuda_lib
    bt = torch.tensor([[4, 9, -1]], dtype=torch.int32, device="cuda")
    pos = torch.tensor([-1, 0, 17, 40, 100], dtype=torch.int32, device="cuda")
    got = pa.slot_mapping(pos, bt, 16)
    # -1: padding; 0 -> page 4; 17 -> page 9 offset 1; 40 -> entry -1 (unmapped);
    # 100 -> logical page 6 beyond the 3-entry row.
    assert got.cpu().tolist() == [-1, 64, 145, -1, -1]
    assert pa.device_errors() == pa.DEVERR_POSITION
    assert pa.device_errors() == 0


def _check_write(pa, case, key, value, slots_gpu, page_stride_mult=1):
    host = _host(case)
    k0, v0 = host["k"].copy(), host["v"].copy()
    pa.reshape_and_cache(key, value, case.k_cache, case.v_cache, slots_gpu)
    torch.cuda.synchronize()
    oracle.reshape_and_cache(bits(key), bits(value), k0, v0, slots_gpu.cpu().numpy(),
                             case.block_size)
    assert np.array_equal(bits(case.k_cache), k0)
    assert np.array_equal(bits(case.v_cache), v0)


@pytest.mark.parametrize("make", ["tiny_decode", "prefill_chunk", "batched_decode"])
def test_reshape_and_cache_bit_exact(cuda_lib, make):
    pa = cuda_lib
    case = getattr(workloads, make)("cuda")
    slots = pa.slot_mapping(case.positions, case.block_table, case.block_size,
                            seq_idx=case.seq_idx)
    _check_write(pa, case, case.new_k, case.new_v, slots)
    assert pa.device_errors() == 0


def test_reshape_and_cache_unbind_views_and_padding(cuda_lib):
    pa = cuda_lib
    g = torch.Generator(device="cuda").manual_seed(5)
    npg, bs, hkv, d = 6, 16, 4, 256
    kv = torch.randn(npg, 2, bs, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    k_cache, v_cache = kv.unbind(1)
    assert k_cache.stride(0) == 2 * bs * hkv * d
    T = 9
    key = torch.randn(T, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    val = torch.randn(T, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    slots = torch.tensor([0, 17, -1, 95, 40, 41, -1, 63, 64], dtype=torch.int64, device="cuda")
    before = bits(kv).copy()
    pa.reshape_and_cache(key, val, k_cache, v_cache, slots)
    after = bits(kv)
    kb, vb = bits(key), bits(val)
    want = before.copy()
    for i, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        want[s // bs, 0, s % bs] = kb[i]
        want[s // bs, 1, s % bs] = vb[i]
    assert np.array_equal(after, want)
    # A slot beyond the pool is skipped and reported.
    bad = torch.tensor([npg * bs + 3], dtype=torch.int64, device="cuda")
    pa.reshape_and_cache(key[:1], val[:1], k_cache, v_cache, bad)
    assert pa.device_errors() == pa.DEVERR_SLOT
    assert np.array_equal(bits(kv), want)
