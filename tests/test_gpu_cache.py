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


def _prep_case(S, block_sizes, seed, pad_every=0):
    """Positions and one random block table per KV-cache group (row s = sequence s)."""
    rng = np.random.default_rng(seed)
    pos = rng.integers(0, 20000, S).astype(np.int32)
    if pad_every:
        pos[::pad_every] = -1
    tables = []
    for bs in block_sizes:
        mb = 20000 // bs + 1
        tables.append(rng.permutation(S * mb + 7)[:S * mb].astype(np.int32).reshape(S, mb))
    sampled = rng.integers(0, 150000, S).astype(np.int32)
    return pos, tables, sampled


@pytest.mark.parametrize("S,block_sizes", [(1, [832]), (1, [832, 16]), (16, [832, 784, 16]),
                                           (300, [64, 832]), (5, [1, 7, 832, 784, 64, 16, 2, 3]),
                                           (1000, [16, 16])])
def test_decode_input_prep_matches_oracle(cuda_lib, S, block_sizes):
    pa = cuda_lib
    pos, tables, sampled = _prep_case(S, block_sizes, 50 + S + len(block_sizes), pad_every=4)
    got = pa.decode_input_prep(torch.from_numpy(pos).cuda(),
                               [torch.from_numpy(t).cuda() for t in tables], block_sizes,
                               sampled_ids=torch.from_numpy(sampled).cuda())
    want = oracle.decode_input_prep(pos, tables, block_sizes, sampled_ids=sampled)
    for k in ("seq_lens", "query_start_loc", "input_ids"):
        assert np.array_equal(got[k].cpu().numpy(), want[k]), k
    for g in range(len(block_sizes)):
        assert np.array_equal(got["slot_mappings"][g].cpu().numpy(), want["slot_mappings"][g])
    assert pa.device_errors() == 0


def test_decode_input_prep_one_request_in_padded_buffers(cuda_lib):
    # The input-prep post's step: one request at position 24576, two groups of block size
    # 16, buffers for 128 requests.  query_start_loc = [0, 1, 1, ...], seq_lens =
    # [24577, 0, 0, ...], bit for bit with the oracle.
    pa = cuda_lib
    pos = np.full(128, -1, np.int32)
    pos[0] = 24576
    cols = np.arange(1600)[None, :]
    rows = np.arange(128)[:, None] * 10000
    tables = [(3 * cols + 1 + rows).astype(np.int32), (2 * cols + 7 + rows).astype(np.int32)]
    sampled = np.zeros(128, np.int32)
    sampled[0] = 42
    got = pa.decode_input_prep(torch.from_numpy(pos).cuda(),
                               [torch.from_numpy(t).cuda() for t in tables], [16, 16],
                               sampled_ids=torch.from_numpy(sampled).cuda())
    want = oracle.decode_input_prep(pos, tables, [16, 16], sampled_ids=sampled)
    assert got["query_start_loc"].tolist() == [0] + [1] * 128
    for k in ("seq_lens", "query_start_loc", "input_ids"):
        assert np.array_equal(got[k].cpu().numpy(), want[k]), k
    for g in range(2):
        assert np.array_equal(got["slot_mappings"][g].cpu().numpy(), want["slot_mappings"][g])
    assert pa.device_errors() == 0


def test_decode_input_prep_reports_positions_past_the_table(cuda_lib):
    pa = cuda_lib
    pos = torch.tensor([100, 5000, 70], dtype=torch.int32, device="cuda")
    t0 = torch.tensor([[3, 4], [5, 6], [-2, 7]], dtype=torch.int32, device="cuda")  # BS 832
    t1 = torch.arange(3 * 400, dtype=torch.int32, device="cuda").reshape(3, 400)    # BS 16
    got = pa.decode_input_prep(pos, [t0, t1], [832, 16])
    # seq 1: 5000 // 832 = 6 >= 2 entries in group 0 -> -1; group 1 entry 312 is fine.
    # seq 2: group 0 entry is negative -> -1.
    assert got["slot_mappings"][0].tolist() == [3 * 832 + 100, -1, -1]
    assert got["slot_mappings"][1].tolist() == [6 * 16 + 4, (400 + 312) * 16 + 8,
                                                (800 + 4) * 16 + 6]
    assert got["seq_lens"].tolist() == [101, 5001, 71]
    assert pa.device_errors() == pa.DEVERR_POSITION


def test_decode_input_prep_feeds_the_fused_decode(cuda_lib):
    # The step of a two-group model: input prep writes seq_lens and both groups' slots in
    # one launch; the attention layer of group 0 then decodes with the fused write.
    pa = cuda_lib
    from _util import assert_attention_close
    case = workloads.batched_decode("cuda")
    k_before, v_before = bits(case.k_cache), bits(case.v_cache)
    positions = (case.seq_lens - 1).to(torch.int32)
    S = positions.shape[0]
    other = torch.arange(S * 2100, dtype=torch.int32, device="cuda").reshape(S, 2100)  # BS 16
    prep = pa.decode_input_prep(positions, [case.block_table, other], [case.block_size, 16])
    assert torch.equal(prep["seq_lens"], case.seq_lens)
    msl = int(case.seq_lens.max())
    out = pa.decode(case.q, case.k_cache, case.v_cache, case.block_table, prep["seq_lens"],
                    case.scale, msl, new_k=case.new_k, new_v=case.new_v,
                    new_slots=prep["slot_mappings"][0])
    torch.cuda.synchronize()
    slots = oracle.slot_mapping(positions.cpu().numpy(), case.block_table.cpu().numpy(),
                                case.block_size, np.arange(S, dtype=np.int32))
    assert np.array_equal(prep["slot_mappings"][0].cpu().numpy(), slots)
    oracle.reshape_and_cache(bits(case.new_k), bits(case.new_v), k_before, v_before, slots,
                             case.block_size)
    assert np.array_equal(bits(case.k_cache), k_before)
    assert np.array_equal(bits(case.v_cache), v_before)
    ref = oracle.decode(bits(case.q), k_before, v_before, case.block_table.cpu().numpy(),
                        case.seq_lens.cpu().numpy(), case.scale)
    assert_attention_close(out, ref, "decode after input prep")
    assert pa.device_errors() == 0
