"""Chunked causal prefill on the GPU vs the fp64 oracle: small shapes compared on every
element (several query and key tiles, ragged tails, page sizes 784/832/64/16); the
full-size chunks (q=4096 over 4096 prior tokens, the q=1685 tail over 12288, the q=4096
first chunk, a mixed batch of four chunks) on every element, and quick variants of them
on sampled (row, head) outputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import assert_attention_close
from workloads import bits

pytestmark = pytest.mark.gpu


def _write_chunk(pa, case):
    """The chunk's own K/V go into the cache first, through the library."""
    slots = pa.slot_mapping(case.positions, case.block_table, case.block_size,
                            seq_idx=case.seq_idx)
    pa.reshape_and_cache(case.new_k, case.new_v, case.k_cache, case.v_cache, slots)
    return slots


def _oracle_caches_after_write(case, k_host, v_host):
    sl = oracle.slot_mapping(case.positions.cpu().numpy(), case.block_table.cpu().numpy(),
                             case.block_size, seq_idx=case.seq_idx.cpu().numpy())
    oracle.reshape_and_cache(bits(case.new_k), bits(case.new_v), k_host, v_host, sl,
                             case.block_size)
    return k_host, v_host


@pytest.mark.parametrize("bs,q_len,q_start", [
    (832, 1, 0), (832, 64, 0), (832, 65, 3), (832, 200, 100), (832, 130, 1000),
    (784, 300, 700), (784, 64, 784), (64, 129, 63), (16, 77, 40), (16, 1, 500),
    # fewer items than SMs over long contexts: items split along the keys into pieces on
    # different SMs, merged afterwards
    (832, 1, 8192), (832, 64, 8192), (784, 200, 3000), (16, 40, 5000),
])
def test_prefill_small_every_element(cuda_lib, bs, q_len, q_start):
    pa = cuda_lib
    npg = -(-(q_start + q_len) // bs) + 3
    case = workloads.paged_case(300 + q_len + q_start, [q_start + q_len], bs, npg,
                                q_rows=q_len, q_start=q_start, device="cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    out = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0], q_start,
                           True, case.scale)
    ref = oracle.prefill(bits(case.q), k_host, v_host, case.block_table[0].cpu().numpy(),
                         q_start, True, case.scale)
    assert_attention_close(out, ref, f"prefill bs={bs} q={q_len}@{q_start}")
    assert pa.device_errors() == 0


@pytest.mark.parametrize("bs,q_len,q_start", [(832, 100, 900), (64, 70, 0)])
def test_prefill_non_causal(cuda_lib, bs, q_len, q_start):
    pa = cuda_lib
    npg = -(-(q_start + q_len) // bs) + 2
    case = workloads.paged_case(500 + q_len, [q_start + q_len], bs, npg, q_rows=q_len,
                                q_start=q_start, device="cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    out = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0], q_start,
                           False, case.scale)
    ref = oracle.prefill(bits(case.q), k_host, v_host, case.block_table[0].cpu().numpy(),
                         q_start, False, case.scale)
    assert_attention_close(out, ref, "non-causal")


@pytest.mark.parametrize("make", ["prefill_chunk", "prefill_tail", "prefill_first"])
def test_prefill_full_chunk_sampled(cuda_lib, make):
    # The q=4096 chunk over 4096 prior tokens, the q=1685 tail chunk over 12288 and the
    # q=4096 first chunk, at full size: sampled rows (the first and last of several
    # 64- and 128-row tiles, and random ones) against the oracle, one by one.
    pa = cuda_lib
    case = getattr(workloads, make)("cuda")
    q_len = case.q.shape[0]
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    out = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0],
                           case.q_start, True, case.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    # The GPU's copy of the cache after its own write is the oracle's copy, bit for bit.
    assert np.array_equal(bits(case.k_cache), k_host)
    assert np.array_equal(bits(case.v_cache), v_host)
    rng = np.random.default_rng(q_len + case.q_start)
    fixed = [r for r in (0, 1, 63, 64, 65, 127, 128, 1536, 1663, 1664, 1684, 2047, 2048,
                         4032, 4094, 4095) if r < q_len]
    rows = np.concatenate([fixed, rng.integers(0, q_len, 180)]).astype(np.int32)
    heads = rng.integers(0, 24, rows.size).astype(np.int32)
    heads[:len(fixed)] = (np.arange(len(fixed)) * 5 + 1) % 24
    ref = oracle.prefill_rows(bits(case.q), k_host, v_host, case.block_table[0].cpu().numpy(),
                              case.q_start, True, case.scale, rows, heads)
    got = out[torch.from_numpy(rows).long().cuda(), torch.from_numpy(heads).long().cuda()]
    assert_attention_close(got, ref, f"{make} (sampled)")
    assert pa.device_errors() == 0
    again = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0],
                             case.q_start, True, case.scale)
    assert torch.equal(out, again)                         # deterministic


def test_prefill_unbind_views(cuda_lib):
    pa = cuda_lib
    q_len, q_start, bs = 150, 900, 832
    case = workloads.paged_case(42, [q_start + q_len], bs, 5, q_rows=q_len, q_start=q_start,
                                device="cuda")
    _write_chunk(pa, case)
    kv = torch.stack([case.k_cache, case.v_cache], dim=1)
    kview, vview = kv.unbind(1)
    a = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0], q_start,
                         True, case.scale)
    b = pa.prefill_chunk(case.q, kview, vview, case.block_table[0], q_start, True, case.scale)
    assert torch.equal(a, b)


def test_prefill_row_equals_decode_of_its_prefix(cuda_lib):
    # The last chunk row at position p attends to the same keys as a decode with p+1 keys.
    pa = cuda_lib
    q_len, q_start, bs = 40, 1200, 832
    case = workloads.paged_case(43, [q_start + q_len], bs, 6, q_rows=q_len, q_start=q_start,
                                device="cuda")
    _write_chunk(pa, case)
    out = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0], q_start,
                           True, case.scale)
    sl = torch.tensor([q_start + q_len], dtype=torch.int32, device="cuda")
    dec = pa.decode(case.q[-1:].contiguous(), case.k_cache, case.v_cache, case.block_table, sl,
                    case.scale, q_start + q_len)
    d = (out[-1].float() - dec[0].float()).abs().max().item()
    assert d <= 1e-2


# ------------------------------------------------------------------ mixed batches (varlen)
VARLEN = [
    # block size, chunk rows per sequence, keys per sequence, causal
    (832, [130, 1, 257], [900, 1, 257], True),
    (784, [64, 0, 300, 5], [784, 100, 1000, 5], True),
    (16, [33, 70], [40, 200], False),
    (64, [1, 2, 3, 200, 129, 128, 127], [1, 70, 64, 200, 500, 128, 1000], True),
]


@pytest.mark.parametrize("bs,q_rows,k_lens,causal", VARLEN)
def test_prefill_varlen_every_element(cuda_lib, bs, q_rows, k_lens, causal):
    pa = cuda_lib
    npg = sum(-(-L // bs) for L in k_lens) + 3
    case = workloads.paged_case(500 + sum(q_rows), k_lens, bs, npg, q_rows=q_rows, device="cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    cu = case.meta["cu_seqlens_q"]
    out = pa.prefill_varlen(case.q, case.k_cache, case.v_cache, case.block_table, cu, k_lens,
                            causal, case.scale)
    ref = oracle.prefill_varlen(bits(case.q), k_host, v_host, case.block_table.cpu().numpy(),
                                cu, k_lens, causal, case.scale)
    assert_attention_close(out, ref, f"varlen bs={bs} {q_rows}")
    assert pa.device_errors() == 0


def test_prefill_varlen_more_chunks_than_one_launch_takes(cuda_lib):
    # 45 non-empty chunks (and 2 empty ones) run as two launches of at most 32 chunks.
    pa = cuda_lib
    rng = np.random.default_rng(45)
    k_lens = rng.integers(1, 300, 47).tolist()
    q_rows = [int(rng.integers(1, L + 1)) for L in k_lens]
    q_rows[5] = q_rows[30] = 0
    bs = 64
    npg = sum(-(-L // bs) for L in k_lens) + 2
    case = workloads.paged_case(4545, k_lens, bs, npg, q_rows=q_rows, device="cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    cu = case.meta["cu_seqlens_q"]
    out = pa.prefill_varlen(case.q, case.k_cache, case.v_cache, case.block_table, cu, k_lens,
                            True, case.scale)
    ref = oracle.prefill_varlen(bits(case.q), k_host, v_host, case.block_table.cpu().numpy(),
                                cu, k_lens, True, case.scale)
    assert_attention_close(out, ref, "varlen, 45 chunks")
    assert pa.device_errors() == 0


def test_prefill_varlen_of_one_sequence_is_prefill_chunk(cuda_lib):
    pa = cuda_lib
    case = workloads.paged_case(77, [1000], 832, 5, q_rows=700, q_start=300, device="cuda")
    _write_chunk(pa, case)
    a = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0], 300, True,
                         case.scale)
    b = pa.prefill_varlen(case.q, case.k_cache, case.v_cache, case.block_table, [0, 700],
                          [1000], True, case.scale)
    assert torch.equal(a, b)


def test_prefill_mixed_batch_full_size_sampled(cuda_lib):
    # Four chunks of a serving step (1024 rows over 3072 keys, 4096 over 8192, the 1685-row
    # tail over 13973, a whole 512-token prompt): sampled rows of every chunk.
    pa = cuda_lib
    case = workloads.prefill_mixed("cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    cu, k_lens = case.meta["cu_seqlens_q"], case.meta["seq_lens"]
    out = pa.prefill_varlen(case.q, case.k_cache, case.v_cache, case.block_table, cu, k_lens,
                            True, case.scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7317)
    bt = case.block_table.cpu().numpy()
    for b in range(len(k_lens)):
        q_len = cu[b + 1] - cu[b]
        rows = np.concatenate([[0, q_len - 1, min(127, q_len - 1), min(128, q_len - 1)],
                               rng.integers(0, q_len, 40)]).astype(np.int32)
        heads = rng.integers(0, 24, rows.size).astype(np.int32)
        ref = oracle.prefill_rows(bits(case.q[cu[b]:cu[b + 1]]), k_host, v_host, bt[b],
                                  k_lens[b] - q_len, True, case.scale, rows, heads)
        got = out[torch.from_numpy(rows + cu[b]).long().cuda(), torch.from_numpy(heads).long().cuda()]
        assert_attention_close(got, ref, f"mixed batch, chunk {b} (sampled)")
    assert pa.device_errors() == 0


# ------------------------------------------------------------------ full size, every element
def _full_chunk(pa, make):
    case = getattr(workloads, make)("cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    return case, k_host, v_host


@pytest.mark.parametrize("make", ["prefill_chunk", "prefill_tail", "prefill_first"])
def test_prefill_full_chunk_every_element(cuda_lib, make):
    # The full-size chunks in the launch the benchmark times (all items of the planned
    # schedule: several items per CTA, items of up to 55 tiles, the ragged last q tile of
    # the tail chunk), every output against the oracle.
    pa = cuda_lib
    case, k_host, v_host = _full_chunk(pa, make)
    out = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0],
                           case.q_start, True, case.scale)
    torch.cuda.synchronize()
    ref = oracle.prefill(bits(case.q), k_host, v_host, case.block_table[0].cpu().numpy(),
                         case.q_start, True, case.scale)
    e = assert_attention_close(out, ref, f"{make} (every element)")
    print(f"{make}: {ref.size} outputs, max_abs={e['max_abs']:.3g} max_rel={e['max_rel']:.3g} "
          f"rel_l2={e['rel_l2']:.3g}")
    assert pa.device_errors() == 0


def test_prefill_mixed_batch_full_size_every_element(cuda_lib):
    pa = cuda_lib
    case, k_host, v_host = _full_chunk(pa, "prefill_mixed")
    cu, k_lens = case.meta["cu_seqlens_q"], case.meta["seq_lens"]
    out = pa.prefill_varlen(case.q, case.k_cache, case.v_cache, case.block_table, cu, k_lens,
                            True, case.scale)
    torch.cuda.synchronize()
    ref = oracle.prefill_varlen(bits(case.q), k_host, v_host, case.block_table.cpu().numpy(),
                                cu, k_lens, True, case.scale)
    e = assert_attention_close(out, ref, "mixed batch (every element)")
    print(f"mixed batch: {ref.size} outputs, max_abs={e['max_abs']:.3g} "
          f"max_rel={e['max_rel']:.3g} rel_l2={e['rel_l2']:.3g}")
    assert pa.device_errors() == 0


@pytest.mark.parametrize("bs,q_len,q_start", [(832, 64, 8192), (784, 200, 3000)])
def test_prefill_split_items_match_the_unsplit_plan(cuda_lib, bs, q_len, q_start):
    # The same chunk with a workspace (items split into pieces and merged) and without
    # (whole items): both within the tolerance of the oracle and of each other, and the
    # split form deterministic.
    pa = cuda_lib
    npg = -(-(q_start + q_len) // bs) + 2
    case = workloads.paged_case(600 + q_len, [q_start + q_len], bs, npg, q_rows=q_len,
                                q_start=q_start, device="cuda")
    _write_chunk(pa, case)
    need = pa.prefill_workspace_size(q_len, q_start, True, 24, 4, 256, bs)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    split = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0], q_start,
                             True, case.scale, workspace=ws)
    ws.fill_(0xFF)  # NaN bytes: the next call must not read what this one left
    again = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0], q_start,
                             True, case.scale, workspace=ws)
    whole = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0], q_start,
                             True, case.scale, workspace=torch.empty(0, dtype=torch.uint8,
                                                                     device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(split, again)
    e = (split.float() - whole.float()).abs().max().item()
    assert e <= 1e-2, e
    assert pa.device_errors() == 0


def test_prefill_varlen_split_items(cuda_lib):
    # Three one-row chunks and a 40-row chunk over 5000-7000 keys: 96 items for 152 SMs,
    # split into pieces; every element against the oracle.
    pa = cuda_lib
    k_lens, q_rows, bs = [6000, 5000, 7000, 5500], [1, 1, 40, 1], 832
    npg = sum(-(-L // bs) for L in k_lens) + 2
    case = workloads.paged_case(4242, k_lens, bs, npg, q_rows=q_rows, device="cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    cu = case.meta["cu_seqlens_q"]
    assert pa.prefill_varlen_workspace_size(cu, k_lens, True, 24, 4, 256, bs) > 0
    out = pa.prefill_varlen(case.q, case.k_cache, case.v_cache, case.block_table, cu, k_lens,
                            True, case.scale)
    ref = oracle.prefill_varlen(bits(case.q), k_host, v_host, case.block_table.cpu().numpy(),
                                cu, k_lens, True, case.scale)
    assert_attention_close(out, ref, "varlen with split items")
    assert pa.device_errors() == 0


def test_prefill_non_causal_split_items(cuda_lib):
    # Non-causal rows see every key; 24 items of ~28 tiles on 152 SMs are split.
    pa = cuda_lib
    q_len, q_start, bs = 100, 6000, 832
    assert pa.prefill_workspace_size(q_len, q_start, False, 24, 4, 256, bs) > 0
    npg = -(-(q_start + q_len) // bs) + 2
    case = workloads.paged_case(7100, [q_start + q_len], bs, npg, q_rows=q_len, q_start=q_start,
                                device="cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    out = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0], q_start,
                           False, case.scale)
    ref = oracle.prefill(bits(case.q), k_host, v_host, case.block_table[0].cpu().numpy(),
                         q_start, False, case.scale)
    assert_attention_close(out, ref, "non-causal, split items")
    assert pa.device_errors() == 0


def test_prefill_varlen_split_items_over_two_launches(cuda_lib):
    # 40 one-row chunks over 2000-4000 keys: two launches (32 + 8 chunks), each with split
    # items, one after the other on the same workspace; every element against the oracle.
    pa = cuda_lib
    rng = np.random.default_rng(40)
    k_lens = rng.integers(2000, 4001, 40).tolist()
    q_rows = [1] * 40
    bs = 832
    npg = sum(-(-L // bs) for L in k_lens) + 2
    case = workloads.paged_case(4040, k_lens, bs, npg, q_rows=q_rows, device="cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    cu = case.meta["cu_seqlens_q"]
    assert pa.prefill_varlen_workspace_size(cu, k_lens, True, 24, 4, 256, bs) > 0
    out = pa.prefill_varlen(case.q, case.k_cache, case.v_cache, case.block_table, cu, k_lens,
                            True, case.scale)
    ref = oracle.prefill_varlen(bits(case.q), k_host, v_host, case.block_table.cpu().numpy(),
                                cu, k_lens, True, case.scale)
    assert_attention_close(out, ref, "varlen, two launches with split items")
    assert pa.device_errors() == 0


@pytest.mark.parametrize("hq,hkv,q_len,q_start,bs", [
    # a short last query tile runs as items of several heads of a KV head
    (24, 4, 21, 700, 832), (24, 4, 22, 700, 832), (24, 4, 149, 900, 784),
    (8, 4, 64, 300, 64), (8, 4, 65, 300, 64), (8, 1, 136, 1000, 832),
    (16, 2, 16, 2000, 16), (4, 4, 1, 900, 832), (32, 4, 16, 0, 832),
    (24, 8, 40, 500, 832), (20, 4, 25, 300, 64), (28, 4, 146, 1000, 784),
    # tails too long for the whole group: 3 heads per item (22..42 rows), 2 (43..64)
    (24, 4, 40, 8000, 832), (24, 4, 60, 900, 784), (24, 4, 128 + 30, 2000, 64),
    (32, 4, 20, 1000, 832), (16, 4, 40, 3000, 832), (24, 4, 64, 7000, 832),
])
def test_prefill_packed_last_tile_every_element(cuda_lib, hq, hkv, q_len, q_start, bs):
    pa = cuda_lib
    npg = -(-(q_start + q_len) // bs) + 2
    case = workloads.paged_case(900 + q_len + hq, [q_start + q_len], bs, npg, q_rows=q_len,
                                q_start=q_start, hq=hq, hkv=hkv, device="cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    ref = oracle.prefill(bits(case.q), k_host, v_host, case.block_table[0].cpu().numpy(),
                         q_start, True, case.scale)
    for ws in (None, torch.empty(0, dtype=torch.uint8, device="cuda")):  # split, whole
        out = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0],
                               q_start, True, case.scale, workspace=ws)
        assert_attention_close(out, ref, f"packed tile hq={hq} hkv={hkv} q={q_len}@{q_start}")
    assert pa.device_errors() == 0


def test_prefill_packed_last_tile_non_causal_and_varlen(cuda_lib):
    # Non-causal packed items, and a mixed batch whose chunks end in short tiles (3, 21
    # and 1 rows, packed) beside one that does not (50 rows).
    pa = cuda_lib
    case = workloads.paged_case(4321, [3021], 832, 6, q_rows=21, q_start=3000, device="cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    out = pa.prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table[0], 3000,
                           False, case.scale)
    ref = oracle.prefill(bits(case.q), k_host, v_host, case.block_table[0].cpu().numpy(),
                         3000, False, case.scale)
    assert_attention_close(out, ref, "packed tile, non-causal")
    k_lens, q_rows, bs = [131, 4000, 6000, 50], [131, 21, 1, 50], 832
    npg = sum(-(-L // bs) for L in k_lens) + 2
    case = workloads.paged_case(4322, k_lens, bs, npg, q_rows=q_rows, device="cuda")
    k_host, v_host = _oracle_caches_after_write(case, bits(case.k_cache), bits(case.v_cache))
    _write_chunk(pa, case)
    cu = case.meta["cu_seqlens_q"]
    out = pa.prefill_varlen(case.q, case.k_cache, case.v_cache, case.block_table, cu, k_lens,
                            True, case.scale)
    ref = oracle.prefill_varlen(bits(case.q), k_host, v_host, case.block_table.cpu().numpy(),
                                cu, k_lens, True, case.scale)
    assert_attention_close(out, ref, "varlen with packed tiles")
    assert pa.device_errors() == 0
