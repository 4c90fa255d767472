"""q=1 paged decode on the GPU vs the fp64 oracle, on the pages' workloads at full size
and on edge cases (page tails, sequence ends on and around page boundaries, unbind
views, group sizes, bad inputs)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import assert_attention_close
from workloads import bits

pytestmark = pytest.mark.gpu


def _oracle_decode(case, k_host=None, v_host=None):
    return oracle.decode(bits(case.q), bits(case.k_cache) if k_host is None else k_host,
                         bits(case.v_cache) if v_host is None else v_host,
                         case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(),
                         case.scale)


def _gpu_decode(pa, case, max_seq_len=None, **kw):
    msl = int(case.seq_lens.max()) if max_seq_len is None else max_seq_len
    return pa.decode(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                     case.scale, msl, **kw)


def test_tiny_decode_with_fused_new_token_write(cuda_lib):
    pa = cuda_lib
    case = workloads.tiny_decode("cuda")
    slots = pa.slot_mapping(case.positions, case.block_table, case.block_size,
                            seq_idx=case.seq_idx)
    out = _gpu_decode(pa, case, new_k=case.new_k, new_v=case.new_v, new_slots=slots)
    torch.cuda.synchronize()
    k_host, v_host = bits(case.k_cache), bits(case.v_cache)
    # The oracle writes the new token into its own copy of the caches (which still have
    # the NaN at that slot, since the GPU copy is read back after the fused write) ...
    k_ref, v_ref = k_host.copy(), v_host.copy()
    oracle.reshape_and_cache(bits(case.new_k), bits(case.new_v), k_ref, v_ref,
                             oracle.slot_mapping(case.positions.cpu().numpy(),
                                                 case.block_table.cpu().numpy(), 832,
                                                 case.seq_idx.cpu().numpy()), 832)
    assert np.array_equal(k_ref, k_host) and np.array_equal(v_ref, v_host)
    ref = _oracle_decode(case, k_ref, v_ref)
    e = assert_attention_close(out, ref, "tiny decode")
    assert e["rel_l2"] < 5e-3
    assert pa.device_errors() == 0


@pytest.mark.parametrize("bs", [832, 784])
@pytest.mark.parametrize("seq_len", [1665 + 16 * k for k in range(-7, 7)] + [1696])
def test_fused_write_when_the_newest_tile_starts_a_split(cuda_lib, seq_len, bs):
    # The kernel loads each split's first stage (two 16-token tiles) before it knows the
    # sequence length.  When that stage also holds the token being decoded (the split's
    # only stage), it has to be loaded again after the fused write; the slot starts as
    # NaN, so a stale copy shows in the output.  These 14 consecutive tile counts put the
    # last split at every length modulo 8 (the smallest split length), with the token on
    # the first row of its tile (and, for 1696, on the last row).  At block size 784 a page
    # holds 49 tiles, so some of these first stages straddle two pages instead.
    pa = cuda_lib
    case = workloads.paged_case(73, [seq_len], bs, 8, new_tokens=1, device="cuda")
    k_ref, v_ref = bits(case.k_cache).copy(), bits(case.v_cache).copy()
    oracle.reshape_and_cache(bits(case.new_k), bits(case.new_v), k_ref, v_ref,
                             oracle.slot_mapping(case.positions.cpu().numpy(),
                                                 case.block_table.cpu().numpy(), bs,
                                                 case.seq_idx.cpu().numpy()), bs)
    slots = pa.slot_mapping(case.positions, case.block_table, bs, seq_idx=case.seq_idx)
    out = _gpu_decode(pa, case, new_k=case.new_k, new_v=case.new_v, new_slots=slots)
    torch.cuda.synchronize()
    assert np.array_equal(bits(case.k_cache), k_ref) and np.array_equal(bits(case.v_cache), v_ref)
    assert_attention_close(out, _oracle_decode(case, k_ref, v_ref), f"fused write, L={seq_len}")
    assert pa.device_errors() == 0


@pytest.mark.parametrize("bs", [832, 784])
def test_decode_8k(cuda_lib, bs):
    pa = cuda_lib
    case = workloads.decode_8k(bs, "cuda")
    out = _gpu_decode(pa, case)
    assert_attention_close(out, _oracle_decode(case), f"decode 8K bs={bs}")
    assert pa.device_errors() == 0


@pytest.mark.parametrize("context", [4096, 8192, 16384, 32768])
def test_decode_sweep_peaked_1gib_pool(cuda_lib, context):
    pa = cuda_lib
    case = workloads.decode_sweep(context, "cuda")
    out = _gpu_decode(pa, case)
    assert_attention_close(out, _oracle_decode(case), f"sweep {context}")
    assert pa.device_errors() == 0


@pytest.mark.parametrize("bs", [16, 64])
def test_decode_32k_small_pages(cuda_lib, bs):
    """Generic small pages: 2048 (16) or 512 (64) scattered pages per 32K sequence; with
    16-token pages every stage's two tiles lie in different pages."""
    pa = cuda_lib
    case = workloads.decode_sweep(32768, "cuda", block_size=bs)
    out = _gpu_decode(pa, case)
    assert_attention_close(out, _oracle_decode(case), f"sweep 32K bs={bs}")
    assert pa.device_errors() == 0


def test_batched_decode_fused_write(cuda_lib):
    pa = cuda_lib
    case = workloads.batched_decode("cuda")
    k_before, v_before = bits(case.k_cache), bits(case.v_cache)
    slots = pa.slot_mapping(case.positions, case.block_table, case.block_size,
                            seq_idx=case.seq_idx)
    out = _gpu_decode(pa, case, new_k=case.new_k, new_v=case.new_v, new_slots=slots)
    torch.cuda.synchronize()
    oracle.reshape_and_cache(bits(case.new_k), bits(case.new_v), k_before, v_before,
                             oracle.slot_mapping(case.positions.cpu().numpy(),
                                                 case.block_table.cpu().numpy(),
                                                 case.block_size, case.seq_idx.cpu().numpy()),
                             case.block_size)
    ref = _oracle_decode(case, k_before, v_before)
    assert_attention_close(out, ref, "batched decode")
    assert pa.device_errors() == 0


EDGE_LENS = [1, 15, 16, 17, 63, 64, 65, 783, 784, 785, 831, 832, 833, 1700]


@pytest.mark.parametrize("bs", [784, 832, 64, 16, 48, 100])
def test_decode_edge_lengths_in_one_batch(cuda_lib, bs):
    # 784 and 48: odd tiles per page (two-tile stages straddle pages); 100: a page ends in
    # a 4-row tile; 16: one tile per page (every stage spans two pages).
    pa = cuda_lib
    npg = sum(-(-L // bs) for L in EDGE_LENS) + 3
    case = workloads.paged_case(77 + bs, EDGE_LENS, bs, npg, device="cuda")
    out = _gpu_decode(pa, case)
    assert_attention_close(out, _oracle_decode(case), f"edge lengths bs={bs}")
    # seq_len 1 returns that token's value row (up to BF16 rounding of an exact copy).
    v = case.v_cache[int(case.block_table[0, 0]), 0]          # [Hkv, D]
    want = v.repeat_interleave(case.q.shape[1] // v.shape[0], dim=0)
    assert torch.equal(out[0], want)
    assert pa.device_errors() == 0


def test_decode_max_seq_len_above_actual_lengths(cuda_lib):
    # The split plan is made for max_seq_len; shorter sequences leave splits empty.
    pa = cuda_lib
    case = workloads.paged_case(5, [100, 5000, 1], 832, 12, device="cuda", max_blocks=40)
    out = _gpu_decode(pa, case, max_seq_len=40 * 832)
    assert_attention_close(out, _oracle_decode(case), "max_seq_len slack")


def test_decode_unbind_view_page_stride(cuda_lib):
    pa = cuda_lib
    case = workloads.decode_8k(832, "cuda")
    kv = torch.stack([case.k_cache, case.v_cache], dim=1)       # [pages, 2, BS, Hkv, D]
    k_view, v_view = kv.unbind(1)
    out = pa.decode(case.q, k_view, v_view, case.block_table, case.seq_lens, case.scale, 8192)
    ref_out = _gpu_decode(pa, case)
    assert torch.equal(out, ref_out)
    assert_attention_close(out, _oracle_decode(case), "unbind view")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 2), (8, 1), (12, 4)])
def test_decode_other_group_sizes(cuda_lib, hq, hkv):
    pa = cuda_lib
    case = workloads.paged_case(900 + hq, [700, 2000], 64, 48, hq=hq, hkv=hkv, device="cuda")
    out = _gpu_decode(pa, case)
    assert_attention_close(out, _oracle_decode(case), f"group {hq}/{hkv}")


def test_decode_is_deterministic(cuda_lib):
    pa = cuda_lib
    case = workloads.decode_sweep(16384, "cuda")
    a = _gpu_decode(pa, case)
    b = _gpu_decode(pa, case)
    assert torch.equal(a, b)


@pytest.mark.parametrize("T", [3000, 8192])
def test_decode_block_size_784_vs_832_bitwise(cuda_lib, T):
    # Same logical tokens, two page sizes: both match the oracle, and the oracle itself
    # gives identical results for both (the definition does not depend on the page size;
    # page832 §9 reports page784 and page832 giving identical bits).  The kernel works in
    # 16-token tiles and 784 = 49 x 16, 832 = 52 x 16, so both sizes give the same tiles,
    # the same splits and the same order of every sum: the outputs are bit for bit equal.
    pa = cuda_lib
    g = torch.Generator(device="cuda").manual_seed(3)
    kc = torch.randn(T, 4, 256, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(T, 4, 256, generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn(1, 24, 256, generator=g, device="cuda").to(torch.bfloat16)
    outs, refs = [], []
    for bs in (784, 832):
        npg = -(-T // bs)
        k_cache = torch.zeros(npg + 2, bs, 4, 256, dtype=torch.bfloat16, device="cuda")
        v_cache = torch.zeros_like(k_cache)
        perm = torch.randperm(npg + 2, generator=torch.Generator().manual_seed(bs))[:npg]
        bt = perm.to(torch.int32).view(1, -1).cuda()
        slots = pa.slot_mapping(torch.arange(T, dtype=torch.int32, device="cuda"), bt, bs)
        pa.reshape_and_cache(kc, vc, k_cache, v_cache, slots)
        sl = torch.tensor([T], dtype=torch.int32, device="cuda")
        outs.append(pa.decode(q, k_cache, v_cache, bt, sl, 1 / 16, T))
        refs.append(oracle.decode(bits(q), bits(k_cache), bits(v_cache), bt.cpu().numpy(),
                                  np.array([T], np.int32), 1 / 16))
    assert np.array_equal(refs[0], refs[1])
    for o in outs:
        assert_attention_close(o, refs[0], "bs invariance")
    assert torch.equal(outs[0], outs[1])


def test_decode_bad_page_is_reported_not_faulted(cuda_lib):
    pa = cuda_lib
    case = workloads.paged_case(9, [2000], 832, 6, device="cuda")
    case.block_table[0, 1] = case.num_pages + 3       # outside the pool: reads zeros
    out = _gpu_decode(pa, case)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert pa.device_errors() & pa.DEVERR_PAGE
    assert pa.device_errors() == 0


def test_decode_seq_len_above_max_is_reported(cuda_lib):
    pa = cuda_lib
    case = workloads.paged_case(10, [900], 832, 4, device="cuda", max_blocks=2)
    case.seq_lens[0] = 5000                            # above max_seq_len = 1664
    out = _gpu_decode(pa, case, max_seq_len=1664)
    torch.cuda.synchronize()
    assert pa.device_errors() & pa.DEVERR_SEQLEN
    assert out.shape == case.q.shape


def test_decode_workspace_too_small_is_rejected(cuda_lib):
    pa = cuda_lib
    case = workloads.decode_8k(832, "cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PAError):
        _gpu_decode(pa, case, workspace=ws)


def test_fused_write_checks_the_slot_of_the_newest_token(cuda_lib):
    # The fused write only lands at the slot the block table gives for position
    # seq_len - 1; any other slot is refused (error bit, nothing written), and a negative
    # slot is padding.
    pa = cuda_lib
    case = workloads.paged_case(71, [900, 1500], 832, 8, new_tokens=1, device="cuda")
    good = pa.slot_mapping(case.positions, case.block_table, 832, seq_idx=case.seq_idx)
    bad = good.clone()
    bad[0] += 1                       # one slot too far for sequence 0
    bad[1] = -1                       # sequence 1: padding, skipped
    before = bits(case.k_cache).copy()
    pa.decode(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, case.scale,
              1500, new_k=case.new_k, new_v=case.new_v, new_slots=bad)
    torch.cuda.synchronize()
    assert pa.device_errors() == pa.DEVERR_SLOT
    assert np.array_equal(bits(case.k_cache), before)      # nothing was written
    pa.decode(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, case.scale,
              1500, new_k=case.new_k, new_v=case.new_v, new_slots=good)
    torch.cuda.synchronize()
    assert pa.device_errors() == 0
    k_ref, v_ref = before.copy(), bits(case.v_cache).copy()
    oracle.reshape_and_cache(bits(case.new_k), bits(case.new_v), k_ref, v_ref,
                             good.cpu().numpy(), 832)
    assert np.array_equal(bits(case.k_cache), k_ref)


@pytest.mark.parametrize("fill", ["nan", "finite"])
@pytest.mark.parametrize("seq_lens", [[8192], [1, 17, 240, 3000, 16000], [1701, 1700]])
def test_decode_ignores_what_the_workspace_held(cuda_lib, fill, seq_lens):
    # The workspace's contents on entry do not matter: the combine reads only the
    # (max, sum) pair and partial sums every split wrote in the same call (an empty split
    # writes (-inf, 0)).  A workspace full of NaN, or of finite values that would pass
    # for a real split's partial (every float pair (30, 1): a large max and a unit sum),
    # must change nothing, with short last splits and splits past a sequence's end among
    # the lengths.  A stale pair read by the combine would outweigh the real splits.
    pa = cuda_lib
    bs = 832
    npg = sum(-(-L // bs) for L in seq_lens) + 2
    msl = max(seq_lens) + 5000  # splits past every sequence's end
    case = workloads.paged_case(900 + sum(seq_lens), seq_lens, bs, npg, device="cuda",
                                max_blocks=-(-msl // bs))
    need = pa.decode_workspace_size(len(seq_lens), 24, 4, 256, bs, msl)
    clean = torch.zeros(need, dtype=torch.uint8, device="cuda")
    want = _gpu_decode(pa, case, max_seq_len=msl, workspace=clean)
    dirty = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    if fill == "nan":
        dirty.fill_(float("nan"))
    else:
        dirty.view(-1, 2)[:, 0] = 30.0
        dirty.view(-1, 2)[:, 1] = 1.0
    got = _gpu_decode(pa, case, max_seq_len=msl, workspace=dirty.view(torch.uint8))
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    assert_attention_close(got, _oracle_decode(case), f"dirty workspace {fill}")
    assert pa.device_errors() == 0
