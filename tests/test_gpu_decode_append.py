"""Decode steps that append the newest token with the slot derived on the device
(pa_decode_append) vs the fp64 oracle: the slots bit-exact against the oracle's slot
mapping of position seq_len - 1, the caches bit-exact against the oracle's KV write,
the attention within the tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import assert_attention_close
from workloads import bits

pytestmark = pytest.mark.gpu


def _append(pa, case, slot_mapping=None, max_seq_len=None):
    msl = int(case.seq_lens.max()) if max_seq_len is None else max_seq_len
    return pa.decode_append(case.q, case.k_cache, case.v_cache, case.block_table,
                            case.seq_lens, case.scale, msl, case.new_k, case.new_v,
                            slot_mapping=slot_mapping)


def _oracle_step(case, k_host, v_host):
    """Oracle slots of each sequence's newest token, its KV write into copies of the
    caches as they were before the step, and the decode over them."""
    S = case.q.shape[0]
    bt = case.block_table.cpu().numpy()
    pos = case.seq_lens.cpu().numpy().astype(np.int64) - 1
    slots = oracle.slot_mapping(pos, bt, case.block_size, np.arange(S))
    k_ref, v_ref = k_host.copy(), v_host.copy()
    oracle.reshape_and_cache(bits(case.new_k), bits(case.new_v), k_ref, v_ref, slots,
                             case.block_size)
    ref = oracle.decode(bits(case.q), k_ref, v_ref, bt, case.seq_lens.cpu().numpy(),
                        case.scale)
    return slots, k_ref, v_ref, ref


def _check_step(pa, case, what):
    k_host, v_host = bits(case.k_cache), bits(case.v_cache)
    slots = torch.full((case.q.shape[0],), -7, dtype=torch.int64, device="cuda")
    out = _append(pa, case, slot_mapping=slots)
    torch.cuda.synchronize()
    want_slots, k_ref, v_ref, ref = _oracle_step(case, k_host, v_host)
    assert np.array_equal(slots.cpu().numpy(), want_slots), f"{what}: slots"
    assert np.array_equal(bits(case.k_cache), k_ref), f"{what}: K cache"
    assert np.array_equal(bits(case.v_cache), v_ref), f"{what}: V cache"
    e = assert_attention_close(out, ref, what)
    assert pa.device_errors() == 0
    return out, e


def test_tiny_decode_append(cuda_lib):
    case = workloads.tiny_decode("cuda")
    _, e = _check_step(cuda_lib, case, "tiny decode append")
    assert e["rel_l2"] < 5e-3


def test_headline_8k_append(cuda_lib):
    case = workloads.paged_case(1002, [8192], 832, 64, new_tokens=1, device="cuda")
    _check_step(cuda_lib, case, "8K append")


@pytest.mark.parametrize("bs", [832, 784])
@pytest.mark.parametrize("seq_len", [1665 + 16 * k for k in range(-7, 7, 3)] + [1696])
def test_append_when_the_newest_tile_starts_a_split(cuda_lib, seq_len, bs):
    # The split holding the newest token may have loaded it before the write (its only
    # stage, loaded ahead of the sequence length); the slot starts as NaN, so a stale
    # copy would show.
    case = workloads.paged_case(73, [seq_len], bs, 8, new_tokens=1, device="cuda")
    _check_step(cuda_lib, case, f"append L={seq_len} bs={bs}")


def test_batched_decode_append(cuda_lib):
    case = workloads.batched_decode("cuda")
    _check_step(cuda_lib, case, "batched append")


EDGE_LENS = [1, 15, 16, 17, 63, 64, 65, 783, 784, 785, 831, 832, 833, 1700]


@pytest.mark.parametrize("bs", [784, 832, 64, 16, 48, 100])
def test_append_edge_lengths_in_one_batch(cuda_lib, bs):
    # A sequence of length 1 consists of its appended token only: the output is that
    # token's value row (BF16 passes through exactly).
    npg = sum(-(-L // bs) for L in EDGE_LENS) + 3
    case = workloads.paged_case(91 + bs, EDGE_LENS, bs, npg, new_tokens=1, device="cuda")
    out, _ = _check_step(cuda_lib, case, f"append edge lengths bs={bs}")
    want = case.new_v[0].repeat_interleave(case.q.shape[1] // case.new_v.shape[1], dim=0)
    assert torch.equal(out[0], want)


def test_append_without_slot_output_matches(cuda_lib):
    pa = cuda_lib
    a = workloads.paged_case(55, [3000, 777], 832, 8, new_tokens=1, device="cuda")
    b = workloads.paged_case(55, [3000, 777], 832, 8, new_tokens=1, device="cuda")
    out_a = _append(pa, a)
    slots = torch.empty(2, dtype=torch.int64, device="cuda")
    out_b = _append(pa, b, slot_mapping=slots)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    # the caches hold NaN in unused slots: compare bits
    assert np.array_equal(bits(a.k_cache), bits(b.k_cache))
    assert np.array_equal(bits(a.v_cache), bits(b.v_cache))
    assert pa.device_errors() == 0


def test_append_replayed_from_a_graph_is_deterministic(cuda_lib):
    pa = cuda_lib
    case = workloads.paged_case(56, [5000, 9000, 2100], 832, 24, new_tokens=1, device="cuda")
    k_host, v_host = bits(case.k_cache), bits(case.v_cache)
    out = torch.empty_like(case.q)
    slots = torch.empty(3, dtype=torch.int64, device="cuda")
    ws = torch.empty(max(256, pa.decode_workspace_size(3, 24, 4, 256, 832, 9000)),
                     dtype=torch.uint8, device="cuda")

    def step():
        pa.decode_append(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                         case.scale, 9000, case.new_k, case.new_v, out=out, workspace=ws,
                         slot_mapping=slots)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    first = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        out.zero_()
        slots.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, first)
    want_slots, k_ref, v_ref, ref = _oracle_step(case, k_host, v_host)
    assert np.array_equal(slots.cpu().numpy(), want_slots)
    assert np.array_equal(bits(case.k_cache), k_ref)
    assert_attention_close(out, ref, "graph replay")
    assert pa.device_errors() == 0


def test_append_bad_page_of_the_newest_token(cuda_lib):
    # The newest token's block-table entry lies past the pool: nothing is written, the
    # page error is set and the reported slot is the formula's value.  A negative entry
    # reports slot -1, as the slot mapping gives it.
    pa = cuda_lib
    case = workloads.paged_case(57, [1000, 1900], 832, 6, new_tokens=1, device="cuda")
    case.block_table[0, 1] = case.num_pages + 3
    case.block_table[1, 2] = -1
    before_k, before_v = bits(case.k_cache).copy(), bits(case.v_cache).copy()
    slots = torch.empty(2, dtype=torch.int64, device="cuda")
    out = _append(pa, case, slot_mapping=slots)
    torch.cuda.synchronize()
    assert pa.device_errors() & pa.DEVERR_PAGE
    assert pa.device_errors() == 0
    assert slots.cpu().tolist() == [(case.num_pages + 3) * 832 + 999 - 832, -1]
    assert np.array_equal(bits(case.k_cache), before_k)
    assert np.array_equal(bits(case.v_cache), before_v)
    assert out.shape == case.q.shape


def test_kernel_events_inside_a_graph(cuda_lib):
    # The measurement hook inside a stream capture: the events become event record nodes,
    # so each replay records them around the split kernel of its own step.
    pa = cuda_lib
    cases = [workloads.paged_case(58 + r, [4000], 832, 8, new_tokens=1, device="cuda")
             for r in range(2)]
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in cases]
    for a, b in evs:
        a.record()
        b.record()
    torch.cuda.synchronize()

    outs = [torch.empty_like(c.q) for c in cases]
    wss = [torch.empty(max(256, pa.decode_workspace_size(1, 24, 4, 256, 832, 4000)),
                       dtype=torch.uint8, device="cuda") for _ in cases]

    def run():
        for c, (a, b), o, w in zip(cases, evs, outs, wss):
            pa.set_kernel_events(a, b)
            pa.decode_append(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens, c.scale,
                             4000, c.new_k, c.new_v, out=o, workspace=w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()                          # outside a capture: plain records
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in evs]
        assert all(0.0 < t < 50.0 for t in ms), ms
    assert pa.device_errors() == 0


def test_append_unbind_view_page_stride(cuda_lib):
    # K and V as the two halves of one [pages, 2, BS, Hkv, D] tensor (page stride twice
    # a page): the same writes and outputs as separate caches.
    pa = cuda_lib
    a = workloads.paged_case(61, [8192], 832, 12, new_tokens=1, device="cuda")
    b = workloads.paged_case(61, [8192], 832, 12, new_tokens=1, device="cuda")
    kv = torch.stack([b.k_cache, b.v_cache], dim=1)
    b.k_cache, b.v_cache = kv.unbind(1)
    out_b = pa.decode_append(b.q, b.k_cache, b.v_cache, b.block_table, b.seq_lens, b.scale,
                             8192, b.new_k, b.new_v)
    out_a, _ = _check_step(pa, a, "append, separate caches")
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert np.array_equal(bits(kv[:, 0]), bits(a.k_cache))
    assert np.array_equal(bits(kv[:, 1]), bits(a.v_cache))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 2), (8, 1), (12, 4)])
def test_append_other_group_sizes(cuda_lib, hq, hkv):
    case = workloads.paged_case(930 + hq, [700, 2000, 1], 64, 48, hq=hq, hkv=hkv,
                                new_tokens=1, device="cuda")
    _check_step(cuda_lib, case, f"append group {hq}/{hkv}")


def test_append_max_seq_len_above_actual_lengths(cuda_lib):
    # The split plan is made for max_seq_len; shorter sequences leave splits empty, and
    # the newest token's tile may sit in any split.
    pa = cuda_lib
    case = workloads.paged_case(62, [100, 5000, 1, 833], 832, 16, new_tokens=1,
                                device="cuda", max_blocks=40)
    k_host, v_host = bits(case.k_cache), bits(case.v_cache)
    slots = torch.empty(4, dtype=torch.int64, device="cuda")
    out = _append(pa, case, slot_mapping=slots, max_seq_len=40 * 832)
    torch.cuda.synchronize()
    want_slots, k_ref, v_ref, ref = _oracle_step(case, k_host, v_host)
    assert np.array_equal(slots.cpu().numpy(), want_slots)
    assert np.array_equal(bits(case.k_cache), k_ref)
    assert_attention_close(out, ref, "append, max_seq_len slack")
    assert pa.device_errors() == 0


@pytest.mark.parametrize("T", [3001, 8192])
def test_append_block_size_784_vs_832_bitwise(cuda_lib, T):
    # The appended token's tile and every sum are the same at both page sizes (784 and
    # 832 are multiples of the 16-token tile): identical output bits.
    pa = cuda_lib
    g = torch.Generator(device="cuda").manual_seed(4)
    kc = torch.randn(T, 4, 256, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(T, 4, 256, generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn(1, 24, 256, generator=g, device="cuda").to(torch.bfloat16)
    outs = []
    for bs in (784, 832):
        npg = -(-T // bs)
        k_cache = torch.zeros(npg + 2, bs, 4, 256, dtype=torch.bfloat16, device="cuda")
        v_cache = torch.zeros_like(k_cache)
        perm = torch.randperm(npg + 2, generator=torch.Generator().manual_seed(bs))[:npg]
        bt = perm.to(torch.int32).view(1, -1).cuda()
        slots = pa.slot_mapping(torch.arange(T - 1, dtype=torch.int32, device="cuda"), bt, bs)
        pa.reshape_and_cache(kc[:T - 1], vc[:T - 1], k_cache, v_cache, slots)
        sl = torch.tensor([T], dtype=torch.int32, device="cuda")
        outs.append(pa.decode_append(q, k_cache, v_cache, bt, sl, 1 / 16, T,
                                     kc[T - 1:].contiguous(), vc[T - 1:].contiguous()))
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    assert pa.device_errors() == 0


def test_append_output_in_pinned_host_memory(cuda_lib):
    # The combine writes the step's result straight into page-locked host memory: the
    # same bits as a device output; pageable host memory is refused.
    pa = cuda_lib
    a = workloads.paged_case(63, [5000, 300], 832, 12, new_tokens=1, device="cuda")
    b = workloads.paged_case(63, [5000, 300], 832, 12, new_tokens=1, device="cuda")
    out_d = _append(pa, a)
    out_h = torch.empty(b.q.shape, dtype=torch.bfloat16).pin_memory()
    pa.decode_append(b.q, b.k_cache, b.v_cache, b.block_table, b.seq_lens, b.scale, 5000,
                     b.new_k, b.new_v, out=out_h)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu())
    with pytest.raises(TypeError):
        pa.decode_append(b.q, b.k_cache, b.v_cache, b.block_table, b.seq_lens, b.scale, 5000,
                         b.new_k, b.new_v, out=torch.empty(b.q.shape, dtype=torch.bfloat16))
    pageable = np.zeros(b.q.numel() + 8, dtype=np.uint16)
    addr = (pageable.ctypes.data + 15) // 16 * 16
    import ctypes
    ws = torch.empty(max(256, pa.decode_workspace_size(2, 24, 4, 256, 832, 5000)),
                     dtype=torch.uint8, device="cuda")
    rc = pa.load().pa_decode(ctypes.c_void_p(b.q.data_ptr()), ctypes.c_void_p(b.k_cache.data_ptr()),
                             ctypes.c_void_p(b.v_cache.data_ptr()), b.k_cache.stride(0),
                             b.k_cache.shape[0], ctypes.c_void_p(b.block_table.data_ptr()),
                             b.block_table.stride(0), ctypes.c_void_p(b.seq_lens.data_ptr()), 2,
                             5000, 24, 4, 256, 832, b.scale, ctypes.c_void_p(addr),
                             ctypes.c_void_p(ws.data_ptr()), ws.numel(), None, None, None,
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 1   # PA_ERR_INVALID_ARG
    assert pa.device_errors() == 0
