"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
hand-worked slot values from the pages' formula, closed forms of softmax attention,
brute force on a contiguous (unpaged) layout, and invariances the definition implies
(page permutation, block size, token order, causal visibility).  CPU only."""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    """float64 array -> BF16 bit patterns, round to nearest even (test-side helper)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def _val(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _paged_from_contiguous(kc, vc, block_size, num_pages, rng):
    """Scatter contiguous [T, Hkv, D] rows into pages by enumerating whole pages (no
    division): logical page p holds tokens p*BS .. p*BS+BS-1 at offsets 0..BS-1."""
    T, hkv, d = kc.shape
    npg = -(-T // block_size)
    phys = rng.permutation(num_pages)[:npg].astype(np.int32)
    k_cache = np.full((num_pages, block_size, hkv, d), 0xFFFF, dtype=np.uint16)
    v_cache = np.full_like(k_cache, 0xFFFF)
    t = 0
    for p in range(npg):
        for o in range(block_size):
            if t < T:
                k_cache[phys[p], o] = kc[t]
                v_cache[phys[p], o] = vc[t]
            t += 1
    return k_cache, v_cache, phys


def _softmax_attention_contiguous(qv, kv, vv, scale):
    s = scale * (kv @ qv)
    w = np.exp(s - s.max())
    w /= w.sum()
    return w @ vv


# ---------------------------------------------------------------- slot mapping
def test_slot_mapping_hand_worked_table():
    rows = [ln.split("#")[0].split() for ln in open(os.path.join(GOLDEN, "slot_mapping_hand.txt"))]
    rows = [r for r in rows if r]
    bt = np.array([5, 2, 7, 0], dtype=np.int32)
    for bs, pos, want in rows:
        got = oracle.slot_mapping(np.array([int(pos)]), bt, int(bs))
        assert int(got[0]) == int(want), (bs, pos)


def _golden_lines(name):
    """Non-empty lines of a golden file, comments (after #) removed, split on blanks."""
    rows = [ln.split("#")[0].split() for ln in open(os.path.join(GOLDEN, name))]
    return [r for r in rows if r]


def test_decode_input_prep_hand_worked_step():
    lines = _golden_lines("decode_input_prep_hand.txt")
    qsl = [list(map(int, r[1:])) for r in lines if r[0] == "query_start_loc"]
    rows = [list(map(int, r)) for r in lines if r[0] != "query_start_loc"]
    g0 = np.array([[5, 2, 7, 0], [3, 1, 6, 4], [9, 8, 11, 10]], dtype=np.int32)
    g1 = np.array([[1000 * (s + 1) + j for j in range(256)] for s in range(3)], dtype=np.int32)
    pos = np.array([r[1] for r in rows], np.int32)
    sampled = np.array([r[2] for r in rows], np.int32)
    got = oracle.decode_input_prep(pos, [g0, g1], [832, 16], sampled_ids=sampled)
    assert got["seq_lens"].tolist() == [r[3] for r in rows]
    assert got["input_ids"].tolist() == [r[2] for r in rows]
    assert got["slot_mappings"][0].tolist() == [r[4] for r in rows]
    assert got["slot_mappings"][1].tolist() == [r[5] for r in rows]
    assert [got["query_start_loc"].tolist()] == qsl


def _expand_runs(tokens):
    """'N*x' -> N copies of x; plain integers as they are."""
    out = []
    for t in tokens:
        if "*" in t:
            n, x = t.split("*")
            out += [int(x)] * int(n)
        else:
            out.append(int(t))
    return out


def test_decode_input_prep_the_pages_step():
    # One request at position 24576, two KV-cache groups of block size 16, buffers for
    # 128 requests: query_start_loc [0, 1, 1, ...] and seq_lens [position + 1, 0, 0, ...].
    f = {r[0]: _expand_runs(r[1:]) for r in _golden_lines("decode_input_prep_pages_step.txt")}
    n = len(f["positions"])
    rows = np.arange(n)[:, None] * 10000
    cols = np.arange(1600)[None, :]
    tables = [(3 * cols + 1 + rows).astype(np.int32), (2 * cols + 7 + rows).astype(np.int32)]
    got = oracle.decode_input_prep(np.array(f["positions"], np.int32), tables, f["block_sizes"],
                                   sampled_ids=np.array(f["sampled_ids"], np.int32))
    assert len(f["query_start_loc"]) == n + 1
    assert got["query_start_loc"].tolist() == f["query_start_loc"]
    assert got["seq_lens"].tolist() == f["seq_lens"]
    assert got["input_ids"].tolist() == f["input_ids"]
    assert got["slot_mappings"][0].tolist() == f["slot_group0"]
    assert got["slot_mappings"][1].tolist() == f["slot_group1"]


def test_page_geometry_from_pages():
    rows = [ln.split("#")[0].split() for ln in open(os.path.join(GOLDEN, "page_geometry.txt"))]
    for bs, groups, tail, nbytes in [r for r in rows if r]:
        bs, groups, tail, nbytes = map(int, (bs, groups, tail, nbytes))
        assert groups * 64 + tail == bs
        assert bs * 4 * 256 * 2 == nbytes


@pytest.mark.parametrize("bs", [784, 832, 64, 16, 1])
def test_slot_mapping_matches_page_enumeration(bs):
    rng = np.random.default_rng(bs)
    S, mb = 3, 9
    bt = rng.permutation(S * mb).astype(np.int32).reshape(S, mb)
    # Enumerate every (sequence, logical page, offset) -> slot without any division.
    want = {}
    for s in range(S):
        for p in range(mb):
            for o in range(bs):
                want[(s, p * bs + o)] = int(bt[s, p]) * bs + o
    keys = list(want.keys())
    pick = rng.choice(len(keys), size=min(400, len(keys)), replace=False)
    seq = np.array([keys[i][0] for i in pick], dtype=np.int32)
    pos = np.array([keys[i][1] for i in pick], dtype=np.int32)
    got = oracle.slot_mapping(pos, bt, bs, seq_idx=seq)
    assert got.dtype == np.int64
    assert [int(x) for x in got] == [want[(int(a), int(b))] for a, b in zip(seq, pos)]


def test_reshape_and_cache_lands_where_enumeration_says():
    rng = np.random.default_rng(7)
    bs, hkv, d, npg = 16, 2, 8, 6
    bt = rng.permutation(npg).astype(np.int32)
    pos = np.array([0, 5, 15, 16, 40, 95], dtype=np.int32)
    key = rng.integers(0, 0x7F00, size=(len(pos), hkv, d)).astype(np.uint16)
    val = rng.integers(0, 0x7F00, size=(len(pos), hkv, d)).astype(np.uint16)
    k_cache = np.zeros((npg, bs, hkv, d), dtype=np.uint16)
    v_cache = np.zeros_like(k_cache)
    slots = oracle.slot_mapping(pos, bt, bs)
    slots_with_pad = np.concatenate([slots, [-1]])
    key_p = np.concatenate([key, np.full((1, hkv, d), 0x1234, np.uint16)])
    val_p = np.concatenate([val, np.full((1, hkv, d), 0x1234, np.uint16)])
    oracle.reshape_and_cache(key_p, val_p, k_cache, v_cache, slots_with_pad, bs)
    written = np.zeros((npg, bs), dtype=bool)
    for i, t in enumerate(pos):
        page, off = bt[t // bs], t % bs
        assert np.array_equal(k_cache[page, off], key[i])
        assert np.array_equal(v_cache[page, off], val[i])
        written[page, off] = True
    assert not k_cache[~written].any() and not v_cache[~written].any()  # nothing else touched
    assert not (k_cache == 0x1234).any()                                # slot -1 skipped


# ---------------------------------------------------------------- attention
@pytest.mark.parametrize("bs", [16, 7, 64])
def test_attend_row_equals_contiguous_bruteforce(bs):
    rng = np.random.default_rng(100 + bs)
    T, hkv, d = 150, 2, 32
    kc = _bf16(rng.standard_normal((T, hkv, d)))
    vc = _bf16(rng.standard_normal((T, hkv, d)))
    q = _bf16(rng.standard_normal(d))
    k_cache, v_cache, phys = _paged_from_contiguous(kc, vc, bs, 40, rng)
    for g in range(hkv):
        for n in (1, 2, bs, bs + 1, T):
            got = oracle.attend_row(q, k_cache, v_cache, phys, bs, g, n, 0.125)
            want = _softmax_attention_contiguous(_val(q), _val(kc[:n, g]), _val(vc[:n, g]), 0.125)
            np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_single_key_returns_its_value_exactly():
    rng = np.random.default_rng(1)
    kc = _bf16(rng.standard_normal((5, 1, 16)))
    vc = _bf16(rng.standard_normal((5, 1, 16)))
    k_cache, v_cache, phys = _paged_from_contiguous(kc, vc, 4, 3, rng)
    out = oracle.attend_row(_bf16(rng.standard_normal(16)), k_cache, v_cache, phys, 4, 0, 1, 0.25)
    assert np.array_equal(out, _val(vc[0, 0]))


@pytest.mark.parametrize("case", ["q_zero", "keys_equal", "scale_zero"])
def test_uniform_weights_give_mean_of_values(case):
    rng = np.random.default_rng(2)
    T, d = 37, 16
    kc = _bf16(rng.standard_normal((T, 1, d)))
    if case == "keys_equal":
        kc[:] = kc[0]
    vc = _bf16(rng.standard_normal((T, 1, d)))
    q = _bf16(rng.standard_normal(d)) if case != "q_zero" else np.zeros(d, np.uint16)
    scale = 0.0 if case == "scale_zero" else 0.5
    k_cache, v_cache, phys = _paged_from_contiguous(kc, vc, 8, 6, rng)
    out, w = oracle.attend_row(q, k_cache, v_cache, phys, 8, 0, T, scale, return_weights=True)
    np.testing.assert_allclose(w, np.full(T, 1.0 / T), rtol=1e-14)
    np.testing.assert_allclose(out, _val(vc[:, 0]).mean(axis=0), rtol=0, atol=1e-13)


def test_two_keys_logistic_closed_form():
    # q = e0, k0 = 2 e0, k1 = 0: scores scale*2 and 0, so w0 = 1 / (1 + exp(-2 scale)).
    d = 8
    q = np.zeros(d, np.uint16); q[0] = _bf16(1.0)
    kc = np.zeros((2, 1, d), np.uint16); kc[0, 0, 0] = _bf16(2.0)
    vc = np.zeros((2, 1, d), np.uint16); vc[0, 0, :] = _bf16(3.0); vc[1, 0, :] = _bf16(-1.0)
    rng = np.random.default_rng(3)
    k_cache, v_cache, phys = _paged_from_contiguous(kc, vc, 1, 4, rng)
    for scale in (0.0625, 1.0, 5.0):
        w0 = 1.0 / (1.0 + math.exp(-2.0 * scale))
        out = oracle.attend_row(q, k_cache, v_cache, phys, 1, 0, 2, scale)
        np.testing.assert_allclose(out, np.full(d, 3.0 * w0 - 1.0 * (1 - w0)), rtol=1e-15)


def test_dominant_key_wins():
    rng = np.random.default_rng(4)
    T, d = 20, 16
    kc = _bf16(rng.standard_normal((T, 1, d)) * 0.01)
    q = np.zeros(d, np.uint16); q[3] = _bf16(1.0)
    kc[11, 0, 3] = _bf16(1000.0)
    vc = _bf16(rng.standard_normal((T, 1, d)))
    k_cache, v_cache, phys = _paged_from_contiguous(kc, vc, 6, 5, rng)
    out = oracle.attend_row(q, k_cache, v_cache, phys, 6, 0, T, 1.0)
    np.testing.assert_allclose(out, _val(vc[11, 0]), rtol=0, atol=1e-300)


def test_softmax_weights_sum_to_one():
    rng = np.random.default_rng(5)
    T, d = 300, 64
    kc = _bf16(rng.standard_normal((T, 1, d)) * 8)
    vc = _bf16(rng.standard_normal((T, 1, d)))
    k_cache, v_cache, phys = _paged_from_contiguous(kc, vc, 13, 30, rng)
    _, w = oracle.attend_row(_bf16(rng.standard_normal(d)), k_cache, v_cache, phys, 13, 0, T,
                             0.125, return_weights=True)
    assert abs(w.sum() - 1.0) < 1e-12 and (w >= 0).all()


def _random_case(rng, T, hkv, d, bs, npg):
    kc = _bf16(rng.standard_normal((T, hkv, d)))
    vc = _bf16(rng.standard_normal((T, hkv, d)))
    k_cache, v_cache, phys = _paged_from_contiguous(kc, vc, bs, npg, rng)
    return kc, vc, k_cache, v_cache, phys


def test_page_permutation_invariance_bitwise():
    rng = np.random.default_rng(6)
    T, hkv, d, bs = 200, 2, 32, 16
    kc = _bf16(rng.standard_normal((T, hkv, d)))
    vc = _bf16(rng.standard_normal((T, hkv, d)))
    q = _bf16(rng.standard_normal(d))
    outs = []
    for trial in range(3):
        k_cache, v_cache, phys = _paged_from_contiguous(kc, vc, bs, 20, np.random.default_rng(trial))
        outs.append(oracle.attend_row(q, k_cache, v_cache, phys, bs, 1, T, 0.2))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_block_size_invariance_bitwise():
    # The pages report page784 and page832 giving bitwise-identical results (page832 post §9):
    # the definition does not depend on the page size.
    rng = np.random.default_rng(8)
    T, hkv, d = 1700, 1, 16
    kc = _bf16(rng.standard_normal((T, hkv, d)))
    vc = _bf16(rng.standard_normal((T, hkv, d)))
    q = _bf16(rng.standard_normal(d))
    outs = []
    for bs in (784, 832, 64):
        k_cache, v_cache, phys = _paged_from_contiguous(kc, vc, bs, 28, rng)
        outs.append(oracle.attend_row(q, k_cache, v_cache, phys, bs, 0, T, 0.0625))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_token_order_invariance():
    rng = np.random.default_rng(9)
    T, d = 64, 32
    kc = _bf16(rng.standard_normal((T, 1, d)))
    vc = _bf16(rng.standard_normal((T, 1, d)))
    q = _bf16(rng.standard_normal(d))
    a = oracle.attend_row(q, *_paged_from_contiguous(kc, vc, 8, 8, rng)[:2],
                          np.arange(8, dtype=np.int32), 8, 0, T, 0.3)
    perm = rng.permutation(T)
    k2, v2, phys2 = _paged_from_contiguous(kc[perm], vc[perm], 8, 8, rng)
    b = oracle.attend_row(q, k2, v2, phys2, 8, 0, T, 0.3)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_decode_gqa_head_mapping_and_sequence_rows():
    # Every token of KV head g of sequence s carries the same V row c[s, g]; the output of
    # query head h of sequence s must then be exactly c[s, h // (Hq/Hkv)].
    rng = np.random.default_rng(10)
    S, hq, hkv, d, bs, npg = 3, 12, 4, 16, 8, 24
    lens = [5, 17, 23]
    c = _bf16(rng.standard_normal((S, hkv, d)))
    k_cache = _bf16(rng.standard_normal((npg, bs, hkv, d)))
    v_cache = np.full((npg, bs, hkv, d), 0xFFFF, np.uint16)
    bt = rng.permutation(npg).astype(np.int32).reshape(S, 8)
    for s in range(S):
        for p in range(-(-lens[s] // bs)):
            v_cache[bt[s, p]] = c[s]
            for o in range(bs):
                if p * bs + o >= lens[s]:
                    v_cache[bt[s, p], o] = 0xFFFF
    q = _bf16(rng.standard_normal((S, hq, d)))
    out = oracle.decode(q, k_cache, v_cache, bt, np.array(lens, np.int32), 0.25)
    for s in range(S):
        for h in range(hq):
            np.testing.assert_allclose(out[s, h], _val(c[s, h // 3]), rtol=1e-15, atol=0)


def test_decode_ignores_slots_past_seq_len():
    rng = np.random.default_rng(11)
    kc, vc, k_cache, v_cache, phys = _random_case(rng, 40, 2, 16, 16, 5)
    q = _bf16(rng.standard_normal((1, 4, 16)))
    out = oracle.decode(q, k_cache, v_cache, phys[None], np.array([33], np.int32), 0.25)
    assert np.isfinite(out).all()   # slots 33..47 of the last page are NaN and unread


def test_prefill_causal_row_equals_decode_of_its_prefix():
    # A chunk row at absolute position p sees keys 0..p: identical to q=1 decode with p+1 keys.
    rng = np.random.default_rng(12)
    hq, hkv, d, bs = 6, 2, 16, 8
    q_start, q_len = 21, 9
    kc, vc, k_cache, v_cache, phys = _random_case(rng, q_start + q_len, hkv, d, bs, 6)
    q = _bf16(rng.standard_normal((q_len, hq, d)))
    full = oracle.prefill(q, k_cache, v_cache, phys, q_start, True, 0.25)
    for i in range(q_len):
        dec = oracle.decode(q[i:i + 1], k_cache, v_cache, phys[None],
                            np.array([q_start + i + 1], np.int32), 0.25)
        assert np.array_equal(full[i], dec[0])
    nc = oracle.prefill(q, k_cache, v_cache, phys, q_start, False, 0.25)
    dec_all = oracle.decode(q[-1:], k_cache, v_cache, phys[None],
                            np.array([q_start + q_len], np.int32), 0.25)
    assert np.array_equal(nc[0], oracle.decode(q[:1], k_cache, v_cache, phys[None],
                                               np.array([q_start + q_len], np.int32), 0.25)[0])
    assert np.array_equal(full[-1], dec_all[0])


def test_prefill_future_tokens_do_not_matter_and_past_ones_do():
    rng = np.random.default_rng(13)
    hq, hkv, d, bs = 4, 1, 16, 8
    q_start, q_len = 10, 6
    T = q_start + q_len
    kc, vc, k_cache, v_cache, phys = _random_case(rng, T, hkv, d, bs, 4)
    q = _bf16(rng.standard_normal((q_len, hq, d)))
    base = oracle.prefill(q, k_cache, v_cache, phys, q_start, True, 0.25)
    i = 2                                   # row at position 12 sees keys 0..12
    k2, v2 = k_cache.copy(), v_cache.copy()
    t = q_start + i + 1                     # first invisible key: position 13
    k2[phys[t // bs], t % bs] = _bf16(50.0)
    v2[phys[t // bs], t % bs] = _bf16(50.0)
    after = oracle.prefill(q, k2, v2, phys, q_start, True, 0.25)
    assert np.array_equal(after[: i + 1], base[: i + 1])
    assert not np.allclose(after[i + 1:], base[i + 1:])
    t = q_start + i                         # last visible key: position 12
    k3 = k_cache.copy()
    k3[phys[t // bs], t % bs] = _bf16(50.0)
    assert not np.allclose(oracle.prefill(q, k3, v_cache, phys, q_start, True, 0.25)[i], base[i])


def test_oracle_reports_unmapped_pages():
    rng = np.random.default_rng(14)
    kc, vc, k_cache, v_cache, phys = _random_case(rng, 20, 1, 8, 8, 3)
    bt = phys.copy()
    bt[1] = 99
    with pytest.raises(ValueError):
        oracle.attend_row(_bf16(rng.standard_normal(8)), k_cache, v_cache, bt, 8, 0, 20, 0.5)


def test_slot_mapping_padding_position():
    bt = np.array([3, 1], dtype=np.int32)
    got = oracle.slot_mapping(np.array([-1, 5, -7], dtype=np.int32), bt, 4)
    assert [int(x) for x in got] == [-1, 1 * 4 + 1, -1]   # 5//4 = 1 -> page 1, offset 1


# ---------------------------------------------------------------- mixed batch (varlen)
def test_prefill_varlen_hand_worked_batch():
    # Equal scores (q = 0) make each row the mean of the V rows it sees: the values in
    # the golden file are those means, worked by hand for each chunk row's position.
    f = {r[0]: r[1:] for r in _golden_lines("prefill_varlen_hand.txt") if r[0] != "row"}
    want = [list(map(float, r[2:])) for r in _golden_lines("prefill_varlen_hand.txt")
            if r[0] == "row"]
    k_lens = [int(x) for x in f["k_lens"]]
    cu = [int(x) for x in f["cu_seqlens_q"]]
    bs, d, npool = 2, 8, 8
    tables = np.array([[4, 0, 6], [2, 7, -1], [5, 1, -1]], dtype=np.int32)
    rng = np.random.default_rng(2)
    k_cache = np.full((npool, bs, 1, d), 0xFFFF, dtype=np.uint16)
    v_cache = np.full_like(k_cache, 0xFFFF)
    for s, L in enumerate(k_lens):
        for t in range(L):  # whole pages enumerated: token t is page t // 2, slot t % 2
            page, off = tables[s][t // bs], t % bs
            k_cache[page, off, 0] = _bf16(rng.standard_normal(d))
            v_cache[page, off, 0] = _bf16(np.full(d, 100.0 * s + t))
    q = np.zeros((cu[-1], 1, d), dtype=np.uint16)  # BF16 +0
    for col, causal in ((0, True), (1, False)):
        got = oracle.prefill_varlen(q, k_cache, v_cache, tables, cu, k_lens, causal, 0.0625)
        for r in range(cu[-1]):
            assert np.all(got[r, 0] == want[r][col]), (causal, r, got[r, 0, 0], want[r][col])


def test_prefill_varlen_chunk_rows_are_decodes_of_their_prefixes():
    # A chunk is the last q_len tokens of its sequence: its first row sees
    # k_len - q_len + 1 keys and its last row all k_len keys, which is what a decode of
    # that many keys over the same block-table row computes.
    rng = np.random.default_rng(11)
    bs, hq, hkv, d = 16, 6, 2, 32
    k_lens, q_rows = [40, 7, 33, 16], [5, 7, 0, 16]
    npg = sum(-(-L // bs) for L in k_lens) + 2
    perm = rng.permutation(npg).astype(np.int32)
    mb = max(-(-L // bs) for L in k_lens)
    tables = np.full((len(k_lens), mb), -1, dtype=np.int32)
    k = 0
    for s, L in enumerate(k_lens):
        n = -(-L // bs)
        tables[s, :n] = perm[k:k + n]
        k += n
    k_cache = _bf16(rng.standard_normal((npg, bs, hkv, d)))
    v_cache = _bf16(rng.standard_normal((npg, bs, hkv, d)))
    cu = np.concatenate([[0], np.cumsum(q_rows)]).astype(np.int32)
    q = _bf16(rng.standard_normal((int(cu[-1]), hq, d)))
    got = oracle.prefill_varlen(q, k_cache, v_cache, tables, cu, k_lens, True, 0.125)
    for s, L in enumerate(k_lens):
        r0, r1 = int(cu[s]), int(cu[s + 1])
        if r1 == r0:
            continue
        for row, keys in ((r0, L - (r1 - r0) + 1), (r1 - 1, L)):
            dec = oracle.decode(q[row:row + 1], k_cache, v_cache, tables[s:s + 1],
                                np.array([keys], np.int32), 0.125)
            np.testing.assert_allclose(got[row], dec[0], rtol=0, atol=1e-12)
    # The rows of an empty chunk's neighbours stay in place: total rows = sum of chunks.
    assert got.shape[0] == sum(q_rows)


def test_prefill_varlen_of_one_sequence_is_its_chunk():
    rng = np.random.default_rng(12)
    bs, hq, hkv, d = 8, 4, 1, 16
    L, ql = 29, 11
    npg = -(-L // bs) + 1
    table = rng.permutation(npg)[:-(-L // bs)].astype(np.int32)
    k_cache = _bf16(rng.standard_normal((npg, bs, hkv, d)))
    v_cache = _bf16(rng.standard_normal((npg, bs, hkv, d)))
    q = _bf16(rng.standard_normal((ql, hq, d)))
    a = oracle.prefill_varlen(q, k_cache, v_cache, table[None, :], [0, ql], [L], True, 0.25)
    b = oracle.prefill(q, k_cache, v_cache, table, L - ql, True, 0.25)
    assert np.array_equal(a, b)
