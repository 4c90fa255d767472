"""Host-only checks of the prefill kernel's static work assignment (pa_prefill_plan).

The plan decides which persistent CTA runs which work item (128 query rows of one head,
or of all heads of a GQA group for a chunk's short last query tile);
it does not change what is computed, so it is checked for validity and balance, with
the item costs recomputed here from the kernel's streaming rule: an item reads the keys
up to its last row (causal) or all keys, in page-local blocks of 64 keys, four blocks
per 256-key tile, and costs its tile count plus one.
"""
import math

import pytest

from test_abi_host import lib  # noqa: F401  (builds and loads libpa.so)


def item_tiles(q_len, q_start, causal, r0, bs):
    rows = min(128, q_len - r0)
    nkeys = q_start + r0 + rows if causal else q_start + q_len
    full, rem = divmod(nkeys, bs)
    nblocks = full * math.ceil(bs / 64) + math.ceil(rem / 64)
    return math.ceil(nblocks / 4)


def tile_heads(q_len, G):
    """Heads per item of a chunk's last query tile: the largest divisor hp of G with
    hp * r <= 128 (r: the tile's rows), 1 if none is above 1."""
    r = q_len - 128 * (math.ceil(q_len / 128) - 1)
    return next((hp for hp in range(G, 1, -1) if G % hp == 0 and hp * r <= 128), 1)


def item_costs(q_len, q_start, causal, hq, bs, hkv=4):
    # Items from the last query tile to the first, one per head; the last tile runs as
    # hq / hp items of hp heads each (hp from tile_heads).
    nqt = math.ceil(q_len / 128)
    hp = tile_heads(q_len, hq // hkv)
    costs = []
    for qt in range(nqt - 1, -1, -1):
        n = hq // hp if qt == nqt - 1 else hq
        costs += [item_tiles(q_len, q_start, causal, qt * 128, bs) + 1] * n
    return costs


def snake_max(costs, G):
    load = [0] * G
    for idx, c in enumerate(costs):
        k, b = divmod(idx, G)
        load[b if k % 2 == 0 else G - 1 - b] += c
    return max(load)


SHAPES = [
    (4096, 4096, True, 24, 832, 152),   # the q=4096 chunk over 4096 prior tokens
    (4096, 0, True, 24, 832, 152),      # first chunk of a prompt
    (1685, 12288, True, 24, 832, 152),  # a tail chunk
    (4096, 4096, True, 24, 784, 152),   # ragged 16-token page tails
    (4096, 4096, False, 24, 832, 152),  # non-causal: all items equal
    (130, 900, True, 24, 832, 152),     # fewer items than CTAs
    (2048, 4096, True, 8, 64, 148),
]


@pytest.mark.parametrize("q_len,q_start,causal,hq,bs,G", SHAPES)
def test_every_item_runs_exactly_once_on_a_valid_cta(lib, q_len, q_start, causal, hq, bs, G):
    import paged_kv_cache_09_gb300 as pa
    cta, max_cost = pa.prefill_plan(q_len, q_start, causal, hq, 4, bs, G)
    costs = item_costs(q_len, q_start, causal, hq, bs)
    assert len(cta) == len(costs)
    ctas = min(G, len(costs))
    assert all(0 <= b < ctas for b in cta)
    load = [0] * ctas
    for i, b in enumerate(cta):
        load[b] += costs[i]
    assert max(load) == max_cost
    assert min(load) > 0  # no CTA is left idle
    # Never worse than the fixed snake order, never below the obvious lower bounds.
    assert max_cost <= snake_max(costs, ctas)
    assert max_cost >= max(max(costs), math.ceil(sum(costs) / ctas))


def test_headline_chunk_is_balanced_to_the_lower_bound(lib):
    import paged_kv_cache_09_gb300 as pa
    costs = item_costs(4096, 4096, True, 24, 832)
    _, max_cost = pa.prefill_plan(4096, 4096, True, 24, 4, 832, 152)
    lb = math.ceil(sum(costs) / 152)
    assert max_cost <= lb + 1
    assert snake_max(costs, 152) - max_cost >= 5  # 143 -> 129 in cost units


def test_plan_is_deterministic_and_cached(lib):
    import paged_kv_cache_09_gb300 as pa
    a = pa.prefill_plan(4096, 4096, True, 24, 4, 832, 152)
    pa.prefill_plan(2048, 0, True, 24, 4, 832, 152)
    b = pa.prefill_plan(4096, 4096, True, 24, 4, 832, 152)
    assert a == b


def test_plan_refuses_bad_sizes_and_oversized_problems(lib):
    import paged_kv_cache_09_gb300 as pa
    with pytest.raises(pa.PAError):
        pa.prefill_plan(0, 0, True, 24, 4, 832, 152)
    with pytest.raises(pa.PAError):
        pa.prefill_plan(128, -1, True, 24, 4, 832, 152)
    with pytest.raises(pa.PAError):  # 33000 rows x 24 heads: 6192 items > 6144
        pa.prefill_plan(33000, 0, True, 24, 4, 832, 152)


SPLIT_SHAPES = SHAPES + [
    (1, 8192, True, 24, 832, 152),      # one row per head over a long context
    (64, 8192, True, 24, 832, 152),
    (200, 3000, True, 24, 784, 152),
    (1685, 12288, True, 24, 832, 148),
]


@pytest.mark.parametrize("q_len,q_start,causal,hq,bs,G", SPLIT_SHAPES)
def test_split_plan_covers_every_key_tile_once(lib, q_len, q_start, causal, hq, bs, G):
    # With a workspace, items may be cut along their key tiles into pieces on different
    # CTAs.  Every split item's pieces must tile [0, n) exactly, in order, each at least 4
    # tiles; every other item runs whole on one CTA; the busiest CTA's cost (tiles + 1 per
    # whole item, + 2 per piece) is the reported one, and never above the unsplit plan's.
    import paged_kv_cache_09_gb300 as pa
    cta, pieces, max_cost = pa.prefill_plan_pieces(q_len, q_start, causal, hq, 4, bs, G)
    costs = item_costs(q_len, q_start, causal, hq, bs)
    assert len(cta) == len(costs)
    _, unsplit = pa.prefill_plan(q_len, q_start, causal, hq, 4, bs, G)
    load = [0] * G
    for i, b in enumerate(cta):
        if b >= 0:
            load[b] += costs[i]
    by_item = {}
    for item, t0, t1, b in pieces:
        assert 0 <= b < G and cta[item] == -1
        assert t1 - t0 >= 4
        load[b] += (t1 - t0) + 2
        by_item.setdefault(item, []).append((t0, t1))
    for item, rs in by_item.items():
        rs.sort()
        assert 2 <= len(rs) <= 16
        assert rs[0][0] == 0 and rs[-1][1] == costs[item] - 1
        assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
    assert set(by_item) == {i for i, b in enumerate(cta) if b < 0}
    assert max(load) == max_cost
    assert max_cost <= unsplit
    if pieces:
        assert max_cost * 100 <= unsplit * 97


def test_split_plan_balances_the_tail_chunk_and_short_chunks(lib):
    import paged_kv_cache_09_gb300 as pa
    # The q=1685 tail: 336 items of ~52 tiles on 152 CTAs; whole items leave the busiest
    # CTA at 149 (three items); pieces bring it near the mean.
    _, pieces, split = pa.prefill_plan_pieces(1685, 12288, True, 24, 4, 832, 152)
    _, whole = pa.prefill_plan(1685, 12288, True, 24, 4, 832, 152)
    mean = sum(item_costs(1685, 12288, True, 24, 832)) / 152
    assert whole >= 140 and pieces and split <= mean + 10
    # 24 one-row items over 8192 keys (33 tiles each) on 152 CTAs: whole items leave 128
    # CTAs idle; pieces spread each item over several CTAs.
    _, pieces, split = pa.prefill_plan_pieces(1, 8192, True, 24, 4, 832, 152)
    _, whole = pa.prefill_plan(1, 8192, True, 24, 4, 832, 152)
    assert pieces and split * 3 <= whole


@pytest.mark.parametrize("q_len,hq,hkv,hp", [
    (21, 24, 4, 6), (22, 24, 4, 3), (42, 24, 4, 3), (43, 24, 4, 2), (64, 24, 4, 2),
    (65, 24, 4, 1), (1, 24, 4, 6), (1685, 24, 4, 6), (1686, 24, 4, 3), (128 + 60, 24, 4, 2),
    (64, 8, 4, 2), (65, 8, 4, 1), (8, 16, 1, 16), (9, 16, 1, 8), (33, 32, 4, 2),
    (5, 4, 4, 1), (128 + 32, 16, 4, 4), (40, 24, 8, 3), (25, 20, 4, 5), (26, 20, 4, 1),
])
def test_short_last_tile_runs_as_items_of_several_heads(lib, q_len, hq, hkv, hp):
    # The last query tile's r rows of hp heads of a KV head share one item, hp the largest
    # divisor of G = hq / hkv with hp * r <= 128: hq / hp items for that tile instead of hq.
    import paged_kv_cache_09_gb300 as pa
    assert tile_heads(q_len, hq // hkv) == hp
    cta, _ = pa.prefill_plan(q_len, 1000, True, hq, hkv, 832, 152)
    nqt = math.ceil(q_len / 128)
    assert len(cta) == (nqt - 1) * hq + hq // hp
    assert len(cta) == len(item_costs(q_len, 1000, True, hq, 832, hkv))
    cta, pieces, _ = pa.prefill_plan_pieces(q_len, 1000, True, hq, hkv, 832, 152)
    assert len(cta) == (nqt - 1) * hq + hq // hp


def test_plan_refuses_a_group_that_does_not_divide(lib):
    import paged_kv_cache_09_gb300 as pa
    with pytest.raises(pa.PAError):
        pa.prefill_plan(100, 0, True, 24, 5, 832, 152)
    with pytest.raises(pa.PAError):
        pa.prefill_plan_pieces(100, 0, True, 24, 0, 832, 152)
