// pa_plan.cu -- static work assignment for the persistent prefill kernel (host only).
//
// The causal chunk's work items (128 query rows of one head, or of several heads of a
// GQA group for a packed last tile) differ in length: row tile r of a chunk at q_start reads
// q_start + r*128 + 128 keys.  With about five items per
// CTA, walking them in a fixed order leaves some CTAs well above the mean (the q=4096
// chunk over 4096 prior tokens: 138 tiles on the busiest CTA against a mean of 123.8).
// This planner assigns items to CTAs up front:
//   1. cost of an item = its K/V tiles + 1 (the per-item Q load and epilogue);
//   2. longest-processing-time first: items by decreasing cost, each to the CTA with the
//      least cost so far;
//   3. local search: while some move of one item off the most loaded CTA, or swap of one
//      of its items with a cheaper item of another CTA, lowers that CTA's cost without
//      raising the other one's to the same level, apply the best such change.
// Whole items cannot always be balanced: the q=1685 tail chunk has 336 items of ~52
// tiles for 152 CTAs, so some CTAs run three items and most two (149 tiles against a
// mean of 114), and a short chunk over a long context has fewer items than CTAs.  When
// the caller provides a workspace, a second plan may split items along the keys:
//   4. with a target T (the mean cost rounded up, then raised step by step until the
//      plan fits), items go by decreasing cost to the least loaded CTA while that stays
//      within T; an item that does not fit is cut into pieces of at least
//      kPfMinPieceTiles tiles that fill the least loaded CTAs up to T (a piece costs its
//      tiles + 2: its Q load, its epilogue and the partial it writes), at most
//      kPfMaxPiecesPerItem pieces per item.
// The split plan is taken when its busiest CTA is at least 3% cheaper.  Each CTA then
// runs its items and pieces longest first.  Plans are cached per shape, since a serving
// loop prefills chunks of the same few shapes over and over.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include "pa.h"
#include "pa_internal.h"

namespace pa {

namespace {

struct PlanKey {
    std::vector<std::pair<int, int>> chunks;  // (q_len, q_start) of each sequence
    int causal, hq, group, bs, ctas;
    bool allow_split;
    bool operator==(const PlanKey &o) const {
        return chunks == o.chunks && causal == o.causal && hq == o.hq && group == o.group &&
               bs == o.bs && ctas == o.ctas && allow_split == o.allow_split;
    }
};

struct CachedPlan {
    PlanKey key;
    int max_cost;
    std::vector<uint16_t> off, items;
    std::vector<PrefillPiece> pieces;
    std::vector<uint16_t> split_item, split_slot0, split_n;
};

// A CTA's list: whole items (index) and pieces (kPfPieceBit | piece), with their costs.
struct Entry {
    uint16_t code;
    int cost;
};

// Fills out.off / out.items from per-CTA lists, each run longest first.
void emit(std::vector<std::vector<Entry>> &bins, CachedPlan &out) {
    const int G = (int)bins.size();
    out.off.assign(G + 1, 0);
    out.items.clear();
    int mx = 0;
    for (int b = 0; b < G; ++b) {
        std::stable_sort(bins[b].begin(), bins[b].end(), [](const Entry &x, const Entry &y) {
            return x.cost != y.cost ? x.cost > y.cost : x.code < y.code;
        });
        int load = 0;
        for (const Entry &e : bins[b]) {
            out.items.push_back(e.code);
            load += e.cost;
        }
        mx = std::max(mx, load);
        out.off[b + 1] = (uint16_t)out.items.size();
    }
    out.max_cost = mx;
}

// Plan 4 of the header: whole items while they fit under the target, pieces otherwise.
// Returns false when no target up to the largest whole-item plan gives a plan within
// the schedule's limits.
bool split_plan(const std::vector<int> &tiles, int G, int limit, CachedPlan &out) {
    const int n = (int)tiles.size();
    long long total = 0;
    for (int t : tiles) total += t + 1;
    std::vector<int> order(n);
    for (int i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return tiles[a] > tiles[b]; });
    using Slot = std::pair<long long, int>;
    for (long long target = (total + G - 1) / G; target < limit; ++target) {
        std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
        for (int b = 0; b < G; ++b) heap.push({0, b});
        std::vector<std::vector<Entry>> bins(G);
        std::vector<long long> load(G, 0);
        std::vector<PrefillPiece> pieces;
        std::vector<uint16_t> si, s0, sn;
        bool ok = true;
        for (int i : order) {
            const int t = tiles[i];
            const int b0 = heap.top().second;
            if (load[b0] + t + 1 <= target) {
                heap.pop();
                bins[b0].push_back({(uint16_t)i, t + 1});
                load[b0] += t + 1;
                heap.push({load[b0], b0});
                continue;
            }
            // Cut the item into pieces that fill the least loaded CTAs up to the target.
            si.push_back((uint16_t)i);
            s0.push_back((uint16_t)pieces.size());
            int begin = 0;
            std::vector<int> used;
            while (begin < t) {
                if (heap.empty()) { ok = false; break; }
                const int b = heap.top().second;
                heap.pop();
                used.push_back(b);
                int take = (int)std::min<long long>(t - begin, target - load[b] - 2);
                if (t - begin - take > 0 && t - begin - take < kPfMinPieceTiles)
                    take = t - begin - kPfMinPieceTiles;
                if (take < kPfMinPieceTiles) { ok = false; break; }
                if ((int)pieces.size() == kPfMaxPieces) { ok = false; break; }
                const uint16_t code = (uint16_t)(kPfPieceBit | pieces.size());
                pieces.push_back({(uint16_t)i, (uint16_t)begin, (uint16_t)(begin + take),
                                  (uint16_t)pieces.size()});
                bins[b].push_back({code, take + 2});
                load[b] += take + 2;
                begin += take;
            }
            for (int b : used) heap.push({load[b], b});
            sn.push_back((uint16_t)(pieces.size() - s0.back()));
            if (!ok || (int)si.size() > kPfMaxSplitItems || sn.back() > kPfMaxPiecesPerItem) {
                ok = false;
                break;
            }
        }
        if (!ok) continue;
        long long entries = 0;
        for (auto &bn : bins) entries += (long long)bn.size();
        if (entries > kPfSchedMaxItems) return false;
        emit(bins, out);
        out.pieces = std::move(pieces);
        out.split_item = std::move(si);
        out.split_slot0 = std::move(s0);
        out.split_n = std::move(sn);
        return true;
    }
    return false;
}

constexpr int kPlanCacheSize = 8;
std::mutex g_plan_mu;
std::vector<CachedPlan> g_plan_cache;  // most recently used last

void compute_plan(const PlanKey &k, CachedPlan &out) {
    // Items sequence by sequence, numbered as prefill_item_at gives them.
    std::vector<int> cost;
    for (const auto &c : k.chunks) {
        const int n = prefill_chunk_items(c.first, k.hq, k.group);
        for (int i = 0; i < n; ++i) {
            int qt, h0, hp;
            prefill_item_at(i, c.first, k.hq, k.group, &qt, &h0, &hp);
            cost.push_back(prefill_item_tiles(c.first, c.second, k.causal, qt * kPfQRows, k.bs) +
                           1);
        }
    }
    const int n = (int)cost.size();
    const int G = std::min(k.ctas, n);
    // 2. LPT.
    std::vector<int> order(n);
    for (int i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int b) { return cost[a] > cost[b]; });
    std::vector<std::vector<int>> bins(G);
    std::vector<long long> load(G, 0);
    using Slot = std::pair<long long, int>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int b = 0; b < G; ++b) heap.push({0, b});
    for (int i : order) {
        const int b = heap.top().second;
        heap.pop();
        bins[b].push_back(i);
        load[b] += cost[i];
        heap.push({load[b], b});
    }
    // 3. Local search on the most loaded CTA (bounded; each step lowers the sum of the
    // squared loads, so it ends well before the bound on any input).
    for (int step = 0; step < 4 * n + 64; ++step) {
        int i = 0;
        for (int b = 1; b < G; ++b)
            if (load[b] > load[i]) i = b;
        const long long Li = load[i];
        long long best_nm = Li;
        int bj = -1, ba = -1, bb = -1;
        for (int j = 0; j < G; ++j) {
            const long long Lj = load[j];
            if (j == i || Lj >= Li - 1) continue;
            for (int ai = 0; ai < (int)bins[i].size(); ++ai) {
                const int ca = cost[bins[i][ai]];
                if (Lj + ca < Li) {  // move
                    const long long nm = std::max(Li - ca, Lj + ca);
                    if (nm < best_nm) best_nm = nm, bj = j, ba = ai, bb = -1;
                }
                for (int bi = 0; bi < (int)bins[j].size(); ++bi) {  // swap
                    const int d = ca - cost[bins[j][bi]];
                    if (d <= 0 || Lj + d >= Li) continue;
                    const long long nm = std::max(Li - d, Lj + d);
                    if (nm < best_nm) best_nm = nm, bj = j, ba = ai, bb = bi;
                }
            }
        }
        if (bj < 0) break;
        const int a = bins[i][ba];
        bins[i].erase(bins[i].begin() + ba);
        if (bb >= 0) {
            const int b = bins[bj][bb];
            bins[bj].erase(bins[bj].begin() + bb);
            bins[i].push_back(b);
            load[i] += cost[b];
            load[bj] -= cost[b];
        }
        bins[bj].push_back(a);
        load[i] -= cost[a];
        load[bj] += cost[a];
    }
    out.key = k;
    std::vector<std::vector<Entry>> entries(G);
    for (int b = 0; b < G; ++b)
        for (int x : bins[b]) entries[b].push_back({(uint16_t)x, cost[x]});
    emit(entries, out);
    out.pieces.clear();
    out.split_item.clear();
    out.split_slot0.clear();
    out.split_n.clear();
    // 4. The split plan, if allowed and at least 3% better.
    if (k.allow_split) {
        std::vector<int> tiles(n);
        for (int i = 0; i < n; ++i) tiles[i] = cost[i] - 1;
        CachedPlan alt;
        if (split_plan(tiles, k.ctas, out.max_cost, alt) &&
            alt.max_cost * 100 <= out.max_cost * 97 && !alt.pieces.empty()) {
            alt.key = k;
            out = std::move(alt);
        }
    }
}

}  // namespace

bool plan_prefill(int num_seqs, const int *q_lens, const int *q_starts, int causal,
                  int num_q_heads, int group, int block_size, int num_ctas, bool allow_split,
                  PrefillSchedule *s, int *max_cost) {
    if (num_seqs < 1 || num_q_heads < 1 || group < 1 || num_q_heads % group || block_size < 1 ||
        num_ctas < 1)
        return false;
    long long n = 0;
    PlanKey key{{}, causal ? 1 : 0, num_q_heads, group, block_size, num_ctas, allow_split};
    for (int b = 0; b < num_seqs; ++b) {
        if (q_lens[b] < 1 || q_starts[b] < 0 || q_lens[b] > (1 << 30)) return false;
        n += (long long)prefill_chunk_items(q_lens[b], num_q_heads, group);
        key.chunks.emplace_back(q_lens[b], q_starts[b]);
    }
    if (n > kPfSchedMaxItems || std::min<long long>(num_ctas, n) > kPfSchedMaxCtas)
        return false;
    std::lock_guard<std::mutex> lock(g_plan_mu);
    auto it = std::find_if(g_plan_cache.begin(), g_plan_cache.end(),
                           [&](const CachedPlan &c) { return c.key == key; });
    if (it == g_plan_cache.end()) {
        CachedPlan fresh;
        compute_plan(key, fresh);
        if ((int)g_plan_cache.size() == kPlanCacheSize) g_plan_cache.erase(g_plan_cache.begin());
        g_plan_cache.push_back(std::move(fresh));
        it = g_plan_cache.end() - 1;
    } else if (it != g_plan_cache.end() - 1) {
        std::rotate(it, it + 1, g_plan_cache.end());  // mark as most recently used
        it = g_plan_cache.end() - 1;
    }
    if (s) {
        const int G = (int)it->off.size() - 1;
        s->num_ctas = G;
        std::memcpy(s->off, it->off.data(), (G + 1) * sizeof(uint16_t));
        std::memcpy(s->items, it->items.data(), it->items.size() * sizeof(uint16_t));
        s->num_pieces = (int)it->pieces.size();
        s->num_split = (int)it->split_item.size();
        if (s->num_pieces)
            std::memcpy(s->pieces, it->pieces.data(), s->num_pieces * sizeof(PrefillPiece));
        for (int x = 0; x < s->num_split; ++x) {
            s->split_item[x] = it->split_item[x];
            s->split_slot0[x] = it->split_slot0[x];
            s->split_n[x] = it->split_n[x];
        }
    }
    if (max_cost) *max_cost = it->max_cost;
    return true;
}

}  // namespace pa

extern "C" int pa_prefill_plan(int q_len, int q_start, int causal, int num_q_heads,
                               int num_kv_heads, int block_size, int num_ctas,
                               int32_t *cta_of_item, int *num_items, int *max_cost) {
    if (q_len < 1 || q_start < 0 || (int64_t)q_start + q_len > INT32_MAX || num_q_heads < 1 ||
        num_kv_heads < 1 || num_q_heads % num_kv_heads || block_size < 1 || num_ctas < 1)
        return PA_ERR_INVALID_ARG;
    static thread_local pa::PrefillSchedule s;
    int mc = 0;
    if (!pa::plan_prefill(1, &q_len, &q_start, causal, num_q_heads, num_q_heads / num_kv_heads,
                          block_size, num_ctas, false, &s, &mc))
        return PA_ERR_UNSUPPORTED;
    const int n = s.off[s.num_ctas];
    if (num_items) *num_items = n;
    if (max_cost) *max_cost = mc;
    if (cta_of_item)
        for (int b = 0; b < s.num_ctas; ++b)
            for (int x = s.off[b]; x < s.off[b + 1]; ++x) cta_of_item[s.items[x]] = b;
    return PA_OK;
}

extern "C" int pa_prefill_plan_pieces(int q_len, int q_start, int causal, int num_q_heads,
                                      int num_kv_heads, int block_size, int num_ctas,
                                      int max_pieces,
                                      int32_t *cta_of_item, int32_t *piece_item,
                                      int32_t *piece_tile_begin, int32_t *piece_tile_end,
                                      int32_t *piece_cta, int *num_items, int *num_pieces,
                                      int *max_cost) {
    if (q_len < 1 || q_start < 0 || (int64_t)q_start + q_len > INT32_MAX || num_q_heads < 1 ||
        num_kv_heads < 1 || num_q_heads % num_kv_heads || block_size < 1 || num_ctas < 1 ||
        max_pieces < 0)
        return PA_ERR_INVALID_ARG;
    static thread_local pa::PrefillSchedule s;
    int mc = 0;
    const int group = num_q_heads / num_kv_heads;
    if (!pa::plan_prefill(1, &q_len, &q_start, causal, num_q_heads, group, block_size, num_ctas,
                          true, &s, &mc))
        return PA_ERR_UNSUPPORTED;
    const int items = pa::prefill_chunk_items(q_len, num_q_heads, group);
    if (num_items) *num_items = items;
    if (num_pieces) *num_pieces = s.num_pieces;
    if (max_cost) *max_cost = mc;
    if (s.num_pieces > max_pieces) return PA_ERR_INVALID_ARG;
    if (cta_of_item)
        for (int i = 0; i < items; ++i) cta_of_item[i] = -1;
    for (int b = 0; b < s.num_ctas; ++b)
        for (int x = s.off[b]; x < s.off[b + 1]; ++x) {
            if (!(s.items[x] & pa::kPfPieceBit)) {
                if (cta_of_item) cta_of_item[s.items[x]] = b;
                continue;
            }
            const int pc = s.items[x] & ~pa::kPfPieceBit;
            if (piece_item) piece_item[pc] = s.pieces[pc].item;
            if (piece_tile_begin) piece_tile_begin[pc] = s.pieces[pc].tile_begin;
            if (piece_tile_end) piece_tile_end[pc] = s.pieces[pc].tile_end;
            if (piece_cta) piece_cta[pc] = b;
        }
    return PA_OK;
}
