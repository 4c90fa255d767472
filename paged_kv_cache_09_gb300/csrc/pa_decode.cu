// pa_decode.cu -- q=1 paged GQA decode: split-context kernel + log-sum-exp combine.
//
// What is computed (page832 post §5, §7): for sequence s and query head h,
//     out[s, h] = softmax_t(scale * q[s, h] . k_t) . v_t,  t < seq_lens[s],
// with k_t, v_t of KV head g = h / G read through the block table (page832 §1).
//
// How (GB300 design, not the pages' DCU design):
//   * grid = (splits, KV heads, sequences).  A CTA owns a contiguous run of page-local
//     16-token tiles of one (sequence, KV head) and all G <= 8 query heads of that KV
//     head, so each K/V byte is read from HBM once for the whole group.
//   * Tiles are 16 page-local tokens; a ring stage holds two consecutive tiles (32 KB).
//     One producer thread reads each block-table entry once and issues the stage's TMA
//     loads: one box per tile for K and one for V, each all 256 dims of the tile's 16
//     rows (8 KB, a 5-D view of the cache whose box is laid out as four 128-byte-swizzled
//     64-dim chunks).  The SM's cost of a TMA box grows slowly with its size, so the box
//     count sets the issue rate: 16 boxes of 16 rows x 64 dims a stage capped an SM below
//     its share of HBM bandwidth; 4 boxes a stage leave room to spare, whether or not the
//     two tiles lie in one page (16-token pages: 32K step 32.3 -> 26.9 us; batched decode
//     195.7 -> 187.3 us).  Rows past a page end come back as zeros and are masked.  The
//     loads mark their L2 lines evict-first: each is read once.
//   * With a new token to append (a decode step), one consumer warp of the CTA holding
//     that token's tile writes its K/V row at the slot the block table gives (or checks
//     a given slot) before the producer loads that tile.
//   * The consumer warps (four with a 4-stage ring for short splits, three with a 6-stage
//     ring for long ones) take tiles round-robin (short splits: tile i -> warp i % C,
//     half i % 2 of ring slot (i / 2) % S, a slot released by the warps of both its tiles;
//     long splits: stage m -> warp m % C).  Per tile: S^T = K Q^T
//     on the tensor cores (mma.m16n8k16, tokens as M, the group's heads as N, two
//     accumulator chains), online softmax over tokens with warp shuffles, then
//     O^T += V^T P^T with P split into a BF16 high part and a BF16 low part (two MMAs),
//     which keeps P to ~16 significant bits.
//   * At the end the warps merge their (max, sum, acc) through shared memory and the
//     CTA writes one fp32 partial per query head; the combine kernel (four CTAs per
//     query head, 64 dims each) merges the splits with a log-sum-exp and writes BF16.
//     Both kernels use programmatic dependent launch, so the combine's launch overlaps
//     the split kernel's tail.
#include <math_constants.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

// A ring stage is [K | V], each [tile of the pair][64-dim chunk][16 rows][128 B]: one TMA
// box (all 256 dims of a tile's 16 rows) fills one tile's K or V.
constexpr int kDecTileBytes = kDecTile * 128;               // one tile's rows of a 64-dim chunk: 2 KB
constexpr int kDecTileKBytes = kChunks * kDecTileBytes;     // one tile's K (or V), all dims: 8 KB
constexpr int kDecHalf = kDecPair * kDecTileKBytes;         // K (or V) of one stage: 16 KB
constexpr int kDecStageBytes = 2 * kDecHalf;                // 32 KB
// Merge buffers, per warp and head: O row (padded by 4 floats, so that the 4 head
// columns a warp stores at once fall in different banks), max and sum.
constexpr int kDecMergeRow = kHeadDim + 4;
template <int kC, int kS>
constexpr int dec_smem_bytes() {
    static_assert(kC * kDecMaxGroup * (kDecMergeRow + 2) * 4 <= kS * kDecStageBytes,
                  "merge buffers reuse the ring");
    return 1024 + kS * kDecStageBytes + (2 * kS + 1) * 8 + 8;  // + the abort flag
}

constexpr int kCombineThreads = 256;
constexpr int kCombineParts = 4;                       // CTAs per (query head, sequence)
constexpr int kCombineDims = kHeadDim / kCombineParts;  // dims one CTA merges: 2 per lane

struct DecodeKParams {
    const uint16_t *q;
    const int32_t *block_table;
    int64_t bt_stride;
    const int32_t *seq_lens;
    int max_seq_len;
    int num_q_heads;
    int group;
    int block_size;
    int tiles_per_page;
    int tiles_per_split;
    int num_splits;
    int64_t num_pages;
    float scale_log2;   // scale * log2(e): scores are kept in base-2 units
    float *part_o;      // [S, Hq, splits, D] unnormalised sums
    float2 *part_ml;    // [S, Hq, splits] (running max in base-2 units, sum of weights)
    uint16_t *out;
    unsigned *err;
    // Fused write of the token being decoded (new_k == nullptr: none).  Its slot comes
    // from new_slots, or, with new_slots == nullptr, from the block table (and is then
    // stored to slot_out when that is set).
    uint16_t *k_cache_w, *v_cache_w;
    const uint16_t *new_k, *new_v;   // [S, Hkv, D]
    const int64_t *new_slots;        // [S]
    int64_t *slot_out;               // [S]
    int64_t page_stride;
    int num_kv_heads;
};

// Fused write of the token being decoded, done by one consumer warp of the CTA that owns
// sequence `seq`'s last tile as soon as the CTA starts: each lane copies 16 bytes of
// the K row and 16 of the V row of KV head g, every lane fences its stores against the
// async proxy, and after the warp has converged lane 0 arrives on `written`.  The
// producer waits on `written` before it issues the TMA load of that last tile.  A given
// slot is written only if it matches the block table's slot for position seq_len - 1;
// without given slots that slot is the one taken (the slot-mapping formula), and the
// CTA of KV head 0 reports it.
__device__ __forceinline__ void write_newest_token(const DecodeKParams &p, const int32_t *bt,
                                                   int seq, int g, int seq_len, int lane,
                                                   uint64_t *written) {
    const int pos = seq_len - 1;
    const int lp = pos / p.block_size;
    const int off = pos - lp * p.block_size;
    const int page = bt[lp];
    const int64_t mapped = page < 0 ? -1 : (int64_t)page * p.block_size + off;
    const bool given = p.new_slots != nullptr;
    const int64_t slot = given ? p.new_slots[seq] : mapped;
    if (!given && g == 0 && lane == 0 && p.slot_out) p.slot_out[seq] = mapped;
    if (slot >= 0 || !given) {  // a negative given slot is padding
        if (page >= 0 && page < p.num_pages && slot == mapped) {
            const int64_t src = ((int64_t)seq * p.num_kv_heads + g) * kHeadDim;
            const int64_t dst =
                page * p.page_stride + ((int64_t)off * p.num_kv_heads + g) * kHeadDim;
            const uint4 k = reinterpret_cast<const uint4 *>(p.new_k + src)[lane];
            const uint4 v = reinterpret_cast<const uint4 *>(p.new_v + src)[lane];
            reinterpret_cast<uint4 *>(p.k_cache_w + dst)[lane] = k;
            reinterpret_cast<uint4 *>(p.v_cache_w + dst)[lane] = v;
        } else if (lane == 0) {
            atomicOr(p.err, given ? kErrSlot : kErrPage);
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(written);
}

// The decode's four tensor maps: K and V with 32-row boxes, and with 16-row boxes.
struct DecMaps {
    CUtensorMap k, v;
};

// Loads the two tiles of a ring stage, rows [off0, off0 + 16) of page0 and rows
// [off1, off1 + 16) of page1 (K and V of KV head g), into ring stage `st`, completing on
// `bar`: four boxes of 8 KB.  Rows past a page end, and a page outside the pool, read as
// zeros.  A decode reads each K/V line once, so the loads mark their L2 lines
// evict-first (measured: the 8K step 12.06 -> 11.47 us, the 32K step 26.4 -> 25.3 us).
__device__ __forceinline__ void load_stage(const DecMaps &mp, uint8_t *st, uint64_t *bar, int g,
                                           int off0, int page0, int off1, int page1) {
    const uint64_t pol = l2_evict_first_policy();
    mbar_arrive_expect_tx(bar, kDecStageBytes);
    tma_load_5d_hint(st, &mp.k, bar, 0, off0, 0, g, page0, pol);
    tma_load_5d_hint(st + kDecTileKBytes, &mp.k, bar, 0, off1, 0, g, page1, pol);
    tma_load_5d_hint(st + kDecHalf, &mp.v, bar, 0, off0, 0, g, page0, pol);
    tma_load_5d_hint(st + kDecHalf + kDecTileKBytes, &mp.v, bar, 0, off1, 0, g, page1, pol);
}

__device__ __forceinline__ int seq_tiles(int seq_len, int block_size, int tiles_per_page) {
    const int full = seq_len / block_size;
    const int rem = seq_len - full * block_size;
    return full * tiles_per_page + (rem + kDecTile - 1) / kDecTile;
}

__device__ __forceinline__ int checked_seq_len(const DecodeKParams &p, int seq, bool report) {
    int L = p.seq_lens[seq];
    if (L < 1 || L > p.max_seq_len) {
        if (report) atomicOr(p.err, kErrSeqLen);
        L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
    }
    return L;
}

// CTA barrier `id` for `threads` threads.  The non-aligned form: the threads may reach it
// from different places in the code (the producer and the consumers do).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

#ifdef PA_TEST_HOOKS
// Test build only: the ring stage whose loads the producer leaves out (-1: none), so
// that the consumer waiting for it runs into its bounded wait; and a delay (ns) before
// the consumer warps other than the one writing the newest token start on their tiles,
// so that every load of the split may land before the first wait.  Set by
// set_decode_test_hook through pa_test_hook.
__device__ int g_test_skip_stage = -1;
__device__ int g_test_consumer_delay_ns = 0;
#endif

// Tiles of its split (two ring stages) that a CTA prefetches into L2 before waiting for
// the previous kernel on the stream, when its split has at most four times as many.
// Measured in streams of steps that rotate over three 1 GiB pools (so that no step finds
// lines an earlier step prefetched), against no prefetch: 4K (8-tile splits) 8.34 ->
// 7.97 us; 8K (14 tiles) 11.06 -> 10.83; 32K (54 tiles) 25.22 -> 25.21.  In rotations
// over one pool the longer splits seemed to gain more (32K 25.45 -> 24.87), but only
// because some prefetched lines stayed in L2 until the same sequence came round again;
// an ncu capture of such a rotation saw a 32K launch read 4.5 of its 134 MB from L2.
// Four tiles gained more than two; eight or sixteen were slower (the prefetch outlasts
// the wait and delays the first loads); six were 1% faster in the 8K sweep but 2-4%
// slower in the 8K legs that rotate 32 copies of a 64-page pool, and in the kernel timed
// alone.
constexpr int kDecPrefetchTiles = 4;

template <int kDecConsumers, int kDecStages>
__global__ void __launch_bounds__((kDecConsumers + 1) * 32, 1)
    decode_split_kernel(const __grid_constant__ DecMaps maps, const DecodeKParams p) {
    (void)DecShape<kDecConsumers, kDecStages>::consumers;  // checks the warp mapping
    static_assert(kDecStages >= 2, "the reload of a one-stage split completes on full[1]");
    constexpr int kDecRingBytes = kDecStages * kDecStageBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kDecRingBytes);
    uint64_t *empty = full + kDecStages;
    uint64_t *written = empty + kDecStages;  // the fused write of the newest token is done
    // Raised by the first bounded wait that runs out; the others then give up at once.
    volatile int *abort = reinterpret_cast<volatile int *>(written + 1);

    const int split = blockIdx.x, g = blockIdx.y, seq = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Prologue: it reads nothing that earlier work on the stream may write but the
    // block-table entries that steer an L2 prefetch (below).
    if (threadIdx.x == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kDecPair);  // released by the warps of both tiles
        }
        mbar_init(written, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kDecConsumers && lane == 0) {
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
        // While the previous kernel on the stream finishes (in a stream of decode steps,
        // the previous step's combine, which leaves HBM idle), warm L2 with the first
        // tiles of this split.  The block-table entries read for this may still be
        // written by that kernel: they only steer the prefetch, which changes no result.
        // Every byte the kernel uses is loaded after the wait, L2 is coherent with the
        // previous kernel's writes, and these reads bypass L1 so that the reads after
        // the wait cannot hit a stale copy.
        const int32_t *bt = p.block_table + (int64_t)seq * p.bt_stride;
        const int tpp = p.tiles_per_page;
        const int t0 = split * p.tiles_per_split;
        const int t_end =
            p.tiles_per_split > 4 * kDecPrefetchTiles
                ? t0
                : min(t0 + kDecPrefetchTiles,
                      seq_tiles(p.max_seq_len, p.block_size, tpp));  // inside the table row
        int lp = t0 / tpp, tip = t0 - lp * tpp;
        int page = t0 < t_end ? __ldcg(bt + lp) : 0;
        // Evict-first, like the loads that use these lines: a prefetched line that
        // outlived its use would otherwise stay in L2 at normal priority.
        const uint64_t pol = l2_evict_first_policy();
        for (int t = t0; t < t_end; ++t) {
            if (page >= 0 && page < p.num_pages) {  // boxes inside the pool only
                tma_prefetch_l2_5d_hint(&maps.k, 0, tip * kDecTile, 0, g, page, pol);
                tma_prefetch_l2_5d_hint(&maps.v, 0, tip * kDecTile, 0, g, page, pol);
            }
            if (++tip == tpp && t + 1 < t_end) {
                tip = 0;
                page = __ldcg(bt + ++lp);
            }
        }
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    const int32_t *bt = p.block_table + (int64_t)seq * p.bt_stride;
    const int tpp = p.tiles_per_page;
    const int t0 = split * p.tiles_per_split;  // a multiple of kDecPair
    const int lp0 = t0 / tpp;
    const int tip0 = t0 - lp0 * tpp;
    const int off0 = tip0 * kDecTile;
    const bool producer = warp == kDecConsumers && lane == 0;
    // The producer loads the split's first stage before the sequence length is known, so
    // that the block-table read and the sequence-length read overlap instead of following
    // one another.  t0 lies below the tile count of the longest allowed sequence and a
    // block-table row holds that many pages, so the read stays inside the table.  Past the
    // sequence's end the entry may hold anything; a page outside the pool only makes the
    // boxes read as zeros, and such a tile is never consumed.  A first stage that would
    // straddle two pages waits for the length instead.
    const bool spec = tip0 + 1 < tpp;
    int page0 = 0;
    if (producer) page0 = bt[lp0];
    const int seq_len = checked_seq_len(p, seq, threadIdx.x == 0 && split == 0 && g == 0);
    if (producer && spec)
        load_stage(maps, smem, &full[0], g, off0, page0, off0 + kDecTile, page0);
    const int ntiles = seq_tiles(seq_len, p.block_size, tpp);
    const int t1 = min(ntiles, t0 + p.tiles_per_split);
    if (t0 >= t1) {
        // This split has no tiles of this sequence (CTA-uniform).  It marks its partials
        // empty (the combine then needs no sequence length), and the first stage's load
        // lands before the CTA exits.
        if (threadIdx.x < p.group)
            p.part_ml[((int64_t)seq * p.num_q_heads + g * p.group + threadIdx.x) * p.num_splits +
                      split] = make_float2(-CUDART_INF_F, 0.f);
        if (producer && spec) mbar_wait(&full[0], 0, p.err);
        return;
    }
    const int n = t1 - t0;                            // tiles of this split
    const int nst = (n + kDecPair - 1) / kDecPair;    // stages of this split
    // This CTA holds the tile of the token being decoded and has to write that token.
    const bool writes_newest = p.new_k != nullptr && t1 == ntiles;
    // ... and if that tile is in the stage loaded ahead, the stage is loaded twice.  The
    // second load completes on full[1] (a split of one stage never uses ring slot 1), so
    // its consumers wait for the first phase of a barrier of its own: an mbarrier wait
    // tells only two phases apart, and a consumer that reached a wait for the second
    // phase of full[0] late, after both loads had landed, could not tell.
    const bool refetch = writes_newest && spec && nst == 1;

    if (warp == kDecConsumers) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
#ifdef PA_TEST_HOOKS
            const int skip_stage = *reinterpret_cast<volatile int *>(&g_test_skip_stage);
#endif
            // Ring slots that received a load (bit s) and the phase parity of the last
            // load issued into each: every one of them lands before the CTA reuses or
            // leaves its shared memory (below), also when a wait gave up.
            uint32_t issued = spec ? 1u : 0u, par = 0;
            // A page outside the pool is reported; the TMA boxes then lie outside the
            // tensor and read as zeros, so nothing faults.
            if (page0 < 0 || page0 >= p.num_pages) atomicOr(p.err, kErrPage);
            // Block-table entries are read once per page and one page ahead, never
            // between two loads of the ring.
            const int lp_last = (t1 - 1) / tpp;
            int lp = lp0, page = page0;
            int page_next = lp0 < lp_last ? bt[lp0 + 1] : 0;
            if (refetch) {
                // The split's only stage holds the token being decoded and was loaded
                // before that token was written: load it again into the same slot once
                // the first load has landed and the write is done, completing on full[1].
                // Its consumers wait for that load only.
                if (mbar_wait_abort(&full[0], 0, p.err, abort) &&
                    mbar_wait_abort(written, 0, p.err, abort)) {
                    load_stage(maps, smem, &full[1], g, off0, page0, off0 + kDecTile,
                               page0);
                    issued |= 2u;  // full[1], phase parity 0
                }
            }
            for (int m = spec ? 1 : 0; m < nst; ++m) {
                const int s = m % kDecStages;
                // The stage's block-table entries are read before the wait for its ring
                // slot, so that their latency overlaps the wait (with small pages a
                // stage needs one or two fresh entries).
                const int j = t0 + m * kDecPair;
                const int l = j / tpp;
                const int tip = j - l * tpp;
                if (l != lp) {
                    // Usually the next page; with one tile per page a stage spans two
                    // pages and the next stage starts two pages further on.
                    page = l == lp + 1 ? page_next : bt[l];
                    lp = l;
                    if (page < 0 || page >= p.num_pages) atomicOr(p.err, kErrPage);
                    if (lp < lp_last) page_next = bt[lp + 1];
                }
                if (m >= kDecStages &&
                    !mbar_wait_abort(&empty[s], ((m / kDecStages) - 1) & 1, p.err, abort))
                    break;
                // The last stage holds the token being decoded: wait until it is written.
                if (writes_newest && m == nst - 1 && !mbar_wait_abort(written, 0, p.err, abort))
                    break;
#ifdef PA_TEST_HOOKS
                if (m == skip_stage) continue;  // its consumer's wait runs out
#endif
                issued |= 1u << s;
                par = (par & ~(1u << s)) | ((uint32_t)((m / kDecStages) & 1) << s);
                uint8_t *st = smem + s * kDecStageBytes;
                if (tip + 1 < tpp) {
                    load_stage(maps, st, &full[s], g, tip * kDecTile, page,
                               (tip + 1) * kDecTile, page);
                } else {
                    // The first tile closes its page: the second opens the next page, or
                    // lies past the split's end and reads as zeros from page -1.
                    const bool second = j + 1 < t1;
                    if (second && (page_next < 0 || page_next >= p.num_pages))
                        atomicOr(p.err, kErrPage);
                    load_stage(maps, st, &full[s], g, tip * kDecTile, page, 0,
                               second ? page_next : -1);
                }
            }
            // Loads always complete, so this wait ends; in a normal run every stage was
            // consumed and it returns at once.
            for (int s = 0; s < kDecStages; ++s)
                if ((issued >> s) & 1u) mbar_wait(&full[s], (par >> s) & 1u, p.err);
        }
        __syncwarp();
        named_bar_sync(1, (kDecConsumers + 1) * 32);  // meets the consumers before the merge
        return;
    }

    // ---------------------------------------------------------------- consumers
    if (writes_newest && warp == kDecConsumers - 1)
        write_newest_token(p, bt, seq, g, seq_len, lane, written);
#ifdef PA_TEST_HOOKS
    else {
        const unsigned long long delay =
            (unsigned)*reinterpret_cast<volatile int *>(&g_test_consumer_delay_ns);
        const unsigned long long t_start = global_ns();
        while (global_ns() - t_start < delay) __nanosleep(256);  // ends after `delay` ns
    }
#endif

    // Q^T as the B operand: lane holds head n = lane/4 and dims 2(lane%4)+{0,1} (+8)
    // of every 16-dim k-step.  Heads past the group are zero columns.
    const int nh = lane >> 2;
    const int qc = (lane & 3) * 2;
    uint32_t qb[16][2];
    {
        const bool hv = nh < p.group;
        const uint16_t *qrow =
            p.q + ((int64_t)seq * p.num_q_heads + g * p.group + (hv ? nh : 0)) * kHeadDim;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            qb[kk][0] = hv ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + qc) : 0u;
            qb[kk][1] = hv ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + qc + 8) : 0u;
        }
    }

    float o[16][4];
#pragma unroll
    for (int mt = 0; mt < 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F;  // heads qc, qc+1 (base-2 units)
    float l0 = 0.f, l1 = 0.f;                        // this lane's share of the sums
    const uint32_t sbase = smem_u32(smem);
    const int r_lo = lane >> 2;  // token rows r_lo and r_lo + 8 of the tile

    // Tile i of the split, held in half h of ring slot s.
    auto tile = [&](int s, int h, int i) {
        const int j = t0 + i;
        const int lp = j / tpp;
        const int off = (j - lp * tpp) * kDecTile;
        const int tok0 = lp * p.block_size + off;
        const int nvalid = min(kDecTile, min(p.block_size - off, seq_len - tok0));
        const uint32_t kb = sbase + s * kDecStageBytes + h * kDecTileKBytes;
        const uint32_t vb = kb + kDecHalf;

        if (nvalid < kDecTile) {
            // Rows past the sequence end may hold anything (even NaN): zero them in V
            // so that a zero weight cannot meet a NaN inside the MMA.
            uint8_t *vp = smem + s * kDecStageBytes + kDecHalf + h * kDecTileKBytes;
            const int per_chunk = (kDecTile - nvalid) * 8;
            for (int u = lane; u < per_chunk * kChunks; u += 32) {
                const int c = u / per_chunk;
                const int r = nvalid + (u - c * per_chunk) / 8;
                const int unit = u & 7;
                *reinterpret_cast<uint4 *>(vp + c * kDecTileBytes + r * 128 + unit * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }

        // S^T (16 tokens x 8 heads) = K (16 x 256) . Q^T (256 x 8), two chains.
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int uhi = lane >> 4;
#pragma unroll
            for (int kk = 0; kk < 16; kk += 2) {
                uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
                ldsm_x4(swz128(kb + (kk >> 2) * kDecTileBytes, row, (kk & 3) * 2 + uhi), a0,
                        a1, a2, a3);
                ldsm_x4(swz128(kb + ((kk + 1) >> 2) * kDecTileBytes, row,
                               ((kk + 1) & 3) * 2 + uhi),
                        c0, c1, c2, c3);
                mma_bf16_16816(sa, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
                mma_bf16_16816(sb, c0, c1, c2, c3, qb[kk + 1][0], qb[kk + 1][1]);
            }
        }

        // Online softmax over the tile's tokens, per head.
        const bool v0 = r_lo < nvalid, v1 = r_lo + 8 < nvalid;
        const float x00 = v0 ? (sa[0] + sb[0]) * p.scale_log2 : -CUDART_INF_F;
        const float x01 = v0 ? (sa[1] + sb[1]) * p.scale_log2 : -CUDART_INF_F;
        const float x10 = v1 ? (sa[2] + sb[2]) * p.scale_log2 : -CUDART_INF_F;
        const float x11 = v1 ? (sa[3] + sb[3]) * p.scale_log2 : -CUDART_INF_F;
        float mx0 = fmaxf(x00, x10), mx1 = fmaxf(x01, x11);
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
        const float mu1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
        const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
        const float p00 = exp2f(x00 - mu0), p01 = exp2f(x01 - mu1);
        const float p10 = exp2f(x10 - mu0), p11 = exp2f(x11 - mu1);
        l0 = l0 * al0 + (p00 + p10);
        l1 = l1 * al1 + (p01 + p11);
        // Rescale the accumulators only when some head's running max moved.
        if (__any_sync(0xffffffffu, mn0 != m0 || mn1 != m1)) {
#pragma unroll
            for (int mt = 0; mt < 16; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
        }
        m0 = mn0;
        m1 = mn1;

        // P^T as the B operand: the S^T fragment holds (token, head pair); the 8x8
        // transpose turns it into (head, token pair).  High and low BF16 parts.
        const uint32_t h0 = pack_bf16x2(p00, p01), h1 = pack_bf16x2(p10, p11);
        const uint32_t e0 = pack_bf16x2(p00 - bf16_lo(h0), p01 - bf16_hi(h0));
        const uint32_t e1 = pack_bf16x2(p10 - bf16_lo(h1), p11 - bf16_hi(h1));
        const uint32_t bh0 = movmatrix_t(h0), bh1 = movmatrix_t(h1);
        const uint32_t bl0 = movmatrix_t(e0), bl1 = movmatrix_t(e1);

        // O^T (256 dims x 8 heads) += V^T (256 x 16 tokens) . P^T (16 x 8)
        {
            const int jm = lane >> 3;
            const int row = (lane & 7) + (jm >> 1) * 8;
            const int ulo = jm & 1;
#pragma unroll
            for (int mt = 0; mt < 16; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(swz128(vb + (mt >> 2) * kDecTileBytes, row, (mt & 3) * 2 + ulo), a0,
                          a1, a2, a3);
                mma_bf16_16816(o[mt], a0, a1, a2, a3, bh0, bh1);
                mma_bf16_16816(o[mt], a0, a1, a2, a3, bl0, bl1);
            }
        }
    };

    // Short splits (the tail of the stream is a large share of their time): tile i is
    // consumed by warp i % C from half i % 2 of stage i / 2 (ring slot (i / 2) % S), so the
    // two tiles of a stage are processed in parallel.  Within a ring round of 2S tiles
    // every (warp, slot, half) is fixed, so each warp waits on its slots in turn and in
    // phase order.  Long splits: stage m is consumed whole by warp m % C, which measured
    // faster over long streams.  The choice is CTA-uniform; a slot is released by two
    // arrivals either way.
    if (n <= kDecShortTiles) {
        for (int i = warp; i < n; i += kDecConsumers) {
            const int m = i / kDecPair, h = i - m * kDecPair;
            const int s = m % kDecStages;
            // (refetch: the split's one stage, reloaded; its second load completes on full[1])
            uint64_t *fb = refetch ? &full[1] : &full[s];
            const uint32_t ph = refetch ? 0u : (uint32_t)(m / kDecStages) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait_abort(fb, ph, p.err, abort))) break;
            tile(s, h, i);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    } else {
        for (int m = warp; m < nst; m += kDecConsumers) {
            const int s = m % kDecStages;
            uint64_t *fb = refetch ? &full[1] : &full[s];  // (refetch: as above)
            const uint32_t ph = refetch ? 0u : (uint32_t)(m / kDecStages) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait_abort(fb, ph, p.err, abort))) break;
            for (int h = 0; h < kDecPair && m * kDecPair + h < n; ++h) tile(s, h, m * kDecPair + h);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s], kDecPair);
        }
    }

#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
        l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
    }

    // ---------------------------------------------------------------- CTA merge
    // Every tile consumed and (the producer joins here after its last load landed) no
    // load in flight: the ring is free.  If a wait gave up (PA_DEVERR_TIMEOUT is set),
    // the split contributes nothing: an empty partial, which the combine skips.
    named_bar_sync(1, (kDecConsumers + 1) * 32);
    if (*abort) {
        if (threadIdx.x < p.group)
            p.part_ml[((int64_t)seq * p.num_q_heads + g * p.group + threadIdx.x) * p.num_splits +
                      split] = make_float2(-CUDART_INF_F, 0.f);
        return;
    }
    float *red_o = reinterpret_cast<float *>(smem);                     // [warp][head][row]
    float *red_m = red_o + kDecConsumers * kDecMaxGroup * kDecMergeRow;  // [warp][head]
    float *red_l = red_m + kDecConsumers * kDecMaxGroup;
    if (lane < 4) {
        red_m[warp * kDecMaxGroup + qc] = m0;
        red_m[warp * kDecMaxGroup + qc + 1] = m1;
        red_l[warp * kDecMaxGroup + qc] = l0;
        red_l[warp * kDecMaxGroup + qc + 1] = l1;
    }
    {
        float *w0 = red_o + (warp * kDecMaxGroup + qc) * kDecMergeRow;
        float *w1 = w0 + kDecMergeRow;
#pragma unroll
        for (int mt = 0; mt < 16; ++mt) {
            const int d = mt * 16 + r_lo;
            w0[d] = o[mt][0];
            w1[d] = o[mt][1];
            w0[d + 8] = o[mt][2];
            w1[d + 8] = o[mt][3];
        }
    }
    named_bar_sync(2, kDecConsumers * 32);
    // Thread t merges the quads (4 consecutive dims of one head) t, t + 32C, ...  Every
    // thread derives its head's CTA max and the warps' weights exp2(m_w - M) itself, so
    // no further barrier is needed and all loads of a quad are independent.
    constexpr int kQuadsPerHead = kHeadDim / 4;
    constexpr int kMergeThreads = kDecConsumers * 32;
    const int nquads = p.group * kQuadsPerHead;
#pragma unroll
    for (int k = 0; k < (kDecMaxGroup * kQuadsPerHead + kMergeThreads - 1) / kMergeThreads;
         ++k) {
        const int q = threadIdx.x + k * kMergeThreads;
        if (q < nquads) {
            const int c = q / kQuadsPerHead, d = (q - c * kQuadsPerHead) * 4;
            float mw[kDecConsumers];
            float M = -CUDART_INF_F;
#pragma unroll
            for (int w = 0; w < kDecConsumers; ++w) {
                mw[w] = red_m[w * kDecMaxGroup + c];
                M = fmaxf(M, mw[w]);
            }
            float L = 0.f;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kDecConsumers; ++w) {
                const float e = M == -CUDART_INF_F ? 0.f : exp2f(mw[w] - M);
                const float4 v = *reinterpret_cast<const float4 *>(
                    red_o + (w * kDecMaxGroup + c) * kDecMergeRow + d);
                L += e * red_l[w * kDecMaxGroup + c];
                O.x += e * v.x;
                O.y += e * v.y;
                O.z += e * v.z;
                O.w += e * v.w;
            }
            const int64_t pi =
                ((int64_t)seq * p.num_q_heads + g * p.group + c) * p.num_splits + split;
            *reinterpret_cast<float4 *>(p.part_o + pi * kHeadDim + d) = O;
            if (d == 0) p.part_ml[pi] = make_float2(M, L);
        }
    }
}

// kCombineParts CTAs per (query head, sequence), each merging 64 of the head's dims, so
// that a CTA reads a quarter of the head's partials (the read of all 37 KB of an 8K
// head through one SM took ~1 us longer).  Warp w merges splits w, w+8, w+16, ...
// against its own running max, each lane owning 2 consecutive dims (one 8-byte load per
// split).  The loads of a batch of up to 8 splits per warp are issued before any of
// their weights is known, so the kernel waits for global memory about once.  The eight
// warp results are then merged through shared memory with one more log-sum-exp step.
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const DecodeKParams p) {
    constexpr int kWarps = kCombineThreads / 32;
    constexpr int kBatch = 8;  // splits per warp whose loads are in flight together
    static_assert(kCombineDims == 64, "a warp covers a CTA's dims with 2 per lane");
    __shared__ __align__(16) float part[kWarps][kCombineDims];
    __shared__ float wm[kWarps], wl[kWarps];
    const int h = blockIdx.x / kCombineParts, d0 = (blockIdx.x % kCombineParts) * kCombineDims;
    const int seq = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    pdl_wait();
    pdl_trigger();
    // Every split wrote its (max, sum); an empty one (max -inf) gets weight 0 and its
    // partial sums, never written, are skipped.
    const int nsplit = p.num_splits;
    const int64_t base = ((int64_t)seq * p.num_q_heads + h) * p.num_splits;
    const float2 *po = reinterpret_cast<const float2 *>(p.part_o + base * kHeadDim + d0) + lane;
    float M = -CUDART_INF_F, L = 0.f;
    float acc0 = 0.f, acc1 = 0.f;
    // Split j of this warp's k-th batch element: warp + kWarps * (b0 + k).
    for (int b0 = 0; warp + kWarps * b0 < nsplit; b0 += kBatch) {
        float2 va[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int j = warp + kWarps * (b0 + k);
            va[k] = j < nsplit ? ld_f2_ordered(po + (int64_t)j * (kHeadDim / 2))
                               : make_float2(0.f, 0.f);
        }
        // Lane k < kBatch holds the (max, sum) of the batch's k-th split (loaded after
        // the sums, so that all of the batch's loads are in flight together).
        const int jl = warp + kWarps * (b0 + lane);
        const float2 ml = lane < kBatch && jl < nsplit ? ld_f2_ordered(p.part_ml + base + jl)
                                                       : make_float2(-CUDART_INF_F, 0.f);
        float bm = ml.x;
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, sh));
        const float mn = fmaxf(M, bm);
        const float f = M == -CUDART_INF_F ? 0.f : exp2f(M - mn);  // rescale of the old sums
        const float e = ml.x == -CUDART_INF_F ? 0.f : exp2f(ml.x - mn);
        float el = e * ml.y;
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) el += __shfl_xor_sync(0xffffffffu, el, sh);
        L = L * f + el;
        M = mn;
        acc0 *= f;
        acc1 *= f;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const float w = __shfl_sync(0xffffffffu, e, k);
            if (w == 0.f) continue;  // warp-uniform: an empty split's sums are not read
            acc0 += w * va[k].x;
            acc1 += w * va[k].y;
        }
    }
    reinterpret_cast<float2 *>(&part[warp][0])[lane] = make_float2(acc0, acc1);
    if (lane == 0) {
        wm[warp] = M;
        wl[warp] = L;
    }
    __syncthreads();
    if (tid < kCombineDims) {
        float Mt = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) Mt = fmaxf(Mt, wm[w]);
        float O = 0.f, Lt = 0.f;
        if (Mt != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float e = wm[w] == -CUDART_INF_F ? 0.f : exp2f(wm[w] - Mt);
                O += e * part[w][tid];
                Lt += e * wl[w];
            }
        }
        const float r = Lt > 0.f ? O / Lt : 0.f;
        const __nv_bfloat16 b = __float2bfloat16_rn(r);
        p.out[((int64_t)seq * p.num_q_heads + h) * kHeadDim + d0 + tid] =
            *reinterpret_cast<const uint16_t *>(&b);
    }
}

}  // namespace

#ifdef PA_TEST_HOOKS
cudaError_t set_decode_test_hook(int skip_stage, int consumer_delay_ns) {
    cudaError_t e = cudaMemcpyToSymbol(g_test_skip_stage, &skip_stage, sizeof skip_stage);
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_test_consumer_delay_ns, &consumer_delay_ns,
                              sizeof consumer_delay_ns);
}
#endif

DecodePlan plan_decode(int num_seqs, int num_kv_heads, int block_size, int max_seq_len,
                       int num_sms) {
    DecodePlan pl;
    pl.tiles_per_page = (block_size + kDecTile - 1) / kDecTile;
    const int full = max_seq_len / block_size;
    const int rem = max_seq_len - full * block_size;
    pl.max_tiles = full * pl.tiles_per_page + (rem + kDecTile - 1) / kDecTile;
    const long long pairs = (long long)num_seqs * num_kv_heads;
    // One CTA per SM across all (sequence, KV head) pairs, whole stages per CTA and at
    // least 8 tiles (4 stages) each.
    long long want = (num_sms + pairs - 1) / pairs;
    if (want < 1) want = 1;
    int tps = (int)((pl.max_tiles + want - 1) / want);
    if (tps < 8) tps = 8;
    if ((pl.max_tiles + tps - 1) / tps > kDecMaxSplits)
        tps = (pl.max_tiles + kDecMaxSplits - 1) / kDecMaxSplits;
    tps = (tps + kDecPair - 1) / kDecPair * kDecPair;
    pl.tiles_per_split = tps;
    pl.num_splits = (pl.max_tiles + tps - 1) / tps;
    return pl;
}

// Workspace layout, the one place that defines it: fp32 partial sums [S, Hq, splits, D],
// then (max, sum) pairs [S, Hq, splits], each region 256-byte aligned.
namespace {
struct DecodeWsLayout {
    size_t o_bytes, ml_bytes;
};
DecodeWsLayout decode_ws_layout(int num_seqs, int num_q_heads, const DecodePlan &plan) {
    const size_t parts = (size_t)num_seqs * num_q_heads * plan.num_splits;
    return {(parts * kHeadDim * sizeof(float) + 255) & ~size_t(255),
            (parts * sizeof(float2) + 255) & ~size_t(255)};
}
}  // namespace

size_t decode_workspace_bytes(int num_seqs, int num_q_heads, const DecodePlan &plan) {
    const DecodeWsLayout l = decode_ws_layout(num_seqs, num_q_heads, plan);
    return l.o_bytes + l.ml_bytes;
}

cudaError_t launch_decode(const CUtensorMap *tmaps, const DecodeArgs &a, const DecodePlan &plan,
                          cudaStream_t stream) {
    // The kernel shape for this plan's split length (see DecShape).
    const bool short_splits = plan.tiles_per_split <= kDecShortTiles;
    void (*split_kernel)(DecMaps, DecodeKParams) =
        short_splits ? decode_split_kernel<kDecShortConsumers, kDecShortStages>
                     : decode_split_kernel<kDecLongConsumers, kDecLongStages>;
    const int smem = short_splits ? dec_smem_bytes<kDecShortConsumers, kDecShortStages>()
                                  : dec_smem_bytes<kDecLongConsumers, kDecLongStages>();
    const int threads = ((short_splits ? kDecShortConsumers : kDecLongConsumers) + 1) * 32;
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(split_kernel), smem,
                                  short_splits ? 0 : 3);
    if (e != cudaSuccess) return e;
    DecodeKParams p;
    p.q = a.q;
    p.block_table = a.block_table;
    p.bt_stride = a.bt_stride;
    p.seq_lens = a.seq_lens;
    p.max_seq_len = a.max_seq_len;
    p.num_q_heads = a.num_q_heads;
    p.group = a.group;
    p.block_size = a.block_size;
    p.tiles_per_page = plan.tiles_per_page;
    p.tiles_per_split = plan.tiles_per_split;
    p.num_splits = plan.num_splits;
    p.num_pages = a.num_pages;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    const DecodeWsLayout ws = decode_ws_layout(a.num_seqs, a.num_q_heads, plan);
    p.part_o = static_cast<float *>(a.workspace);
    p.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(a.workspace) + ws.o_bytes);
    p.out = a.out;
    p.err = a.err;
    p.k_cache_w = a.k_cache_w;
    p.v_cache_w = a.v_cache_w;
    p.new_k = a.new_k;
    p.new_v = a.new_v;
    p.new_slots = a.new_slots;
    p.slot_out = a.slot_out;
    p.page_stride = a.page_stride;
    p.num_kv_heads = a.num_kv_heads;
    const dim3 grid(plan.num_splits, a.num_kv_heads, a.num_seqs);
    if (a.ev_start && (e = record_event(a.ev_start, stream)) != cudaSuccess) return e;
    DecMaps maps;
    maps.k = tmaps[0];
    maps.v = tmaps[1];
    e = launch_pdl(split_kernel, grid, dim3(threads), smem, stream, maps, p);
    if (e != cudaSuccess) return e;
    if (a.ev_stop && (e = record_event(a.ev_stop, stream)) != cudaSuccess) return e;
    return launch_pdl(decode_combine_kernel, dim3(a.num_q_heads * kCombineParts, a.num_seqs),
                      dim3(kCombineThreads), 0, stream, p);
}

}  // namespace pa
