// pa_prefill.cu -- chunked-prefill attention of one sequence over its paged cache, on
// the tcgen05 tensor cores with TMEM accumulators.
//
// What is computed (page832 post §6): query row i of the chunk sits at absolute
// position q_start + i and, with causal masking, attends to keys 0..q_start+i of the
// same sequence (earlier chunks and the chunk itself, already written to the cache);
// without it, to all q_start + q_len keys.  K/V are read through the block table
// (page832 §1) in page-local blocks of 64 keys; four blocks form a 256-key tile.
//
// Shape choices.  A tcgen05.mma with M=128 and K=16 occupies the tensor core for about
// the same time for any N up to 256, so every MMA here has N = 256: S = Q K^T runs over
// 256 keys at a time, and O += P V covers all 256 output dims in one MMA per 16 keys.
// With O (256 columns) and S (256 columns) TMEM is full, so S is single-buffered.  To
// keep the tensor core busy while the softmax runs, P is handed over in 64-key quarters:
// the PV of quarter q runs while the softmax of quarter q+1 is computed, and the tensor
// core only waits for the softmax of each tile's first quarter.
//
// Work item = (128 query rows of one head).  A chunk's last query tile of r rows runs
// instead as packed items of hp heads, hp the largest divisor of the GQA group G with
// hp * r <= 128: TMEM lane x holds tile row x / hp of query head h0 + x % hp (Q comes in
// as boxes of hp heads x 128/hp rows), so the heads of a group share passes over their
// K/V rather than each taking a 128-row item with r rows present.  Persistent CTAs, one per SM, run the items
// the host planner assigned to them (a static schedule that balances the causal items'
// unequal lengths across CTAs, passed in the kernel parameters), longest first.
// Problems too large for the schedule arrays walk the items longest first in a snake
// order instead (item k of CTA b: k*G + b for even k, k*G + G-1-b for odd k).
//
// Warp roles (576 threads):
//   warp 0    TMA producer: the item's Q tile (4 boxes of 64 dims x 128 rows, 64 KB),
//             then per tile four K units (one 64-dim chunk x 256 keys, 32 KB each) and
//             four V units (64 keys x 256 dims) into a 5-slot ring of 32 KB.  Boxes are
//             64 keys of one page; keys of the sequence's last page come through tensor
//             maps cut at the last token, so rows past it (and past a page end) are zeros.
//   warp 1    MMA issuer (one thread) and TMEM owner: S = Q K^T (A, B K-major in shared
//             memory), then O += P V per 64-key quarter (A = P from TMEM, B = V unit
//             MN-major, 8 KB between 64-dim atoms).
//   warps 2-9 softmax: warps w and w+4 share query rows 32*(w%4) .. +31 (TMEM lanes),
//             one thread per row, and split each 64-key quarter into two 32-key halves
//             (and O into two 128-column halves).  Per quarter each warp reads its 32 S
//             values, masks (page end, sequence end, causal) where needed, and the pair
//             agrees on the quarter's row max through shared memory.  The running max
//             moves only when it grows by more than 8 (log2 units; then both warps
//             rescale their half of the O row in TMEM).  Each warp writes P = P_hi + P_lo
//             (two BF16 parts, so that P keeps ~16 significant bits) for its keys over
//             that quarter of S.  At the end the pair adds its two partial row sums,
//             hands them to the epilogue warps through shared memory and starts on its
//             next item.
//   warps 10-17 epilogue: two per TMEM lane quarter (128 O columns each); when an
//             item's last PV is done, they load O into registers (BF16, normalised),
//             release O to the next item's PVs, then store the rows to out (a piece of a
//             split item: fp32 partials to the workspace).
// TMEM columns: O [0, 256), S [256, 512); P of quarter q: hi at 256+64q, lo at +32.
//
// Every wait is bounded; a wait that runs out sets PA_DEVERR_TIMEOUT, flags the CTA to
// stop, and the CTA drains its tensor-core work and frees TMEM before it returns.
#include <float.h>
#include <math_constants.h>
#include <string.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kBM = kPfQRows;                 // 128 query rows
constexpr int kBN = kPfKvTile;                // 256 keys per tile
constexpr int kBlk = 64;                      // keys per TMA box (page-local block)
constexpr int kBlkBytes = kBlk * 128;         // one box: 64 rows x 128 B = 8 KB
constexpr int kUnit = 4 * kBlkBytes;          // 32 KB ring slot
constexpr int kQChunk = kBM * 128;            // 64 dims x 128 rows: 16 KB
constexpr int kQBytes = kChunks * kQChunk;    // 64 KB
constexpr int kRing = kPfRing;
constexpr int kSoftmaxWarps = 8;              // two per TMEM lane quarter
constexpr int kEpilogueWarps = 8;             // two per TMEM lane quarter
constexpr int kThreads = (2 + kSoftmaxWarps + kEpilogueWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256;
static_assert(kBN == 4 * kBlk && kBN == 256, "tile = four 64-key blocks");

// Shared memory.  Its dynamic part starts 1024-byte aligned on this GPU (right after the
// 1 KB the hardware reserves per block), which the 128-byte swizzle of the TMA tiles
// needs; the kernel checks this and reports PA_DEVERR_LAYOUT rather than run otherwise.
constexpr int kOffQ = 0;
constexpr int kOffRing = kQBytes;
constexpr int kOffXchg = kOffRing + kRing * kUnit;  // row maxima / sums of warp pairs
constexpr int kXchgBytes = 4 * 2 * 2 * 32 * 4;      // [lane quarter][phase][half][lane]
constexpr int kOffRowSum = kOffXchg + kXchgBytes;   // an item's row sums, to the epilogue
constexpr int kOffBars = kOffRowSum + kBM * 4;
enum Bar {
    kRingFull = 0,
    kRingEmpty = kRingFull + kRing,
    kQFull = kRingEmpty + kRing,
    kQEmpty,
    kSFull,
    kPFull,               // [4] quarters
    kPvDone = kPFull + 4, // [4] quarters
    kOEmpty = kPvDone + 4,
    kEpiReady,            // the softmax warps handed an item's row sums to the epilogue
    kDrain,
    kPair,                // [4] the two softmax warps of a lane quarter meet here
    kNumBars = kPair + 4
};
constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// One sequence of the launch: its chunk is rows q_off .. q_off + q_len - 1 of q / out, at
// absolute positions q_start .. q_start + q_len - 1 of a sequence of seq_len_k keys.
struct SeqInfo {
    int q_off, q_len, q_start, seq_len_k;
    int last_page;    // logical index of the sequence's last page
    int item_off;     // its first work item (items numbered as prefill_item_at gives them)
    int bt_row;       // its row of the block table
};

// The schedule as the kernel reads it: the CTA -> entries lists, and the pieces only in
// the extended build (the kernel parameters of plain plans stay small).
struct DevSchedule {
    int num_ctas;                        // 0: none (the kernel walks a snake order)
    uint16_t off[kPfSchedMaxCtas + 1];
    uint16_t items[kPfSchedMaxItems];
};
template <bool kExt>
struct DevPieces {
    PrefillPiece pieces[kPfMaxPieces];
};
template <>
struct DevPieces<false> {};

template <int kSeqs, bool kExt>
struct TcParams {
    const int32_t *block_table;  // row b of sequence b, bt_stride entries apart
    int64_t bt_stride;
    int causal, num_seqs, num_items;
    int num_q_heads, group;
    // packed items: heads per item of each packed Q map, and the bytes of its Q tile
    // (hp heads x 128/hp rows, four 64-dim chunks); 0 past the group's divisors
    int qp_hp[kPfMaxPackMaps], qp_bytes[kPfMaxPackMaps];
    int block_size, blocks_per_page;
    int64_t num_pages;
    float sc;             // |scale| * log2(e), at least FLT_MIN
    int neg;              // scale < 0
    uint16_t *out;
    unsigned *err;
    float *ws_o;    // piece partials: O [slot][128 rows][256] (only with split items)
    float2 *ws_ml;  // piece partials: (running max, sum of weights) [slot][128 rows]
    SeqInfo seq[kSeqs];
    DevSchedule sched;       // static item -> CTA assignment
    DevPieces<kExt> pc;   // pieces of split items (extended build only)
};

template <int kSeqs>
struct TcMaps {
    CUtensorMap q;
    CUtensorMap qp[kPfMaxPackMaps];  // Q in boxes of hp heads x 128/hp rows (packed items)
    CUtensorMap k, v;
    CUtensorMap k_last[kSeqs], v_last[kSeqs];  // cut at each sequence's last token
};

static_assert(sizeof(TcMaps<kPfMaxSeqs>) + sizeof(TcParams<kPfMaxSeqs, true>) <= 32764,
              "the kernel's parameters fit the 32 KB parameter space");

struct Item {
    // head (the first of its heads for a packed item), KV head, first row of the query
    // tile, its rows present (per head), key blocks, tiles
    int h, g, r0, rows, nblocks, n;
    int hp;   // heads of the item: 1, or a packed item's (lane x: row x / hp, head h + x % hp)
    int qpi;  // a packed item's Q map
    int b, q_off, q_start, seq_len_k, last_page, bt_row;  // its sequence
    // The tiles [jb, je) this CTA runs: all n of a whole item, or one piece's range; a
    // piece writes its partial to workspace slot `slot` (-1: a whole item, normalised
    // output stored to out).
    int jb, je, slot;
};

// kExt: the launch may hold pieces of split items and packed last tiles.  Launches with
// neither use the kernel built without them, so plain plans run the plain code (piece
// support measured 1.6% slower on the q=4096 chunk when always compiled in, packed
// tiles another 1.5%).
template <int kSeqs, bool kExt>
__device__ __forceinline__ bool item_of(const TcParams<kSeqs, kExt> &p, int k, Item &it) {
    const int G = gridDim.x, b = blockIdx.x;
    int idx, piece = -1;
    if (p.sched.num_ctas) {
        const int x = p.sched.off[b] + k;
        if (x >= p.sched.off[b + 1]) return false;
        idx = p.sched.items[x];
        if constexpr (kExt) {
            if (idx & kPfPieceBit) {
                piece = idx & ~kPfPieceBit;
                idx = p.pc.pieces[piece].item;
            }
        }
    } else {
        idx = (k & 1) ? k * G + (G - 1 - b) : k * G + b;
        if (idx >= p.num_items) return false;
    }
    int sb = 0;
    while (sb + 1 < p.num_seqs && idx >= p.seq[sb + 1].item_off) ++sb;
    const SeqInfo &sq = p.seq[sb];
    const int local = idx - sq.item_off;
    int qt;
    it.qpi = 0;
    if constexpr (kExt) {
        prefill_item_at(local, sq.q_len, p.num_q_heads, p.group, &qt, &it.h, &it.hp);
        while (it.qpi + 1 < kPfMaxPackMaps && p.qp_hp[it.qpi] != it.hp) ++it.qpi;
    } else {  // no packed tile: item i is tile nqt - 1 - i / Hq of head i % Hq
        qt = (sq.q_len + kBM - 1) / kBM - 1 - local / p.num_q_heads;
        it.h = local % p.num_q_heads;
        it.hp = 1;
    }
    it.g = it.h / p.group;
    it.r0 = qt * kBM;
    it.rows = min(kBM, sq.q_len - it.r0);
    it.b = sb;
    it.q_off = sq.q_off;
    it.q_start = sq.q_start;
    it.seq_len_k = sq.seq_len_k;
    it.last_page = sq.last_page;
    it.bt_row = sq.bt_row;
    const int nkeys = p.causal ? sq.q_start + it.r0 + it.rows : sq.seq_len_k;
    const int full = nkeys / p.block_size;
    const int rem = nkeys - full * p.block_size;
    it.nblocks = full * p.blocks_per_page + (rem + kBlk - 1) / kBlk;
    it.n = (it.nblocks + 3) / 4;
    it.jb = 0;
    it.je = it.n;
    it.slot = -1;
    if constexpr (kExt) {
        if (piece >= 0) {
            it.jb = p.pc.pieces[piece].tile_begin;
            it.je = p.pc.pieces[piece].tile_end;
            it.slot = p.pc.pieces[piece].slot;
        }
    }
    return true;
}

#ifdef PA_TEST_HOOKS
// Test build only: the K/V ring unit (counted over the CTA's whole run) whose loads the
// producer leaves out (-1: none), so that the MMA thread's wait for it runs out.  Set by
// set_prefill_test_hook through pa_test_hook.
__device__ int g_test_skip_unit = -1;
#endif

template <int kSeqs, bool kExt>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ TcMaps<kSeqs> maps,
                      const __grid_constant__ TcParams<kSeqs, kExt> p) {
    extern __shared__ __align__(16) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {  // CTA-uniform; nothing has been set up yet
        if (threadIdx.x == 0) atomicOr(p.err, kErrLayout);
        return;
    }
    uint8_t *qs = smem + kOffQ;
    uint8_t *ring = smem + kOffRing;
    float *xchg = reinterpret_cast<float *>(smem + kOffXchg);
    float *rowsum = reinterpret_cast<float *>(smem + kOffRowSum);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---------------------------------------------------------------- prologue
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bars[kRingFull + i], 1);
            mbar_init(&bars[kRingEmpty + i], 1);
        }
        mbar_init(&bars[kQFull], 1);
        mbar_init(&bars[kQEmpty], 1);
        mbar_init(&bars[kSFull], 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&bars[kPFull + i], kSoftmaxWarps);  // one elected lane per warp
            mbar_init(&bars[kPvDone + i], 1);
            mbar_init(&bars[kPair + i], 2);
        }
        mbar_init(&bars[kOEmpty], kEpilogueWarps);
        mbar_init(&bars[kEpiReady], kSoftmaxWarps / 2);  // one warp of each pair
        mbar_init(&bars[kDrain], 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
#ifdef PA_TEST_HOOKS
            const int skip_unit = *reinterpret_cast<volatile int *>(&g_test_skip_unit);
#endif
            uint32_t u = 0;
            // Ring slots that received a load (bit s), the phase parity of the last load
            // issued into each, and the Q loads issued: all of them land before the CTA
            // leaves, also when a wait gave up.
            uint32_t issued = 0, par = 0;
            int q_loads = 0;
            Item it;
            bool stop = false;
            for (int k = 0; !stop && (item_of<kSeqs, kExt>(p, k, it)); ++k) {
                if (k > 0 && !mbar_wait_abort(&bars[kQEmpty], (k - 1) & 1, p.err, abort)) break;
                ++q_loads;
                const bool pk = kExt && it.hp > 1;
                mbar_arrive_expect_tx(&bars[kQFull], pk ? p.qp_bytes[it.qpi] : kQBytes);
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
                    tma_load_3d(qs + c * kQChunk, pk ? &maps.qp[it.qpi] : &maps.q,
                                &bars[kQFull], c * kChunkElems, it.h, it.q_off + it.r0);
                const int32_t *bt = p.block_table + (int64_t)it.bt_row * p.bt_stride;
                // Page and in-page index of block kb, advanced block by block: a division
                // per block would take the MUFU, which the softmax warps keep busy (one
                // per item places the first block of a piece).
                int blk_lp = kExt && it.jb ? (4 * it.jb) / p.blocks_per_page : 0;
                int blk_in = 4 * it.jb - blk_lp * p.blocks_per_page;
                for (int j = it.jb; j < it.je && !stop; ++j) {
                    // Page, offset and map of each of the tile's four blocks; blocks past the
                    // item's last are read from outside the pool (zeros) and masked.
                    int pg[4], of[4];
                    const CUtensorMap *mk[4], *mv[4];
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) {
                        const int kb = 4 * j + bb;
                        const int lp = blk_lp;
                        of[bb] = blk_in * kBlk;
                        if (++blk_in == p.blocks_per_page) {
                            blk_in = 0;
                            ++blk_lp;
                        }
                        if (kb < it.nblocks) {
                            pg[bb] = bt[lp];
                            if (pg[bb] < 0 || pg[bb] >= p.num_pages) atomicOr(p.err, kErrPage);
                            mk[bb] = lp == it.last_page ? &maps.k_last[it.b] : &maps.k;
                            mv[bb] = lp == it.last_page ? &maps.v_last[it.b] : &maps.v;
                        } else {
                            pg[bb] = (int)p.num_pages;
                            of[bb] = 0;
                            mk[bb] = &maps.k;
                            mv[bb] = &maps.v;
                        }
                    }
                    // 4 K units (dim chunk c: the four blocks stacked), then 4 V units
                    // (block bb: the four dim chunks side by side).
                    for (int x = 0; x < 8; ++x, ++u) {
                        const int s = u % kRing;
                        if (u >= kRing &&
                            !mbar_wait_abort(&bars[kRingEmpty + s], ((u / kRing) - 1) & 1, p.err,
                                           abort)) {
                            stop = true;
                            break;
                        }
#ifdef PA_TEST_HOOKS
                        if ((int)u == skip_unit) continue;  // the MMA thread's wait runs out
#endif
                        issued |= 1u << s;
                        par = (par & ~(1u << s)) | (((u / kRing) & 1u) << s);
                        uint8_t *dst = ring + s * kUnit;
                        mbar_arrive_expect_tx(&bars[kRingFull + s], kUnit);
                        if (x < 4) {
#pragma unroll
                            for (int bb = 0; bb < 4; ++bb)
                                tma_load_4d(dst + bb * kBlkBytes, mk[bb], &bars[kRingFull + s],
                                            x * kChunkElems, it.g, of[bb], pg[bb]);
                        } else {
                            const int bb = x - 4;
#pragma unroll
                            for (int c = 0; c < kChunks; ++c)
                                tma_load_4d(dst + c * kBlkBytes, mv[bb], &bars[kRingFull + s],
                                            c * kChunkElems, it.g, of[bb], pg[bb]);
                        }
                    }
                }
            }
            // Loads always complete, so these waits end; in a normal run every unit and Q
            // tile was consumed and they return at once.
            for (int s = 0; s < kRing; ++s)
                if ((issued >> s) & 1u) mbar_wait(&bars[kRingFull + s], (par >> s) & 1u, p.err);
            if (q_loads > 0) mbar_wait(&bars[kQFull], (q_loads - 1) & 1, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdQK = umma_idesc_bf16(kBM, kBN, 0, 0);
            constexpr uint32_t kIdPV = umma_idesc_bf16(kBM, kHeadDim, 0, 1);
            const uint32_t q_addr = smem_u32(qs), ring_addr = smem_u32(ring);
            const uint32_t sbuf = tmem + kColS, obuf = tmem + kColO;
            uint32_t u = 0, jt = 0;
            Item it;
            bool stop = false;
            for (int k = 0; !stop && (item_of<kSeqs, kExt>(p, k, it)); ++k) {
                if (!mbar_wait_abort(&bars[kQFull], k & 1, p.err, abort)) break;
                tc_fence_after();
                for (int j = it.jb; j < it.je && !stop; ++j) {
                    const uint32_t jr = (uint32_t)(j - it.jb);  // tile of this item or piece
                    // S = Q K^T over the tile's 256 keys.
                    for (int c = 0; c < kChunks; ++c, ++u) {
                        const int s = u % kRing;
                        if (!mbar_wait_abort(&bars[kRingFull + s], (u / kRing) & 1, p.err, abort)) {
                            stop = true;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
                            umma_ss(sbuf, umma_sdesc_sw128(q_addr + c * kQChunk + k4 * 32),
                                    umma_sdesc_sw128(ring_addr + s * kUnit + k4 * 32), kIdQK,
                                    (c | k4) != 0);
                        umma_commit(&bars[kRingEmpty + s]);
                    }
                    if (stop) break;
                    if (j == it.je - 1) umma_commit(&bars[kQEmpty]);
                    umma_commit(&bars[kSFull]);
                    // O += P V, one 64-key quarter (one V unit) at a time.  The V unit and
                    // the O buffer are usually ready long before P: their waits (each
                    // costs this thread a few hundred cycles even when already complete)
                    // and the descriptors come first, so that only the P hand-off sits
                    // between one quarter's MMAs and the next.
                    for (int qq = 0; qq < 4; ++qq, ++u) {
                        const int s = u % kRing;
                        if (!mbar_wait_abort(&bars[kRingFull + s], (u / kRing) & 1, p.err, abort)) {
                            stop = true;
                            break;
                        }
                        if (jr == 0 && qq == 0 && k > 0 &&
                            !mbar_wait_abort(&bars[kOEmpty], (k - 1) & 1, p.err, abort)) {
                            stop = true;
                            break;
                        }
                        uint64_t vd[kBlk / 16];
#pragma unroll
                        for (int ks = 0; ks < kBlk / 16; ++ks)
                            vd[ks] = umma_sdesc_sw128(ring_addr + s * kUnit + ks * 2048, kBlkBytes);
                        if (!mbar_wait_abort(&bars[kPFull + qq], (jt + jr) & 1, p.err, abort)) {
                            stop = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t phi = sbuf + 64 * qq;
#pragma unroll
                        for (int ks = 0; ks < kBlk / 16; ++ks) {
                            umma_ts(obuf, phi + 8 * ks, vd[ks], kIdPV, (jr | qq | ks) != 0);
                            umma_ts(obuf, phi + 32 + 8 * ks, vd[ks], kIdPV, 1);
                        }
                        umma_commit(&bars[kRingEmpty + s]);
                        umma_commit(&bars[kPvDone + qq]);
                    }
                }
                jt += it.je - it.jb;
            }
            // Drain: every tensor-core operation issued by this thread is complete before
            // the CTA frees TMEM.
            umma_commit(&bars[kDrain]);
            mbar_wait(&bars[kDrain], 0, p.err);
        }
    } else if (warp < 2 + kSoftmaxWarps) {
        // ------------------------------------------------------------ softmax
        // Two warps per TMEM lane quarter: warp sw (0..7) owns rows 32*(warp % 4) + lane
        // and half hf = sw / 4 of every 64-key quarter (keys 32*hf .. 32*hf + 31) and of
        // the O columns (128*hf .. 128*hf + 127).  The pair agrees on each quarter's row
        // max through shared memory and its kPair barrier.
        const int lq = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int row = lq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(lq * 32) << 16;
        const uint32_t obase = tmem + lane_off + kColO + 128 * hf;
        const uint32_t sbase = tmem + lane_off + kColS;
        float *xq = xchg + lq * 128;  // [phase][half][lane]
        // Loop-invariant parameters, read once into registers.
        const int block_size = p.block_size, blocks_per_page = p.blocks_per_page;
        const bool causal = p.causal != 0, neg = p.neg != 0;
        const float sc = p.sc;
        uint64_t *pair = &bars[kPair + lq];
        uint32_t pc = 0;  // exchanges done by this pair (both warps count alike)
        // Publishes v, meets the partner warp, returns the partner's value.  The meeting
        // also orders each warp's (completed) TMEM loads of its S half before the
        // partner's P stores, which land partly in those columns.
        auto exchange = [&](float v, bool &ok) -> float {
            const uint32_t ph = pc & 1;
            xq[ph * 64 + hf * 32 + lane] = v;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pair);
            ok = mbar_wait_abort(pair, ph, p.err, abort);
            tc_fence_after();
            ++pc;
            return xq[ph * 64 + (hf ^ 1) * 32 + lane];
        };
        uint32_t jt = 0;
        Item it;
        bool stop = false;
        for (int k = 0; !stop && (item_of<kSeqs, kExt>(p, k, it)); ++k) {
            // This lane's query row is tile row rpos (of head it.h + row % hp in a packed
            // item; lanes past hp * rows, and rows past the chunk's end, are computed but
            // not stored).
            int rpos = row;
            if constexpr (kExt) {
                if (it.hp > 1) rpos = row / it.hp;
            }
            const int qpos = it.q_start + it.r0 + rpos;
            float m_used = -CUDART_INF_F, l = 0.f;
            // First token of block kb = 4j + qq and its in-page index, advanced quarter by
            // quarter (no division: it would wait behind the partner warp's exps on the MUFU).
            int blk_in = 0, blk_tok0 = 0;
            if (kExt && it.jb) {  // a piece starts at block 4 * jb
                const int lp0 = (4 * it.jb) / blocks_per_page;
                blk_in = 4 * it.jb - lp0 * blocks_per_page;
                blk_tok0 = lp0 * block_size + blk_in * kBlk;
            }
            for (int j = it.jb; j < it.je && !stop; ++j) {
                const uint32_t jr = (uint32_t)(j - it.jb);  // tile of this item or piece
                if (!__all_sync(0xffffffffu,
                                mbar_wait_abort(&bars[kSFull], (jt + jr) & 1, p.err, abort))) {
                    stop = true;
                    break;
                }
                tc_fence_after();
                for (int qq = 0; qq < 4; ++qq) {
                    float x[32];
                    {
                        uint32_t r[32];
                        tmem_ld32(sbase + 64 * qq + 32 * hf, r);
                        tc_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
                    }
                    if (neg) {  // a negative scale reverses the order of the raw scores
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[i] = -x[i];
                    }
                    // The quarter is one 64-key block; its valid keys form a prefix [0, lim).
                    // Only quarters with a page tail, the sequence end or the causal
                    // diagonal in them need the mask.
                    const int kb = 4 * j + qq;
                    int lim = 0;
                    if (kb < it.nblocks) {
                        const int off = blk_in * kBlk, tok0 = blk_tok0;
                        lim = min(kBlk, min(block_size - off, it.seq_len_k - tok0));
                        if (causal) lim = min(lim, qpos - tok0 + 1);
                    }
                    if (++blk_in == blocks_per_page) {  // the next block opens a page
                        blk_tok0 += block_size - (blocks_per_page - 1) * kBlk;
                        blk_in = 0;
                    } else {
                        blk_tok0 += kBlk;
                    }
                    lim -= 32 * hf;  // valid keys of this warp's half
                    if (!__all_sync(0xffffffffu, lim >= 32)) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[i] = i < lim ? x[i] : -CUDART_INF_F;
                    }
                    float mp[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        mp[i] = fmax3(fmax3(x[i], x[i + 4], x[i + 8]),
                                      fmax3(x[i + 12], x[i + 16], x[i + 20]),
                                      fmaxf(x[i + 24], x[i + 28]));
                    float mh = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3]));
                    bool ok = true;
                    mh = fmaxf(mh, exchange(mh, ok));
                    if (!__all_sync(0xffffffffu, ok)) {
                        stop = true;
                        break;
                    }
                    const float mx = mh * sc;
                    const float m_new = fmaxf(m_used, mx);
                    const bool need = m_new > m_used + 8.f;  // also true for the first finite max
                    const float alpha =
                        !need ? 1.f
                              : (m_used == -CUDART_INF_F ? 0.f : ex2_approx(m_used - m_new));
                    if (need) {
                        l *= alpha;
                        m_used = m_new;
                    }
                    const float nmu = m_used == -CUDART_INF_F ? 0.f : -m_used;
                    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float e0, e1;
                        fma2_bc(e0, e1, x[2 * i], x[2 * i + 1], sc, nmu);
                        const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
                        add2(sa[i & 3], sb[i & 3], sa[i & 3], sb[i & 3], p0, p1);
                        hi[i] = pack_bf16x2(p0, p1);
                        float r0, r1;
                        sub2(r0, r1, p0, p1, bf16_lo(hi[i]), bf16_hi(hi[i]));
                        lo[i] = pack_bf16x2(r0, r1);
                    }
                    tmem_st16(sbase + 64 * qq + 16 * hf, hi);
                    tmem_st16(sbase + 64 * qq + 32 + 16 * hf, lo);
                    l += ((sa[0] + sb[0]) + (sa[1] + sb[1])) + ((sa[2] + sb[2]) + (sa[3] + sb[3]));
                    // Moving the running max rescales this row of O (this warp's half of the
                    // columns), which the PVs of the tile's earlier quarters may still be
                    // accumulating: wait for them first (their completion covers every
                    // earlier tensor op).  At quarter 0 no wait is needed: S_j being ready
                    // means every tensor op issued before QK_j has completed.  Either way
                    // the parity wait is never two phases behind its barrier.
                    if ((jr > 0 || qq > 0) && __any_sync(0xffffffffu, need)) {
                        ok = qq == 0 || mbar_wait_abort(&bars[kPvDone + qq - 1], (jt + jr) & 1,
                                                      p.err, abort);
                        if (!__all_sync(0xffffffffu, ok)) {
                            stop = true;
                            break;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < 4; ++c) {
                            uint32_t r[32];
                            tmem_ld32(obase + 32 * c, r);
                            tc_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                            tmem_st32(obase + 32 * c, r);
                        }
                    }
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[kPFull + qq]);
                }
            }
            if (stop) break;
            // The row sum is the pair's two partial sums.  One warp of the pair hands it to
            // the epilogue warps (and, for a piece, stores the row's running max and sum
            // to the workspace), and the pair goes on with its next item at once.  The
            // epilogue reads the sums before it releases O, and the next item's sums are
            // written only after that item's first PV, which waits for that release.
            bool ok = true;
            const float lt = l + exchange(l, ok);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (hf == 0) {
                rowsum[row] = lt;
                if (kExt && it.slot >= 0 && rpos < it.rows)
                    p.ws_ml[(int64_t)it.slot * kBM + row] = make_float2(m_used, lt);
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kEpiReady]);
            }
            jt += it.je - it.jb;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Two warps per TMEM lane quarter: warp ew (0..7) takes rows 32*(warp % 4) + lane
        // and O columns 128*eh .. 128*eh + 127, eh = ew / 4.  Once the softmax warps have
        // handed over an item's row sums and its last PV is done, a whole item's warp
        // loads its 128 columns (four loads of 32), normalises them into BF16 registers,
        // releases O to the next item's PVs and only then stores its rows to out: the next
        // item's first PV waits for that release.  A piece of a split item keeps fp32 (its
        // unnormalised partial goes to the workspace slot, and the merge kernel combines
        // the item's pieces), so it stores each column block as it loads it and releases
        // O after the last load.  (tcgen05.ld is warp-wide: every lane loads; only rows
        // present store.)
        const int lq = warp & 3;
        const int eh = (warp - 2 - kSoftmaxWarps) >> 2;
        const int row = lq * 32 + lane;
        const uint32_t obase = tmem + ((uint32_t)(lq * 32) << 16) + kColO + 128 * eh;
        uint32_t jt = 0;
        Item it;
        for (int k = 0; item_of<kSeqs, kExt>(p, k, it); ++k) {
            if (!__all_sync(0xffffffffu,
                            mbar_wait_abort(&bars[kEpiReady], k & 1, p.err, abort) &&
                                mbar_wait_abort(&bars[kPvDone + 3],
                                                (jt + (it.je - it.jb) - 1) & 1, p.err, abort)))
                break;
            tc_fence_after();
            const float lt = rowsum[row];
            int rpos = row, rhead = it.h;
            if constexpr (kExt) {
                if (it.hp > 1) {
                    rpos = row / it.hp;
                    rhead = it.h + (row - rpos * it.hp);
                }
            }
            const bool present = rpos < it.rows;
            if (kExt && it.slot >= 0) {
                float *po = p.ws_o + ((int64_t)it.slot * kBM + row) * kHeadDim + 128 * eh;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld32(obase + 32 * c, r);
                    tc_wait_ld();
                    if (c == 3) {  // O is read: the next item may overwrite it
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars[kOEmpty]);
                    }
                    if (present) {
                        float4 *d4 = reinterpret_cast<float4 *>(po + 32 * c);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            d4[q4] = make_float4(__uint_as_float(r[4 * q4]),
                                                 __uint_as_float(r[4 * q4 + 1]),
                                                 __uint_as_float(r[4 * q4 + 2]),
                                                 __uint_as_float(r[4 * q4 + 3]));
                    }
                }
            } else {
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                uint32_t b[64];  // this warp's 128 columns of the row as BF16 pairs
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t r[16];
                    tmem_ld16(obase + 16 * c, r);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        b[8 * c + i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv,
                                                   __uint_as_float(r[2 * i + 1]) * inv);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kOEmpty]);  // O is read
                if (present) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(
                        p.out +
                        ((int64_t)(it.q_off + it.r0 + rpos) * p.num_q_heads + rhead) * kHeadDim +
                        128 * eh);
#pragma unroll
                    for (int q4 = 0; q4 < 16; ++q4)
                        d4[q4] = make_uint4(b[4 * q4], b[4 * q4 + 1], b[4 * q4 + 2],
                                            b[4 * q4 + 3]);
                }
            }
            jt += it.je - it.jb;
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

}  // namespace

// Merge of split items: item s's pieces each left, per query row, an unnormalised O row
// (sum over the piece's keys of 2^(score - m) v) with its running max m and sum of
// weights l.  The row's output is sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k with
// M = max_k m_k (a piece in which the row sees no key has m = -inf and weight 0), stored
// as BF16.  A CTA takes kMergeRows rows of one split item, 16 threads per row, each
// thread 16 dims: it reads its row's (m, l) pairs of all pieces at once, then four
// pieces' O values per round, 16 bytes at a time, so that many loads are in flight (the
// partials are read once).  Measured on the tail chunk's 22 MB (ncu, cold L2): one
// thread per dim and row ~44 us, 8 threads per row with two pieces per round ~14.6 us.
constexpr int kMergeRows = 16;
constexpr int kMergeThreadsPerRow = 16;
constexpr int kMergeDims = kHeadDim / kMergeThreadsPerRow;  // 16 dims per thread
constexpr int kMergeThreads = kMergeRows * kMergeThreadsPerRow;
constexpr int kMergeRound = 4;  // pieces whose loads are in flight together
struct MergeSplit {
    int out_row0;   // the item's first row in out
    int rows;       // its rows present (TMEM lanes: rows x hp for a packed item)
    int head;       // its head (the group's first, for a packed item)
    int pack;       // hp for a packed item (lane x: row x / hp, head + x % hp), else 0
    int slot0, npieces;
};
struct MergeParams {
    const float *ws_o;
    const float2 *ws_ml;
    uint16_t *out;
    int num_q_heads, num_split;
    MergeSplit s[kPfMaxSplitItems];
};

__global__ void __launch_bounds__(kMergeThreads) prefill_merge_kernel(
    const __grid_constant__ MergeParams p) {
    static_assert(kPfMaxPiecesPerItem <= 16, "a row's (m, l) pairs are kept in registers");
    static_assert(kPfMaxPiecesPerItem % kMergeRound == 0, "whole rounds of pieces");
    pdl_wait();  // the pieces' partials come from the prefill kernel before it
    pdl_trigger();
    const int si = blockIdx.x / (kBM / kMergeRows);
    const int r = (blockIdx.x % (kBM / kMergeRows)) * kMergeRows +
                  threadIdx.x / kMergeThreadsPerRow;
    const int d0 = (threadIdx.x % kMergeThreadsPerRow) * kMergeDims;
    if (si >= p.num_split) return;
    const MergeSplit d = p.s[si];
    if (r >= d.rows) return;
    float w[kPfMaxPiecesPerItem], lk[kPfMaxPiecesPerItem];
    float M = -CUDART_INF_F;
#pragma unroll
    for (int k = 0; k < kPfMaxPiecesPerItem; ++k) {
        const float2 ml = k < d.npieces ? p.ws_ml[(int64_t)(d.slot0 + k) * kBM + r]
                                        : make_float2(-CUDART_INF_F, 0.f);
        w[k] = ml.x;
        lk[k] = ml.y;
        M = fmaxf(M, ml.x);
    }
    float L = 0.f;
#pragma unroll
    for (int k = 0; k < kPfMaxPiecesPerItem; ++k) {
        w[k] = w[k] == -CUDART_INF_F ? 0.f : exp2f(w[k] - M);  // no key of piece k: weight 0
        L += w[k] * lk[k];
    }
    float acc[kMergeDims];
#pragma unroll
    for (int i = 0; i < kMergeDims; ++i) acc[i] = 0.f;
    // A piece in which the row sees no key holds zeros there (its weights were all 0),
    // so weight 0 times its values is 0; a slot past the item's pieces is not read.
#pragma unroll
    for (int k0 = 0; k0 < kPfMaxPiecesPerItem; k0 += kMergeRound) {
        if (k0 >= d.npieces) break;  // the same for every thread of the CTA
        float4 v[kMergeRound][kMergeDims / 4];
#pragma unroll
        for (int k = 0; k < kMergeRound; ++k) {
            const float4 *src = reinterpret_cast<const float4 *>(
                p.ws_o + ((int64_t)(d.slot0 + k0 + k) * kBM + r) * kHeadDim + d0);
#pragma unroll
            for (int i = 0; i < kMergeDims / 4; ++i)
                v[k][i] = k0 + k < d.npieces ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < kMergeRound; ++k) {
            const float wk = k0 + k < d.npieces ? w[k0 + k] : 0.f;
#pragma unroll
            for (int i = 0; i < kMergeDims / 4; ++i) {
                acc[4 * i] += wk * v[k][i].x;
                acc[4 * i + 1] += wk * v[k][i].y;
                acc[4 * i + 2] += wk * v[k][i].z;
                acc[4 * i + 3] += wk * v[k][i].w;
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int rp = d.pack ? r / d.pack : r;
    const int hh = d.pack ? d.head + (r - rp * d.pack) : d.head;
    uint4 *dst = reinterpret_cast<uint4 *>(
        p.out + ((int64_t)(d.out_row0 + rp) * p.num_q_heads + hh) * kHeadDim + d0);
#pragma unroll
    for (int i = 0; i < kMergeDims / 8; ++i)
        dst[i] = make_uint4(pack_bf16x2(acc[8 * i] * inv, acc[8 * i + 1] * inv),
                            pack_bf16x2(acc[8 * i + 2] * inv, acc[8 * i + 3] * inv),
                            pack_bf16x2(acc[8 * i + 4] * inv, acc[8 * i + 5] * inv),
                            pack_bf16x2(acc[8 * i + 6] * inv, acc[8 * i + 7] * inv));
}

#ifdef PA_TEST_HOOKS
cudaError_t set_prefill_test_hook(int skip_unit) {
    return cudaMemcpyToSymbol(g_test_skip_unit, &skip_unit, sizeof skip_unit);
}
#endif

namespace {

template <int kSeqs, bool kExt>
cudaError_t launch_prefill_n(const CUtensorMap *tmaps, const PrefillArgs &a, int slot,
                             cudaStream_t stream) {
    cudaError_t e = set_smem_once(
        reinterpret_cast<const void *>(prefill_tc_kernel<kSeqs, kExt>), kSmemBytes, slot);
    if (e != cudaSuccess) return e;
    TcMaps<kSeqs> maps;
    constexpr int kM = 3 + kPfMaxPackMaps;  // the first per-sequence map
    maps.q = tmaps[0];
    for (int i = 0; i < kPfMaxPackMaps; ++i) maps.qp[i] = tmaps[1 + i];
    maps.k = tmaps[kM - 2];
    maps.v = tmaps[kM - 1];
    TcParams<kSeqs, kExt> p;
    p.block_table = a.block_table;
    p.bt_stride = a.bt_stride;
    p.causal = a.causal;
    p.num_seqs = a.num_seqs;
    int items = 0;
    for (int b = 0; b < a.num_seqs; ++b) {
        const PrefillSeq &sq = a.seqs[b];
        maps.k_last[b] = tmaps[kM + 2 * b];
        maps.v_last[b] = tmaps[kM + 1 + 2 * b];
        SeqInfo &si = p.seq[b];
        si.q_off = sq.q_off;
        si.q_len = sq.q_len;
        si.q_start = sq.q_start;
        si.seq_len_k = sq.q_start + sq.q_len;
        si.last_page = (si.seq_len_k - 1) / a.block_size;
        si.item_off = items;
        si.bt_row = sq.bt_row;
        items += prefill_chunk_items(sq.q_len, a.num_q_heads, a.group);
    }
    p.num_items = items;
    p.num_q_heads = a.num_q_heads;
    p.group = a.group;
    // The packed Q maps' heads per item: the group's divisors > 1, largest first (as the
    // maps were made).
    int npack = 0;
    for (int hp = a.group; hp > 1 && npack < kPfMaxPackMaps; --hp)
        if (a.group % hp == 0) {
            p.qp_hp[npack] = hp;
            p.qp_bytes[npack++] = kChunks * 128 * hp * (kBM / hp);
        }
    for (; npack < kPfMaxPackMaps; ++npack) p.qp_hp[npack] = p.qp_bytes[npack] = 0;
    p.block_size = a.block_size;
    p.blocks_per_page = (a.block_size + kBlk - 1) / kBlk;
    p.num_pages = a.num_pages;
    p.sc = fmaxf(fabsf(a.scale) * 1.4426950408889634f, FLT_MIN);
    p.neg = a.scale < 0.f;
    p.out = a.out;
    p.err = a.err;
    int grid = min(p.num_items, a.num_sms > 0 ? a.num_sms : 1);
    int num_split = 0;
    p.ws_o = nullptr;
    p.ws_ml = nullptr;
    if (a.sched && a.sched->num_ctas > 0) {
        const PrefillSchedule &sc = *a.sched;
        const int G = sc.num_ctas;
        p.sched.num_ctas = G;
        memcpy(p.sched.off, sc.off, (G + 1) * sizeof(uint16_t));
        memcpy(p.sched.items, sc.items, sc.off[G] * sizeof(uint16_t));
        grid = G;
        if (sc.num_pieces > 0) {
            if (!kExt || !a.workspace) return cudaErrorInvalidValue;
            if constexpr (kExt)
                memcpy(p.pc.pieces, sc.pieces, sc.num_pieces * sizeof(PrefillPiece));
            p.ws_o = static_cast<float *>(a.workspace);
            p.ws_ml = reinterpret_cast<float2 *>(p.ws_o + (size_t)sc.num_pieces * kBM * kHeadDim);
            num_split = sc.num_split;
        }
    } else {
        p.sched.num_ctas = 0;
    }
    if (a.ev_start && (e = record_event(a.ev_start, stream)) != cudaSuccess) return e;
    e = launch_pdl(prefill_tc_kernel<kSeqs, kExt>, dim3(grid), dim3(kThreads), kSmemBytes, stream,
                   maps, p);
    if (e != cudaSuccess) return e;
    if (num_split > 0) {
        // The split items' pieces are merged into their rows of out.
        MergeParams mp;
        mp.ws_o = p.ws_o;
        mp.ws_ml = p.ws_ml;
        mp.out = a.out;
        mp.num_q_heads = a.num_q_heads;
        mp.num_split = num_split;
        for (int x = 0; x < num_split; ++x) {
            const int idx = a.sched->split_item[x];
            int b = 0;
            while (b + 1 < a.num_seqs && idx >= p.seq[b + 1].item_off) ++b;
            const SeqInfo &sq = p.seq[b];
            int qt, h0, hp;
            prefill_item_at(idx - sq.item_off, sq.q_len, a.num_q_heads, a.group, &qt, &h0, &hp);
            const int rows = min(kBM, sq.q_len - qt * kBM);
            mp.s[x].out_row0 = sq.q_off + qt * kBM;
            mp.s[x].rows = rows * hp;
            mp.s[x].head = h0;
            mp.s[x].pack = hp > 1 ? hp : 0;
            mp.s[x].slot0 = a.sched->split_slot0[x];
            mp.s[x].npieces = a.sched->split_n[x];
        }
        e = launch_pdl(prefill_merge_kernel, dim3(num_split * (kBM / kMergeRows)),
                       dim3(kMergeThreads), 0, stream, mp);
        if (e != cudaSuccess) return e;
    }
    if (a.ev_stop) e = record_event(a.ev_stop, stream);
    return e;
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap *tmaps, const PrefillArgs &a, cudaStream_t stream) {
    if (a.num_seqs < 1 || a.num_seqs > kPfMaxSeqs) return cudaErrorInvalidValue;
    // The extended kernel when the plan has pieces of split items or a chunk ends in a
    // packed query tile.
    bool ext = a.sched && a.sched->num_ctas > 0 && a.sched->num_pieces > 0;
    for (int b = 0; b < a.num_seqs; ++b)
        ext = ext || prefill_tile_heads(a.seqs[b].q_len, a.group) > 1;
    if (a.num_seqs == 1)
        return ext ? launch_prefill_n<1, true>(tmaps, a, 4, stream)
                   : launch_prefill_n<1, false>(tmaps, a, 1, stream);
    return ext ? launch_prefill_n<kPfMaxSeqs, true>(tmaps, a, 5, stream)
               : launch_prefill_n<kPfMaxSeqs, false>(tmaps, a, 2, stream);
}

}  // namespace pa
