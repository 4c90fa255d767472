// pa_internal.h -- host-side declarations shared between the C-ABI layer (pa_api.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

// The calling thread's current CUDA context as a number (0 if none).  Host-side caches
// of per-device facts (symbol addresses, function attributes) are keyed on it: after
// cudaDeviceReset the device gets a new primary context with the module loaded afresh.
uintptr_t current_context();

// Raises a kernel's dynamic shared-memory limit once per (kernel slot, device context),
// so that later launches (possibly under stream capture) make no attribute call.  Slots:
// 0 and 3 the two decode kernel shapes, 1, 2, 4, 5 the four prefill kernel variants.
constexpr int kSmemSlots = 8;
cudaError_t set_smem_once(const void *kernel, int bytes, int slot);

// Launches a kernel with programmatic dependent launch allowed: it may start while the
// previous kernel on the stream is still running.  Every library kernel calls
// pdl_wait() before it reads memory that earlier work on the stream may produce, and
// pdl_trigger() once its own dependents may start their prologue.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Records a measurement event on the stream.  Under stream capture it becomes an event
// record node of the graph (cudaEventRecordExternal), so that each replay records it; a
// plain record in a capturing stream would only order the capture.  Outside a capture it
// is a plain record (the runtime refuses the external flag there).
inline cudaError_t record_event(cudaEvent_t ev, cudaStream_t stream) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return e;
    return cs == cudaStreamCaptureStatusActive
               ? cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal)
               : cudaEventRecord(ev, stream);
}

// Kernel copy of bytes (a multiple of 16) between 16-byte aligned device-accessible
// addresses.
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream);

// ----------------------------------------------------------------- cache write
cudaError_t launch_slot_mapping(const int32_t *positions, const int32_t *seq_idx,
                                const int32_t *block_table, int num_seqs, int64_t bt_stride,
                                int max_blocks,
                                int num_tokens, int block_size, int64_t *slot_mapping,
                                unsigned *err, cudaStream_t stream);

// Decode input preparation for several KV-cache groups in one launch.
constexpr int kPrepMaxGroups = 8;
struct PrepGroup {
    const int32_t *block_table;
    int64_t bt_stride;
    int max_blocks, block_size;
    int64_t *slot_mapping;
};
struct PrepArgs {
    const int32_t *positions, *sampled_ids;
    int32_t *input_ids, *seq_lens, *query_start_loc;
    int num_seqs, num_groups;
    PrepGroup g[kPrepMaxGroups];
    unsigned *err;
};
cudaError_t launch_decode_input_prep(const PrepArgs &a, cudaStream_t stream);

cudaError_t launch_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                                     uint16_t *k_cache, uint16_t *v_cache, int64_t page_stride,
                                     int64_t num_pages, const int64_t *slot_mapping,
                                     int num_tokens, int row_elems, int block_size,
                                     unsigned *err, cudaStream_t stream);

// ----------------------------------------------------------------- decode
constexpr int kDecTile = 16;       // tokens per MMA tile (page-local)
constexpr int kDecPair = 2;        // tiles per ring stage
// Two shapes of the split kernel (consumer warps, 32 KB ring stages): splits of up to
// kDecShortTiles tiles (the tail of the stream and the CTA merge are a large share of their
// time) run with four consumer warps and a 4-stage ring; longer splits with three consumer
// warps and a 6-stage ring (measured fastest for each; fewer warps means less to merge).
constexpr int kDecShortConsumers = 4, kDecShortStages = 4;
constexpr int kDecLongConsumers = 3, kDecLongStages = 6;
constexpr int kDecShortTiles = 64;
// Stage m holds tiles 2m and 2m + 1 of the split and uses ring slot m % stages.  In a short
// split tile i is consumed by warp i % consumers; in a long one stage m by warp
// m % consumers.  An mbarrier wait only tells the last two phases apart, so a warp must
// visit each of its slots once per ring round, in phase order: the ring round (stages *
// kDecPair tiles, or stages stages) is a multiple of the consumer count.
template <int kC, int kS>
struct DecShape {
    static_assert((kS * kDecPair) % kC == 0 && kS % kC == 0, "tile -> warp mapping must be fixed");
    static constexpr int consumers = kC, stages = kS;
};
constexpr int kDecMaxSplits = 1024;  // upper bound on CTAs per (sequence, KV head)
constexpr int kDecMaxGroup = 8;    // query heads per KV head handled by one MMA column tile

struct DecodePlan {
    int tiles_per_page;   // ceil(block_size / kDecTile)
    int max_tiles;        // tiles of the longest allowed sequence
    int tiles_per_split;  // tiles one CTA processes (a multiple of kDecPair)
    int num_splits;       // CTAs per (sequence, KV head)
};

DecodePlan plan_decode(int num_seqs, int num_kv_heads, int block_size, int max_seq_len,
                       int num_sms);
size_t decode_workspace_bytes(int num_seqs, int num_q_heads, const DecodePlan &plan);

struct DecodeArgs {
    const uint16_t *q;
    const int32_t *block_table;
    int64_t bt_stride;
    const int32_t *seq_lens;
    int num_seqs, max_seq_len;
    int num_q_heads, num_kv_heads, group;
    int block_size;
    int64_t num_pages;
    float scale;
    uint16_t *out;
    void *workspace;
    unsigned *err;
    cudaEvent_t ev_start, ev_stop;  // optional: recorded around the split kernel
    // Optional fused write of each sequence's newest token (all NULL when unused).  With
    // new_k set and new_slots NULL the slots come from the block table, and are stored
    // to slot_out when that is set.
    uint16_t *k_cache_w, *v_cache_w;
    const uint16_t *new_k, *new_v;
    const int64_t *new_slots;
    int64_t *slot_out;
    int64_t page_stride;            // elements between consecutive pages
};

// tmaps: K and V as 5-D views whose boxes hold one 16-token tile of one KV head, all
// dims (the two tiles of a ring stage are two boxes, from one page or from two).
cudaError_t launch_decode(const CUtensorMap *tmaps, const DecodeArgs &a, const DecodePlan &plan,
                          cudaStream_t stream);

// ----------------------------------------------------------------- prefill
constexpr int kPfQRows = 128;      // query rows per work item (one TMEM lane each)
constexpr int kPfKvTile = 256;     // keys per K/V tile: four page-local blocks
constexpr int kPfBlock = 64;       // keys per TMA box (one page-local block)
constexpr int kPfRing = 5;         // 32 KB K/V unit slots in the shared-memory ring

// Keys one work item (kPfQRows query rows of one head) reads, counted in kPfKvTile-key
// tiles of page-local kPfBlock-key blocks: what the kernel streams for that item.
__host__ __device__ inline int prefill_item_tiles(int q_len, int q_start, int causal, int r0,
                                                  int block_size) {
    const int rows = q_len - r0 < kPfQRows ? q_len - r0 : kPfQRows;
    const int nkeys = causal ? q_start + r0 + rows : q_start + q_len;
    const int blocks_per_page = (block_size + kPfBlock - 1) / kPfBlock;
    const int full = nkeys / block_size;
    const int rem = nkeys - full * block_size;
    const int nblocks = full * blocks_per_page + (rem + kPfBlock - 1) / kPfBlock;
    return (nblocks + kPfKvTile / kPfBlock - 1) / (kPfKvTile / kPfBlock);
}

// Packed last query tile.  A chunk's last query tile holds r = q_len - 128 * (tiles - 1)
// rows.  It runs as items of hp query heads each, hp the largest divisor of the GQA group
// G = Hq / Hkv with hp * r <= 128 (hp = 1: one head per item, not packed): item row x is
// tile row x / hp of query head h0 + x % hp, and Q is read as one box of hp heads x
// 128 / hp rows.  The hp heads of an item share one KV head (hp divides G), so the tile
// runs as Hq / hp items instead of Hq items of r rows: the q=1685 tail chunk (21 rows,
// G = 6) as 4 items instead of 24, a 40-row tail as 8 (hp = 3), a 60-row tail as 12.
constexpr int kPfMaxPackMaps = 3;  // divisors > 1 of a group of at most 8: {8, 4, 2}, {6, 3, 2}
__host__ __device__ inline int prefill_tile_heads(int q_len, int group) {
    const int r = q_len - ((q_len - 1) / kPfQRows) * kPfQRows;  // rows of the last tile
    for (int hp = group; hp > 1; --hp)
        if (group % hp == 0 && hp * r <= kPfQRows) return hp;
    return 1;
}
// Work items of one chunk, and what item i of it is: query tile *qt, its first query
// head *h0 and its heads *hp (1 unless it is one of the packed last tile's items).  Items
// run from the chunk's last (longest, under causal masking) query tile to its first.
__host__ __device__ inline int prefill_chunk_items(int q_len, int num_q_heads, int group) {
    const int nqt = (q_len + kPfQRows - 1) / kPfQRows;
    return (nqt - 1) * num_q_heads + num_q_heads / prefill_tile_heads(q_len, group);
}
__host__ __device__ inline void prefill_item_at(int i, int q_len, int num_q_heads, int group,
                                                int *qt, int *h0, int *hp) {
    const int nqt = (q_len + kPfQRows - 1) / kPfQRows;
    const int php = prefill_tile_heads(q_len, group);
    if (php > 1) {
        const int n_last = num_q_heads / php;
        if (i < n_last) {
            *qt = nqt - 1;
            *h0 = i * php;
            *hp = php;
            return;
        }
        i -= n_last;
        *qt = nqt - 2 - i / num_q_heads;
    } else {
        *qt = nqt - 1 - i / num_q_heads;
    }
    *h0 = i % num_q_heads;
    *hp = 1;
}

// Static assignment of prefill work items to the persistent CTAs (items numbered as
// prefill_item_at gives them, sequence by sequence).
// When a workspace is given and the items do not divide evenly over the CTAs, some
// items are split along the keys into pieces (ranges of their 256-key tiles) that run on
// different CTAs; each piece writes an unnormalised partial (fp32 O rows, and per row
// the running max and the sum of weights) into its workspace slot, and a merge kernel
// combines an item's pieces afterwards.
constexpr int kPfSchedMaxCtas = 256;
constexpr int kPfSchedMaxItems = 6144;     // schedule entries (whole items and pieces)
constexpr int kPfMaxPieces = 480;          // pieces of split items
constexpr int kPfMaxSplitItems = 160;      // split items
constexpr uint16_t kPfPieceBit = 0x8000;   // schedule entry kPfPieceBit | p: piece p
constexpr int kPfMinPieceTiles = 4;        // no piece is shorter
constexpr int kPfMaxPiecesPerItem = 16;    // no item is cut into more pieces

struct PrefillPiece {
    uint16_t item;                  // the split item
    uint16_t tile_begin, tile_end;  // its 256-key tiles [tile_begin, tile_end)
    uint16_t slot;                  // its partial's workspace slot
};

struct PrefillSchedule {
    int num_ctas;                        // 0: none (the kernel walks a snake order)
    int num_pieces, num_split;           // pieces, and the items they split
    uint16_t off[kPfSchedMaxCtas + 1];   // CTA b runs items[off[b] .. off[b+1]) in order
    uint16_t items[kPfSchedMaxItems];    // an item index, or kPfPieceBit | piece index
    PrefillPiece pieces[kPfMaxPieces];
    // Split item s: item split_item[s], whose pieces own slots split_slot0[s] .. + split_n[s].
    uint16_t split_item[kPfMaxSplitItems], split_slot0[kPfMaxSplitItems],
        split_n[kPfMaxSplitItems];
};

// Bytes of one piece's partial in the prefill workspace: 128 rows x 256 fp32 O values,
// plus a (running max, sum of weights) pair per row.
constexpr size_t kPfSlotBytes = (size_t)kPfQRows * 256 * 4 + (size_t)kPfQRows * 8;  // head dim 256

// Plans the schedule (cached per shape) for one launch over num_seqs chunks (chunk b:
// q_lens[b] rows at positions q_starts[b]..; work items numbered sequence by sequence,
// each sequence's longest query tile first); false when the problem exceeds the arrays.
// allow_split: items may be split into pieces (the launch has a workspace of
// s->num_pieces * kPfSlotBytes bytes).  max_cost (optional): the largest per-CTA cost, in
// tiles plus one per item (two per piece).
bool plan_prefill(int num_seqs, const int *q_lens, const int *q_starts, int causal,
                  int num_q_heads, int group, int block_size, int num_ctas, bool allow_split,
                  PrefillSchedule *s, int *max_cost);

// Sequences one prefill launch takes (their chunks' tensor maps travel in the launch's
// parameters); a larger batch is split into several launches.
constexpr int kPfMaxSeqs = 32;

struct PrefillSeq {
    int q_off;    // first row of the chunk in q / out
    int q_len;    // rows of the chunk (>= 1)
    int q_start;  // absolute position of the chunk's first row
    int bt_row;   // its row of the block table
};

struct PrefillArgs {
    const PrefillSchedule *sched;  // host copy, passed to the kernel by value (or NULL)
    void *workspace;               // piece partials (sched->num_pieces slots), or NULL
    const int32_t *block_table;    // [num_seqs, bt_stride]: row b for sequence b
    int64_t bt_stride;
    int num_seqs;                  // 1 .. kPfMaxSeqs
    const PrefillSeq *seqs;        // host array of num_seqs entries
    int causal;
    int num_q_heads, num_kv_heads, group;
    int block_size;
    int64_t num_pages;
    float scale;
    uint16_t *out;
    unsigned *err;
    cudaEvent_t ev_start, ev_stop;  // optional: recorded around the prefill kernel
    int num_sms;                    // persistent grid size bound
};

// tmaps: Q (boxes of 1 head x 128 rows); kPfMaxPackMaps maps of Q for packed items, one
// per divisor hp > 1 of the group, largest first (boxes of hp heads x 128 / hp rows;
// copies of the first map where the group has fewer such divisors); K, V; then the K and
// V maps cut at each sequence's last token (2 per sequence).
cudaError_t launch_prefill(const CUtensorMap *tmaps, const PrefillArgs &a, cudaStream_t stream);

#ifdef PA_TEST_HOOKS
// Test build only (libpa_test.so, compiled with -DPA_TEST_HOOKS and a short wait limit):
// the decode producer leaves out the loads of ring stage `skip_stage` of every CTA, the
// prefill producer those of ring unit `skip_unit` (-1: none), so that a consumer's
// bounded wait runs out; and the decode consumer warps (but the one writing the newest
// token) start `consumer_delay_ns` late, after the split's loads may all have landed.
// Exported to the failure-path tests as
//     extern "C" int pa_test_hook(int decode_skip_stage, int prefill_skip_unit,
//                                 int decode_consumer_delay_ns);
// The product library has neither the hooks nor this entry point.
cudaError_t set_decode_test_hook(int skip_stage, int consumer_delay_ns);
cudaError_t set_prefill_test_hook(int skip_unit);
#endif

}  // namespace pa
