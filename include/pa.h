/*
 * pa.h -- C ABI of the paged-KV GQA attention library for one GB300 (sm_103a).
 *
 * The library computes grouped-query attention over a paged BF16 KV cache addressed
 * through a block table, in two shapes -- q=1 decode and a causal prefill chunk over
 * earlier paged context -- plus the slot-mapping computation and the KV write of new
 * tokens.  Sources, cited by page and section:
 *   page832 post   = luanjiahao.me feed, "784 -> 832 KV page for the DCU vendor paged
 *                    attention" (sections 1, 4, 5, 6, 7);
 *   input-prep post = jsqmd.com, "single-token decode input preparation on DCU" (3.2, 5).
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library never
 *     allocates, frees or keeps a tensor; a call only reads and writes what it is given.
 *   - BF16 values are passed as raw 16-bit patterns (pa_bf16).
 *   - Cache layout [page832 §4]: K and V are separate arrays, each
 *     [num_pages, block_size, num_kv_heads, head_dim] in the last three dimensions,
 *     with the distance between consecutive pages given by page_stride (in elements):
 *     block_size * num_kv_heads * head_dim for a plain tensor, twice that for the
 *     unbind(1) views of a [num_pages, 2, block_size, Hkv, D] tensor.
 *   - Address translation [page832 §1]: token t of a sequence lives in page
 *     block_table[t / block_size] at offset t % block_size.
 *   - Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns a status code.  Arguments are checked on the host before any
 *     work is queued; a bad argument returns an error and queues nothing.  No call
 *     throws, traps or asserts on the device.
 *   - Device-side checks: a block-table entry outside [0, num_pages), a slot outside
 *     the pool, a sequence length outside [1, max_seq_len] or a bounded wait that ran
 *     out do not fault: the access is skipped (a tile read outside the pool reads
 *     zeros) and a bit is set in the library's device error word, which
 *     pa_get_device_errors() reads.
 *   - Supported shapes: head_dim 256 and num_q_heads / num_kv_heads in 1..8 for the
 *     attention calls (anything else returns PA_ERR_UNSUPPORTED: there is no fallback
 *     path).  Pointers must be 16-byte aligned.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pa_bf16;

enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, bad workspace */
    PA_ERR_UNSUPPORTED = 2,   /* valid but outside the shapes the kernels are built for */
    PA_ERR_CUDA = 3,          /* the CUDA runtime or driver reported an error */
    PA_ERR_TIMEOUT = 4,       /* pa_get_device_errors: a bounded wait inside a kernel ran
                                 out (PA_DEVERR_TIMEOUT is set in the error word) */
};

/* Bits of the device error word (pa_get_device_errors). */
enum pa_device_error {
    PA_DEVERR_PAGE = 1u,      /* block-table entry outside [0, num_pages) */
    PA_DEVERR_SEQLEN = 2u,    /* sequence length outside [1, max_seq_len] */
    PA_DEVERR_SLOT = 4u,      /* slot (or its page) outside the pool */
    PA_DEVERR_TIMEOUT = 8u,   /* a bounded wait inside a kernel ran out */
    PA_DEVERR_POSITION = 16u, /* a position past the block table's capacity */
    PA_DEVERR_LAYOUT = 32u,   /* a kernel found its shared memory misaligned; it did nothing */
};

/*
 * pa_slot_mapping -- slot of each new token [input-prep §3.2]:
 *     slot[i] = block_table[s, p / block_size] * block_size + p % block_size
 * with p = positions[i] and s = seq_idx[i] (seq_idx may be NULL: every token belongs
 * to sequence 0).  block_table is int32 [num_seqs, bt_stride] row-major, of which the
 * first max_blocks entries of a row are valid.  slot_mapping is int64 [num_tokens].
 * A negative position is a padding token and gets slot -1.  A token whose sequence is
 * outside [0, num_seqs), whose logical page is >= max_blocks, or whose block-table
 * entry is negative gets slot -1 and sets PA_DEVERR_POSITION.  num_tokens == 0 is a
 * no-op.
 */
int pa_slot_mapping(const int32_t *positions, const int32_t *seq_idx,
                    const int32_t *block_table, int num_seqs, int64_t bt_stride,
                    int max_blocks, int num_tokens, int block_size, int64_t *slot_mapping,
                    void *stream);

/*
 * pa_decode_input_prep -- the inputs of one decode step, computed on the device in one
 * launch for every KV-cache group [input-prep §2, §4, §5]: num_seqs entries, each a
 * sequence that decodes one new token at positions[s] (the number of tokens already in
 * its cache) or a padding entry (positions[s] < 0).  Writes
 *   seq_lens[s]          = positions[s] + 1    (0 for a padding entry)
 *   input_ids[s]         = sampled_ids[s]      (the token sampled by the previous step)
 *   query_start_loc[0]   = 0, query_start_loc[s + 1] = query_start_loc[s] + (1 for a
 *                          sequence, 0 for a padding entry): a padded entry owns no query
 *                          row, so one request in padded buffers gives [0, 1, 1, ...]
 *                          beside seq_lens [position + 1, 0, 0, ...] (§2)
 *   slot_mappings[g][s]  = block_tables[g][s * bt_strides[g] + p / block_sizes[g]]
 *                          * block_sizes[g] + p % block_sizes[g],   p = positions[s]
 * for each group g, with the checks of pa_slot_mapping (slot -1 for padding; -1 and
 * PA_DEVERR_POSITION for a logical page >= max_blocks[g] or a negative table entry).
 *   positions        int32 [num_seqs], device
 *   sampled_ids, input_ids   int32 [num_seqs], device; both NULL to skip the copy
 *   seq_lens         int32 [num_seqs], device, or NULL (not written)
 *   query_start_loc  int32 [num_seqs + 1], device, or NULL (not written)
 *   block_tables, bt_strides, max_blocks, block_sizes, slot_mappings: HOST arrays of
 *                    num_groups entries (1 <= num_groups <= 8); block_tables[g] points to
 *                    the group's int32 [num_seqs, bt_strides[g]] table on the device,
 *                    slot_mappings[g] to its int64 [num_seqs] output on the device.  The
 *                    pointers are read during the call only (under stream capture they
 *                    are baked into the captured launch).
 * The groups may differ in block size (a model whose layers keep separate caches).
 * Returns PA_ERR_INVALID_ARG for a bad count, a NULL pointer, or bt_strides[g] <
 * max_blocks[g]; num_seqs == 0 is a no-op.
 */
int pa_decode_input_prep(const int32_t *positions, const int32_t *sampled_ids,
                         int32_t *input_ids, int32_t *seq_lens, int32_t *query_start_loc,
                         int num_seqs, int num_groups, const int32_t *const *block_tables,
                         const int64_t *bt_strides, const int *max_blocks,
                         const int *block_sizes, int64_t *const *slot_mappings, void *stream);

/*
 * pa_reshape_and_cache -- KV write of new tokens.  key and value are BF16
 * [num_tokens, num_kv_heads, head_dim], contiguous; token i's rows are copied bit for
 * bit to page slot_mapping[i] / block_size, offset slot_mapping[i] % block_size of
 * k_cache and v_cache [page832 §4 layout].  A negative slot is skipped (padding); a
 * slot whose page is >= num_pages is skipped and sets PA_DEVERR_SLOT.
 * num_kv_heads * head_dim must be a multiple of 8.  num_tokens == 0 is a no-op.
 */
int pa_reshape_and_cache(const pa_bf16 *key, const pa_bf16 *value, pa_bf16 *k_cache,
                         pa_bf16 *v_cache, int64_t page_stride, int64_t num_pages,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, void *stream);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs for this
 * problem size on the current device.  Returns 0 for invalid sizes.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                int head_dim, int block_size, int max_seq_len);

/*
 * pa_decode -- q=1 paged attention for a batch [page832 §5, §7]: for each sequence s
 * and query head h,
 *     out[s, h] = softmax_t( scale * q[s, h] . k_t ) . v_t,   t in [0, seq_lens[s])
 * with k_t, v_t of KV head h / (Hq / Hkv) fetched through row s of block_table.
 *   q, out       BF16 [num_seqs, num_q_heads, head_dim], contiguous.  out may also be
 *                page-locked host memory (cudaHostAlloc or cudaHostRegister): the combine
 *                kernel then writes the result straight to the host.  Other host memory
 *                is refused (PA_ERR_INVALID_ARG).
 *   block_table  int32 [num_seqs, bt_stride]; entries past a sequence's last page unused
 *   seq_lens     int32 [num_seqs], device; each in [1, max_seq_len]
 *   workspace    device scratch of >= pa_decode_workspace_size(...) bytes, 256-byte
 *                aligned; its contents on entry do not matter.
 * Optional fused write of each sequence's newest token (a serving step): when new_k,
 * new_v and new_slots are all non-NULL, the token being decoded -- position
 * seq_lens[s] - 1 of sequence s -- is written into the caches from new_k / new_v
 * ([num_seqs, Hkv, D]) at new_slots[s] (int64 [num_seqs], as pa_slot_mapping gives it),
 * bit for bit as pa_reshape_and_cache would, and the attention includes it.  The
 * write happens inside the decode kernel, by the CTA that reads that token's tile, just
 * before it loads the tile.  A negative new_slots[s] is skipped (padding).  A slot that
 * is not the one the block table gives for position seq_lens[s] - 1 is not written and
 * sets PA_DEVERR_SLOT.  Pass all three NULL to skip.
 * The split-context kernel processes page-local tiles of 16 tokens, so any block_size
 * works (one that is not a multiple of 16 leaves a ragged tile at each page end; 784
 * and 832 are both multiples of 16).
 */
int pa_decode(const pa_bf16 *q, const pa_bf16 *k_cache, const pa_bf16 *v_cache,
              int64_t page_stride, int64_t num_pages, const int32_t *block_table,
              int64_t bt_stride, const int32_t *seq_lens, int num_seqs, int max_seq_len,
              int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
              pa_bf16 *out, void *workspace, size_t workspace_bytes,
              const pa_bf16 *new_k, const pa_bf16 *new_v, const int64_t *new_slots,
              void *stream);

/*
 * pa_decode_append -- one decode step in which each sequence's newest token is appended
 * to the cache and attended to, with its slot derived on the device [input-prep §3.2,
 * §5: the slot-mapping formula; page832 §5, §7].  For each sequence s, the token being
 * decoded sits at position p = seq_lens[s] - 1 and its slot is
 *     slot_mapping[s] = block_table[s][p / block_size] * block_size + p % block_size,
 * the value pa_slot_mapping gives for (p, s).  The kernel writes new_k[s] / new_v[s]
 * ([num_seqs, Hkv, D], contiguous) there, bit for bit as pa_reshape_and_cache would,
 * then decodes as pa_decode does; no separate slot-mapping launch is needed.
 *   slot_mapping  int64 [num_seqs], device, 8-byte aligned, OUTPUT, may be NULL: the
 *                 slots written, for callers that reuse them (for example for the other
 *                 layers' pa_reshape_and_cache of the same step).
 * Every sequence has a newest token (no padding).  A block-table entry for that token
 * outside [0, num_pages) writes nothing and sets PA_DEVERR_PAGE; slot_mapping[s] then
 * holds -1 for a negative entry (as pa_slot_mapping gives) and the formula's value for
 * one past the pool.  All other arguments, checks and errors are those of
 * pa_decode; new_k and new_v must be non-NULL and 16-byte aligned.
 */
int pa_decode_append(const pa_bf16 *q, pa_bf16 *k_cache, pa_bf16 *v_cache, int64_t page_stride,
                     int64_t num_pages, const int32_t *block_table, int64_t bt_stride,
                     const int32_t *seq_lens, int num_seqs, int max_seq_len, int num_q_heads,
                     int num_kv_heads, int head_dim, int block_size, float scale, pa_bf16 *out,
                     void *workspace, size_t workspace_bytes, const pa_bf16 *new_k,
                     const pa_bf16 *new_v, int64_t *slot_mapping, void *stream);

/*
 * pa_decode_noalloc -- the same decode as pa_decode (without the fused write), for
 * callers that cannot allocate device memory on the decode path: for example a serving
 * runtime that gives almost all device memory to its KV-cache pool at start-up and
 * allows no allocation afterwards, or plain C code with no device allocator at hand.
 * The pages describe nothing like it; it exists only for such callers.
 *
 * Instead of a caller-provided workspace it uses one fixed scratch array of
 * PA_DECODE_NOALLOC_SCRATCH_BYTES (4 MiB) that is part of the library's device image:
 * every GPU that loads the library holds that memory until the process exits.  The call
 * allocates and frees nothing.  The caller still passes all inputs and the output.
 *   - Problems whose split partials need more than that (pa_decode_workspace_size >
 *     PA_DECODE_NOALLOC_SCRATCH_BYTES; about 160 sequences of 24 heads, or fewer with
 *     long contexts on few sequences) are refused with PA_ERR_UNSUPPORTED and nothing
 *     is queued.  Other bad arguments return what pa_decode returns for them.
 *   - The first call on each device looks up the array's device address (with that
 *     device current) and keeps it; make that first call before any stream capture.
 *     After cudaDeviceReset the device's next context loads the array afresh; the next
 *     call sees the new context and looks the address up again (so, after a reset too,
 *     make one call before capturing).
 *   - All calls on a device share the one array, and it keeps whatever the last call
 *     wrote.  Nothing in it needs to start at zero: every value a call reads from it was
 *     written earlier in the same call.  Calls whose work overlaps on the GPU (different
 *     streams, or different host threads, without ordering between them) race on the
 *     array and can produce wrong outputs; order them, e.g. on one stream.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES (4u << 20)

int pa_decode_noalloc(const pa_bf16 *q, const pa_bf16 *k_cache, const pa_bf16 *v_cache,
                      int64_t page_stride, int64_t num_pages, const int32_t *block_table,
                      int64_t bt_stride, const int32_t *seq_lens, int num_seqs,
                      int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, float scale, pa_bf16 *out, void *stream);

/*
 * pa_prefill_workspace_size -- bytes of device workspace with which pa_prefill_chunk
 * may split work items along the keys for this chunk shape on the current device; 0 when
 * no split would pay (or for invalid sizes).  The kernel's work item is 128 query rows of
 * one head; when the items do not divide evenly over the SMs (the q=1685 tail chunk over
 * 12288 tokens has 336 items of ~52 key tiles for 152 SMs; a short chunk over a long
 * context has fewer items than SMs), pieces of the longest items run on different SMs
 * and a merge kernel combines them (about 129 KB per piece).  At most a few tens of MB.
 */
size_t pa_prefill_workspace_size(int q_len, int q_start, int causal, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size);

/*
 * pa_prefill_chunk -- attention of a chunk of q_len query rows of ONE sequence over
 * that sequence's paged cache [page832 §6].  Row i sits at absolute position
 * q_start + i; with causal != 0 it sees keys 0..q_start+i (diagonal included),
 * otherwise all q_start + q_len keys.  The chunk's own K/V must already be in the cache
 * (pa_slot_mapping + pa_reshape_and_cache first).
 *   q, out       BF16 [q_len, num_q_heads, head_dim], contiguous
 *   block_table  int32, the sequence's row: ceil((q_start + q_len) / block_size) entries
 *   workspace    device scratch of workspace_bytes bytes, 256-byte aligned, or NULL (then
 *                no item is split).  With at least pa_prefill_workspace_size(...) bytes
 *                the call may split items (its contents on entry do not matter); with
 *                less it runs as with NULL.  Calls that run at the same time need
 *                separate workspaces.
 * Shapes accepted: 1 <= q_len, 0 <= q_start, q_start + q_len <= 2^31 - 1.
 */
int pa_prefill_chunk(const pa_bf16 *q, const pa_bf16 *k_cache, const pa_bf16 *v_cache,
                     int64_t page_stride, int64_t num_pages, const int32_t *block_table,
                     int q_len, int q_start, int causal, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, float scale, pa_bf16 *out, void *workspace,
                     size_t workspace_bytes, void *stream);

/*
 * pa_prefill_varlen -- pa_prefill_chunk for a mixed batch: the chunks of num_seqs
 * sequences, stacked row-wise, in one call [page832 §6: the vendor kernel's
 * cu_seqlens_q / seqused_k / block_table interface].  Sequence b's chunk is rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q and out; they are the LAST
 * q_len_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] tokens of the sequence's seq_lens_k[b]
 * keys, i.e. row i of the chunk sits at absolute position seq_lens_k[b] - q_len_b + i and,
 * with causal != 0, sees keys 0 .. that position; otherwise all seq_lens_k[b] keys.  The
 * chunk's own K/V must already be in the cache.
 *   q, out         BF16 [cu_seqlens_q[num_seqs], num_q_heads, head_dim], contiguous
 *   block_table    int32 [num_seqs, bt_stride], device; row b for sequence b; bt_stride
 *                  >= ceil(seq_lens_k[b] / block_size) for every b
 *   cu_seqlens_q   int32 [num_seqs + 1], HOST, cu_seqlens_q[0] = 0, non-decreasing
 *   seq_lens_k     int32 [num_seqs], HOST, each >= its chunk's rows
 *   workspace      as for pa_prefill_chunk, sized by pa_prefill_varlen_workspace_size
 * The lengths are host arrays because the library plans the work on the host (which
 * CTA runs which 128-row tile of which sequence and head).  Sequences with an empty chunk
 * are skipped; more than 32 non-empty chunks run as several launches, 32 chunks each,
 * one after another on the stream.  num_seqs == 0 or no rows at all is a no-op.
 */
size_t pa_prefill_varlen_workspace_size(const int32_t *cu_seqlens_q, const int32_t *seq_lens_k,
                                        int num_seqs, int causal, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size);

int pa_prefill_varlen(const pa_bf16 *q, const pa_bf16 *k_cache, const pa_bf16 *v_cache,
                      int64_t page_stride, int64_t num_pages, const int32_t *block_table,
                      int64_t bt_stride, const int32_t *cu_seqlens_q, const int32_t *seq_lens_k,
                      int num_seqs, int causal, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, float scale, pa_bf16 *out, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * pa_prefill_plan -- the static work assignment pa_prefill_chunk uses without a workspace
 * (whole items only), for inspection.  The pages have no counterpart: it describes how
 * this library spreads one chunk over the GPU, not what the attention computes.  Host
 * only; touches no device.
 *
 * Work items run from the chunk's last query tile (the longest under causal masking) to
 * its first; within a tile, one item per query head: item i is the 128 query rows of tile
 * ceil(q_len / 128) - 1 - i / num_q_heads of head i % num_q_heads.  One exception: the
 * last tile, of r rows, runs as items of hp query heads, hp the largest divisor of
 * G = num_q_heads / num_kv_heads with hp * r <= 128, when that is more than 1 (items
 * 0 .. num_q_heads / hp - 1, then the other tiles as above, shifted): packed item j holds
 * the r rows of query heads j*hp .. j*hp + hp - 1, which share one KV head (its row x is
 * tile row x / hp of query head j*hp + x % hp).  An item's cost is the number of 256-key
 * tiles it reads (64-key page-local blocks, four per tile) plus one.  pa_prefill_chunk
 * runs min(num_ctas, items) persistent CTAs, with num_ctas = the device's SM count.
 *   cta_of_item  int32 [items] (host) or NULL: the CTA each item runs on
 *   num_items    (host, or NULL) the item count
 *   max_cost     (host, or NULL) the largest per-CTA total cost
 * Returns PA_ERR_INVALID_ARG for bad sizes (num_q_heads not a multiple of num_kv_heads
 * included), PA_ERR_UNSUPPORTED when the problem has more than 6144 items or 256 CTAs
 * (pa_prefill_chunk then walks the items in a fixed order).
 */
int pa_prefill_plan(int q_len, int q_start, int causal, int num_q_heads, int num_kv_heads,
                    int block_size, int num_ctas, int32_t *cta_of_item, int *num_items,
                    int *max_cost);

/*
 * pa_prefill_plan_pieces -- the plan pa_prefill_chunk uses when given a workspace of
 * pa_prefill_workspace_size bytes, for inspection (host only; the pages have no
 * counterpart).  cta_of_item[i] (num_items entries) is the CTA that runs item i whole, or
 * -1 for an item split into pieces: piece p covers 256-key tiles [piece_tile_begin[p],
 * piece_tile_end[p]) of item piece_item[p] (items numbered as for pa_prefill_plan) and
 * runs on CTA piece_cta[p].  *num_pieces is 0 when no split pays (the plan is then that
 * of pa_prefill_plan); *max_cost is the busiest CTA's cost (tiles + 1 per whole item,
 * tiles + 2 per piece).  Any array may be NULL; the piece arrays hold max_pieces entries
 * (PA_ERR_INVALID_ARG if the plan has more pieces).
 */
int pa_prefill_plan_pieces(int q_len, int q_start, int causal, int num_q_heads,
                           int num_kv_heads, int block_size, int num_ctas, int max_pieces,
                           int32_t *cta_of_item,
                           int32_t *piece_item, int32_t *piece_tile_begin,
                           int32_t *piece_tile_end, int32_t *piece_cta, int *num_items,
                           int *num_pieces, int *max_cost);

/*
 * pa_copy -- copies `bytes` bytes from src to dst with a kernel on `stream` (ordered like
 * the library's other launches, and capturable into a CUDA graph).  Each address may be
 * device memory or page-locked host memory (cudaHostAlloc / cudaMallocHost / registered
 * with cudaHostRegister), which the kernel reaches through its device mapping; for a
 * step's few kilobytes of inputs and results this avoids a copy-engine node, whose fixed
 * cost on this system is several microseconds.  Both addresses must be 16-byte aligned
 * and bytes a multiple of 16; the ranges must not overlap.  Returns PA_ERR_INVALID_ARG
 * for a NULL or misaligned pointer, a bad size, or an address the device cannot reach
 * (pageable host memory); bytes == 0 is a no-op.
 */
int pa_copy(void *dst, const void *src, size_t bytes, void *stream);

/*
 * pa_get_device_errors -- waits for `stream`, then returns in *bits the device error
 * word of the current device (PA_DEVERR_* bits set by any call since the last clear)
 * and, if clear != 0, resets it to zero.
 * Returns PA_ERR_TIMEOUT (with *bits filled in) when PA_DEVERR_TIMEOUT is set: a wait
 * inside a kernel gave up after its limit (2 s), so some outputs of the calls since the
 * last clear are incomplete.  The kernel that gave up let every copy it had started
 * land, freed what it held and returned, so the context stays usable; a decode split
 * that gave up contributes nothing to its outputs, a prefill CTA that gave up leaves its
 * remaining rows unwritten.  PA_OK otherwise (PA_ERR_CUDA if the stream or the read
 * failed).
 */
int pa_get_device_errors(unsigned int *bits, int clear, void *stream);

/*
 * pa_set_kernel_events -- measurement hook.  The next pa_decode, pa_decode_append,
 * pa_prefill_chunk or pa_prefill_varlen call made by this host thread records `start` on
 * its stream immediately before it launches its main kernel (the split-context decode
 * kernel, or the prefill kernel) and `stop` immediately after that launch, then forgets
 * both.  Inside a stream capture the records carry cudaEventRecordExternal, so they
 * become event record nodes that every replay of the graph records.  The arguments are
 * cudaEvent_t handles owned by the caller; passing NULL, NULL cancels a pending hook.
 * Both or neither must be NULL.
 */
int pa_set_kernel_events(void *start, void *stop);

/* Human-readable name of a pa_status value (static storage). */
const char *pa_status_string(int status);

/* Build identity: target architecture, kernel tile sizes and compiler version. */
const char *pa_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
