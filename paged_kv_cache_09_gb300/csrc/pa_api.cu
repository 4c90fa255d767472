// pa_api.cu -- the C ABI declared in include/pa.h: host-side argument checks, TMA
// descriptor construction, the device error word and kernel dispatch.  No call
// allocates device memory; every call is asynchronous on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

// The library's device error word (one per device that loads the library).
__device__ unsigned int g_pa_device_errors;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    uintptr_t ctx = 0;  // the context these facts belong to (0: not looked up)
    int num_sms = 0;
    unsigned *err = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Per-device facts, looked up with the device current, again whenever the device's
// context has changed (the error word's address belongs to one context's module).
int device_info(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    const uintptr_t ctx = pa::current_context();  // 0 until the thread has a context
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (ctx == 0 || d.ctx != ctx) {
        int sms = 0;
        void *ptr = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PA_ERR_CUDA;
        if (cudaGetSymbolAddress(&ptr, g_pa_device_errors) != cudaSuccess) return PA_ERR_CUDA;
        d.num_sms = sms;
        d.err = static_cast<unsigned *>(ptr);
        d.ctx = pa::current_context();  // the symbol lookup made the device's context current
    }
    *out = d;
    return PA_OK;
}

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so the library
// does not link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// K or V cache as a 4-D tensor {D, Hkv, rows, pages}; boxes of 64 dims x 1 head x
// box_rows tokens x 1 page, 128-byte swizzle.  rows < block_size cuts the page short
// (used for the last page of a sequence).
bool make_cache_map(CUtensorMap *m, const void *base, int head_dim, int num_kv_heads,
                    int rows, int64_t num_pages, int64_t page_stride, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads, (cuuint64_t)rows,
                          (cuuint64_t)num_pages};
    cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_kv_heads * head_dim * 2,
                             (cuuint64_t)page_stride * 2};
    cuuint32_t box[4] = {(cuuint32_t)pa::kChunkElems, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K or V cache as a 5-D view {64 dims, rows, D / 64 chunks, Hkv, pages} for the decode:
// one box of 64 dims x 16 rows x all D / 64 chunks x 1 head x 1 page holds a whole
// 16-token tile of one KV head, laid out [chunk][row][128 B] with the 128-byte swizzle,
// the same bytes four 64-dim boxes of the {D, Hkv, rows, pages} view would give.  The
// dims are not in stride order (rows step Hkv * D elements, chunks 64); the tensor map
// takes each dim's stride as given.
bool make_tile_map(CUtensorMap *m, const void *base, int head_dim, int num_kv_heads,
                   int rows, int64_t num_pages, int64_t page_stride, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int chunks = head_dim / pa::kChunkElems;
    cuuint64_t dims[5] = {(cuuint64_t)pa::kChunkElems, (cuuint64_t)rows, (cuuint64_t)chunks,
                          (cuuint64_t)num_kv_heads, (cuuint64_t)num_pages};
    cuuint64_t strides[4] = {(cuuint64_t)num_kv_heads * head_dim * 2,
                             (cuuint64_t)pa::kChunkElems * 2, (cuuint64_t)head_dim * 2,
                             (cuuint64_t)page_stride * 2};
    cuuint32_t box[5] = {(cuuint32_t)pa::kChunkElems, (cuuint32_t)box_rows, (cuuint32_t)chunks,
                         1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Query rows [q_len, Hq, D] as {D, Hq, q_len}; boxes of 64 dims x box_heads heads x
// box_rows rows (in shared memory: box_heads * box_rows rows of 128 bytes, heads fastest).
bool make_rows_map(CUtensorMap *m, const void *base, int head_dim, int num_heads, int rows,
                   int box_heads, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_heads * head_dim * 2};
    cuuint32_t box[3] = {(cuuint32_t)pa::kChunkElems, (cuuint32_t)box_heads,
                         (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A small per-thread cache of decode descriptors: encoding costs host time and the
// same cache pointers come back call after call.
struct MapKey {
    const void *base;
    int head_dim, num_kv_heads, rows, box_rows;
    int64_t num_pages, page_stride;
    bool operator==(const MapKey &o) const {
        return base == o.base && head_dim == o.head_dim && num_kv_heads == o.num_kv_heads &&
               rows == o.rows && box_rows == o.box_rows && num_pages == o.num_pages &&
               page_stride == o.page_stride;
    }
};

bool cached_cache_map(CUtensorMap *m, const MapKey &k) {
    struct Entry {
        MapKey key;
        CUtensorMap map;
        bool used;
    };
    thread_local Entry entries[16] = {};
    thread_local int next = 0;
    for (auto &e : entries)
        if (e.used && e.key == k) {
            *m = e.map;
            return true;
        }
    if (!make_tile_map(m, k.base, k.head_dim, k.num_kv_heads, k.rows, k.num_pages,
                       k.page_stride, k.box_rows))
        return false;
    entries[next] = Entry{k, *m, true};
    next = (next + 1) % 16;
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Pending measurement events of this host thread (pa_set_kernel_events).
thread_local cudaEvent_t t_ev_start = nullptr, t_ev_stop = nullptr;

void take_kernel_events(cudaEvent_t *start, cudaEvent_t *stop) {
    *start = t_ev_start;
    *stop = t_ev_stop;
    t_ev_start = t_ev_stop = nullptr;
}

bool diag_enabled() {
    static int on = -1;
    if (on < 0) {
        const char *v = getenv("PA_DIAG");
        on = (v && v[0] && v[0] != '0') ? 1 : 0;
    }
    return on == 1;
}

// Checks shared by the two attention calls.
int check_attention_shape(int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int64_t num_pages, int64_t page_stride) {
    if (num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 ||
        num_pages < 1)
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
    if (num_q_heads > 65535 || num_kv_heads > 65535) return PA_ERR_INVALID_ARG;
    if (page_stride < (int64_t)block_size * num_kv_heads * head_dim) return PA_ERR_INVALID_ARG;
    if ((page_stride * 2) % 16) return PA_ERR_INVALID_ARG;
    if (num_pages > 0x7fffffffLL) return PA_ERR_INVALID_ARG;
    if (head_dim != pa::kHeadDim) return PA_ERR_UNSUPPORTED;
    const int group = num_q_heads / num_kv_heads;
    if (group > pa::kDecMaxGroup) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

}  // namespace

extern "C" {

const char *pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
        default: return "PA_ERR_UNKNOWN";
    }
}

// The address through which the device reaches p: p itself for device and managed
// memory, the device mapping of page-locked host memory; false for memory the device
// cannot reach (pageable host memory) or an unknown address.
static bool device_address(const void *p, const void **dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of the query
        return false;
    }
    switch (a.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged: *dev = p; return true;
        case cudaMemoryTypeHost:
            if (!a.devicePointer) return false;
            *dev = a.devicePointer;
            return true;
        default: return false;
    }
}

int pa_copy(void *dst, const void *src, size_t bytes, void *stream) {
    if (bytes == 0) return PA_OK;
    if (!dst || !src || (bytes & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u) ||
        (reinterpret_cast<uintptr_t>(src) & 15u) || bytes > ((size_t)1 << 40))
        return PA_ERR_INVALID_ARG;
    const void *d = nullptr, *s = nullptr;
    if (!device_address(dst, &d) || !device_address(src, &s)) return PA_ERR_INVALID_ARG;
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(d), s0 = reinterpret_cast<uintptr_t>(s);
    if (d0 < s0 + bytes && s0 < d0 + bytes) return PA_ERR_INVALID_ARG;  // overlapping ranges
    return pa::launch_copy(const_cast<void *>(d), s, bytes, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

const char *pa_build_info(void) {
    static char buf[256];
    static std::once_flag once;
    std::call_once(once, [] {
        snprintf(buf, sizeof buf,
                 "paged_kv_cache_09_gb300: sm_103a; decode tiles of %d tokens, two per stage, "
                 "%d warps x %d stages (splits <= %d tiles) or %d x %d; prefill %dx%d tcgen05 "
                 "tiles; nvcc %d.%d",
                 pa::kDecTile, pa::kDecShortConsumers, pa::kDecShortStages, pa::kDecShortTiles,
                 pa::kDecLongConsumers, pa::kDecLongStages, pa::kPfQRows, pa::kPfKvTile,
                 __CUDACC_VER_MAJOR__, __CUDACC_VER_MINOR__);
    });
    return buf;
}

int pa_slot_mapping(const int32_t *positions, const int32_t *seq_idx,
                    const int32_t *block_table, int num_seqs, int64_t bt_stride,
                    int max_blocks, int num_tokens, int block_size, int64_t *slot_mapping,
                    void *stream) {
    if (num_tokens < 0 || block_size < 1 || max_blocks < 1 || bt_stride < max_blocks ||
        num_seqs < 1)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!positions || !block_table || !slot_mapping) return PA_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (int rc = device_info(&dev)) return rc;
    cudaError_t e = pa::launch_slot_mapping(positions, seq_idx, block_table, num_seqs,
                                            bt_stride, max_blocks, num_tokens, block_size,
                                            slot_mapping,
                                            dev.err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_decode_input_prep(const int32_t *positions, const int32_t *sampled_ids,
                         int32_t *input_ids, int32_t *seq_lens, int32_t *query_start_loc,
                         int num_seqs, int num_groups, const int32_t *const *block_tables,
                         const int64_t *bt_strides, const int *max_blocks,
                         const int *block_sizes, int64_t *const *slot_mappings, void *stream) {
    if (num_seqs < 0 || num_groups < 1 || num_groups > pa::kPrepMaxGroups)
        return PA_ERR_INVALID_ARG;
    if (!block_tables || !bt_strides || !max_blocks || !block_sizes || !slot_mappings)
        return PA_ERR_INVALID_ARG;
    if ((sampled_ids == nullptr) != (input_ids == nullptr)) return PA_ERR_INVALID_ARG;
    pa::PrepArgs a = {};
    for (int g = 0; g < num_groups; ++g) {
        if (!block_tables[g] || !slot_mappings[g] || block_sizes[g] < 1 || max_blocks[g] < 1 ||
            bt_strides[g] < max_blocks[g])
            return PA_ERR_INVALID_ARG;
        a.g[g] = pa::PrepGroup{block_tables[g], bt_strides[g], max_blocks[g], block_sizes[g],
                               slot_mappings[g]};
    }
    if (num_seqs == 0) return PA_OK;
    if (!positions) return PA_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (int rc = device_info(&dev)) return rc;
    a.positions = positions;
    a.sampled_ids = sampled_ids;
    a.input_ids = input_ids;
    a.seq_lens = seq_lens;
    a.query_start_loc = query_start_loc;
    a.num_seqs = num_seqs;
    a.num_groups = num_groups;
    a.err = dev.err;
    return pa::launch_decode_input_prep(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int pa_reshape_and_cache(const pa_bf16 *key, const pa_bf16 *value, pa_bf16 *k_cache,
                         pa_bf16 *v_cache, int64_t page_stride, int64_t num_pages,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, void *stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_pages < 1)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (row % 8 || row > 0x7fffffffLL) return PA_ERR_INVALID_ARG;
    if (page_stride < row * block_size || (page_stride * 2) % 16) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (int rc = device_info(&dev)) return rc;
    cudaError_t e = pa::launch_reshape_and_cache(key, value, k_cache, v_cache, page_stride,
                                                 num_pages, slot_mapping, num_tokens, (int)row,
                                                 block_size, dev.err,
                                                 static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_seq_len) {
    if (num_seqs < 1 || num_q_heads < 1 || num_kv_heads < 1 || head_dim != pa::kHeadDim ||
        block_size < 1 || max_seq_len < 1 || num_q_heads % num_kv_heads)
        return 0;
    DeviceInfo dev;
    if (device_info(&dev)) return 0;
    const pa::DecodePlan plan =
        pa::plan_decode(num_seqs, num_kv_heads, block_size, max_seq_len, dev.num_sms);
    return pa::decode_workspace_bytes(num_seqs, num_q_heads, plan);
}

// pa_decode and pa_decode_append.  fused: the newest tokens are written (new_k and new_v
// set); their slots are new_slots when given, else derived in the kernel and stored to
// slot_out (when set).
static int decode_impl(const pa_bf16 *q, const pa_bf16 *k_cache, const pa_bf16 *v_cache,
                       int64_t page_stride, int64_t num_pages, const int32_t *block_table,
                       int64_t bt_stride, const int32_t *seq_lens, int num_seqs,
                       int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, float scale, pa_bf16 *out, void *workspace,
                       size_t workspace_bytes, bool fused, const pa_bf16 *new_k,
                       const pa_bf16 *new_v, const int64_t *new_slots, int64_t *slot_out,
                       void *stream) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !workspace)
        return PA_ERR_INVALID_ARG;
    if (num_seqs < 1 || num_seqs > 65535 || max_seq_len < 1) return PA_ERR_INVALID_ARG;
    if (int rc = check_attention_shape(num_q_heads, num_kv_heads, head_dim, block_size,
                                       num_pages, page_stride))
        return rc;
    const int64_t max_blocks = ((int64_t)max_seq_len + block_size - 1) / block_size;
    if (bt_stride < max_blocks) return PA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PA_ERR_INVALID_ARG;
    if (fused && (!new_k || !new_v || !aligned16(new_k) || !aligned16(new_v)))
        return PA_ERR_INVALID_ARG;

    // The output may be page-locked host memory (the combine then writes the step's
    // result straight to the host); pageable or unknown memory is refused.
    const void *out_dev = nullptr;
    if (!device_address(out, &out_dev)) return PA_ERR_INVALID_ARG;

    DeviceInfo dev;
    if (int rc = device_info(&dev)) return rc;
    const pa::DecodePlan plan =
        pa::plan_decode(num_seqs, num_kv_heads, block_size, max_seq_len, dev.num_sms);
    if (workspace_bytes < pa::decode_workspace_bytes(num_seqs, num_q_heads, plan))
        return PA_ERR_INVALID_ARG;

    // Tile boxes: one 16-row box per tile of K or V (two tiles of a stage may lie in
    // different pages).
    CUtensorMap maps[2];
    if (!cached_cache_map(&maps[0], MapKey{k_cache, head_dim, num_kv_heads, block_size,
                                           pa::kDecTile, num_pages, page_stride}) ||
        !cached_cache_map(&maps[1], MapKey{v_cache, head_dim, num_kv_heads, block_size,
                                           pa::kDecTile, num_pages, page_stride}))
        return PA_ERR_CUDA;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    pa::DecodeArgs a;
    a.k_cache_w = fused ? const_cast<pa_bf16 *>(k_cache) : nullptr;
    a.v_cache_w = fused ? const_cast<pa_bf16 *>(v_cache) : nullptr;
    a.new_k = fused ? new_k : nullptr;
    a.new_v = fused ? new_v : nullptr;
    a.new_slots = fused ? new_slots : nullptr;
    a.slot_out = fused && !new_slots ? slot_out : nullptr;
    a.page_stride = page_stride;
    a.q = q;
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.max_seq_len = max_seq_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = num_q_heads / num_kv_heads;
    a.block_size = block_size;
    a.num_pages = num_pages;
    a.scale = scale;
    a.out = static_cast<uint16_t *>(const_cast<void *>(out_dev));
    a.workspace = workspace;
    a.err = dev.err;
    take_kernel_events(&a.ev_start, &a.ev_stop);
    if (diag_enabled())
        fprintf(stderr, "[pa] decode: seqs=%d max_seq_len=%d bs=%d splits=%d tiles/split=%d\n",
                num_seqs, max_seq_len, block_size, plan.num_splits, plan.tiles_per_split);
    return pa::launch_decode(maps, a, plan, st) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_decode(const pa_bf16 *q, const pa_bf16 *k_cache, const pa_bf16 *v_cache,
              int64_t page_stride, int64_t num_pages, const int32_t *block_table,
              int64_t bt_stride, const int32_t *seq_lens, int num_seqs, int max_seq_len,
              int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
              pa_bf16 *out, void *workspace, size_t workspace_bytes, const pa_bf16 *new_k,
              const pa_bf16 *new_v, const int64_t *new_slots, void *stream) {
    const int nfused = (new_k != nullptr) + (new_v != nullptr) + (new_slots != nullptr);
    if (nfused != 0 && nfused != 3) return PA_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, page_stride, num_pages, block_table, bt_stride,
                       seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                       block_size, scale, out, workspace, workspace_bytes, nfused == 3, new_k,
                       new_v, new_slots, nullptr, stream);
}

int pa_decode_append(const pa_bf16 *q, pa_bf16 *k_cache, pa_bf16 *v_cache, int64_t page_stride,
                     int64_t num_pages, const int32_t *block_table, int64_t bt_stride,
                     const int32_t *seq_lens, int num_seqs, int max_seq_len, int num_q_heads,
                     int num_kv_heads, int head_dim, int block_size, float scale, pa_bf16 *out,
                     void *workspace, size_t workspace_bytes, const pa_bf16 *new_k,
                     const pa_bf16 *new_v, int64_t *slot_mapping, void *stream) {
    if (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) return PA_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, page_stride, num_pages, block_table, bt_stride,
                       seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                       block_size, scale, out, workspace, workspace_bytes, true, new_k, new_v,
                       nullptr, slot_mapping, stream);
}

// The schedule of one prefill launch over nseq chunks: with split items when the
// workspace (workspace_bytes; 0 for none) holds their pieces' partials.
static bool prefill_schedule(const pa::PrefillSeq *seqs, int nseq, int causal, int num_q_heads,
                             int group, int block_size, int num_sms, size_t workspace_bytes,
                             pa::PrefillSchedule *sched) {
    int q_lens[pa::kPfMaxSeqs], q_starts[pa::kPfMaxSeqs];
    for (int b = 0; b < nseq; ++b) {
        q_lens[b] = seqs[b].q_len;
        q_starts[b] = seqs[b].q_start;
    }
    if (workspace_bytes >= pa::kPfSlotBytes &&
        pa::plan_prefill(nseq, q_lens, q_starts, causal, num_q_heads, group, block_size, num_sms,
                         true, sched, nullptr) &&
        (size_t)sched->num_pieces * pa::kPfSlotBytes <= workspace_bytes)
        return true;
    return pa::plan_prefill(nseq, q_lens, q_starts, causal, num_q_heads, group, block_size,
                            num_sms, false, sched, nullptr);
}

// One prefill launch over 1 .. kPfMaxSeqs chunks whose rows lie in q / out of total_q rows.
static int prefill_launch(const pa_bf16 *q, int total_q, const pa_bf16 *k_cache,
                          const pa_bf16 *v_cache, int64_t page_stride, int64_t num_pages,
                          const int32_t *block_table, int64_t bt_stride,
                          const pa::PrefillSeq *seqs, int nseq, int causal, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, float scale,
                          pa_bf16 *out, void *workspace, size_t workspace_bytes,
                          const DeviceInfo &dev, cudaEvent_t ev_start, cudaEvent_t ev_stop,
                          cudaStream_t stream) {
    constexpr int kM = 3 + pa::kPfMaxPackMaps;  // index of the first per-sequence map
    CUtensorMap maps[kM + 2 * pa::kPfMaxSeqs];
    const int group = num_q_heads / num_kv_heads;
    if (!make_rows_map(&maps[0], q, head_dim, num_q_heads, total_q, 1, pa::kPfQRows))
        return PA_ERR_CUDA;
    // Q for packed items: one map per divisor hp > 1 of the group, largest first.
    int npack = 0;
    for (int hp = group; hp > 1 && npack < pa::kPfMaxPackMaps; --hp)
        if (group % hp == 0 &&
            !make_rows_map(&maps[1 + npack++], q, head_dim, num_q_heads, total_q, hp,
                           pa::kPfQRows / hp))
            return PA_ERR_CUDA;
    for (int i = npack; i < pa::kPfMaxPackMaps; ++i) maps[1 + i] = maps[0];
    if (!make_cache_map(&maps[kM - 2], k_cache, head_dim, num_kv_heads, block_size, num_pages,
                        page_stride, pa::kPfBlock) ||
        !make_cache_map(&maps[kM - 1], v_cache, head_dim, num_kv_heads, block_size, num_pages,
                        page_stride, pa::kPfBlock))
        return PA_ERR_CUDA;
    for (int b = 0; b < nseq; ++b) {
        // The sequence's last page is read through maps whose rows end at its last token,
        // so rows past it come back as zeros.
        const int seq_len_k = seqs[b].q_start + seqs[b].q_len;
        const int last_rows = seq_len_k - ((seq_len_k - 1) / block_size) * block_size;
        if (!make_cache_map(&maps[kM + 2 * b], k_cache, head_dim, num_kv_heads, last_rows,
                            num_pages, page_stride, pa::kPfBlock) ||
            !make_cache_map(&maps[kM + 1 + 2 * b], v_cache, head_dim, num_kv_heads, last_rows,
                            num_pages, page_stride, pa::kPfBlock))
            return PA_ERR_CUDA;
    }
    // The static work assignment (cached per shape); problems too large for its arrays
    // run without one.
    static thread_local pa::PrefillSchedule sched;
    const bool planned = prefill_schedule(seqs, nseq, causal, num_q_heads, group, block_size,
                                          dev.num_sms, workspace ? workspace_bytes : 0, &sched);
    pa::PrefillArgs a;
    a.sched = planned ? &sched : nullptr;
    a.workspace = workspace;
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.num_seqs = nseq;
    a.seqs = seqs;
    a.causal = causal;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = group;
    a.block_size = block_size;
    a.num_pages = num_pages;
    a.scale = scale;
    a.out = out;
    a.err = dev.err;
    a.num_sms = dev.num_sms;
    a.ev_start = ev_start;
    a.ev_stop = ev_stop;
    if (diag_enabled())
        fprintf(stderr, "[pa] prefill: %d chunk(s), first q_len=%d q_start=%d causal=%d bs=%d\n",
                nseq, seqs[0].q_len, seqs[0].q_start, causal, block_size);
    return pa::launch_prefill(maps, a, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_prefill_workspace_size(int q_len, int q_start, int causal, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size) {
    if (q_len < 1 || q_start < 0 || (int64_t)q_start + q_len > 0x7fffffffLL ||
        num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads ||
        head_dim != pa::kHeadDim || block_size < 1)
        return 0;
    DeviceInfo dev;
    if (device_info(&dev)) return 0;
    const pa::PrefillSeq seq{0, q_len, q_start, 0};
    static thread_local pa::PrefillSchedule sched;
    if (!prefill_schedule(&seq, 1, causal ? 1 : 0, num_q_heads, num_q_heads / num_kv_heads,
                          block_size, dev.num_sms,
                          (size_t)pa::kPfMaxPieces * pa::kPfSlotBytes, &sched))
        return 0;
    return (size_t)sched.num_pieces * pa::kPfSlotBytes;
}

int pa_prefill_chunk(const pa_bf16 *q, const pa_bf16 *k_cache, const pa_bf16 *v_cache,
                     int64_t page_stride, int64_t num_pages, const int32_t *block_table,
                     int q_len, int q_start, int causal, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, float scale, pa_bf16 *out, void *workspace,
                     size_t workspace_bytes, void *stream) {
    if (!q || !k_cache || !v_cache || !block_table || !out) return PA_ERR_INVALID_ARG;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PA_ERR_INVALID_ARG;
    if (q_len < 1 || q_start < 0 || (int64_t)q_start + q_len > 0x7fffffffLL)
        return PA_ERR_INVALID_ARG;
    if (int rc = check_attention_shape(num_q_heads, num_kv_heads, head_dim, block_size,
                                       num_pages, page_stride))
        return rc;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return PA_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (int rc = device_info(&dev)) return rc;
    cudaEvent_t e0, e1;
    take_kernel_events(&e0, &e1);
    const pa::PrefillSeq seq{0, q_len, q_start, 0};
    return prefill_launch(q, q_len, k_cache, v_cache, page_stride, num_pages, block_table, 0,
                          &seq, 1, causal ? 1 : 0, num_q_heads, num_kv_heads, head_dim,
                          block_size, scale, out, workspace, workspace ? workspace_bytes : 0, dev,
                          e0, e1, static_cast<cudaStream_t>(stream));
}

// The non-empty chunks of a mixed batch, in launch order; false for bad lengths.
static bool varlen_chunks(const int32_t *cu_seqlens_q, const int32_t *seq_lens_k, int num_seqs,
                          std::vector<pa::PrefillSeq> *seqs) {
    if (num_seqs < 0 || !cu_seqlens_q || (num_seqs > 0 && !seq_lens_k) || cu_seqlens_q[0] != 0)
        return false;
    for (int b = 0; b < num_seqs; ++b) {
        const int64_t ql = (int64_t)cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        if (ql < 0 || seq_lens_k[b] < 0 || ql > seq_lens_k[b]) return false;
        if (ql > 0) seqs->push_back(pa::PrefillSeq{cu_seqlens_q[b], (int)ql, seq_lens_k[b] - (int)ql, b});
    }
    return true;
}

size_t pa_prefill_varlen_workspace_size(const int32_t *cu_seqlens_q, const int32_t *seq_lens_k,
                                        int num_seqs, int causal, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size) {
    std::vector<pa::PrefillSeq> seqs;
    if (!varlen_chunks(cu_seqlens_q, seq_lens_k, num_seqs, &seqs) || num_q_heads < 1 ||
        num_kv_heads < 1 || num_q_heads % num_kv_heads || head_dim != pa::kHeadDim ||
        block_size < 1)
        return 0;
    DeviceInfo dev;
    if (device_info(&dev)) return 0;
    static thread_local pa::PrefillSchedule sched;
    size_t need = 0;
    const int n = (int)seqs.size();
    for (int s0 = 0; s0 < n; s0 += pa::kPfMaxSeqs) {
        const int cnt = std::min(pa::kPfMaxSeqs, n - s0);
        if (prefill_schedule(&seqs[s0], cnt, causal ? 1 : 0, num_q_heads,
                             num_q_heads / num_kv_heads, block_size,
                             dev.num_sms, (size_t)pa::kPfMaxPieces * pa::kPfSlotBytes, &sched))
            need = std::max(need, (size_t)sched.num_pieces * pa::kPfSlotBytes);
    }
    return need;
}

int pa_prefill_varlen(const pa_bf16 *q, const pa_bf16 *k_cache, const pa_bf16 *v_cache,
                      int64_t page_stride, int64_t num_pages, const int32_t *block_table,
                      int64_t bt_stride, const int32_t *cu_seqlens_q, const int32_t *seq_lens_k,
                      int num_seqs, int causal, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, float scale, pa_bf16 *out, void *workspace,
                      size_t workspace_bytes, void *stream) {
    if (num_seqs < 0 || !cu_seqlens_q || (num_seqs > 0 && !seq_lens_k)) return PA_ERR_INVALID_ARG;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PA_ERR_INVALID_ARG;
    if (cu_seqlens_q[0] != 0) return PA_ERR_INVALID_ARG;
    int64_t max_pages = 0;
    for (int b = 0; b < num_seqs; ++b) {
        const int64_t ql = (int64_t)cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        if (ql < 0 || seq_lens_k[b] < 0 || ql > seq_lens_k[b]) return PA_ERR_INVALID_ARG;
        if (block_size >= 1)
            max_pages = std::max<int64_t>(max_pages, (seq_lens_k[b] + block_size - 1) / block_size);
    }
    const int total_q = num_seqs > 0 ? cu_seqlens_q[num_seqs] : 0;
    if (int rc = check_attention_shape(num_q_heads, num_kv_heads, head_dim, block_size,
                                       num_pages, page_stride))
        return rc;
    if (total_q == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_table || !out || bt_stride < max_pages)
        return PA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return PA_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (int rc = device_info(&dev)) return rc;
    cudaEvent_t e0, e1;
    take_kernel_events(&e0, &e1);
    // The non-empty chunks, kPfMaxSeqs per launch (each launch spreads its chunks over all
    // SMs; the launches run back to back on the stream, and a later one reuses the
    // workspace only after the one before has been merged).
    std::vector<pa::PrefillSeq> seqs;
    varlen_chunks(cu_seqlens_q, seq_lens_k, num_seqs, &seqs);
    const int n = (int)seqs.size();
    for (int s0 = 0; s0 < n; s0 += pa::kPfMaxSeqs) {
        const int cnt = std::min(pa::kPfMaxSeqs, n - s0);
        if (int rc = prefill_launch(q, total_q, k_cache, v_cache, page_stride, num_pages,
                                    block_table, bt_stride, &seqs[s0], cnt, causal ? 1 : 0,
                                    num_q_heads, num_kv_heads, head_dim, block_size, scale, out,
                                    workspace, workspace ? workspace_bytes : 0, dev,
                                    s0 == 0 ? e0 : nullptr,
                                    s0 + cnt == n ? e1 : nullptr,
                                    static_cast<cudaStream_t>(stream)))
            return rc;
    }
    return PA_OK;
}

int pa_set_kernel_events(void *start, void *stop) {
    if ((start == nullptr) != (stop == nullptr)) return PA_ERR_INVALID_ARG;
    t_ev_start = static_cast<cudaEvent_t>(start);
    t_ev_stop = static_cast<cudaEvent_t>(stop);
    return PA_OK;
}

int pa_get_device_errors(unsigned int *bits, int clear, void *stream) {
    if (!bits) return PA_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (int rc = device_info(&dev)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, dev.err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PA_ERR_CUDA;
    if (clear && cudaMemset(dev.err, 0, sizeof v) != cudaSuccess) return PA_ERR_CUDA;
    *bits = v;
    return (v & pa::kErrTimeout) ? PA_ERR_TIMEOUT : PA_OK;
}

#ifdef PA_TEST_HOOKS
int pa_test_hook(int decode_skip_stage, int prefill_skip_unit, int decode_consumer_delay_ns) {
    if (decode_consumer_delay_ns < 0 || decode_consumer_delay_ns > 1000000) return PA_ERR_INVALID_ARG;
    if (pa::set_decode_test_hook(decode_skip_stage, decode_consumer_delay_ns) != cudaSuccess ||
        pa::set_prefill_test_hook(prefill_skip_unit) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}
#endif

}  // extern "C"
