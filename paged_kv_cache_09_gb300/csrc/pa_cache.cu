// pa_cache.cu -- slot mapping and KV write of new tokens.
//
// Slot mapping follows the input-prep post §3.2 (slot = block_table[pos / bs] * bs +
// pos % bs) and §5 (computed on the device from the resident block table, one launch).
// The KV write copies each token's [Hkv, D] BF16 row, bit for bit, to its slot in the
// page layout of the page832 post §4.  Both are pure integer / byte work.
#include "pa_device.cuh"
#include "pa_internal.h"

#include <atomic>
#include <mutex>

namespace pa {

// Byte copy between two device-accessible ranges (device memory or page-locked host
// memory through its device mapping), 16 bytes per thread and step.
__global__ void __launch_bounds__(256) copy_kernel(const uint4 *__restrict__ src,
                                                   uint4 *__restrict__ dst, int64_t n16) {
    pdl_wait();  // the source may be written by earlier work on the stream
    pdl_trigger();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream) {
    const int64_t n16 = (int64_t)(bytes / 16);
    const int64_t blocks = (n16 + 255) / 256;
    return launch_pdl(copy_kernel, dim3((unsigned)(blocks < 1024 ? blocks : 1024)), dim3(256),
                      0, stream, static_cast<const uint4 *>(src), static_cast<uint4 *>(dst),
                      n16);
}

// The calling thread's current CUDA context, through the driver entry point the runtime
// hands out (the library does not link libcuda).  0 when there is none or on failure.
uintptr_t current_context() {
    typedef CUresult (*GetCurrentFn)(CUcontext *);
    static GetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<GetCurrentFn>(p);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return 0;
    return reinterpret_cast<uintptr_t>(c);
}

cudaError_t set_smem_once(const void *kernel, int bytes, int slot) {
    // Per (kernel slot, device): the context in which the limit was last raised.  A new
    // context for the device (after cudaDeviceReset the module is loaded afresh and the
    // attribute is gone) raises it again.
    constexpr int kDevices = 64;
    if (slot < 0 || slot >= kSmemSlots) return cudaErrorInvalidValue;
    static std::atomic<uintptr_t> done[kSmemSlots][kDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uintptr_t ctx = current_context();
    if (dev >= kDevices || ctx == 0)
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (done[slot][dev].load(std::memory_order_acquire) == ctx) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[slot][dev].store(ctx, std::memory_order_release);
    return e;
}

// Slot of position pos of sequence s (row s of the block table), or -1: a negative
// position is padding; a logical page past max_blocks, a sequence outside the table or a
// negative table entry gives -1 and sets kErrPosition.
__device__ __forceinline__ int64_t slot_of(int32_t pos, int64_t s, const int32_t *block_table,
                                           int num_seqs, int64_t bt_stride, int max_blocks,
                                           int block_size, unsigned *err) {
    if (pos < 0) return -1;
    const int logical_block = pos / block_size;
    if (logical_block < max_blocks && s >= 0 && s < num_seqs) {
        const int32_t block_number = block_table[s * bt_stride + logical_block];
        if (block_number >= 0) return (int64_t)block_number * block_size + pos % block_size;
    }
    atomicOr(err, kErrPosition);
    return -1;
}

__global__ void slot_mapping_kernel(const int32_t *__restrict__ positions,
                                    const int32_t *__restrict__ seq_idx,
                                    const int32_t *__restrict__ block_table, int num_seqs,
                                    int64_t bt_stride, int max_blocks, int num_tokens,
                                    int block_size,
                                    int64_t *__restrict__ slot_mapping, unsigned *err) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    pdl_wait();
    pdl_trigger();
    if (i >= num_tokens) return;
    slot_mapping[i] = slot_of(positions[i], seq_idx ? seq_idx[i] : 0, block_table, num_seqs,
                              bt_stride, max_blocks, block_size, err);
}

// Decode input preparation (input-prep post §2, §4, §5): grid (sequence blocks, groups)
// of kPrepThreads threads.  The blocks of group 0 also write the step's shared metadata;
// every group writes its own slots from its own block table and block size.  An entry
// with a negative position is padding: seq_lens 0, slot -1, and no query row, so
// query_start_loc is the running count of query rows ([0, 1, 1, ...] for one request in
// padded buffers, as §2 gives it).  Block (0, 0) computes that count for all entries,
// kPrepThreads at a time: a ballot per warp, then the warps' totals in shared memory.
constexpr int kPrepThreads = 128;

__global__ void __launch_bounds__(kPrepThreads) decode_input_prep_kernel(
    const __grid_constant__ PrepArgs a) {
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    const int grp = blockIdx.y;
    pdl_wait();
    pdl_trigger();
    if (grp == 0 && blockIdx.x == 0 && a.query_start_loc) {
        __shared__ int warp_rows[kPrepThreads / 32];
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        if (threadIdx.x == 0) a.query_start_loc[0] = 0;
        int carry = 0;  // query rows of the entries before this round
        for (int base = 0; base < a.num_seqs; base += kPrepThreads) {
            const int e = base + threadIdx.x;
            const bool row = e < a.num_seqs && a.positions[e] >= 0;
            const unsigned b = __ballot_sync(0xffffffffu, row);
            if (lane == 0) warp_rows[w] = __popc(b);
            __syncthreads();
            int before = carry, round = 0;
#pragma unroll
            for (int i = 0; i < kPrepThreads / 32; ++i) {
                before += i < w ? warp_rows[i] : 0;
                round += warp_rows[i];
            }
            // rows of entries base .. e inclusive (lane mask up to and including this lane)
            const unsigned upto = lane == 31 ? 0xffffffffu : (2u << lane) - 1u;
            if (e < a.num_seqs) a.query_start_loc[e + 1] = before + __popc(b & upto);
            __syncthreads();  // warp_rows is rewritten by the next round
            carry += round;
        }
    }
    if (s >= a.num_seqs) return;
    const int32_t pos = a.positions[s];
    if (grp == 0) {
        if (a.input_ids) a.input_ids[s] = a.sampled_ids[s];
        if (a.seq_lens) a.seq_lens[s] = pos >= 0 ? pos + 1 : 0;
    }
    const PrepGroup &g = a.g[grp];
    g.slot_mapping[s] = slot_of(pos, s, g.block_table, a.num_seqs, g.bt_stride, g.max_blocks,
                                g.block_size, a.err);
}

cudaError_t launch_decode_input_prep(const PrepArgs &a, cudaStream_t stream) {
    const dim3 grid((a.num_seqs + kPrepThreads - 1) / kPrepThreads, a.num_groups);
    return launch_pdl(decode_input_prep_kernel, grid, dim3(kPrepThreads), 0, stream, a);
}

cudaError_t launch_slot_mapping(const int32_t *positions, const int32_t *seq_idx,
                                const int32_t *block_table, int num_seqs, int64_t bt_stride,
                                int max_blocks, int num_tokens, int block_size,
                                int64_t *slot_mapping, unsigned *err, cudaStream_t stream) {
    const int threads = 128;
    const int blocks = (num_tokens + threads - 1) / threads;
    return launch_pdl(slot_mapping_kernel, dim3(blocks), dim3(threads), 0, stream, positions,
                      seq_idx, block_table, num_seqs, bt_stride, max_blocks, num_tokens,
                      block_size, slot_mapping, err);
}

// One warp-group per token row pair: each thread moves 16 bytes of K and 16 of V per
// step.  Rows are row_elems BF16 long (Hkv * D, a multiple of 8).
__global__ void __launch_bounds__(128) reshape_and_cache_kernel(
    const uint4 *__restrict__ key, const uint4 *__restrict__ value, uint16_t *k_cache,
    uint16_t *v_cache, int64_t page_stride, int64_t num_pages,
    const int64_t *__restrict__ slot_mapping, int num_tokens, int row_elems, int block_size,
    unsigned *err) {
    const int t = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (t >= num_tokens) return;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;
    const int64_t page = slot / block_size;
    const int64_t offset = slot - page * block_size;
    if (page >= num_pages) {
        if (threadIdx.x == 0) atomicOr(err, kErrSlot);
        return;
    }
    const int64_t dst = page * page_stride + offset * row_elems;  // in BF16 elements
    uint4 *kd = reinterpret_cast<uint4 *>(k_cache + dst);
    uint4 *vd = reinterpret_cast<uint4 *>(v_cache + dst);
    const int vecs = row_elems / 8;
    const uint4 *ks = key + (int64_t)t * vecs;
    const uint4 *vs = value + (int64_t)t * vecs;
    for (int i = threadIdx.x; i < vecs; i += blockDim.x) {
        const uint4 a = __ldg(ks + i);
        const uint4 b = __ldg(vs + i);
        kd[i] = a;
        vd[i] = b;
    }
}

cudaError_t launch_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                                     uint16_t *k_cache, uint16_t *v_cache, int64_t page_stride,
                                     int64_t num_pages, const int64_t *slot_mapping,
                                     int num_tokens, int row_elems, int block_size,
                                     unsigned *err, cudaStream_t stream) {
    return launch_pdl(reshape_and_cache_kernel, dim3(num_tokens), dim3(128), 0, stream,
                      reinterpret_cast<const uint4 *>(key), reinterpret_cast<const uint4 *>(value),
                      k_cache, v_cache, page_stride, num_pages, slot_mapping, num_tokens,
                      row_elems, block_size, err);
}

}  // namespace pa
