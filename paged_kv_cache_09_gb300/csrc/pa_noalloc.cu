// pa_noalloc.cu -- decode without a caller-provided workspace.
//
// pa_decode needs device scratch for its split partials, and expects the caller to
// allocate it.  Some callers cannot: a serving runtime that hands nearly all device
// memory to its KV-cache pool up front and allows no allocation afterwards, or plain C
// code that has no device allocator of its own on the decode path.  For them,
// pa_decode_noalloc runs the same decode with its scratch taken from one fixed
// array that lives in this library's device image.
//
// The array is a file-scope __device__ variable of PA_DECODE_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds one copy of it until the process exits.
// Host code cannot use the array's name as a device address: on the host that name is
// only a stand-in.  So, once per device and with that device current, the first call
// looks up the real device address with cudaGetSymbolAddress, checks the result, and
// keeps it with the context it belongs to.  Later calls on that device reuse it while the
// device's context stays the same, and look it up again after a cudaDeviceReset.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
    uintptr_t ctx;  // the context whose module the address belongs to (0: none yet)
    void *ptr;
};
ScratchAddr g_scratch[kMaxScratchDevices];

// Device address of this device's scratch array.  It is looked up with the device
// current on the first call, and again whenever the device's context has changed (after
// cudaDeviceReset the module, and with it the array, is loaded afresh).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices)
        return PA_ERR_CUDA;
    const uintptr_t ctx = pa::current_context();  // 0 until the thread has a context
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr &a = g_scratch[dev];
    if (ctx == 0 || a.ctx != ctx || !a.ptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr)
            return PA_ERR_CUDA;
        a.ptr = ptr;
        a.ctx = pa::current_context();  // the lookup made the device's context current
    }
    *out = a.ptr;
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_noalloc(const pa_bf16 *q, const pa_bf16 *k_cache,
                                 const pa_bf16 *v_cache, int64_t page_stride, int64_t num_pages,
                                 const int32_t *block_table, int64_t bt_stride,
                                 const int32_t *seq_lens, int num_seqs, int max_seq_len,
                                 int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, float scale, pa_bf16 *out, void *stream) {
    // A problem whose partials do not fit the fixed array is refused up front.  Any other
    // bad argument is reported by pa_decode's own checks below (the size query returns 0
    // for those, which always fits).
    const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 block_size, max_seq_len);
    if (need > PA_DECODE_NOALLOC_SCRATCH_BYTES) return PA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (int rc = scratch_address(&scratch)) return rc;
    return pa_decode(q, k_cache, v_cache, page_stride, num_pages, block_table, bt_stride,
                     seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                     block_size, scale, out, scratch, PA_DECODE_NOALLOC_SCRATCH_BYTES, nullptr,
                     nullptr, nullptr, stream);
}
