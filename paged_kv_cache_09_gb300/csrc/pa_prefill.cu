// pa_prefill.cu -- chunked-prefill attention of one sequence over its paged cache.
//
// What is computed (page832 post §6): query row i of the chunk sits at absolute
// position q_start + i and, with causal masking, attends to keys 0..q_start+i of the
// same sequence (earlier chunks and the chunk itself, already written to the cache);
// without it, to all q_start + q_len keys.  K/V are read through the block table
// (page832 §1) in page-local 64-token tiles.
//
// Kernel shape: one CTA per (64-row query tile, query head); the longest (latest)
// query tiles are launched first.  A producer warp loads the query tile once and
// streams K/V tiles with TMA into a 2-stage ring.  Keys of the sequence's last page
// are read through tensor maps whose row extent ends at the sequence's last token, so
// rows past it arrive as zeros (never stale or NaN data).  Four consumer warps each own
// 16 query rows: S = Q K^T and O += P V on mma.m16n8k16 tensor-core tiles, online
// softmax in registers, fp32 accumulation, BF16 output.
#include <math_constants.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kPfConsumers = kPfQRows / 16;
constexpr int kPfThreads = (kPfConsumers + 1) * 32;
constexpr int kPfQChunk = kPfQRows * 128;       // one 64-dim box of the query tile
constexpr int kPfQBytes = kChunks * kPfQChunk;  // 32 KB
constexpr int kPfKvChunk = kPfKvTile * 128;
constexpr int kPfHalf = kChunks * kPfKvChunk;   // K (or V) of one tile: 32 KB
constexpr int kPfStageBytes = 2 * kPfHalf;
constexpr int kPfSmemBytes = 1024 + kPfQBytes + kPfStages * kPfStageBytes + 64;

struct PfKParams {
    const int32_t *block_table;
    int q_len, q_start, causal, seq_len_k;
    int num_q_heads, group;
    int block_size, tiles_per_page, last_page, num_q_tiles;
    int64_t num_pages;
    float scale_log2;
    uint16_t *out;
    unsigned *err;
};

struct PfMaps {
    CUtensorMap q, k, v, k_last, v_last;
};

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ PfMaps maps, const PfKParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qs = smem;
    uint8_t *ring = smem + kPfQBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + kPfStages * kPfStageBytes);
    uint64_t *qbar = bars;
    uint64_t *full = bars + 1;
    uint64_t *empty = full + kPfStages;

    const int qt = p.num_q_tiles - 1 - blockIdx.x;  // latest rows (most keys) first
    const int h = blockIdx.y;
    const int g = h / p.group;
    const int row0 = qt * kPfQRows;
    const int rows_here = min(kPfQRows, p.q_len - row0);
    const int nkeys = p.causal ? p.q_start + row0 + rows_here : p.seq_len_k;
    const int full_pages = nkeys / p.block_size;
    const int rem = nkeys - full_pages * p.block_size;
    const int ntiles = full_pages * p.tiles_per_page + (rem + kPfKvTile - 1) / kPfKvTile;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(qbar, 1);
        for (int s = 0; s < kPfStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPfConsumers);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kPfConsumers) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(qbar, kPfQBytes);
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
                tma_load_3d(qs + c * kPfQChunk, &maps.q, qbar, c * kChunkElems, h, row0);
            for (int i = 0; i < ntiles; ++i) {
                const int s = i % kPfStages;
                if (i >= kPfStages && !mbar_wait(&empty[s], ((i / kPfStages) - 1) & 1, p.err))
                    break;
                const int lp = i / p.tiles_per_page;
                const int off = (i - lp * p.tiles_per_page) * kPfKvTile;
                const int page = p.block_table[lp];
                if (page < 0 || page >= p.num_pages) atomicOr(p.err, kErrPage);
                const CUtensorMap *mk = lp == p.last_page ? &maps.k_last : &maps.k;
                const CUtensorMap *mv = lp == p.last_page ? &maps.v_last : &maps.v;
                uint8_t *st = ring + s * kPfStageBytes;
                mbar_arrive_expect_tx(&full[s], kPfStageBytes);
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    tma_load_4d(st + c * kPfKvChunk, mk, &full[s], c * kChunkElems, g, off, page);
                    tma_load_4d(st + kPfHalf + c * kPfKvChunk, mv, &full[s], c * kChunkElems, g,
                                off, page);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int wr = warp * 16;                // this warp's rows within the tile
    const int ra = lane >> 2;                // fragment rows ra and ra + 8
    const int qpos_a = p.q_start + row0 + wr + ra;
    const int qpos_b = qpos_a + 8;
    const uint32_t qbase = smem_u32(qs);
    const uint32_t rbase = smem_u32(ring);

    float o[32][4];
#pragma unroll
    for (int nt = 0; nt < 32; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_a = -CUDART_INF_F, m_b = -CUDART_INF_F, l_a = 0.f, l_b = 0.f;

    const bool ok = __all_sync(0xffffffffu, mbar_wait(qbar, 0, p.err));
    for (int i = 0; ok && i < ntiles; ++i) {
        const int s = i % kPfStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (i / kPfStages) & 1, p.err))) break;
        const int lp = i / p.tiles_per_page;
        const int off = (i - lp * p.tiles_per_page) * kPfKvTile;
        const int tok0 = lp * p.block_size + off;
        const uint32_t kb = rbase + s * kPfStageBytes;
        const uint32_t vb = kb + kPfHalf;

        // S (16 rows x 64 keys) = Q (16 x 256) . K^T (256 x 64)
        float sacc[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const int c = kk >> 2;
            const int u0 = (kk & 3) * 2;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(swz128(qbase + c * kPfQChunk, wr + (lane & 7) + ((lane >> 3) & 1) * 8,
                           u0 + (lane >> 4)),
                    a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(swz128(kb + c * kPfKvChunk, np * 16 + (lane & 7) + (lane >> 4) * 8,
                               u0 + ((lane >> 3) & 1)),
                        b0, b1, b2, b3);
                mma_bf16_16816(sacc[2 * np], a0, a1, a2, a3, b0, b1);
                mma_bf16_16816(sacc[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }

        // Mask (page tail, sequence end, causal) and online softmax per row.
        float mx_a = -CUDART_INF_F, mx_b = -CUDART_INF_F;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = nt * 8 + (lane & 3) * 2 + (e & 1);
                const int t = tok0 + col;
                const int qpos = (e >> 1) ? qpos_b : qpos_a;
                const bool valid = (off + col < p.block_size) && (t < p.seq_len_k) &&
                                   (!p.causal || t <= qpos);
                const float x = valid ? sacc[nt][e] * p.scale_log2 : -CUDART_INF_F;
                sacc[nt][e] = x;
                if (e >> 1) mx_b = fmaxf(mx_b, x); else mx_a = fmaxf(mx_a, x);
            }
        }
#pragma unroll
        for (int sh = 1; sh < 4; sh <<= 1) {
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, sh));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, sh));
        }
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float mu_a = mn_a == -CUDART_INF_F ? 0.f : mn_a;
        const float mu_b = mn_b == -CUDART_INF_F ? 0.f : mn_b;
        const float al_a = exp2f(m_a - mu_a), al_b = exp2f(m_b - mu_b);
        m_a = mn_a;
        m_b = mn_b;
        float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            sacc[nt][0] = exp2f(sacc[nt][0] - mu_a);
            sacc[nt][1] = exp2f(sacc[nt][1] - mu_a);
            sacc[nt][2] = exp2f(sacc[nt][2] - mu_b);
            sacc[nt][3] = exp2f(sacc[nt][3] - mu_b);
            rs_a += sacc[nt][0] + sacc[nt][1];
            rs_b += sacc[nt][2] + sacc[nt][3];
        }
        l_a = l_a * al_a + rs_a;
        l_b = l_b * al_b + rs_b;
#pragma unroll
        for (int nt = 0; nt < 32; ++nt) {
            o[nt][0] *= al_a;
            o[nt][1] *= al_a;
            o[nt][2] *= al_b;
            o[nt][3] *= al_b;
        }

        // O (16 x 256) += P (16 x 64) . V (64 x 256), with P = P_hi + P_lo in two BF16
        // parts: a single BF16 P carries a relative error up to 2^-8 per weight, which
        // rows with few or peaked keys turn into output errors above the tolerance.
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
            uint32_t ah[4], al[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float x0 = sacc[2 * kt + (r >> 1)][(r & 1) * 2];
                const float x1 = sacc[2 * kt + (r >> 1)][(r & 1) * 2 + 1];
                ah[r] = pack_bf16x2(x0, x1);
                al[r] = pack_bf16x2(x0 - bf16_lo(ah[r]), x1 - bf16_hi(ah[r]));
            }
#pragma unroll
            for (int dp = 0; dp < 16; ++dp) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(swz128(vb + (dp >> 2) * kPfKvChunk,
                                 kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8,
                                 (dp & 3) * 2 + (lane >> 4)),
                          b0, b1, b2, b3);
                mma_bf16_16816(o[2 * dp], ah[0], ah[1], ah[2], ah[3], b0, b1);
                mma_bf16_16816(o[2 * dp + 1], ah[0], ah[1], ah[2], ah[3], b2, b3);
                mma_bf16_16816(o[2 * dp], al[0], al[1], al[2], al[3], b0, b1);
                mma_bf16_16816(o[2 * dp + 1], al[0], al[1], al[2], al[3], b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

#pragma unroll
    for (int sh = 1; sh < 4; sh <<= 1) {
        l_a += __shfl_xor_sync(0xffffffffu, l_a, sh);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, sh);
    }
    const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f;
    const float inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
    const int row_a = row0 + wr + ra, row_b = row_a + 8;
    const int dc = (lane & 3) * 2;
    if (row_a < p.q_len) {
        uint16_t *dst = p.out + ((int64_t)row_a * p.num_q_heads + h) * kHeadDim + dc;
#pragma unroll
        for (int nt = 0; nt < 32; ++nt)
            *reinterpret_cast<uint32_t *>(dst + nt * 8) =
                pack_bf16x2(o[nt][0] * inv_a, o[nt][1] * inv_a);
    }
    if (row_b < p.q_len) {
        uint16_t *dst = p.out + ((int64_t)row_b * p.num_q_heads + h) * kHeadDim + dc;
#pragma unroll
        for (int nt = 0; nt < 32; ++nt)
            *reinterpret_cast<uint32_t *>(dst + nt * 8) =
                pack_bf16x2(o[nt][2] * inv_b, o[nt][3] * inv_b);
    }
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap *tmaps, const PrefillArgs &a, cudaStream_t stream) {
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(prefill_kernel),
                                  kPfSmemBytes, 1);
    if (e != cudaSuccess) return e;
    PfMaps maps;
    maps.q = tmaps[0];
    maps.k = tmaps[1];
    maps.v = tmaps[2];
    maps.k_last = tmaps[3];
    maps.v_last = tmaps[4];
    PfKParams p;
    p.block_table = a.block_table;
    p.q_len = a.q_len;
    p.q_start = a.q_start;
    p.causal = a.causal;
    p.seq_len_k = a.q_start + a.q_len;
    p.num_q_heads = a.num_q_heads;
    p.group = a.group;
    p.block_size = a.block_size;
    p.tiles_per_page = (a.block_size + kPfKvTile - 1) / kPfKvTile;
    p.last_page = a.last_page;
    p.num_q_tiles = (a.q_len + kPfQRows - 1) / kPfQRows;
    p.num_pages = a.num_pages;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.out = a.out;
    p.err = a.err;
    const dim3 grid(p.num_q_tiles, a.num_q_heads);
    if (a.ev_start && (e = cudaEventRecord(a.ev_start, stream)) != cudaSuccess) return e;
    prefill_kernel<<<grid, kPfThreads, kPfSmemBytes, stream>>>(maps, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.ev_stop) e = cudaEventRecord(a.ev_stop, stream);
    return e;
}

}  // namespace pa
