// Lightning-indexer score on tcgen05 tensor cores (mlx-native deepseek_rows.metal,
// kernel deepseek_indexer_score_mma_rows_bf16):
//   s[j] = sum_h w[h] * max(0, q_h . k_j)   (64 heads, 128 dims, per key j)
//
// GB300 design. The work is a stream of 128-key tiles over all rows (a row's
// tile t covers keys [128 t, 128 t + 128) of that row). A persistent CTA takes
// a contiguous range of tiles. Per tile, one tcgen05.mma chain computes
// D[128 keys x 64 heads] = K_tile[128 x 128] * Q[64 x 128]^T into TMEM
// (M=128, N=64, K=128 as 8 steps of 16). Operands sit in shared memory in the
// 128-byte-swizzled K-major layout written by TMA. The epilogue gives each
// thread one key (one TMEM lane): it reads the key's 64 head dot products and
// sums relu(x_h) * w_h as four interleaved partial sums (heads h = i mod 4,
// each in head order) added pairwise, so the score of a key depends only on
// the key's data and the query (bitwise, wherever the tile sits).
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs, warps 2..5 run the epilogue. Key tiles flow through a
// 5-stage ring; the query of the current row is double-buffered; the
// accumulator is double-buffered in TMEM so the epilogue of tile i overlaps
// the MMAs of tile i+1. Keys are streamed with an L2 evict-first policy.
//
// Optional fused output: a 2048-bin histogram of the order-preserving score
// keys per row (top 11 bits), used by the top-k stage to find its threshold.

#include "common.cuh"
#include "kernels.h"

namespace dsrows {

namespace {

constexpr int kThreads = 192;
constexpr int kTileKeys = 128;
constexpr int kStages = 5;
constexpr int kHalfBytes = kTileKeys * 64 * 2;  // one 64-column SW128 box of a key tile
constexpr int kTileBytes = 2 * kHalfBytes;      // 32 KiB
constexpr int kQHalfBytes = 64 * 64 * 2;        // 8 KiB
constexpr int kQBytes = 2 * kQHalfBytes;        // 16 KiB
constexpr int kAccCols = 64;
constexpr int kAccBufs = 2;
constexpr uint32_t kTmemCols = kAccCols * kAccBufs;  // 128 (power of two >= 32)

struct __align__(8) Barriers {
    uint64_t k_full[kStages];
    uint64_t k_empty[kStages];
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t acc_full[kAccBufs];
    uint64_t acc_empty[kAccBufs];
    uint32_t tmem_base;
    uint32_t abort_flag;
};

struct SmemLayout {
    static constexpr size_t keys = 0;
    static constexpr size_t q = keys + (size_t)kStages * kTileBytes;
    static constexpr size_t w = q + 2 * (size_t)kQBytes;
    static constexpr size_t hist = w + (size_t)kRowsMax * kIdxHeads * 4;
    static constexpr size_t bars = hist + (size_t)kHistBins * 4;
    static constexpr size_t total = bars + sizeof(Barriers);
};
constexpr size_t kSmemBytes = SmemLayout::total + 1024;  // + alignment slack

__device__ __forceinline__ int entry_of_tile(const IndexerParams& p, uint32_t g) {
    int e = 0;
#pragma unroll
    for (int i = 1; i < kRowsMax; ++i)
        if (i < (int)p.rows && g >= p.tile_begin[i]) e = i;
    return e;
}

__device__ __forceinline__ float relu_nan(float x) {
    // max(0, x) that keeps NaN (a NaN dot product must poison the score).
    return (x > 0.0f || x != x) ? x : 0.0f;
}

__device__ __forceinline__ void named_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) indexer_score_kernel(const __grid_constant__ IndexerParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* keys_s = smem + SmemLayout::keys;
    uint8_t* q_s = smem + SmemLayout::q;
    float* w_s = reinterpret_cast<float*>(smem + SmemLayout::w);
    uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + SmemLayout::hist);
    Barriers* bar = reinterpret_cast<Barriers*>(smem + SmemLayout::bars);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t G = gridDim.x;
    const uint32_t T = p.total_tiles;
    const uint32_t g_begin = (uint32_t)(((uint64_t)blockIdx.x * T) / G);
    const uint32_t g_end = (uint32_t)(((uint64_t)(blockIdx.x + 1) * T) / G);

    // Inputs may still be in flight from the previous kernel (programmatic
    // launch): then nothing is read before it completes.
    if (!p.inputs_ready) pdl_wait();

    // ---- setup -------------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar->k_full[s], 1);
            mbar_init(&bar->k_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar->q_full[b], 1);
            mbar_init(&bar->q_empty[b], 1);
        }
        for (int a = 0; a < kAccBufs; ++a) {
            mbar_init(&bar->acc_full[a], 1);
            mbar_init(&bar->acc_empty[a], 4);
        }
        bar->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int e = 0; e < (int)p.rows; ++e) tma_prefetch_map(&p.kmap[e]);
        tma_prefetch_map(&p.qmap);
    }
    if (warp == 1) {
        tmem_alloc(&bar->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    for (int i = threadIdx.x; i < (int)p.rows * kIdxHeads; i += kThreads) {
        const int e = i / kIdxHeads, h = i % kIdxHeads;
        w_s[i] = p.w[(size_t)p.q_row[e] * kIdxHeads + h];
    }
    for (int i = threadIdx.x; i < kHistBins; i += kThreads) hist_s[i] = 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = bar->tmem_base;
    pdl_trigger();

    if (warp == 0) {
        // ---- TMA producer ----------------------------------------------------
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            const uint64_t q_policy = l2_policy_evict_last();
            int cur = -1;
            uint32_t q_uses = 0, it = 0;
            uint32_t last_parity[kStages];
            bool used[kStages];
            for (int s = 0; s < kStages; ++s) used[s] = false;
            bool ok = true;
            for (uint32_t g = g_begin; g < g_end && ok; ++g, ++it) {
                const int e = entry_of_tile(p, g);
                const uint32_t tile = g - p.tile_begin[e];
                if (e != cur) {
                    cur = e;
                    const uint32_t qb = q_uses & 1;
                    if (!mbar_wait(&bar->q_empty[qb], ((q_uses >> 1) & 1) ^ 1, p.status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bar->q_full[qb], kQBytes);
                    uint8_t* dst = q_s + (size_t)qb * kQBytes;
                    const int y = (int)(p.q_row[e] * kIdxHeads);
                    tma_load_2d(dst, &p.qmap, &bar->q_full[qb], 0, y, q_policy);
                    tma_load_2d(dst + kQHalfBytes, &p.qmap, &bar->q_full[qb], 64, y, q_policy);
                    ++q_uses;
                }
                const uint32_t s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!mbar_wait(&bar->k_empty[s], ph ^ 1, p.status)) { ok = false; break; }
                mbar_arrive_expect_tx(&bar->k_full[s], kTileBytes);
                uint8_t* dst = keys_s + (size_t)s * kTileBytes;
                const int y = (int)(tile * kTileKeys);
                tma_load_2d(dst, &p.kmap[e], &bar->k_full[s], 0, y, policy);
                tma_load_2d(dst + kHalfBytes, &p.kmap[e], &bar->k_full[s], 64, y, policy);
                used[s] = true;
                last_parity[s] = ph;
            }
            if (!ok) atomicExch(&bar->abort_flag, 1u);
            // Drain: every load this thread issued has landed before the CTA exits.
            for (int s = 0; s < kStages; ++s)
                if (used[s]) (void)mbar_wait(&bar->k_full[s], last_parity[s], p.status);
        }
    } else if (warp == 1) {
        // ---- MMA issuer --------------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 64);
            int cur = -1;
            uint32_t q_uses = 0, qb = 0, it = 0;
            for (uint32_t g = g_begin; g < g_end; ++g, ++it) {
                if (*(volatile uint32_t*)&bar->abort_flag) break;
                const int e = entry_of_tile(p, g);
                if (e != cur) {
                    if (cur >= 0) umma_commit(&bar->q_empty[qb]);
                    qb = q_uses & 1;
                    if (!mbar_wait(&bar->q_full[qb], (q_uses >> 1) & 1, p.status)) break;
                    ++q_uses;
                    cur = e;
                }
                const uint32_t s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                const uint32_t a = it % kAccBufs;
                const uint32_t aph = (it / kAccBufs) & 1;
                if (!mbar_wait(&bar->k_full[s], ph, p.status)) break;
                if (!mbar_wait(&bar->acc_empty[a], aph ^ 1, p.status)) break;
                tc_fence_after();
                const uint32_t a_base = smem_u32(keys_s + (size_t)s * kTileBytes);
                const uint32_t b_base = smem_u32(q_s + (size_t)qb * kQBytes);
                const uint32_t d_tmem = tmem_base + a * kAccCols;
#pragma unroll
                for (int kk = 0; kk < kIdxDim / 16; ++kk) {
                    const uint32_t koff = (uint32_t)(kk & 3) * 32;  // 16 bf16 = 32 B inside the 128-B row
                    const uint64_t adesc = smem_desc_sw128_kmajor(a_base + (kk >> 2) * kHalfBytes + koff);
                    const uint64_t bdesc = smem_desc_sw128_kmajor(b_base + (kk >> 2) * kQHalfBytes + koff);
                    umma_bf16(d_tmem, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
                }
                umma_commit(&bar->k_empty[s]);
                umma_commit(&bar->acc_full[a]);
            }
        }
        __syncwarp();
    } else {
        // ---- epilogue: one key per thread --------------------------------------
        const int quarter = warp & 3;          // TMEM lanes [32*quarter, 32*quarter+32)
        const int ep_tid = threadIdx.x - 64;   // 0..127
        const bool want_hist = p.hist != nullptr;
        // The histogram may still be being cleared by the previous kernel (PDL):
        // the producer and MMA warps start streaming, the epilogue waits here.
        pdl_wait();
        // The scores are read back by the next kernel: keep them in L2 while the
        // key stream (evict-first) passes through.
        const uint64_t keep = l2_policy_evict_last();
        int cur = -1;
        uint32_t it = 0;
        for (uint32_t g = g_begin; g < g_end; ++g, ++it) {
            const int e = entry_of_tile(p, g);
            const uint32_t tile = g - p.tile_begin[e];
            if (want_hist && e != cur && cur >= 0) {
                named_bar(1, 128);
                for (int b = ep_tid; b < kHistBins; b += 128) {
                    const uint32_t v = hist_s[b];
                    if (v) {
                        atomicAdd(&p.hist[(size_t)cur * kHistBins + b], v);
                        hist_s[b] = 0;
                    }
                }
                named_bar(1, 128);
            }
            cur = e;
            const uint32_t a = it % kAccBufs;
            const uint32_t aph = (it / kAccBufs) & 1;
            if (!mbar_wait(&bar->acc_full[a], aph, p.status)) break;
            tc_fence_after();
            uint32_t v[64];
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + a * kAccCols;
            tmem_ld_x16(taddr + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
            tmem_ld_x16(taddr + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
            tmem_ld_x16(taddr + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
            tmem_ld_x16(taddr + 48, *reinterpret_cast<uint32_t(*)[16]>(&v[48]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->acc_empty[a]);

            const float* w = w_s + e * kIdxHeads;
            // Four independent chains: a quarter of the dependent FMA latency.
            float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int h = 0; h < kIdxHeads; ++h) s4[h & 3] = fmaf(relu_nan(__uint_as_float(v[h])), w[h], s4[h & 3]);
            const float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
            const uint32_t j = tile * kTileKeys + quarter * 32 + lane;
            if (j < p.kv_len[e]) {
                const bool fin = finite_f(s);
                st_global_hint(p.scores + (size_t)e * p.score_stride + j, fin ? s : -INFINITY, keep);
                if (want_hist && fin) atomicAdd(&hist_s[score_key(s) >> 21], 1u);
            }
        }
        if (want_hist && cur >= 0) {
            named_bar(1, 128);
            for (int b = ep_tid; b < kHistBins; b += 128) {
                const uint32_t v = hist_s[b];
                if (v) atomicAdd(&p.hist[(size_t)cur * kHistBins + b], v);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

size_t indexer_smem_bytes() { return kSmemBytes; }

cudaError_t launch_indexer(const IndexerParams& p, int num_sms, cudaStream_t stream, bool pdl) {
    static bool configured = false;
    if (!configured) {
        cudaError_t err = cudaFuncSetAttribute(indexer_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kSmemBytes);
        if (err != cudaSuccess) return err;
        configured = true;
    }
    if (p.total_tiles == 0) return cudaSuccess;
    const uint32_t grid = p.total_tiles < (uint32_t)num_sms ? p.total_tiles : (uint32_t)num_sms;
    return launch_kernel(indexer_score_kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, pdl, p);
}

uint32_t indexer_tile_keys() { return kTileKeys; }

}  // namespace dsrows
