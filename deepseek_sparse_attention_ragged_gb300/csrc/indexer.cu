// Lightning-indexer score on tcgen05 tensor cores (mlx-native deepseek_rows.metal,
// kernel deepseek_indexer_score_mma_rows_bf16):
//   s[j] = sum_h w[h] * max(0, q_h . k_j)   (64 heads, 128 dims, per key j)
//
// GB300 design. The work is a stream of 128-key tiles over all rows (a row's
// tile t covers keys [128 t, 128 t + 128) of that row). A persistent CTA takes
// every n-th tile of one row (one query per row: n CTAs per row, in proportion
// to the row's tiles) or a contiguous range of the stream. Per tile, one tcgen05.mma chain computes
// D[128 keys x 64 heads] = K_tile[128 x 128] * Q[64 x 128]^T into TMEM
// (M=128, N=64, K=128 as 8 steps of 16). Operands sit in shared memory in the
// 128-byte-swizzled K-major layout written by TMA. The epilogue gives each
// thread one key (one TMEM lane): it reads the key's 64 head dot products and
// sums relu(x_h) * w_h as four interleaved partial sums (heads h = i mod 4,
// each in head order) added pairwise, so the score of a key depends only on
// the key's data and the query (bitwise, wherever the tile sits).
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs, warps 2..5 run the epilogue. Warp 0 starts loading key
// tiles as soon as the barriers exist, while the other warps allocate TMEM
// and stage the head weights. Key tiles flow through a
// 4-stage ring (with the HBM saturated by all SMs, a fifth or sixth stage in
// flight per SM only lengthened the memory queues); the query of the current
// row is double-buffered; the accumulator is double-buffered in TMEM so the
// epilogue of tile i overlaps the MMAs of tile i+1. Keys are streamed with an
// L2 evict-first policy.
//
// Optional fused output: a 2048-bin histogram of the order-preserving score
// keys per row (top 11 bits), used by the top-k stage to find its threshold.
//
// Several queries per row (the kernel's query loop on the pages; query i of an
// entry sits at its position + i and scores its own causal count of keys): a
// segment is an entry with up to four consecutive queries, whose query rows
// stack along N, so each key tile is read from HBM once for all of them:
// D[128 keys x 64 nq] = K_tile . [q_0; ...; q_{nq-1}]^T. Eight epilogue warps
// split the queries, two warps per TMEM lane quarter; a warp reads one query's
// columns at a time, its first query's head weights held in registers for the
// segment. Each query's score of a key is the same arithmetic as with one
// query, so it does not depend on its neighbours.

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace dsrows {

namespace {

constexpr int kTileKeys = 128;
constexpr int kHalfBytes = kTileKeys * 64 * 2;  // one 64-column SW128 box of a key tile
constexpr int kTileBytes = 2 * kHalfBytes;      // 32 KiB
constexpr int kQBoxBytes = 64 * 64 * 2;         // one query's 64 heads x 64 columns: 8 KiB

// Shape of the kernel for G queries per key tile.
//   G = 1: 4-stage key ring, double-buffered query, 4 epilogue warps (one
//          key per thread), accumulators 2 x 64 TMEM columns, the head
//          weights of every row and a 2048-bin u32 histogram in shared memory;
//   G = 4: 4-stage key ring, one query buffer (up to 4 x 16 KiB), 8 epilogue
//          warps (two per TMEM lane quarter, splitting the segment's queries
//          evenly), accumulators 2 x 256 columns, the head weights of the
//          current segment, and per query a 2048-bin histogram of 16-bit
//          counts packed two to a word (flushed at least every kFlushTiles
//          tiles, so a count stays below 2^16).
template <int G>
struct Shape {
    static constexpr int kStages = 4;
    static constexpr int kQBufs = G == 1 ? 2 : 1;
    static constexpr int kEpiWarps = G == 1 ? 4 : 8;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    static constexpr int kQPerWarp = G * 4 / kEpiWarps;  // queries per epilogue thread, at most
    static constexpr int kSegs = G == 1 ? kRowsMax : kSegMax;
    static constexpr int kVRows = G == 1 ? kRowsMax : kVRowsMax;
    static constexpr int kWRows = G == 1 ? kRowsMax : G;  // rows of head weights held
    static constexpr int kHistWords = G == 1 ? kHistBins : G * kHistBins / 2;
    static constexpr uint32_t kFlushTiles = 256;           // 256 x 128 keys < 2^16
    static constexpr int kQHalfBytes = G * kQBoxBytes;    // 64 columns of G x 64 query rows
    static constexpr int kQBytes = 2 * kQHalfBytes;
    static constexpr uint32_t kAccCols = 64 * G;
    static constexpr uint32_t kTmemCols = 2 * kAccCols;   // double-buffered; a power of two >= 32
    // shared memory
    static constexpr size_t keys = 0;
    static constexpr size_t q = keys + (size_t)kStages * kTileBytes;
    static constexpr size_t w = q + (size_t)kQBufs * kQBytes;
    static constexpr size_t hist = w + (size_t)kWRows * kIdxHeads * 4;
    static constexpr size_t bars = hist + (size_t)kHistWords * 4;
};

template <int G>
struct __align__(8) Barriers {
    uint64_t k_full[Shape<G>::kStages];
    uint64_t k_empty[Shape<G>::kStages];
    uint64_t q_full[Shape<G>::kQBufs];
    uint64_t q_empty[Shape<G>::kQBufs];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    uint32_t abort_flag;
};

template <int G>
constexpr size_t smem_bytes() {
    return Shape<G>::bars + sizeof(Barriers<G>) + 1024;  // + alignment slack
}
static_assert(smem_bytes<1>() <= 227 * 1024 && smem_bytes<kIndexerGroup>() <= 227 * 1024, "shared memory");

template <int S, int V>
__device__ __forceinline__ int segment_of_tile(const IndexerParamsT<S, V>& p, uint32_t g) {
    int s = 0;
#pragma unroll
    for (int i = 1; i < S; ++i)
        if (i < (int)p.segs && g >= p.tile_begin[i]) s = i;
    return s;
}

__device__ __forceinline__ float relu_nan(float x) {
    // max(0, x) that keeps NaN (a NaN dot product must poison the score).
    float r;
    asm("max.NaN.f32 %0, %1, 0f00000000;" : "=f"(r) : "f"(x));
    return r;
}

// sum_h w[h] relu(x[h]) over the 64 head dot products x of one key, with w in
// registers (wr) or shared memory (w_s): four chains (heads h = c mod 4, in
// head order), added pairwise.
// Two fp32 FMAs in one instruction (each rounded as fmaf): d = a * b + c lane-wise.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
          "l"(*reinterpret_cast<const uint64_t*>(&c)));
    return *reinterpret_cast<const float2*>(&d);
}

__device__ __forceinline__ float head_sum(const uint32_t (&x)[64], const float* wr, const float* w_s) {
    if (wr) {
        // Weights in registers: chains 0 and 1 (heads h = 0, 1 mod 4) and chains
        // 2 and 3 advance in pairs, two FMAs per instruction.
        float2 s01 = make_float2(0.0f, 0.0f), s23 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int h = 0; h < kIdxHeads; h += 4) {
            const float2 r01 = make_float2(relu_nan(__uint_as_float(x[h])), relu_nan(__uint_as_float(x[h + 1])));
            const float2 r23 = make_float2(relu_nan(__uint_as_float(x[h + 2])), relu_nan(__uint_as_float(x[h + 3])));
            s01 = fma2(r01, make_float2(wr[h], wr[h + 1]), s01);
            s23 = fma2(r23, make_float2(wr[h + 2], wr[h + 3]), s23);
        }
        return (s01.x + s01.y) + (s23.x + s23.y);
    }
    float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int h = 0; h < kIdxHeads; h += 4) {
        const float4 w4 = *reinterpret_cast<const float4*>(w_s + h);
        s4[0] = fmaf(relu_nan(__uint_as_float(x[h])), w4.x, s4[0]);
        s4[1] = fmaf(relu_nan(__uint_as_float(x[h + 1])), w4.y, s4[1]);
        s4[2] = fmaf(relu_nan(__uint_as_float(x[h + 2])), w4.z, s4[2]);
        s4[3] = fmaf(relu_nan(__uint_as_float(x[h + 3])), w4.w, s4[3]);
    }
    return (s4[0] + s4[1]) + (s4[2] + s4[3]);
}

__device__ __forceinline__ void named_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void named_bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace

template <int G>
using ParamsOf = IndexerParamsT<Shape<G>::kSegs, Shape<G>::kVRows>;

template <int G>
__device__ __forceinline__ void indexer_score_body(const ParamsOf<G>& p) {
    using S = Shape<G>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* keys_s = smem + S::keys;
    uint8_t* q_s = smem + S::q;
    float* w_s = reinterpret_cast<float*>(smem + S::w);
    uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + S::hist);
    Barriers<G>* bar = reinterpret_cast<Barriers<G>*>(smem + S::bars);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t NB = gridDim.x;
    const uint32_t T = p.total_tiles;
    // This CTA's k-th tile. One query per entry: the CTAs are split over the
    // entries in proportion to their tiles, and an entry's CTAs take every n-th
    // of its tiles, so they sweep the cache side by side and finish together
    // (contiguous ranges ended up to 4 us apart) while each CTA keeps one query
    // and one histogram. Grouped: a contiguous range of the whole stream.
    const uint32_t g_begin = (uint32_t)(((uint64_t)blockIdx.x * T) / NB);
    const uint32_t g_end = (uint32_t)(((uint64_t)(blockIdx.x + 1) * T) / NB);
    int my_seg = 0;
    if (G == 1)
        for (int i = 1; i < (int)p.segs; ++i)
            if (blockIdx.x >= p.cta_begin[i]) my_seg = i;
    const uint32_t seg_j = blockIdx.x - p.cta_begin[my_seg];
    const uint32_t seg_n = p.cta_begin[my_seg + 1] - p.cta_begin[my_seg];
    const uint32_t seg_end = my_seg + 1 < (int)p.segs ? p.tile_begin[my_seg + 1] : T;
    auto tile_of = [&](uint32_t k) -> uint32_t {
        const uint32_t g = G == 1 ? p.tile_begin[my_seg] + seg_j + k * seg_n : g_begin + k;
        return g < (G == 1 ? seg_end : g_end) ? g : T;
    };

    // Inputs may still be in flight from the previous kernel (programmatic
    // launch): then nothing is read before it completes. With inputs_ready 2
    // only the query and head weights are: the CTA sets up at once, and the
    // producer (after the first stages of key tiles, before its first query
    // load) and the epilogue (before the weights) wait.
    if (!p.inputs_ready) pdl_wait();

    // ---- setup -------------------------------------------------------------
    // The producer warp only initialises the barriers: it announces them on the
    // setup barrier without waiting and starts the key stream at once, while
    // the other warps allocate TMEM, load the head weights and zero the
    // histogram, then wait on the setup barrier.
    constexpr int kSetupBar = 2;
    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < S::kStages; ++s) {
                mbar_init(&bar->k_full[s], 1);
                mbar_init(&bar->k_empty[s], 1);
            }
            for (int b = 0; b < S::kQBufs; ++b) {
                mbar_init(&bar->q_full[b], 1);
                mbar_init(&bar->q_empty[b], 1);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(&bar->acc_full[a], 1);
                mbar_init(&bar->acc_empty[a], S::kEpiWarps);
            }
            bar->abort_flag = 0;
            fence_barrier_init();
            for (int e = 0; e < (int)p.rows; ++e) tma_prefetch_map(&p.kmap[e]);
            tma_prefetch_map(&p.qmap);
        }
        __syncwarp();
        named_bar_arrive(kSetupBar, S::kThreads);
    } else {
        if (warp == 1) {
            tmem_alloc(&bar->tmem_base, S::kTmemCols);
            tmem_relinquish();
        }
        const int tid = threadIdx.x - 32;
        if (G == 1 && p.inputs_ready != 2)
            for (int i = tid; i < (int)p.vrows * kIdxHeads; i += S::kThreads - 32) {
                const int v = i / kIdxHeads, h = i % kIdxHeads;
                w_s[i] = p.w[(size_t)p.q_row[v] * kIdxHeads + h];
            }
        for (int i = tid; i < S::kHistWords; i += S::kThreads - 32) hist_s[i] = 0;
        tc_fence_before();
        named_bar(kSetupBar, S::kThreads);
        tc_fence_after();
    }
    const uint32_t tmem_base = warp == 0 ? 0u : bar->tmem_base;
    pdl_trigger();

    if (warp == 0) {
        // ---- TMA producer ----------------------------------------------------
        if (lane == 0) {
            // A key tile is read once per segment; with several segments per
            // entry (more than G queries) it is read again and may come from L2.
            const uint64_t policy = l2_policy_evict_first();
            const uint64_t q_policy = l2_policy_evict_last();
            int cur = -1;
            uint32_t q_uses = 0, it = 0;
            uint32_t last_parity[S::kStages];
            bool used[S::kStages];
            for (int s = 0; s < S::kStages; ++s) used[s] = false;
            bool ok = true;
            // The queries of segment sg into the next query buffer.
            auto load_query = [&](int sg) -> bool {
                const uint32_t qb = q_uses % S::kQBufs, use = q_uses / S::kQBufs;
                if (!mbar_wait(&bar->q_empty[qb], (use & 1) ^ 1, p.status)) return false;
                const int nq = G == 1 ? 1 : p.seg_queries[sg];
                mbar_arrive_expect_tx(&bar->q_full[qb], (uint32_t)nq * 2 * kQBoxBytes);
                uint8_t* dst = q_s + (size_t)qb * S::kQBytes;
                for (int i = 0; i < nq; ++i) {
                    const int y = (int)(p.q_row[p.seg_vrow[sg] + i] * kIdxHeads);
                    tma_load_2d(dst + i * kQBoxBytes, &p.qmap, &bar->q_full[qb], 0, y, q_policy);
                    tma_load_2d(dst + S::kQHalfBytes + i * kQBoxBytes, &p.qmap, &bar->q_full[qb], 64, y, q_policy);
                }
                ++q_uses;
                return true;
            };
            // With inputs_ready 2 the first query is still being written by the
            // previous kernel: the key tiles of the first stages (complete
            // inputs) are requested first, then the wait, then that query.
            bool q_deferred = false;
            for (;; ++it) {
                const uint32_t g = tile_of(it);
                if (g >= T || !ok) break;
                const int sg = segment_of_tile(p, g);
                const int e = G == 1 ? sg : p.seg_entry[sg];  // one segment per entry with one query
                const uint32_t tile = g - p.tile_begin[sg];
                if (sg != cur) {
                    cur = sg;
                    if (p.inputs_ready == 2 && q_uses == 0) q_deferred = true;
                    else if (!load_query(sg)) { ok = false; break; }
                }
                const uint32_t s = it % S::kStages;
                const uint32_t ph = (it / S::kStages) & 1;
                if (!mbar_wait(&bar->k_empty[s], ph ^ 1, p.status)) { ok = false; break; }
                mbar_arrive_expect_tx(&bar->k_full[s], kTileBytes);
                uint8_t* dst = keys_s + (size_t)s * kTileBytes;
                const int y = (int)(tile * kTileKeys);
                tma_load_2d(dst, &p.kmap[e], &bar->k_full[s], 0, y, policy);
                tma_load_2d(dst + kHalfBytes, &p.kmap[e], &bar->k_full[s], 64, y, policy);
                used[s] = true;
                last_parity[s] = ph;
                if (q_deferred) {
                    // Before the ring would wait, or before another segment's query.
                    const uint32_t gn = tile_of(it + 1);
                    if (it + 1 == (uint32_t)S::kStages || gn >= T || segment_of_tile(p, gn) != cur) {
                        pdl_wait();
                        q_deferred = false;
                        if (!load_query(cur)) { ok = false; break; }
                    }
                }
            }
            if (!ok) atomicExch(&bar->abort_flag, 1u);
            // Drain: every load this thread issued has landed before the CTA exits.
            for (int s = 0; s < S::kStages; ++s)
                if (used[s]) (void)mbar_wait(&bar->k_full[s], last_parity[s], p.status);
        }
    } else if (warp == 1) {
        // ---- MMA issuer --------------------------------------------------------
        if (lane == 0) {
            int cur = -1;
            uint32_t q_uses = 0, qb = 0, it = 0, idesc = 0;
            for (;; ++it) {
                const uint32_t g = tile_of(it);
                if (g >= T) break;
                if (*(volatile uint32_t*)&bar->abort_flag) break;
                const int sg = segment_of_tile(p, g);
                if (sg != cur) {
                    if (cur >= 0) umma_commit(&bar->q_empty[qb]);
                    qb = q_uses % S::kQBufs;
                    if (!mbar_wait(&bar->q_full[qb], (q_uses / S::kQBufs) & 1, p.status)) break;
                    ++q_uses;
                    cur = sg;
                    // D[128 keys x 64 nq] = K_tile . [q_0; ...; q_{nq-1}]^T
                    if (G != 1) idesc = idesc_bf16_f32(128, 64 * (int)p.seg_queries[sg]);
                }
                const uint32_t s = it % S::kStages;
                const uint32_t ph = (it / S::kStages) & 1;
                const uint32_t a = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                if (!mbar_wait(&bar->k_full[s], ph, p.status)) break;
                if (!mbar_wait(&bar->acc_empty[a], aph ^ 1, p.status)) break;
                tc_fence_after();
                const uint32_t a_base = smem_u32(keys_s + (size_t)s * kTileBytes);
                const uint32_t b_base = smem_u32(q_s + (size_t)qb * S::kQBytes);
                const uint32_t d_tmem = tmem_base + a * S::kAccCols;
#pragma unroll
                for (int kk = 0; kk < kIdxDim / 16; ++kk) {
                    const uint32_t koff = (uint32_t)(kk & 3) * 32;  // 16 bf16 = 32 B inside the 128-B row
                    const uint64_t adesc = smem_desc_sw128_kmajor(a_base + (kk >> 2) * kHalfBytes + koff);
                    const uint64_t bdesc = smem_desc_sw128_kmajor(b_base + (kk >> 2) * S::kQHalfBytes + koff);
                    umma_bf16(d_tmem, adesc, bdesc, G == 1 ? idesc_bf16_f32(128, 64) : idesc, kk > 0 ? 1u : 0u);
                }
                umma_commit(&bar->k_empty[s]);
                umma_commit(&bar->acc_full[a]);
            }
        }
        __syncwarp();
    } else {
        // ---- epilogue: one key per thread, kQPerWarp queries ---------------------
        constexpr int kEpiThreads = 32 * S::kEpiWarps;
        const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter+32)
        const int ep_tid = threadIdx.x - 64;
        constexpr int kGroups = S::kEpiWarps / 4;  // warps per TMEM lane quarter: they split the queries
        const int sub = G == 1 ? 0 : (warp - 2) >> 2;
        const bool want_hist = p.hist != nullptr;
        // The histogram may still be being cleared by the previous kernel (PDL):
        // the producer and MMA warps start streaming, the epilogue waits here.
        pdl_wait();
        for (uint32_t i = blockIdx.x * kEpiThreads + ep_tid; i < p.side_n16; i += NB * kEpiThreads)
            p.side_dst[i] = p.side_src[i];
        if (G == 1 && p.inputs_ready == 2) {
            for (int i = ep_tid; i < (int)p.vrows * kIdxHeads; i += kEpiThreads) {
                const int v = i / kIdxHeads, h = i % kIdxHeads;
                w_s[i] = p.w[(size_t)p.q_row[v] * kIdxHeads + h];
            }
            named_bar(1, kEpiThreads);
        }
        // The scores are read back by the next kernel: keep them in L2 while the
        // key stream (evict-first) passes through.
        const uint64_t keep = l2_policy_evict_last();
        // Add this CTA's counts of segment `sg` to the row histograms and zero them.
        auto flush = [&](int sg) {
            const int nq = G == 1 ? 1 : (int)p.seg_queries[sg];
            for (int i = 0; i < nq; ++i) {
                uint32_t* dst = p.hist + (size_t)(p.seg_vrow[sg] + i) * kHistBins;
                if (G == 1) {
                    // All of this thread's bins are read first, so the reads overlap.
                    constexpr int kPer = kHistBins / kEpiThreads;
                    uint32_t hv[kPer];
#pragma unroll
                    for (int k = 0; k < kPer; ++k) hv[k] = hist_s[ep_tid + k * kEpiThreads];
#pragma unroll
                    for (int k = 0; k < kPer; ++k)
                        if (hv[k]) {
                            atomicAdd(dst + ep_tid + k * kEpiThreads, hv[k]);
                            hist_s[ep_tid + k * kEpiThreads] = 0;
                        }
                } else {
                    uint32_t* h = hist_s + i * (kHistBins / 2);
                    for (int b = ep_tid; b < kHistBins / 2; b += kEpiThreads) {
                        const uint32_t v = h[b];
                        if (v) {
                            if (v & 0xFFFFu) atomicAdd(dst + 2 * b, v & 0xFFFFu);
                            if (v >> 16) atomicAdd(dst + 2 * b + 1, v >> 16);
                            h[b] = 0;
                        }
                    }
                }
            }
        };
        int cur = -1;
        uint32_t it = 0, since_flush = 0;
        // One query: the row's head weights stay in registers. Several: the weights
        // of this warp's first query of the segment do.
        float wr[G == 1 ? kIdxHeads : 4];
        float wq0[G == 1 ? 4 : kIdxHeads];
        for (;; ++it) {
            const uint32_t g = tile_of(it);
            if (g >= T) break;
            const int sg = segment_of_tile(p, g);
            const uint32_t tile = g - p.tile_begin[sg];
            if (G == 1) {
                if (want_hist && sg != cur && cur >= 0) {
                    named_bar(1, kEpiThreads);
                    flush(cur);
                    named_bar(1, kEpiThreads);
                }
                if (sg != cur)
#pragma unroll
                    for (int h = 0; h < kIdxHeads; h += 4)
                        *reinterpret_cast<float4*>(&wr[h]) = *reinterpret_cast<const float4*>(w_s + sg * kIdxHeads + h);
            } else if (sg != cur || (want_hist && since_flush == S::kFlushTiles)) {
                named_bar(1, kEpiThreads);  // every thread is done with the weights and counts
                if (want_hist && cur >= 0) flush(cur);
                if (sg != cur) {
                    const int nq = p.seg_queries[sg];
                    for (int i = ep_tid; i < nq * kIdxHeads; i += kEpiThreads)
                        w_s[i] = p.w[(size_t)p.q_row[p.seg_vrow[sg] + i / kIdxHeads] * kIdxHeads + i % kIdxHeads];
                }
                named_bar(1, kEpiThreads);
                if (G != 1 && sg != cur) {
                    const int nq_n = p.seg_queries[sg];
                    const int q0_n = sub * ((nq_n + kGroups - 1) / kGroups);
                    if (q0_n < nq_n)
#pragma unroll
                        for (int h = 0; h < kIdxHeads; h += 4)
                            *reinterpret_cast<float4*>(&wq0[h]) =
                                *reinterpret_cast<const float4*>(w_s + q0_n * kIdxHeads + h);
                }
                since_flush = 0;
            }
            cur = sg;
            ++since_flush;
            const int nq = G == 1 ? 1 : (int)p.seg_queries[sg];
            // This warp's queries of the segment: [q0, q0 + nk).
            const int per = (nq + kGroups - 1) / kGroups;
            const int q0 = sub * per;
            const int nk = nq - q0 < 0 ? 0 : (nq - q0 < per ? nq - q0 : per);
            const uint32_t a = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            if (!mbar_wait(&bar->acc_full[a], aph, p.status)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + a * S::kAccCols;
            const uint32_t j = tile * kTileKeys + quarter * 32 + lane;
            float scs[S::kQPerWarp];
            if constexpr (G == 1) {
                uint32_t v[64];
                tmem_ld_x16(taddr + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                tmem_ld_x16(taddr + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                tmem_ld_x16(taddr + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
                tmem_ld_x16(taddr + 48, *reinterpret_cast<uint32_t(*)[16]>(&v[48]));
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->acc_empty[a]);
                scs[0] = head_sum(v, wr, nullptr);
            } else {
                // One query's 64 columns at a time: the first query's sum uses the
                // weights in registers, the second's those in shared memory.
                static_assert(S::kQPerWarp == 2, "two queries per epilogue thread");
                uint32_t v[64];
                auto load = [&](int k) {
                    const uint32_t c = taddr + 64 * (q0 + k);
                    tmem_ld_x16(c + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                    tmem_ld_x16(c + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                    tmem_ld_x16(c + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
                    tmem_ld_x16(c + 48, *reinterpret_cast<uint32_t(*)[16]>(&v[48]));
                    tmem_ld_wait();
                };
                if (nk > 0) {
                    load(0);
                    scs[0] = head_sum(v, wq0, nullptr);
                }
                if (nk > 1) load(1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->acc_empty[a]);
                if (nk > 1) scs[1] = head_sum(v, nullptr, w_s + (q0 + 1) * kIdxHeads);
            }
#pragma unroll
            for (int k = 0; k < S::kQPerWarp; ++k) {
                if (k >= nk) break;
                const int vr = G == 1 ? sg : p.seg_vrow[sg] + q0 + k;
                const float sc = scs[k];
                if (j < p.valid[vr]) {
                    const bool fin = finite_f(sc);
                    st_global_hint(p.scores + (size_t)vr * p.score_stride + j, fin ? sc : -INFINITY, keep);
                    if (want_hist && fin) {
                        const uint32_t bin = score_key(sc) >> 21;
                        if (G == 1) atomicAdd(&hist_s[bin], 1u);
                        else atomicAdd(&hist_s[(q0 + k) * (kHistBins / 2) + (bin >> 1)], (bin & 1) ? 0x10000u : 1u);
                    }
                }
            }
        }
        if (want_hist && cur >= 0) {
            named_bar(1, kEpiThreads);
            flush(cur);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, S::kTmemCols);
    }
}

// One query per entry (decode) and up to kIndexerGroup queries per segment.
__global__ void __launch_bounds__(Shape<1>::kThreads, 1) indexer_score_kernel(const __grid_constant__ IndexerParams1 p) {
    indexer_score_body<1>(p);
}

__global__ void __launch_bounds__(Shape<kIndexerGroup>::kThreads, 1)
    indexer_score_group_kernel(const __grid_constant__ IndexerParamsG p) {
    indexer_score_body<kIndexerGroup>(p);
}

template <int G, class K>
static cudaError_t launch_group(K kernel, const ParamsOf<G>& p, int num_sms, cudaStream_t stream, bool pdl) {
    static std::atomic<uint64_t> smem_set{0};
    constexpr size_t bytes = smem_bytes<G>();
    const cudaError_t err = set_smem_limit_once(kernel, bytes, smem_set);
    if (err != cudaSuccess) return err;
    const uint32_t grid = p.total_tiles < (uint32_t)num_sms ? p.total_tiles : (uint32_t)num_sms;
    return launch_kernel(kernel, dim3(grid), dim3(Shape<G>::kThreads), bytes, stream, pdl, p);
}

static_assert(std::is_same<ParamsOf<1>, IndexerParams1>::value, "one-query table");
static_assert(std::is_same<ParamsOf<kIndexerGroup>, IndexerParamsG>::value, "grouped table");

cudaError_t launch_indexer(const IndexerParams1& p, int num_sms, cudaStream_t stream, bool pdl) {
    if (p.total_tiles == 0) return cudaSuccess;
    return launch_group<1>(indexer_score_kernel, p, num_sms, stream, pdl);
}

cudaError_t launch_indexer(const IndexerParamsG& p, int num_sms, cudaStream_t stream, bool pdl) {
    if (p.total_tiles == 0) return cudaSuccess;
    return launch_group<kIndexerGroup>(indexer_score_group_kernel, p, num_sms, stream, pdl);
}

uint32_t indexer_tile_keys() { return kTileKeys; }

}  // namespace dsrows
