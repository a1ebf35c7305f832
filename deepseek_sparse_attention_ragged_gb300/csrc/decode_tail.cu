// Top-k selection and sink-softmax sparse attention of each row in one kernel
// (mlx-native deepseek_rows.metal: the top-k kernels
// deepseek_indexer_topk_*_rows_i32 followed by
// deepseek_sparse_attention_score_rows_bf16 / _reduce_rows_bf16; gather
// semantics of deepseek_sparse_attention_gather_rows_bf16).
//
// Per row e and head h over the selected slots t (index i_t):
//   l_t = scale * q_h . KV[i_t],  m = max(sink_h, max l_t),
//   den = exp(sink_h - m) + sum exp(l_t - m),  out_h = sum exp(l_t - m) KV[i_t] / den.
//
// One 8-CTA thread-block cluster per row, 512 threads per CTA. CTA r owns the
// 128-slot chunk c = r / 2 and the head half r % 2 (32 heads).
//   1. select (decode only): every CTA streams its slice of the row's scores
//      and stores the candidates at or above the level-0 threshold bin, in
//      index order, into the shared memory of every CTA of the cluster (an
//      all-gather); after one cluster barrier each CTA refines the exact
//      threshold over the gathered candidates and places the winners in index
//      order: slot t holds the winner with the t-th smallest index. Every CTA
//      computes the same selection, so no winner or slot crosses the cluster.
//      The caller's best-first index list comes from a ninth cluster, which
//      sorts each row's published winners best first (or, without attention,
//      from each CTA ranking its 64 slots). With indices given by the caller,
//      each CTA sorts them ascending (sentinels last) into the same slot order;
//   2. attend, on tcgen05 tensor cores with fp32 accumulators in TMEM: gather
//      the chunk's 128 KV rows into the 128-byte-swizzled K-major layout, then
//        logits  D[128 slots x 32 heads] = KV_chunk . Q_half^T   (K = 512,
//                as four accumulators over the K-steps k = a mod 4, added
//                as (D0 + D1) + (D2 + D3)),
//      the chunk softmax (max and sum over the 128 slots, per head), and
//        P G     D[128 features x 64] = KV_chunk^T . [P_hi; P_lo]^T  (K = 128 slots)
//      for the four 128-feature blocks, where the same KV buffer is the
//      MN-major operand and P enters as a bf16 hi + lo pair stacked along N
//      (acc = D[:, h] + D[:, 32 + h]);
//   3. combine: the chunk partials go to the workspace (the feature block a
//      CTA combines itself stays in its shared memory); after a cluster
//      barrier CTA r combines feature columns [128 c, 128 c + 128) of its 32
//      heads over the chunks in chunk order:
//        m = max(sink, m_c), den = exp(sink - m) + sum_c l_c exp(m_c - m),
//        out = sum_c acc_c exp(m_c - m) / den.
// Every reduction order depends on the row's width and its indices alone, and
// the stand-alone attention runs this kernel on the caller's indices in the
// same ascending order, so the decode's output is bitwise the attention of
// its own best-first index list.
//
// Fail-closed rules: a caller's index < -1 or >= kv_len flags the whole row; a
// non-finite logit (non-finite q or KV element, or overflow) flags its head;
// a non-finite sink or denominator flags the head; a flagged head is written
// as zeros, and any non-finite output element is written as zero.
//
// Bounded waits: a wait for the tensor cores that gives up (DS_STATUS_WAIT_TIMEOUT)
// stops the CTA's attention work (no further MMA, no TMEM read) and flags the
// row, so every head of it is written as zeros; the CTA still takes part in
// every cluster barrier, and before it frees TMEM it waits (bounded) once more
// for the MMAs it issued.

#include <cooperative_groups.h>

#include "attend.cuh"
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace dsrows {

namespace cg = cooperative_groups;
using attend::combine_slice;
using attend::cp_async16;
using attend::cp_async4;
using attend::cp_async_commit;
using attend::cp_async_wait_all;
using namespace rowsel;

namespace {

constexpr int kChunkSlots = 128;                         // slots per chunk (UMMA M of the logits)
constexpr int kHalfHeads = kHeads / 2;                   // heads per CTA (UMMA N)
constexpr uint32_t kTmemCols = 512;                      // logits (4 x 32) + P G (4 x 64)
constexpr uint32_t kPvCol = 128;                         // first TMEM column of P G
// MMAs are issued by one thread in each of this many warps, into independent
// accumulators: one thread issues a tcgen05.mma in about 80 cycles, far longer
// than these N=32/64 MMAs take, so the issue rate sets the phase's time.
constexpr int kIssuers = 4;
constexpr int kGBlock = kChunkSlots * 128;               // one 64-column block of the KV rows: 16 KiB
constexpr int kQBlock = kHalfHeads * 128;                // one 64-column block of the query half: 4 KiB
constexpr int kPBlock = 2 * kHalfHeads * 128;            // 64 slots of [P_hi; P_lo] (64 rows): 8 KiB
static_assert(kCluster * kChunkSlots == 2 * kTopK, "4 chunks x 2 head halves per row");
static_assert(kThreads == 512, "16 warps");

struct TailLayout {
    static constexpr size_t g = 0;                                     // KV rows [128][512], K-major SW128
    static constexpr size_t q = g + 8 * (size_t)kGBlock;               // query half [32][512], K-major SW128
    static constexpr size_t pmat = q + 8 * (size_t)kQBlock;            // [P_hi; P_lo] [64][128 slots], K-major SW128
    static constexpr size_t idx = pmat + 2 * (size_t)kPBlock;          // i32 [128] this chunk's slots
    static constexpr size_t sel = idx + (size_t)kChunkSlots * 4;       // u64 [512] the row's winners
    static constexpr size_t red = sel + (size_t)kTopK * 8;             // [4 quarters][32 heads] max, sum, bad
    static constexpr size_t misc = red + 3 * 4 * (size_t)kHalfHeads * 4;
    static constexpr size_t sinks = misc + 64;                         // f32 [32] this head half's sinks
    static constexpr size_t ranks = sinks + (size_t)kHalfHeads * 4;    // u32 [64] best-first ranks
    static constexpr size_t total = ranks + 64 * 4;
    // Aliases used before the KV rows are gathered and P is written: the
    // gathered candidates ([8][kCandCap] u64) and the selection state.
    static constexpr size_t regions = g;
    static constexpr size_t gather = pmat;
};
static_assert(TailLayout::regions + (size_t)kCluster * kCandCap * 8 <= TailLayout::q, "candidates overlap the query");
static_assert(TailLayout::gather + sizeof(GatherSmem) <= TailLayout::idx, "selection state overlaps the slots");
static_assert(TailLayout::misc % 8 == 0, "alignment");
constexpr size_t kTailSmem = TailLayout::total + 1024;  // + slack to align the swizzled buffers to 1 KiB
static_assert(kTailSmem <= 227 * 1024, "shared memory");

// Maximum over the warp, in the integer reduction unit: finite values and
// -inf map order-preservingly to int (no NaN reaches here).
__device__ __forceinline__ float warp_max(float x) {
    const int i = __float_as_int(x);
    const int r = __reduce_max_sync(0xFFFFFFFFu, i >= 0 ? i : i ^ 0x7FFFFFFF);
    return __int_as_float(r >= 0 ? r : r ^ 0x7FFFFFFF);
}

// Byte offset of 16-byte chunk ch (0..63) of row r in a K-major SW128 buffer of
// 64-column blocks `block` bytes apart (rows of 128 B per block).
__device__ __forceinline__ uint32_t sw128_chunk(int r, int ch, int block) {
    return (uint32_t)((ch >> 3) * block + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

}  // namespace

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tail_kernel(const TailParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using T = TailLayout;
    uint8_t* g_s = smem + T::g;
    uint8_t* q_s = smem + T::q;
    uint8_t* p_s = smem + T::pmat;
    int* idx_s = reinterpret_cast<int*>(smem + T::idx);
    uint64_t* sel = reinterpret_cast<uint64_t*>(smem + T::sel);
    float* red_max = reinterpret_cast<float*>(smem + T::red);
    float* red_sum = red_max + 4 * kHalfHeads;
    uint32_t* red_bad = reinterpret_cast<uint32_t*>(red_sum + 4 * kHalfHeads);
    uint32_t* tmem_s = reinterpret_cast<uint32_t*>(smem + T::misc);
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(smem + T::misc + 8);
    float* sinks_s = reinterpret_cast<float*>(smem + T::sinks);
    uint64_t* regions = reinterpret_cast<uint64_t*>(smem + T::regions);
    float* own_s = reinterpret_cast<float*>(smem + T::g);  // after P·G: this CTA's combined feature block
    GatherSmem& gs = *reinterpret_cast<GatherSmem*>(smem + T::gather);

    // The stream's next kernel may launch while this one runs: it waits for this
    // grid to complete (griddepcontrol.wait) before it reads or writes anything
    // this kernel uses.
    pdl_trigger();
    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t rank = cluster.block_rank();
    const int e = blockIdx.x / kCluster;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    // With attention: [8] "winners published" flags after the row flags, and the
    // winners' numbers after the published winners.
    auto pub_flag = [&](uint32_t r) { return p.flags + kRowsMax * kHeads + kRowsMax + r; };
    auto pub_n = [&](uint32_t r) { return reinterpret_cast<uint32_t*>(p.pub + (size_t)kRowsMax * kTopK) + r; };

    if (e >= (int)p.rows) {
        // ---- one more cluster ranks the rows' winners (decode with attention):
        // CTA r waits for row r to publish its winners in index order, sorts
        // them best first and writes the row's index list. No row waits for it.
        const uint32_t re = rank;
        if (re >= p.rows) return;
        pdl_wait();  // the publish flags were zeroed by earlier work
        uint32_t ok = 1;
        if (t == 0) {
            const uint64_t start = global_timer_ns();
            while (ld_acquire_gpu(pub_flag(re)) == 0)
                if (global_timer_ns() - start > kWaitBudgetNs) {
                    atomicOr(p.status, kStatusWaitTimeout);
                    ok = 0;
                    break;
                }
        }
        ok = __syncthreads_and(t != 0 || ok);
        __threadfence();
        const uint64_t x0 = ok ? __ldcg(p.pub + (size_t)re * kTopK + t) : 0ull;
        const uint32_t nsel = ok ? __ldcg(pub_n(re)) : 0u;
        const uint64_t x = bitonic512_desc(x0, reinterpret_cast<uint64_t*>(gs.h));
        if ((uint32_t)t < p.width[re])
            p.indices[p.index_offset[re] + t] = (uint32_t)t < nsel ? (int32_t)(~(uint32_t)x) + p.offset[re] : -1;
        return;
    }

    const uint32_t c = rank >> 1;          // chunk: slots [128 c, 128 c + 128)
    const int half = (int)(rank & 1);      // heads [32 half, 32 half + 32)
    const int head0 = half * kHalfHeads;
    const uint32_t L = p.kv_len[e];
    const uint32_t W = p.width[e];
    const uint32_t q_row = p.q_row[e];
    const uint32_t nchunks = (W + kChunkSlots - 1) / kChunkSlots;
    const bool has_chunk = c < nchunks;

    // ---- setup: counters, barrier, TMEM, and the query (an input of the call) --
    if (t == 0) {
        mbar_init(mma_bar, kIssuers);
        fence_barrier_init();
    }
    if (t < kChunkSlots) idx_s[t] = -1;  // slots past the last winner stay empty
    sel[t] = 0;
    if (warp == 0 && p.attend) {
        tmem_alloc(tmem_s, kTmemCols);
        tmem_relinquish();
    }
    // The query half (cp.async into the swizzled layout; waited for before the
    // logits) and the sinks (possibly in host memory; the combine uses them last).
    auto fetch_inputs = [&]() {
        const __nv_bfloat16* qh = p.q + ((size_t)q_row * kHeads + head0) * kDim;
        for (int k = t; k < kHalfHeads * (kDim / 8); k += kThreads) {
            const int h = k >> 6, ch = k & 63;
            cp_async16(q_s + sw128_chunk(h, ch, kQBlock), qh + (size_t)h * kDim + ch * 8);
        }
        if (t < kHalfHeads) cp_async4(sinks_s + t, p.sinks + (size_t)q_row * p.sinks_row_stride + head0 + t);
        cp_async_commit();
    };
    if (p.attend && !p.q_after_wait) fetch_inputs();
    tc_fence_before();
    cluster.sync();  // every CTA's counters are set before anyone stores into them
    tc_fence_after();
    const uint32_t tmem = p.attend ? *tmem_s : 0u;
    pdl_wait();  // scores and histogram (decode) or indices (caller) come from earlier work
    if (p.attend && p.q_after_wait) fetch_inputs();

    const uint32_t first = c * kChunkSlots;
    uint32_t nsel = 0;
    if (p.given == nullptr) {
        // ---- select: gather the candidates, then every CTA selects the same winners
        const float* s = p.scores + (size_t)e * p.score_stride;
        const Gathered gat = select_collect_all(s, L, W, p.hist + (size_t)e * kHistBins, rank, gs, regions);
        cluster.sync();  // every CTA's candidates are in every CTA; no CTA touches
                         // another's shared memory after this barrier
        nsel = select_slots(gat, s, L, W, gs, regions, sel, idx_s, first, p.status);
    } else {
        // ---- the caller's indices, in ascending order (sentinels last): the
        // attention is a function of the index multiset. An index < -1 or
        // >= kv_len flags the row (it is written as zeros) and takes no slot.
        uint64_t v = 0;
        if ((uint32_t)t < W) {
            const int g = __ldcg(p.given + p.index_offset[e] + t);
            if (g < -1 || g >= (int)L) atomicOr(&p.flags[kRowsMax * kHeads + e], 1u);
            else if (g >= 0) v = (uint64_t)(~(uint32_t)g);
        }
        v = bitonic512_desc(v, reinterpret_cast<uint64_t*>(gs.h));
        if ((uint32_t)t - first < (uint32_t)kChunkSlots && v != 0) idx_s[t - first] = (int32_t)(~(uint32_t)v);
    }
    __syncthreads();  // this chunk's slots are in place (and the candidates consumed)
    // Publish the winners (index order) for the ranking cluster. The flag that
    // releases them is set after the gather is issued, by a thread that issues
    // no MMA, so the fence does not delay this CTA's attention.
    constexpr int kPublisher = kThreads - 32;
    const bool publish = p.ranker && rank == 0;
    if (publish) {
        p.pub[(size_t)e * kTopK + t] = sel[t];
        if (t == 0) *pub_n(e) = nsel;
    }
    // The gather of the chunk's KV rows starts now.
    const size_t part0_off = ((size_t)2 * p.chunk_begin[e] + (size_t)half * nchunks) * kPartFloats;
    if (has_chunk && p.attend) {
        const __nv_bfloat16* kv = p.kv[e];
        for (int k = t; k < kChunkSlots * (kDim / 8); k += kThreads) {
            const int r = k >> 6, ch = k & 63;
            const int i = idx_s[r];
            uint8_t* dst = g_s + sw128_chunk(r, ch, kGBlock);
            if (i >= 0 && (uint32_t)i < L) cp_async16(dst, kv + (size_t)i * kDim + ch * 8);
            else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
    }
    // Best-first ranks (decode): CTA `rank` ranks the winners of slots
    // [64 rank, 64 rank + 64) against all of them (group t / 64 of 64 each) and
    // writes their indices at their ranks; slots past the last winner (up to
    // the width) are -1. With attention this runs inside the cluster barrier
    // that precedes the combine.
    auto rank_indices = [&]() {
        uint32_t* rk = reinterpret_cast<uint32_t*>(smem + T::ranks);
        if (t < 64) rk[t] = 0;
        __syncthreads();
        const uint32_t k = rank * 64 + (uint32_t)(t & 63);
        const uint64_t ck = sel[k];
        const uint64_t* grp = sel + (t >> 6) * 64;
        uint32_t nb = 0;
#pragma unroll 16
        for (int j = 0; j < 64; ++j) nb += grp[j] > ck ? 1u : 0u;
        atomicAdd(&rk[t & 63], nb);
        __syncthreads();
        if (t < 64) {
            int32_t* out = p.indices + p.index_offset[e];
            if (k < nsel) out[rk[t]] = (int32_t)(~(uint32_t)ck) + p.offset[e];
            else if (k < W) out[k] = -1;
        }
    };
    const bool want_ranks = p.given == nullptr && p.indices != nullptr && !p.ranker;
    if (!p.attend) {
        if (want_ranks) rank_indices();
        return;
    }

    // ---- attend: 128 slots x 32 heads on the tensor cores ------------------------
    cp_async_wait_all();      // the query and the KV rows
    fence_proxy_async_smem();  // ... are visible to the tensor cores
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (publish && t == kPublisher) {
        // Every thread's winner store precedes the barrier above.
        __threadfence();
        st_release_gpu(pub_flag(e), 1u);
    }

    // `alive`: every tensor-core wait of this CTA has succeeded (uniform over the
    // CTA); `pending`: the mma_bar phase of MMAs whose completion was not seen.
    bool alive = true;
    int pending = -1;
    if (has_chunk) {
        const uint32_t g_addr = smem_u32(g_s), q_addr = smem_u32(q_s);
        if (lane == 0 && warp < kIssuers) {
            // Accumulator a = warp takes the K-steps kk = 4 j + a.
            constexpr uint32_t idesc = idesc_bf16_f32(128, kHalfHeads);
            const uint32_t koff = (uint32_t)warp * 32;  // 16 bf16 = 32 B inside the 128-B row
#pragma unroll
            for (int j = 0; j < kDim / 64; ++j)
                umma_bf16(tmem + 32 * warp, smem_desc_sw128_kmajor(g_addr + j * kGBlock + koff),
                          smem_desc_sw128_kmajor(q_addr + j * kQBlock + koff), idesc, j > 0 ? 1u : 0u);
            umma_commit(mma_bar);
        }
    }
    if (has_chunk) {
        alive = __syncthreads_and(mbar_wait(mma_bar, 0, p.status)) != 0;
        if (!alive) pending = 0;
    }
    if (has_chunk && alive) {
        tc_fence_after();
        // ---- chunk softmax: warp -> (32 slots, 8 heads), lane -> one slot ----------
        const int qt = warp & 3, hg = warp >> 2;
        const int slot = 32 * qt + lane;
        uint32_t v[4][8];
#pragma unroll
        for (int a = 0; a < 4; ++a) tmem_ld_x8(tmem + ((uint32_t)(32 * qt) << 16) + 32 * a + 8 * hg, v[a]);
        tmem_ld_wait();
        const bool live = idx_s[slot] >= 0;
        float l[8], m[8];
        uint32_t bad_bits = 0;  // head i of this warp's 8 has a non-finite live logit
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            l[i] = ((__uint_as_float(v[0][i]) + __uint_as_float(v[1][i])) +
                    (__uint_as_float(v[2][i]) + __uint_as_float(v[3][i]))) * p.scale;
            const bool ok = live && finite_f(l[i]);
            bad_bits |= (live && !ok) ? 1u << i : 0u;
            if (!ok) l[i] = -INFINITY;
            m[i] = warp_max(l[i]);
        }
        bad_bits = __reduce_or_sync(0xFFFFFFFFu, bad_bits);
        if (lane == 0)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                red_max[qt * kHalfHeads + 8 * hg + i] = m[i];
                red_bad[qt * kHalfHeads + 8 * hg + i] = (bad_bits >> i) & 1u;
            }
        __syncthreads();
        float sum[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int h = 8 * hg + i;
            const float mh = fmaxf(fmaxf(red_max[h], red_max[kHalfHeads + h]),
                                   fmaxf(red_max[2 * kHalfHeads + h], red_max[3 * kHalfHeads + h]));
            const float w = l[i] == -INFINITY ? 0.0f : expf(l[i] - mh);
            const __nv_bfloat16 hi = __float2bfloat16_rn(w);
            const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
            // Row h holds P_hi, row 32 + h P_lo (same swizzle phase: 32 is a multiple of 8).
            const uint32_t off = (uint32_t)((slot >> 6) * kPBlock + h * 128 +
                                            ((((slot & 63) >> 3) ^ (h & 7)) << 4) + ((slot & 7) << 1));
            *reinterpret_cast<__nv_bfloat16*>(p_s + off) = hi;
            *reinterpret_cast<__nv_bfloat16*>(p_s + off + kHalfHeads * 128) = lo;
            sum[i] = w;
        }
        fence_proxy_async_smem();  // P is visible to the tensor cores
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t g_addr = smem_u32(g_s);
        if (lane == 0 && warp < kIssuers) {
            // Feature block b = warp: features [128 b, 128 b + 128).
            constexpr uint32_t idesc = idesc_bf16_f32(128, 2 * kHalfHeads) | kIdescAMnMajor;
            const uint32_t p_addr = smem_u32(p_s);
            const int b = warp;
#pragma unroll
            for (int ks = 0; ks < kChunkSlots / 16; ++ks) {
                // A: features [128 b, 128 b + 128) x slots [16 ks, 16 ks + 16), MN-major.
                const uint64_t ad = smem_desc_sw128_mnmajor(g_addr + 2 * b * kGBlock + ks * 2048, kGBlock, 1024);
                const uint64_t bd = smem_desc_sw128_kmajor(p_addr + (ks >> 2) * kPBlock + (ks & 3) * 32);
                umma_bf16(tmem + kPvCol + 64 * b, ad, bd, idesc, ks != 0 ? 1u : 0u);
            }
            umma_commit(mma_bar);
        }
        // While the tensor cores run P G: the chunk's sum per head (a fixed warp
        // tree, then the four quarters) and the head flags.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i) sum[i] += __shfl_xor_sync(0xFFFFFFFFu, sum[i], o);
        if (lane == 0)
#pragma unroll
            for (int i = 0; i < 8; ++i) red_sum[qt * kHalfHeads + 8 * hg + i] = sum[i];
        __syncthreads();
        float* part = p.part + part0_off + (size_t)c * kPartFloats;
        if (t < kHalfHeads) {
            const float mh = fmaxf(fmaxf(red_max[t], red_max[kHalfHeads + t]),
                                   fmaxf(red_max[2 * kHalfHeads + t], red_max[3 * kHalfHeads + t]));
            part[t] = mh;
            part[kHalfHeads + t] = (red_sum[t] + red_sum[kHalfHeads + t]) +
                                   (red_sum[2 * kHalfHeads + t] + red_sum[3 * kHalfHeads + t]);
            if (red_bad[t] | red_bad[kHalfHeads + t] | red_bad[2 * kHalfHeads + t] | red_bad[3 * kHalfHeads + t])
                atomicOr(&p.flags[e * kHeads + head0 + t], 1u);
        }
        alive = __syncthreads_and(mbar_wait(mma_bar, 1, p.status)) != 0;
        if (!alive) pending = 1;
        if (alive) {
            tc_fence_after();
            // ---- partial: warp -> (32 features, 32 heads) of block warp / 4 -------------
            const int b = warp >> 2;
            uint32_t ahi[32], alo[32];
            const uint32_t tcol = tmem + ((uint32_t)(32 * qt) << 16) + kPvCol + 64 * b;
            tmem_ld_x32(tcol, ahi);
            tmem_ld_x32(tcol + kHalfHeads, alo);
            tmem_ld_wait();
            if (b == (int)c) {
                // Feature block c is combined by this CTA: it stays in shared
                // memory (the KV buffer is free once P·G is done), [32 heads][128].
                float* o = own_s + 32 * qt + lane;
#pragma unroll
                for (int h = 0; h < kHalfHeads; ++h) o[h * 128] = __uint_as_float(ahi[h]) + __uint_as_float(alo[h]);
            } else {
                float* pacc = part + 2 * kHalfHeads + 128 * b + 32 * qt + lane;
#pragma unroll
                for (int h = 0; h < kHalfHeads; ++h)
                    pacc[(size_t)h * kDim] = __uint_as_float(ahi[h]) + __uint_as_float(alo[h]);
            }
        }
    }
    // A CTA whose tensor-core wait gave up has no valid partial: the whole row
    // is written as zeros.
    if (!alive && t == 0) atomicOr(&p.flags[kRowsMax * kHeads + e], 1u);
    tc_fence_before();
    // Every chunk's partial and flags are visible to the cluster after this
    // barrier; the best-first ranks are written while it completes.
    cluster_arrive_release();
    if (want_ranks) rank_indices();
    cluster_wait_acquire();
    tc_fence_after();

    // ---- combine: feature columns [128 c, 128 c + 128) of the 32 heads ----------
    combine_slice<kHalfHeads, kThreads, 128>(
        p.part + part0_off, kPartFloats, (int)nchunks, (int)(128 * c), own_s, has_chunk ? (int)c : -1, sinks_s,
        p.flags + kRowsMax * kHeads + e, p.flags + e * kHeads + head0,
        p.out + ((size_t)q_row * kHeads + head0) * kDim,
        p.invalid && c == 0 ? p.invalid + (size_t)q_row * kHeads + head0 : nullptr);

    // MMAs whose completion was not seen may still write TMEM: wait once more
    // (bounded) before it is freed.
    if (pending >= 0) (void)mbar_wait(mma_bar, (uint32_t)pending, nullptr);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

size_t decode_tail_smem_bytes() { return kTailSmem; }

cudaError_t launch_decode_tail(const TailParams& p, cudaStream_t stream, bool pdl) {
    static std::atomic<uint64_t> smem_set{0};
    const cudaError_t err = set_smem_limit_once(decode_tail_kernel, kTailSmem, smem_set);
    if (err != cudaSuccess) return err;
    if (p.rows == 0) return cudaSuccess;
    const uint32_t clusters = p.rows + (p.ranker ? 1u : 0u);
    return launch_kernel(decode_tail_kernel, dim3(clusters * kCluster), dim3(kThreads), kTailSmem, stream, pdl, p);
}

}  // namespace dsrows
