// The decode step after the indexer: top-k selection and sink-softmax sparse
// attention of each row in one kernel (mlx-native deepseek_rows.metal: the
// top-k kernels deepseek_indexer_topk_*_rows_i32 followed by
// deepseek_sparse_attention_score_rows_bf16 / _reduce_rows_bf16).
//
// One 8-CTA thread-block cluster per row, 512 threads per CTA:
//   1. select: every CTA streams its slice of the row's scores and appends the
//      candidates at or above the level-0 threshold bin to the leader's shared
//      memory; the leader refines and keeps the winners' composites;
//   2. place: every CTA ranks 64 of the winners against all of them by
//      composite (score descending, lower index first): that rank is the
//      winner's slot, both in the caller's best-first index list and in the
//      attention, and the CTA stores the index into the shared memory of the
//      CTA that owns the slot;
//   3. attend: CTA r takes slots [64 r, 64 r + 64) for all 64 heads:
//      bulk-copies the 64 KV rows, then logits, chunk softmax and P G (the
//      query was fetched while the indexer was running); the chunk partial
//      goes to the workspace;
//   4. combine: after a cluster barrier CTA r combines feature columns
//      [64 r, 64 r + 64) of every head over the chunks, in chunk order.
// Per output element the operations and their order are those of the
// stand-alone attention kernels, so the decode's output is bitwise the
// attention of its own best-first index list.

#include <cooperative_groups.h>

#include "attend.cuh"
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace dsrows {

namespace cg = cooperative_groups;
using namespace attend;
using namespace rowsel;

namespace {

constexpr int kRowBytes = kDim * 2;
constexpr size_t kTailPartFloats = 2 * kHeads + (size_t)kHeads * kDim;  // m[64], l[64], acc[64][512]
static_assert(kTailPartFloats == 2 * kPartFloats, "a chunk's partial fills the space of its two head halves");

struct TailLayout {
    static constexpr size_t q = 0;                                       // bf16 [64][kQStride]
    static constexpr size_t g = q + (size_t)kHeads * kQStride * 2;       // bf16 [64][kQStride]
    static constexpr size_t lg = g + (size_t)kSlots * kQStride * 2;      // f32 [64][kLgStride]
    static constexpr size_t p_hi = lg + (size_t)kHeads * kLgStride * 4;  // bf16 [64][kPStride]
    static constexpr size_t p_lo = p_hi + (size_t)kHeads * kPStride * 2;
    static constexpr size_t idx = p_lo + (size_t)kHeads * kPStride * 2;  // i32 [64] this CTA's slots
    static constexpr size_t sel = idx + (size_t)kSlots * 4;              // u64 [512] winners (leader)
    static constexpr size_t nsel = sel + (size_t)kTopK * 8;              // u32 number of winners (leader)
    static constexpr size_t gbar = nsel + 16;                            // mbarrier of the KV copies
    static constexpr size_t cs = gbar + 16;                              // CombineSmem<64>
    static constexpr size_t total = cs + sizeof(CombineSmem<kHeads>);
    // Aliases of the KV rows' space, used before the copies land.
    static constexpr size_t select = g;                                  // SelectSmem (select phase)
    static constexpr size_t selcopy = g;                                 // u64 [512] (place phase)
    static constexpr size_t ranks = g + (size_t)kTopK * 8;               // u32 [64] (place phase)
};
static_assert(TailLayout::select + sizeof(SelectSmem) <= TailLayout::p_hi, "select state overlaps P");
static_assert(TailLayout::gbar % 8 == 0 && TailLayout::sel % 8 == 0, "alignment");
static_assert(TailLayout::total <= 227 * 1024, "shared memory");
static_assert(kThreads == 512 && kCluster * kSlots == kTopK, "one 64-slot chunk per CTA");

}  // namespace

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tail_kernel(const TailParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    using T = TailLayout;
    __nv_bfloat16* q_s = reinterpret_cast<__nv_bfloat16*>(smem + T::q);
    __nv_bfloat16* g_s = reinterpret_cast<__nv_bfloat16*>(smem + T::g);
    float* lg_s = reinterpret_cast<float*>(smem + T::lg);
    __nv_bfloat16* ph_s = reinterpret_cast<__nv_bfloat16*>(smem + T::p_hi);
    __nv_bfloat16* pl_s = reinterpret_cast<__nv_bfloat16*>(smem + T::p_lo);
    int* idx_s = reinterpret_cast<int*>(smem + T::idx);
    uint64_t* sel = reinterpret_cast<uint64_t*>(smem + T::sel);
    uint32_t* nsel_s = reinterpret_cast<uint32_t*>(smem + T::nsel);
    uint64_t* gbar = reinterpret_cast<uint64_t*>(smem + T::gbar);
    CombineSmem<kHeads>& cs = *reinterpret_cast<CombineSmem<kHeads>*>(smem + T::cs);
    SelectSmem& sm = *reinterpret_cast<SelectSmem*>(smem + T::select);

    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t rank = cluster.block_rank();
    const int e = blockIdx.x / kCluster;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const uint32_t L = p.kv_len[e];
    const uint32_t W = p.width[e];
    const uint32_t q_row = p.q_row[e];
    const float* s = p.scores + (size_t)e * p.score_stride;
    SelectSmem& leader = *cluster.map_shared_rank(&sm, 0);

    // ---- select --------------------------------------------------------------
    if (t == 0) {
        sm.ncand = 0;
        mbar_init(gbar, 1);
        fence_barrier_init();
    }
    // The query is an input of the call: fetch it while the indexer finishes.
    load_q<kHeads, kThreads>(q_s, p.q + (size_t)q_row * kHeads * kDim, t);
    cp_async_commit();
    cluster.sync();  // the leader's counters are zero before anyone appends
    pdl_wait();      // scores and histogram come from the indexer
    const Collected col = select_collect(s, L, W, p.hist + (size_t)e * kHistBins, rank, sm, leader);
    cluster.sync();  // every append into the leader is visible to it
    if (rank == 0) {
        const uint32_t n = select_finish(col, s, L, W, false, nullptr, sm, sel, p.status);
        if (t == 0) *nsel_s = n;
    }
    cluster.sync();  // the winners are visible to the cluster

    // ---- place: rank 64 winners, store them in their slots ---------------------
    {
        const uint32_t nsel = *cluster.map_shared_rank(nsel_s, 0);
        uint64_t* sc = reinterpret_cast<uint64_t*>(smem + T::selcopy);
        uint32_t* rk = reinterpret_cast<uint32_t*>(smem + T::ranks);
        sc[t] = (uint32_t)t < nsel ? cluster.map_shared_rank(sel, 0)[t] : 0ull;
        if (t < kSlots) rk[t] = 0;
        // Slots of this CTA past the last winner are empty.
        if (t < kSlots && rank * kSlots + (uint32_t)t >= nsel) idx_s[t] = -1;
        __syncthreads();
        // Winner k against the 64 winners of group t / 64: how many are better
        // (the zero padding never is; composites are distinct).
        const uint32_t k = rank * kSlots + (uint32_t)(t & (kSlots - 1));
        const uint64_t ck = sc[k];
        const uint64_t* grp = sc + (t >> 6) * kSlots;
        uint32_t nb = 0;
#pragma unroll 16
        for (int j = 0; j < kSlots; ++j) nb += grp[j] > ck ? 1u : 0u;
        atomicAdd(&rk[t & (kSlots - 1)], nb);
        __syncthreads();
        if (t < kSlots) {
            int32_t* out = p.indices ? p.indices + p.index_offset[e] : nullptr;
            if (k < nsel) {
                const uint32_t pos = rk[t];
                const int32_t j = (int32_t)(~(uint32_t)ck);
                if (out) out[pos] = j;
                cluster.map_shared_rank(idx_s, pos / kSlots)[pos % kSlots] = j;
            } else if (out && k < W) {
                out[k] = -1;
            }
        }
    }
    cluster.sync();  // every CTA's slots are in place

    // ---- attend: slots [64 rank, 64 rank + 64) for all 64 heads ----------------
    const uint32_t nchunks = (W + kSlots - 1) / kSlots;
    const bool has_chunk = rank < nchunks;
    float* part0 = p.part + (size_t)p.chunk_begin[e] * kTailPartFloats;  // this row's first partial
    if (has_chunk) {
        // The KV rows' space held generic-proxy data: order it before the copies.
        fence_proxy_async_smem();
        const int live = __syncthreads_count(t < kSlots && idx_s[t] >= 0);
        if (t == 0) mbar_arrive_expect_tx(gbar, (uint32_t)live * kRowBytes);
        if (t < kSlots) {
            const int i = idx_s[t];
            __nv_bfloat16* dst = g_s + t * kQStride;
            if (i >= 0) {
                bulk_copy_g2s(dst, p.kv[e] + (size_t)i * kDim, kRowBytes, gbar);
            } else {
                for (int c = 0; c < kDim / 8; ++c) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
            }
        }
        mbar_wait(gbar, 0, p.status);
        cp_async_wait_all();  // the query
        __syncthreads();

        logits<kHeads>(q_s, g_s, lg_s, p.scale, warp, lane);
        __syncthreads();
        float* part = part0 + (size_t)rank * kTailPartFloats;
        softmax<4>(lg_s, idx_s, ph_s, pl_s, warp, lane, [&](int h, float m, float l, bool bad) {
            if (bad) atomicOr(&p.flags[e * kHeads + h], 1u);
            part[h] = m;
            part[kHeads + h] = l;
        });
        __syncthreads();
        float acc[16][4];
        pv<128>(ph_s, pl_s, g_s, warp, lane, acc);
        float* pacc = part + 2 * kHeads;
        const int h0 = 16 * (warp >> 2) + (lane >> 2);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int f = (warp & 3) * 128 + nt * 8 + 2 * (lane & 3);
            *reinterpret_cast<float2*>(pacc + (size_t)h0 * kDim + f) = make_float2(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<float2*>(pacc + (size_t)(h0 + 8) * kDim + f) = make_float2(acc[nt][2], acc[nt][3]);
        }
    }
    cluster.sync();  // every chunk's partial and head flags are visible to the cluster

    // ---- combine: feature columns [64 rank, 64 rank + 64) of every head --------
    combine_slice<kHeads, kThreads>(part0, kTailPartFloats, (int)nchunks, (int)rank * 64,
                                    p.sinks + (size_t)q_row * p.sinks_row_stride, false, p.flags + e * kHeads,
                                    p.out + (size_t)q_row * kHeads * kDim,
                                    p.invalid && rank == 0 ? p.invalid + (size_t)q_row * kHeads : nullptr, cs);
}

size_t decode_tail_smem_bytes() { return TailLayout::total; }

cudaError_t launch_decode_tail(const TailParams& p, cudaStream_t stream, bool pdl) {
    static bool configured = false;
    if (!configured) {
        cudaError_t err = cudaFuncSetAttribute(decode_tail_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)TailLayout::total);
        if (err != cudaSuccess) return err;
        configured = true;
    }
    if (p.rows == 0) return cudaSuccess;
    return launch_kernel(decode_tail_kernel, dim3(p.rows * kCluster), dim3(kThreads), TailLayout::total, stream, pdl,
                         p);
}

}  // namespace dsrows
