// Deterministic top-k over fp32 scores (mlx-native deepseek_rows.metal:
// index_rows_better and kernels deepseek_indexer_topk_block/merge/finalize_rows_i32).
//
// Order: score descending, then lower index; only finite scores take part;
// slots past the number of finite scores hold -1; -0.0 ties +0.0.
//
// GB300 design (no sort network over every score): each score is mapped to an
// order-preserving 32-bit key, and (key, index) to the 64-bit composite
//   c = key << 32 | ~index,
// which is distinct per element, so "the best `width`" is the set of the
// `width` largest composites, a pure function of the scores. The selection is
// a radix select that keeps each row on chip:
//   1. a 2048-bin histogram of the top 11 key bits per row (fused into the
//      indexer epilogue in the decode step, or the histogram kernel here);
//   2. one 8-CTA thread-block cluster per row: every CTA picks the bin of the
//      width-th best score from the histogram, streams its slice of the row
//      once, and appends the elements at or above that bin (typically width +
//      a few hundred) into the leader CTA's shared memory through distributed
//      shared memory;
//   3. after one cluster barrier the leader refines the threshold digit by
//      digit over its candidates (11/11/10 key bits, then the index bits,
//      stopping as soon as a bin is taken whole), keeps the `width` winners
//      and sorts them: 16 warp-level 32-element shuffle sorts, then four
//      merge rounds by binary search.
// A row whose threshold bin overflows the leader's candidate space is refined
// by the leader from the row's full score array (correct, slower).
// This kernel serves row sets of more than 8 rows (several queries per row).
// Up to 8 rows, the library selects with the attention kernel in
// selection-only mode instead: there every CTA of the cluster gathers all
// candidates and ranks its own slots, which beats one leader's sort.

#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace dsrows {

using namespace rowsel;

namespace {

constexpr int kChunk = 8192;
constexpr size_t kSelectSmemBytes = sizeof(SelectSmem) + kTopK * sizeof(uint64_t);  // + the winners

__device__ __forceinline__ int entry_of_chunk(const TopkParams& p, uint32_t c) {
    int e = 0;
    for (int i = 1; i < (int)p.rows; ++i)
        if (c >= p.chunk_begin[i]) e = i;
    return e;
}

}  // namespace

// Level-0 histogram of one chunk of a row's scores (stand-alone top-k).
__global__ void __launch_bounds__(kThreads) topk_hist_kernel(const TopkParams p) {
    __shared__ uint32_t h[kHistBins];
    pdl_trigger();
    pdl_wait();  // the histogram is being cleared by the previous kernel
    const int e = entry_of_chunk(p, blockIdx.x);
    const uint32_t c = blockIdx.x - p.chunk_begin[e];
    const uint32_t L = p.kv_len[e];
    const uint32_t begin = c * kChunk;
    const uint32_t end = min(L, begin + kChunk);
    for (int i = threadIdx.x; i < kHistBins; i += kThreads) h[i] = 0;
    __syncthreads();
    const float* s = p.scores + (size_t)e * p.score_stride;
    float v[kChunk / kThreads];
#pragma unroll
    for (int i = 0; i < kChunk / kThreads; ++i) {
        const uint32_t j = begin + threadIdx.x + i * kThreads;
        v[i] = j < end ? s[j] : __int_as_float(0x7FC00000);
    }
#pragma unroll
    for (int i = 0; i < kChunk / kThreads; ++i)
        if (finite_f(v[i])) atomicAdd(&h[score_key(v[i]) >> 21], 1u);
    __syncthreads();
    for (int i = threadIdx.x; i < kHistBins; i += kThreads)
        if (h[i]) atomicAdd(&p.hist[(size_t)e * kHistBins + i], h[i]);
}

// One 8-CTA cluster per row. Every CTA takes the level-0 threshold bin from
// the row's histogram, streams its slice of the scores once, and appends the
// candidates (finite, top 11 key bits >= that bin) and the level-1 histogram
// of the bin straight into the leader CTA's shared memory; after one cluster
// barrier the leader refines, sorts and writes the row.
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    topk_select_kernel(const TopkParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SelectSmem& sm = *reinterpret_cast<SelectSmem*>(smem_raw);
    uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw + sizeof(SelectSmem));
    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t rank = cluster.block_rank();
    const int e = blockIdx.x / kCluster;
    const uint32_t L = p.kv_len[e];
    const uint32_t width = p.width[e];
    const float* s = p.scores + (size_t)e * p.score_stride;
    SelectSmem& leader = *cluster.map_shared_rank(&sm, 0);

    if (threadIdx.x == 0) sm.ncand = 0;
    pdl_trigger();
    cluster.sync();  // the leader's counters are zero before anyone appends
    pdl_wait();      // scores and histogram come from the previous kernel
    const Collected c = select_collect(s, L, width, p.hist + (size_t)e * kHistBins, rank, sm, leader);
    cluster.sync();  // every append into the leader is visible to it
    if (rank != 0) return;
    select_finish(c, s, L, width, p.out + p.out_offset[e], sm, sel, p.status, p.offset[e]);
}

uint32_t topk_chunk() { return kChunk; }

cudaError_t launch_topk_hist(const TopkParams& p, cudaStream_t stream, bool pdl) {
    if (p.total_chunks == 0) return cudaSuccess;
    return launch_kernel(topk_hist_kernel, dim3(p.total_chunks), dim3(kThreads), 0, stream, pdl, p);
}

cudaError_t launch_topk_select(const TopkParams& p, cudaStream_t stream, bool pdl) {
    static std::atomic<uint64_t> smem_set{0};
    const cudaError_t err = set_smem_limit_once(topk_select_kernel, kSelectSmemBytes, smem_set);
    if (err != cudaSuccess) return err;
    return launch_kernel(topk_select_kernel, dim3(p.rows * kCluster), dim3(kThreads), kSelectSmemBytes, stream,
                         pdl, p);
}

// The first kernel of a call. It may be launched while the stream's previous
// kernel runs (programmatic launch); it waits for that kernel to complete
// before it writes anything, and only then lets the next kernel launch, so
// every input of the call is complete when that one starts.
__global__ void __launch_bounds__(1024) clear_kernel(uint32_t* __restrict__ p, uint32_t words) {
    pdl_wait();
    pdl_trigger();
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < words; i += gridDim.x * blockDim.x) p[i] = 0;
}

cudaError_t launch_clear(uint32_t* p, uint32_t words, cudaStream_t stream) {
    return launch_kernel(clear_kernel, dim3(16), dim3(1024), 0, stream, true, p, words);
}

// The library's bounded mbarrier wait on two phases of a shared-memory barrier
// with one expected arrival: phase 0, which this thread completes, and phase 1,
// which nothing completes (the wait must give up after budget_ns).
__global__ void wait_selftest_kernel(uint32_t* __restrict__ status, uint32_t* __restrict__ result,
                                     uint64_t budget_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_arrive(&bar);
    result[0] = mbar_wait(&bar, 0, status, budget_ns) ? 1u : 0u;
    result[1] = mbar_wait(&bar, 1, status, budget_ns) ? 0u : 1u;
}

cudaError_t launch_wait_selftest(uint32_t* status, uint32_t* result, uint64_t budget_ns, cudaStream_t stream) {
    return launch_kernel(wait_selftest_kernel, dim3(1), dim3(32), 0, stream, false, status, result, budget_ns);
}

// clear_kernel plus two 16-byte-granular copies (the indexer's query and head
// weights, from pinned host memory into device staging), with the same launch
// rules. The next kernel may start early; it waits for this one
// (griddepcontrol.wait) before it reads the copies.
__global__ void __launch_bounds__(1024) clear_copy_kernel(uint32_t* __restrict__ p, uint32_t words,
                                                          const uint4* __restrict__ a_src, uint4* __restrict__ a_dst,
                                                          uint32_t a_n, const uint4* __restrict__ b_src,
                                                          uint4* __restrict__ b_dst, uint32_t b_n) {
    pdl_wait();
    pdl_trigger();
    const uint32_t stride = gridDim.x * blockDim.x;
    const uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t n = a_n > b_n ? a_n : b_n;
    // Both host loads of an element are in flight before either store: one
    // round trip over the host link per element, not two.
    for (uint32_t i = i0; i < n; i += stride) {
        const bool ha = i < a_n, hb = i < b_n;
        uint4 av = make_uint4(0, 0, 0, 0), bv = av;
        if (ha) av = a_src[i];
        if (hb) bv = b_src[i];
        if (ha) a_dst[i] = av;
        if (hb) b_dst[i] = bv;
    }
    for (uint32_t i = i0; i < words; i += stride) p[i] = 0;
}

// 64 CTAs of 256 threads: the host loads go out from 64 SMs. The CTAs are
// small enough to share an SM with the indexer's.
cudaError_t launch_clear_copy(uint32_t* p, uint32_t words, const void* a_src, void* a_dst, size_t a_bytes,
                              const void* b_src, void* b_dst, size_t b_bytes, cudaStream_t stream) {
    return launch_kernel(clear_copy_kernel, dim3(64), dim3(256), 0, stream, true, p, words,
                         static_cast<const uint4*>(a_src), static_cast<uint4*>(a_dst), (uint32_t)(a_bytes / 16),
                         static_cast<const uint4*>(b_src), static_cast<uint4*>(b_dst), (uint32_t)(b_bytes / 16));
}

}  // namespace dsrows
