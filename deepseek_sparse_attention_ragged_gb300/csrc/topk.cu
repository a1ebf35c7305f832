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
// a radix select:
//   1. a 2048-bin histogram of the top 11 key bits per row (fused into the
//      indexer epilogue in the decode step, or the histogram kernel here);
//   2. one pass of CTAs over each row: from the histogram every CTA finds the
//      bin of the width-th best score and appends the elements at or above it
//      to a per-row candidate list (typically width + a few hundred);
//   3. the last CTA of a row to finish (an atomic arrival counter; nothing
//      waits) refines the threshold digit by digit (11/11/10 key bits, then
//      the index bits, stopping as soon as a bin is taken whole), keeps the
//      `width` winners, sorts them with a 512-wide bitonic network (warp
//      shuffles for partners closer than 32) and writes them best first.
// A row whose threshold bin alone overflows the candidate list falls back to
// the same refinement over the row's full score array.

#include "common.cuh"
#include "kernels.h"

namespace dsrows {

namespace {

constexpr int kChunk = 8192;
constexpr int kThreads = 512;
constexpr uint32_t kFull = 0xFFFFFFFFu;

struct LevelSpec {
    int shift;
    int bits;
};
// Digits of the composite, most significant first.
__constant__ LevelSpec kLevels[6] = {{53, 11}, {42, 11}, {32, 10}, {21, 11}, {10, 11}, {0, 10}};

__device__ __forceinline__ int entry_of_chunk(const TopkParams& p, uint32_t c) {
    int e = 0;
#pragma unroll
    for (int i = 1; i < kRowsMax; ++i)
        if (i < (int)p.rows && c >= p.chunk_begin[i]) e = i;
    return e;
}

__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t index) {
    return ((uint64_t)key << 32) | (uint64_t)(~index);
}

struct BinPick {
    int bin;        // -1 when the histogram holds fewer than `need` elements
    uint32_t gt;    // elements in bins above `bin`
    uint32_t eq;    // elements in `bin`
    uint32_t total; // elements in all bins
};

// Block-wide (512 threads, 4 bins each): the bin b with
//   count(bins >= b) >= need > count(bins > b).
// `scratch` is >= 24 words of shared memory.
__device__ BinPick pick_bin(const uint32_t* h, uint32_t need, uint32_t* scratch) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const uint32_t v0 = h[4 * t], v1 = h[4 * t + 1], v2 = h[4 * t + 2], v3 = h[4 * t + 3];
    const uint32_t tot = v0 + v1 + v2 + v3;
    uint32_t x = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(kFull, x, off);
        if (lane + off < 32) x += y;
    }
    if (t == 0) scratch[16] = 0xFFFFFFFFu;
    if (lane == 0) scratch[w] = x;
    __syncthreads();
    uint32_t after = 0;
    for (int w2 = w + 1; w2 < kThreads / 32; ++w2) after += scratch[w2];
    const uint32_t excl = x - tot + after;  // elements in bins > 4t+3
    const uint32_t ge3 = excl + v3, ge2 = ge3 + v2, ge1 = ge2 + v1, ge0 = ge1 + v0;
    int b = -1;
    uint32_t gt = 0, eq = 0;
    if (ge3 >= need && excl < need) { b = 4 * t + 3; gt = excl; eq = v3; }
    else if (ge2 >= need && ge3 < need) { b = 4 * t + 2; gt = ge3; eq = v2; }
    else if (ge1 >= need && ge2 < need) { b = 4 * t + 1; gt = ge2; eq = v1; }
    else if (ge0 >= need && ge1 < need) { b = 4 * t; gt = ge1; eq = v0; }
    if (b >= 0) {
        scratch[16] = (uint32_t)b;
        scratch[17] = gt;
        scratch[18] = eq;
    }
    if (t == 0) scratch[19] = ge0;  // thread 0 covers bin 0: ge0 is the total
    __syncthreads();
    BinPick r;
    r.bin = (int)scratch[16];
    r.gt = scratch[17];
    r.eq = scratch[18];
    r.total = scratch[19];
    if (r.bin < 0) r.gt = r.eq = 0;
    __syncthreads();
    return r;
}


// Element sources for the refinement: candidates in shared or global memory, or a full score row.
struct SmemCandSource {
    const uint64_t* c;  // composites
    uint32_t n;
    __device__ __forceinline__ uint32_t size() const { return n; }
    __device__ __forceinline__ bool get(uint32_t i, uint64_t& v) const {
        v = c[i];
        return true;
    }
};

struct CandSource {
    const uint64_t* cand;  // key << 32 | index
    uint32_t n;
    __device__ __forceinline__ uint32_t size() const { return n; }
    __device__ __forceinline__ bool get(uint32_t i, uint64_t& c) const {
        const uint64_t v = __ldcg(cand + i);
        c = composite((uint32_t)(v >> 32), (uint32_t)v);
        return true;
    }
};

struct RowSource {
    const float* s;
    uint32_t n;
    __device__ __forceinline__ uint32_t size() const { return n; }
    __device__ __forceinline__ bool get(uint32_t i, uint64_t& c) const {
        const float x = __ldcg(s + i);
        if (!finite_f(x)) return false;
        c = composite(score_key(x), i);
        return true;
    }
};

constexpr int kSmemCand = 4096;  // candidates the finishing CTA stages in shared memory

struct FinishSmem {
    uint32_t h[kHistBins];
    uint32_t scratch[32];
    uint64_t cand[kSmemCand];
    uint64_t sel[kTopK];
    uint32_t nsel;
};

// Sort the 512 composites of sm.sel in descending order; thread t ends with element t.
// Bitonic network: partners closer than 32 exchange by warp shuffle, the rest through shared memory.
__device__ __forceinline__ uint64_t bitonic_desc_512(FinishSmem& sm) {
    const int t = threadIdx.x;
    uint64_t x = sm.sel[t];
    for (int k = 2; k <= kTopK; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            uint64_t y;
            if (j >= 32) {
                __syncthreads();
                sm.sel[t] = x;
                __syncthreads();
                y = sm.sel[t ^ j];
            } else {
                y = __shfl_xor_sync(kFull, x, j);
            }
            const bool desc = (t & k) == 0;
            const bool lower = (t & j) == 0;
            const uint64_t hi = x > y ? x : y, lo = x > y ? y : x;
            x = (lower == desc) ? hi : lo;
        }
    }
    return x;
}

// Refine from the level-0 pick, select the winners, sort and write them best first.
template <class Src>
__device__ void finish_row(const Src& src, const BinPick& l0, uint32_t width, int32_t* out, FinishSmem& sm,
                           uint32_t* status) {
    const int t = threadIdx.x, lane = t & 31;
    const bool take_all = l0.total <= width;
    int level = 0;
    uint64_t prefix = (uint64_t)(l0.bin < 0 ? 0 : l0.bin);
    uint32_t need = take_all ? 0 : width - l0.gt;
    bool done = take_all || l0.eq == need;
    for (int lv = 1; lv < 6 && !done; ++lv) {
        const LevelSpec up = kLevels[lv - 1];
        const LevelSpec cur = kLevels[lv];
        const uint32_t mask = (1u << cur.bits) - 1;
        for (int i = t; i < kHistBins; i += kThreads) sm.h[i] = 0;
        __syncthreads();
        const uint32_t n = src.size();
        for (uint32_t i = t; i < n; i += kThreads) {
            uint64_t c;
            if (src.get(i, c) && (c >> up.shift) == prefix) atomicAdd(&sm.h[(c >> cur.shift) & mask], 1u);
        }
        __syncthreads();
        const BinPick pk = pick_bin(sm.h, need, sm.scratch);
        if (pk.bin < 0) {  // inconsistent counts: keep what is certain
            if (t == 0) atomicOr(status, kStatusCandOverflow);
            break;
        }
        need -= pk.gt;
        prefix = (prefix << cur.bits) | (uint64_t)pk.bin;
        level = lv;
        done = pk.eq == need;
    }
    const int shift = kLevels[level].shift;

    if (t == 0) sm.nsel = 0;
    sm.sel[t] = 0;  // below every finite element's composite
    __syncthreads();
    const uint32_t n = src.size();
    for (uint32_t base = 0; base < n; base += kThreads) {
        const uint32_t i = base + t;
        uint64_t c = 0;
        const bool take = i < n && src.get(i, c) && (take_all || (c >> shift) >= prefix);
        const uint32_t m = __ballot_sync(kFull, take);
        if (m) {
            uint32_t pos = 0;
            if (lane == 0) pos = atomicAdd(&sm.nsel, (uint32_t)__popc(m));
            pos = __shfl_sync(kFull, pos, 0) + __popc(m & ((1u << lane) - 1u));
            if (take && pos < (uint32_t)kTopK) sm.sel[pos] = c;
        }
    }
    __syncthreads();
    const uint32_t got = sm.nsel;
    const uint32_t nsel = got < width ? got : width;
    if (got > width && t == 0) atomicOr(status, kStatusCandOverflow);
    const uint64_t x = bitonic_desc_512(sm);
    if ((uint32_t)t < width) out[t] = (uint32_t)t < nsel ? (int32_t)(~(uint32_t)x) : -1;
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

// Candidate collection for one chunk; the row's last CTA finishes the row.
__global__ void __launch_bounds__(kThreads) topk_select_kernel(const TopkParams p) {
    __shared__ FinishSmem sm;
    __shared__ uint32_t is_last;
    const int e = entry_of_chunk(p, blockIdx.x);
    const uint32_t c = blockIdx.x - p.chunk_begin[e];
    const uint32_t L = p.kv_len[e];
    const uint32_t width = p.width[e];
    const uint32_t nchunks = (L + kChunk - 1) / kChunk;
    const uint32_t* hist = p.hist + (size_t)e * kHistBins;
    uint32_t* ctl = p.ctl + (size_t)e * kCtlWords;
    uint64_t* cand = p.cand + (size_t)e * kCandCap;
    const float* s = p.scores + (size_t)e * p.score_stride;
    const int t = threadIdx.x, lane = t & 31;
    pdl_trigger();
    pdl_wait();  // scores and histogram come from the previous kernel

    // Issue this thread's 16 score loads before anything waits on them.
    constexpr int kPer = kChunk / kThreads;  // 16
    const uint32_t begin = c * kChunk;
    const uint32_t end = min(L, begin + kChunk);
    const bool vec = (reinterpret_cast<uintptr_t>(s) & 15) == 0;
    float v[kPer];
#pragma unroll
    for (int i = 0; i < kPer / 4; ++i) {
        const uint32_t j = begin + 4 * t + 4 * kThreads * i;
        if (vec && j + 3 < end) {
            const float4 q = __ldcg(reinterpret_cast<const float4*>(s + j));
            v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) v[4 * i + u] = j + u < end ? __ldcg(s + j + u) : __int_as_float(0x7FC00000);
        }
    }
    for (int i = t; i < kHistBins; i += kThreads) sm.h[i] = __ldcg(hist + i);
    __syncthreads();
    const BinPick l0 = pick_bin(sm.h, width, sm.scratch);
    const bool take_all = l0.total <= width;
    const uint32_t n_cand = take_all ? l0.total : l0.gt + l0.eq;
    const uint32_t b0 = take_all ? 0u : (uint32_t)l0.bin;
    const bool fast = n_cand <= (uint32_t)kCandCap;

    if (fast) {
        uint32_t take = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) take |= (finite_f(v[i]) && (score_key(v[i]) >> 21) >= b0) ? (1u << i) : 0u;
        const uint32_t cnt = __popc(take);
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        const uint32_t total = __shfl_sync(kFull, incl, 31);
        uint32_t base = 0;
        if (lane == 31 && total) base = atomicAdd(&ctl[0], total);
        uint32_t at = __shfl_sync(kFull, base, 31) + incl - cnt;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            if (take & (1u << i)) {
                const uint32_t j = begin + 4 * t + 4 * kThreads * (i >> 2) + (i & 3);
                if (at < (uint32_t)kCandCap) cand[at] = ((uint64_t)score_key(v[i]) << 32) | j;
                ++at;
            }
        }
    }

    // Arrival: the last CTA of the row sees every other CTA's candidates.
    __threadfence();
    __syncthreads();
    if (t == 0) is_last = (atomicAdd(&ctl[1], 1u) == nchunks - 1) ? 1u : 0u;
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    int32_t* out = p.out + p.out_offset[e];
    if (fast) {
        const uint32_t got = __ldcg(&ctl[0]);
        if (got != n_cand && t == 0) atomicOr(p.status, kStatusCandOverflow);
        const uint32_t n = got < (uint32_t)kCandCap ? got : (uint32_t)kCandCap;
        BinPick l0f = l0;
        l0f.bin = (int)b0;
        if (n <= (uint32_t)kSmemCand) {
            for (uint32_t i = t; i < n; i += kThreads) {
                const uint64_t x = __ldcg(cand + i);
                sm.cand[i] = composite((uint32_t)(x >> 32), (uint32_t)x);
            }
            __syncthreads();
            finish_row(SmemCandSource{sm.cand, n}, l0f, width, out, sm, p.status);
        } else {
            finish_row(CandSource{cand, n}, l0f, width, out, sm, p.status);
        }
    } else {
        finish_row(RowSource{s, L}, l0, width, out, sm, p.status);
    }
}

uint32_t topk_chunk() { return kChunk; }

cudaError_t launch_topk_hist(const TopkParams& p, cudaStream_t stream, bool pdl) {
    if (p.total_chunks == 0) return cudaSuccess;
    return launch_kernel(topk_hist_kernel, dim3(p.total_chunks), dim3(kThreads), 0, stream, pdl, p);
}

cudaError_t launch_topk_select(const TopkParams& p, cudaStream_t stream, bool pdl) {
    if (p.total_chunks == 0) return cudaSuccess;
    return launch_kernel(topk_select_kernel, dim3(p.total_chunks), dim3(kThreads), 0, stream, pdl, p);
}

__global__ void __launch_bounds__(1024) clear_kernel(uint32_t* __restrict__ p, uint32_t words) {
    pdl_trigger();
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < words; i += gridDim.x * blockDim.x) p[i] = 0;
}

cudaError_t launch_clear(uint32_t* p, uint32_t words, cudaStream_t stream) {
    return launch_kernel(clear_kernel, dim3(4), dim3(1024), 0, stream, false, p, words);
}

}  // namespace dsrows
