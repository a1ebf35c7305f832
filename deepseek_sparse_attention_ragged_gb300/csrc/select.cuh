// Row selection building blocks (radix select over fp32 scores) shared by the
// stand-alone top-k kernel and the decode's fused select + attend kernel.
//
// Order: score descending, then lower index; only finite scores take part.
// Each score maps to an order-preserving 32-bit key, and (key, index) to the
// 64-bit composite c = key << 32 | ~index, distinct per element, so the best
// `width` elements are the `width` largest composites.
#pragma once

#include <cfloat>
#include <cooperative_groups.h>

#include "common.cuh"

namespace dsrows {
namespace rowsel {

namespace cg = cooperative_groups;

constexpr int kThreads = 512;
constexpr uint32_t kFull = 0xFFFFFFFFu;

// Digits of the composite, most significant first: level lv covers bits
// [level_shift(lv), level_shift(lv) + level_bits(lv)).
__device__ __forceinline__ int level_shift(int lv) {
    return lv == 0 ? 53 : lv == 1 ? 42 : lv == 2 ? 32 : lv == 3 ? 21 : lv == 4 ? 10 : 0;
}
__device__ __forceinline__ int level_bits(int lv) { return (lv == 2 || lv == 5) ? 10 : 11; }

struct BinPick {
    int bin;        // -1 when the histogram holds fewer than `need` elements
    uint32_t gt;    // elements in bins above `bin`
    uint32_t eq;    // elements in `bin`
    uint32_t total; // elements in all bins
};

// Block-wide (512 threads, 4 bins each): the bin b with
//   count(bins >= b) >= need > count(bins > b).
// `scratch` is >= 24 words of shared memory; h is 16-byte aligned. Every
// thread has read h when the call returns, so h may be overwritten then.
// Without `sync_after`, the next call must use other scratch words.
// The same, with thread t's bins 4t..4t+3 already in registers.
__device__ inline BinPick pick_bin_regs(const uint4 hv, uint32_t need, uint32_t* scratch, bool sync_after = true) {
    static_assert(4 * kThreads == kHistBins, "four bins per thread");
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const uint32_t v0 = hv.x, v1 = hv.y, v2 = hv.z, v3 = hv.w;
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
    uint32_t after = 0;  // elements in the bins of later warps (16 independent loads)
#pragma unroll
    for (int w2 = 0; w2 < kThreads / 32; ++w2) after += w2 > w ? scratch[w2] : 0u;
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
    if (sync_after) __syncthreads();
    return r;
}

__device__ inline BinPick pick_bin(const uint32_t* h, uint32_t need, uint32_t* scratch, bool sync_after = true) {
    return pick_bin_regs(reinterpret_cast<const uint4*>(h)[threadIdx.x], need, scratch, sync_after);
}


// Element sources for the refinement: candidates in shared memory, or a full score row.
struct SmemCandSource {
    const uint64_t* c;  // composites
    uint32_t n;
    __device__ __forceinline__ uint32_t size() const { return n; }
    __device__ __forceinline__ bool get(uint32_t i, uint64_t& v) const {
        v = c[i];
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

constexpr int kCluster = 8;        // CTAs per row in the select kernel
constexpr uint32_t kChunkSlotsSel = 128;  // attention slots per CTA chunk
constexpr int kLeaderCap = 8192;   // candidates the leader CTA holds in shared memory

constexpr uint32_t kRankDirect = 128;  // a threshold bin this small is ranked element by element

struct SelectSmem;
__device__ __forceinline__ uint32_t* pick_scratch(SelectSmem& sm);
struct SelectSmem {
    __align__(16) uint32_t h[kHistBins];  // level-0 histogram (each CTA), then refinement levels (leader),
                             // then the threshold bin's elements when they are ranked directly
    uint32_t scratch[32];
    uint64_t cand[kLeaderCap];
    uint32_t ncand;
    uint32_t nsel;
    uint32_t nres;
};
__device__ __forceinline__ uint32_t* pick_scratch(SelectSmem& sm) { return sm.scratch; }

// Where the refinement stands: the last digit level fixed, the composite
// prefix through that level, and how many elements of that prefix are needed.
struct Refine {
    bool take_all;  // fewer finite scores than the width: keep them all
    int level;
    uint64_t prefix;
    uint32_t need;
    uint32_t eq;    // elements in the prefix's bin
    bool done;      // the prefix's whole bin is taken
};

__device__ __forceinline__ Refine refine_from_level0(const BinPick& l0, uint32_t width) {
    Refine r;
    r.take_all = l0.total <= width;
    r.level = 0;
    r.prefix = (uint64_t)(l0.bin < 0 ? 0 : l0.bin);
    r.need = r.take_all ? 0 : width - l0.gt;
    r.eq = l0.eq;
    r.done = r.take_all || l0.eq == r.need;
    return r;
}

// Write the nsel winners of sel (composites), as index + offset, to
// out[0, width) best first (sorted by composite), then -1; `out` may point to
// global or shared memory, and sel is left unchanged.
__device__ __forceinline__ void write_winners(SelectSmem& sm, const uint64_t* sel, uint32_t nsel, uint32_t width,
                                              int32_t* out, int32_t offset) {
    const int t = threadIdx.x;
    uint64_t x[1] = {sel[t]};
    __syncthreads();  // every thread holds its element before the buffer is reused
    sort512_desc<kThreads>(x, sm.cand);  // the candidates are consumed
    // ~(low word) of a composite is its index.
    if ((uint32_t)t < width) out[t] = (uint32_t)t < nsel ? (int32_t)(~(uint32_t)x[0]) + offset : -1;
}

// Ranks inside a threshold bin of nr <= kRankDirect elements bin[0, nr):
// element i = threadIdx.x / 4 (held in `ck`) is compared with every element
// of the bin by four threads, each taking every fourth one (the four
// addresses of a load fall in different banks), and their counts are summed
// by shuffles. Returns how many elements of the bin are greater than element
// i, valid in threads with threadIdx.x % 4 == 0 and i < nr. Called by whole
// warps: those holding elements, warps w with 8 w < nr; the bin may hold
// anything past nr.
__device__ __forceinline__ uint32_t count_better(const uint64_t* bin, uint32_t nr, uint64_t& ck) {
    static_assert(kThreads >= 4 * kRankDirect, "four threads per element of the bin");
    const uint32_t t = threadIdx.x, i = t >> 2, q = t & 3;
    ck = i < nr ? bin[i] : 0ull;
    uint32_t better = 0;
    const uint32_t iters = (nr + 3) >> 2;  // 4 iters <= kRankDirect: j stays inside the bin buffer
#pragma unroll 4
    for (uint32_t u = 0; u < iters; ++u) {
        const uint32_t j = 4 * u + q;
        const uint64_t y = bin[j];
        better += j < nr && y > ck ? 1u : 0u;
    }
    better += __shfl_xor_sync(kFull, better, 1);
    better += __shfl_xor_sync(kFull, better, 2);
    return better;
}

// Refine digit by digit until the threshold bin is taken whole or holds at
// most kRankDirect elements, then keep the winners' composites in sel[0, 512)
// (zero past the last): every element above the bin, and the `need` best of
// the bin's elements, found by counting for each how many of them are better.
// `sm` provides h[kHistBins], scratch[32], nsel and nres. Returns the number of
// winners (their order in sel is arbitrary).
template <class Src, class Smem>
__device__ inline uint32_t finish_row(const Src& src, Refine st, uint32_t width, Smem& sm, uint64_t* sel,
                                      uint32_t* status) {
    const int t = threadIdx.x, lane = t & 31;
    const bool take_all = st.take_all;
    int level = st.level;
    uint64_t prefix = st.prefix;
    uint32_t need = st.need;
    uint32_t eq = st.eq;
    bool done = st.done;
    for (int lv = level + 1; lv < 6 && !done && eq > kRankDirect; ++lv) {
        const int up_shift = level_shift(lv - 1), cur_shift = level_shift(lv), cur_bits = level_bits(lv);
        const uint32_t mask = (1u << cur_bits) - 1;
        for (int i = t; i < kHistBins; i += kThreads) sm.h[i] = 0;
        __syncthreads();
        const uint32_t n = src.size();
        for (uint32_t i = t; i < n; i += kThreads) {
            uint64_t c;
            if (src.get(i, c) && (c >> up_shift) == prefix) atomicAdd(&sm.h[(c >> cur_shift) & mask], 1u);
        }
        __syncthreads();
        const BinPick pk = pick_bin(sm.h, need, pick_scratch(sm));
        if (pk.bin < 0) {  // inconsistent counts: keep what is certain
            if (t == 0) atomicOr(status, kStatusCandOverflow);
            done = true;
            break;
        }
        need -= pk.gt;
        prefix = (prefix << cur_bits) | (uint64_t)pk.bin;
        level = lv;
        eq = pk.eq;
        done = pk.eq == need;
    }
    const bool direct = !done;  // the bin's eq (<= kRankDirect) elements are ranked below
    const int shift = level_shift(level);
    uint64_t* bin_el = reinterpret_cast<uint64_t*>(sm.h);  // the threshold bin's elements

    if (t == 0) {
        sm.nsel = 0;
        sm.nres = 0;
    }
    sel[t] = 0;  // below every finite element's composite
    __syncthreads();
    const uint32_t n = src.size();
    for (uint32_t base = 0; base < n; base += kThreads) {
        const uint32_t i = base + t;
        uint64_t c = 0;
        const bool valid = i < n && src.get(i, c);
        const uint64_t d = c >> shift;
        const bool take = valid && (take_all || (direct ? d > prefix : d >= prefix));
        const bool in_bin = valid && direct && !take_all && d == prefix;
        uint32_t m = __ballot_sync(kFull, take);
        if (m) {
            uint32_t pos = 0;
            if (lane == 0) pos = atomicAdd(&sm.nsel, (uint32_t)__popc(m));
            pos = __shfl_sync(kFull, pos, 0) + __popc(m & ((1u << lane) - 1u));
            if (take && pos < (uint32_t)kTopK) sel[pos] = c;
        }
        m = __ballot_sync(kFull, in_bin);
        if (m) {
            uint32_t pos = 0;
            if (lane == 0) pos = atomicAdd(&sm.nres, (uint32_t)__popc(m));
            pos = __shfl_sync(kFull, pos, 0) + __popc(m & ((1u << lane) - 1u));
            if (in_bin && pos < kRankDirect) bin_el[pos] = c;
        }
    }
    __syncthreads();
    if (direct) {
        const uint32_t nr = sm.nres < kRankDirect ? sm.nres : kRankDirect;
        if (sm.nres != eq && t == 0) atomicOr(status, kStatusCandOverflow);
        if ((uint32_t)(t >> 5) * 8 < nr) {  // warp-uniform: the warps holding elements
            uint64_t ck;
            const uint32_t better = count_better(bin_el, nr, ck);
            if ((t & 3) == 0 && (uint32_t)(t >> 2) < nr && better < need) {
                const uint32_t pos = atomicAdd(&sm.nsel, 1u);
                if (pos < (uint32_t)kTopK) sel[pos] = ck;
            }
        }
        __syncthreads();
    }
    const uint32_t got = sm.nsel;
    const uint32_t nsel = got < width ? got : width;
    if (got > width && t == 0) atomicOr(status, kStatusCandOverflow);
    return nsel;
}

// The result of a row's collection phase (the same in every CTA of the cluster).
struct Collected {
    BinPick l0;     // level-0 pick from the row's histogram
    uint32_t b0;    // threshold bin (0 when every finite score is taken)
    bool take_all;  // no more finite scores than the width
    bool fast;      // the candidates fit the leader's shared memory
};

// Collection phase of a row's select cluster (kCluster CTAs of kThreads):
// every CTA picks the level-0 threshold bin from the row's histogram, streams
// its slice of the scores once and appends the candidates (finite, top 11 key
// bits >= that bin) as composites into the leader's shared memory.
// Before the call the leader's ncand is zero and visible cluster-wide; after
// it a cluster barrier makes the appends visible to the leader.
__device__ __forceinline__ Collected select_collect(const float* s, uint32_t L, uint32_t width,
                                                    const uint32_t* hist_row, uint32_t rank, SelectSmem& sm,
                                                    SelectSmem& leader) {
    const int t = threadIdx.x, lane = t & 31;
    // This CTA's slice: a multiple of 2048 scores (512 threads x float4).
    const uint32_t per = (((L + kCluster - 1) / kCluster) + 2047) & ~2047u;
    const uint32_t begin = min(L, rank * per);
    const uint32_t end = min(L, begin + per);
    const bool vec = (reinterpret_cast<uintptr_t>(s) & 15) == 0;
    constexpr int kBatch = 8;  // float4 loads in flight per thread
    float v[kBatch * 4];
    auto load_batch = [&](uint32_t base) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const uint32_t j = base + 4 * t + 4 * kThreads * i;
            if (vec && j + 3 < end) {
                const float4 q = __ldcg(reinterpret_cast<const float4*>(s + j));
                v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    v[4 * i + u] = j + u < end ? __ldcg(s + j + u) : __int_as_float(0x7FC00000);
            }
        }
    };
    // The histogram first (the threshold pick waits for it), then the slice's
    // scores, which stay in flight while the threshold is picked.
    uint32_t hv[kHistBins / kThreads];
#pragma unroll
    for (int i = 0; i < kHistBins / kThreads; ++i) hv[i] = __ldcg(hist_row + t + i * kThreads);
    load_batch(begin);
#pragma unroll
    for (int i = 0; i < kHistBins / kThreads; ++i) sm.h[t + i * kThreads] = hv[i];
    __syncthreads();
    Collected r;
    r.l0 = pick_bin(sm.h, width, pick_scratch(sm));
    r.take_all = r.l0.total <= width;
    const uint32_t n_cand = r.take_all ? r.l0.total : r.l0.gt + r.l0.eq;
    r.b0 = r.take_all ? 0u : (uint32_t)r.l0.bin;
    r.fast = n_cand <= (uint32_t)kLeaderCap;

    if (r.fast) {
        // The smallest score whose key falls in bin b0: for finite scores,
        // key >= b0 << 21 is the same as score >= this value (-0.0 ties +0.0).
        float thr = -FLT_MAX;
        if (!r.take_all) {
            const uint32_t k0 = r.b0 << 21;
            const float f = __uint_as_float((k0 & 0x80000000u) ? (k0 & 0x7FFFFFFFu) : ~k0);
            if (finite_f(f)) thr = f;
        }
        for (uint32_t base = begin; base < end; base += kBatch * 4 * kThreads) {
            if (base != begin) load_batch(base);
            uint32_t take = 0;
#pragma unroll
            for (int i = 0; i < kBatch * 4; ++i) take |= (v[i] >= thr && v[i] < INFINITY) ? (1u << i) : 0u;
            const uint32_t cnt = __popc(take);
            uint32_t incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t total = __shfl_sync(kFull, incl, 31);
            uint32_t at = 0;
            if (lane == 31 && total) at = atomicAdd(&leader.ncand, total);
            at = __shfl_sync(kFull, at, 31) + incl - cnt;
#pragma unroll
            for (int i = 0; i < kBatch * 4; ++i) {
                if (take & (1u << i)) {
                    const uint32_t j = base + 4 * t + 4 * kThreads * (i >> 2) + (i & 3);
                    if (at < (uint32_t)kLeaderCap) leader.cand[at] = composite(score_key(v[i]), j);
                    ++at;
                }
            }
        }
    }
    return r;
}

// The leader's half of a row's selection, after the collection phase and a
// cluster barrier: refine, keep the winners in sel and write their indices.
__device__ __forceinline__ uint32_t select_finish(const Collected& c, const float* s, uint32_t L, uint32_t width,
                                                  int32_t* out, SelectSmem& sm, uint64_t* sel,
                                                  uint32_t* status, int32_t offset = 0) {
    if (c.fast) {
        const uint32_t got = sm.ncand;
        const uint32_t n_cand = c.take_all ? c.l0.total : c.l0.gt + c.l0.eq;
        if (got != n_cand && threadIdx.x == 0) atomicOr(status, kStatusCandOverflow);
        BinPick l0f = c.l0;
        l0f.bin = (int)c.b0;
        const Refine st = refine_from_level0(l0f, width);
        const uint32_t nsel = finish_row(
            SmemCandSource{sm.cand, got < (uint32_t)kLeaderCap ? got : (uint32_t)kLeaderCap}, st, width, sm, sel,
            status);
        if (out) write_winners(sm, sel, nsel, width, out, offset);
        return nsel;
    }
    const uint32_t nsel = finish_row(RowSource{s, L}, refine_from_level0(c.l0, width), width, sm, sel, status);
    if (out) write_winners(sm, sel, nsel, width, out, offset);
    return nsel;
}

// ---- all-gather selection: every CTA of the row's cluster selects locally ----
//
// Every CTA of a row's cluster gathers all of the row's candidates, in index
// order, and computes the same exact threshold T (the composite of the
// width-th best score): the winners are the candidates >= T. A winner's slot
// is its place among the winners in index order (the attention's slot order).

constexpr uint32_t kCandCap = 2048;  // candidates one CTA may contribute to its cluster
constexpr int kRegCandSmall = 4;     // candidates per thread in registers while they fit
constexpr int kRegCandMid = 5;       // then this many,
constexpr int kRegCandLarge = 9;     // this many,
constexpr int kRegCand = 12;         // and at most this many per thread, else the general path

// State of the all-gather selection in each CTA of a row's cluster.
struct GatherSmem {
    __align__(16) uint32_t h[kHistBins];  // level-0 histogram, the refinement levels, sort buffers
    uint32_t pick[2][32];                 // two alternating pick_bin scratch areas
    uint32_t scan[2][16];                 // two alternating block_excl_scan scratch areas
    uint32_t count[kCluster];             // candidates contributed by each CTA (written by that CTA)
    uint32_t nres;                        // elements of the final threshold bin (zeroed by the collection)
    uint32_t nsel;
    uint64_t thr;
    uint64_t bin[kRankDirect];            // the final threshold bin's elements
};
__device__ __forceinline__ uint32_t* pick_scratch(GatherSmem& sm) { return sm.pick[0]; }
static_assert(kHistBins * 4 >= 2 * kTopK * 8, "the sorts use h as two 512-entry buffers");

// Exclusive prefix over the block's threads, in thread order, of one count
// per thread, and the block's total, with one barrier. `scratch` (16 words) is
// rewritten only after the next block barrier.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t& total, uint32_t* scratch) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) scratch[w] = inc;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w2 = 0; w2 < kThreads / 32; ++w2) {
        const uint32_t y = scratch[w2];
        all += y;
        before += w2 < w ? y : 0u;
    }
    total = all;
    return before + inc - v;
}

// The cluster's candidates in this CTA's shared memory: region r (kCandCap
// composites from its start) holds the count[r] contributed by CTA r, in index
// order; position i of the source is in the region r with b[r] <= i < b[r + 1],
// so positions follow the index.
struct RegionSource {
    const uint64_t* c;
    uint32_t b[kCluster + 1];
    __device__ __forceinline__ uint32_t size() const { return b[kCluster]; }
    __device__ __forceinline__ bool get(uint32_t i, uint64_t& v) const {
        uint32_t r = 0, base = 0;
#pragma unroll
        for (int k = 1; k < kCluster; ++k)
            if (i >= b[k]) { r = (uint32_t)k; base = b[k]; }
        v = c[(size_t)r * kCandCap + (i - base)];
        return true;
    }
};

struct Gathered {
    BinPick l0;     // level-0 pick from the row's histogram
    uint32_t b0;    // threshold bin (0 when every finite score is taken)
    bool take_all;  // no more finite scores than the width
    bool fast;      // the candidates were gathered (else the full row is refined)
};

// Collection phase of a row's cluster (kCluster CTAs of kThreads): every CTA
// picks the level-0 threshold bin from the row's histogram and compacts the
// candidates of its slice of the row (finite scores whose top 11 key bits are
// >= that bin), as composites in index order, into region `rank` of `regions`
// in its own shared memory (a slice is a multiple of 128 scores). The slice's
// first 16384 scores are loaded with the histogram, before the threshold is
// known; warp w holds scores
// [1024 w, 1024 w + 1024) of a batch, thread t of it [128 i + 4 t, +4) for
// i < 8, so every load of a warp is 512 contiguous bytes. Then each CTA copies
// its candidates, densely, into region `rank` of every other CTA of the
// cluster, and its count into count[rank] of every CTA. Before the call every
// CTA has passed a cluster barrier; after it a cluster barrier makes every
// CTA's candidates visible to all. h is left zero.
__device__ __forceinline__ Gathered select_collect_all(const float* s, uint32_t L, uint32_t width,
                                                       const uint32_t* hist_row, uint32_t rank, GatherSmem& sm,
                                                       uint64_t* regions) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    constexpr int kSub = 8;                                   // 128-score sub-blocks per warp and batch
    constexpr uint32_t kBatchScores = 128 * kSub * (kThreads / 32);  // 16384
    // A multiple of 128 scores per CTA: short rows spread over the cluster.
    const uint32_t per = (((L + kCluster - 1) / kCluster) + 127) & ~127u;
    const uint32_t begin = min(L, rank * per);
    const uint32_t end = min(L, begin + per);
    const bool vec = (reinterpret_cast<uintptr_t>(s) & 15) == 0;
    float v[kSub * 4];
    auto load_batch = [&](uint32_t base) {
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
            const uint32_t j = base + 1024 * w + 128 * i + 4 * lane;
            if (vec && j + 3 < end) {
                const float4 q = __ldcg(reinterpret_cast<const float4*>(s + j));
                v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    v[4 * i + u] = j + u < end ? __ldcg(s + j + u) : __int_as_float(0x7FC00000);
            }
        }
    };
    // The histogram first (the threshold pick waits for it; thread t takes bins
    // 4t..4t+3 straight into registers), then the slice's scores, which stay in
    // flight while the threshold is picked.
    const uint4 hv = __ldcg(reinterpret_cast<const uint4*>(hist_row) + t);
    __syncthreads();  // every warp's histogram load is issued before any score load
    load_batch(begin);
    // The refinement's first level counts into h (not used by the pick): zero
    // it, and the final bin's count.
#pragma unroll
    for (int i = 0; i < kHistBins / kThreads; ++i) sm.h[t + i * kThreads] = 0;
    if (t == 0) sm.nres = 0;
    Gathered r;
    r.l0 = pick_bin_regs(hv, width, sm.pick[0], false);
    r.take_all = r.l0.total <= width;
    const uint32_t n_cand = r.take_all ? r.l0.total : r.l0.gt + r.l0.eq;
    r.b0 = r.take_all ? 0u : (uint32_t)r.l0.bin;
    r.fast = n_cand <= (uint32_t)kCluster * kCandCap;

    uint64_t* own = regions + (size_t)rank * kCandCap;
    uint32_t n_local = 0;
    if (r.fast) {
        // The smallest score whose key falls in bin b0: for finite scores,
        // key >= b0 << 21 is the same as score >= this value (-0.0 ties +0.0).
        float thr = -FLT_MAX;
        if (!r.take_all) {
            const uint32_t k0 = r.b0 << 21;
            const float f = __uint_as_float((k0 & 0x80000000u) ? (k0 & 0x7FFFFFFFu) : ~k0);
            if (finite_f(f)) thr = f;
        }
        const uint32_t below = (1u << lane) - 1u;
        int par = 0;
        for (uint32_t base = begin; base < end; base += kBatchScores) {
            if (base != begin) load_batch(base);
            // Within the warp, index order is (i, lane, u): ballots per (i, u).
            uint32_t bal[kSub * 4];
            uint32_t cnt = 0;
#pragma unroll
            for (int i = 0; i < kSub * 4; ++i) {
                bal[i] = __ballot_sync(kFull, v[i] >= thr && v[i] < INFINITY);
                cnt += __popc(bal[i]);
            }
            // The warp's candidates follow those of the warps before it.
            uint32_t total;
            uint32_t at = n_local + block_excl_scan(lane == 0 ? cnt : 0u, total, sm.scan[par]);
            at = __shfl_sync(kFull, at, 0);
            par ^= 1;
            n_local += total;
#pragma unroll
            for (int i = 0; i < kSub; ++i) {
                const uint32_t b0 = bal[4 * i], b1 = bal[4 * i + 1], b2 = bal[4 * i + 2], b3 = bal[4 * i + 3];
                if (b0 | b1 | b2 | b3) {  // warp-uniform; the stores below are predicated, not branched
                    uint32_t pos = at + __popc(b0 & below) + __popc(b1 & below) + __popc(b2 & below) +
                                   __popc(b3 & below);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t bit = (bal[4 * i + u] >> lane) & 1u;
                        const uint64_t c = composite(score_key(v[4 * i + u]), base + 1024 * w + 128 * i + 4 * lane + u);
                        if (bit != 0 && pos < kCandCap) own[pos] = c;
                        pos += bit;
                    }
                    at += __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
                }
            }
        }
    }
    __syncthreads();  // this CTA's candidates are in place
    // Dense copy into the other CTAs: 16 bytes per store, consecutive threads
    // on consecutive addresses.
    const uint32_t m = n_local < kCandCap ? n_local : kCandCap;
    const uint32_t own_addr = smem_u32(own);
    for (uint32_t i = 2 * t; i < m; i += 2 * kThreads) {
        const uint64_t a = own[i], b = i + 1 < m ? own[i + 1] : 0ull;
#pragma unroll
        for (int q = 1; q < kCluster; ++q) {
            const uint32_t d = cluster_addr(own_addr, (rank + q) % kCluster) + 8 * i;
            if (i + 1 < m) asm volatile("st.shared::cluster.v2.u64 [%0], {%1, %2};" ::"r"(d), "l"(a), "l"(b) : "memory");
            else st_cluster_u64(d, a);
        }
    }
    if (t < kCluster) st_cluster_u32(cluster_addr(smem_u32(&sm.count[rank]), (uint32_t)t), n_local);
    return r;
}

// The exact threshold of the winners among the gathered candidates held in
// registers, R per thread (each candidate in one x[k] of one thread, the
// unused entries zero),
// from the refinement state `st`: the winners are the candidates with a
// composite >= the returned value (1 when every candidate is taken). h and
// nres are zero on entry.
template <int R>
__device__ __forceinline__ uint64_t refine_threshold(const uint64_t (&x)[R], Refine st, GatherSmem& sm,
                                                     uint32_t* status) {
    const int t = threadIdx.x, lane = t & 31;
    if (st.take_all) return 1ull;
    int level = st.level;
    uint64_t prefix = st.prefix;
    uint32_t need = st.need;
    uint32_t eq = st.eq;
    bool done = st.done;
    int par = 0;
    for (int lv = level + 1; lv < 6 && !done && eq > kRankDirect; ++lv) {
        const int up_shift = level_shift(lv - 1), cur_shift = level_shift(lv), cur_bits = level_bits(lv);
        const uint32_t mask = (1u << cur_bits) - 1;
        if (lv > st.level + 1) {
            for (int i = t; i < kHistBins; i += kThreads) sm.h[i] = 0;
            __syncthreads();
        }
#pragma unroll
        for (int k = 0; k < R; ++k)
            if (x[k] != 0 && (x[k] >> up_shift) == prefix) atomicAdd(&sm.h[(x[k] >> cur_shift) & mask], 1u);
        __syncthreads();
        const BinPick pk = pick_bin(sm.h, need, sm.pick[par], false);
        par ^= 1;
        if (pk.bin < 0) {  // inconsistent counts: keep what is certain
            if (t == 0) atomicOr(status, kStatusCandOverflow);
            done = true;
            break;
        }
        need -= pk.gt;
        prefix = (prefix << cur_bits) | (uint64_t)pk.bin;
        level = lv;
        eq = pk.eq;
        done = pk.eq == need;
    }
    const int shift = level_shift(level);
    const uint64_t whole = prefix << shift;  // the bin taken whole: every composite >= this
    if (done) return whole;
    // The threshold bin's eq (<= kRankDirect) elements go to their own buffer
    // (no barrier against the last pick's reads of h; nres was zeroed by the
    // collection), and the need-th best of them is the threshold.
    if (t == 0) sm.thr = whole;  // kept if the counts disagree
#pragma unroll
    for (int k = 0; k < R; ++k) {
        const bool in_bin = x[k] != 0 && (x[k] >> shift) == prefix;
        const uint32_t m = __ballot_sync(kFull, in_bin);
        if (m) {
            uint32_t pos = 0;
            if (lane == 0) pos = atomicAdd(&sm.nres, (uint32_t)__popc(m));
            pos = __shfl_sync(kFull, pos, 0) + __popc(m & ((1u << lane) - 1u));
            if (in_bin && pos < kRankDirect) sm.bin[pos] = x[k];
        }
    }
    __syncthreads();
    const uint32_t nres = sm.nres;
    const uint32_t nr = nres < kRankDirect ? nres : kRankDirect;
    if (nres != eq && t == 0) atomicOr(status, kStatusCandOverflow);
    if ((uint32_t)(t >> 5) * 8 < nr) {  // warp-uniform: the warps holding elements
        uint64_t ck;
        const uint32_t better = count_better(sm.bin, nr, ck);
        if ((t & 3) == 0 && (uint32_t)(t >> 2) < nr && better == need - 1) sm.thr = ck;
    }
    __syncthreads();
    return sm.thr;
}

// Slots of the winners (candidates >= T) in candidate order, for candidates in
// registers as for refine_threshold, where thread t's candidates follow those
// of threads < t and x[k] precedes x[k + 1]: slot[k] of x[k] (-1 for a
// non-winner). Returns the number of winners. One barrier.
template <int R>
__device__ __forceinline__ uint32_t winner_slots(const uint64_t (&x)[R], uint64_t T, int32_t (&slot)[R],
                                                 uint32_t* scratch) {
    bool f[R];
    uint32_t cnt = 0;
#pragma unroll
    for (int k = 0; k < R; ++k) {
        f[k] = x[k] != 0 && x[k] >= T;
        cnt += f[k] ? 1u : 0u;
    }
    uint32_t total;
    uint32_t at = block_excl_scan(cnt, total, scratch);
#pragma unroll
    for (int k = 0; k < R; ++k) {
        slot[k] = f[k] ? (int32_t)at : -1;
        at += f[k] ? 1u : 0u;
    }
    return total;
}

// Sort 512 values in descending order, one per thread (bitonic network): the
// strides below 32 exchange through warp shuffles, the larger ones through
// shared memory (two 512-entry buffers of `buf`, alternating: one barrier per
// stage, and every access of a warp is to consecutive words). Returns the
// value of rank threadIdx.x.
__device__ __forceinline__ uint64_t bitonic512_desc(uint64_t x, uint64_t* buf) {
    const uint32_t t = threadIdx.x;
    int b = 0;
#pragma unroll
    for (uint32_t k = 2; k <= 512; k <<= 1) {
#pragma unroll
        for (uint32_t j = k >> 1; j > 0; j >>= 1) {
            uint64_t y;
            if (j >= 32) {
                buf[b * 512 + t] = x;
                __syncthreads();
                y = buf[b * 512 + (t ^ j)];
                b ^= 1;
            } else {
                y = __shfl_xor_sync(kFull, x, j);
            }
            // The lower position of a pair keeps the larger value in blocks
            // (of k) sorted descending, the smaller in the others.
            const bool keep_max = ((t & j) == 0) == ((t & k) == 0);
            x = keep_max ? (x > y ? x : y) : (x < y ? x : y);
        }
    }
    return x;
}

// sel[0, 512) holds the winners' composites in any order, zero past the last:
// returns the winner of slot threadIdx.x in index order (zero past the last).
// Uses `buf` (1024 entries) for the sort; sel is read once per thread.
__device__ __forceinline__ uint64_t winner_by_index(const uint64_t* sel, uint64_t* buf) {
    const uint64_t c = sel[threadIdx.x];
    // ~index in the high word: descending order is ascending index; zero last.
    uint64_t k = c ? ((c << 32) | (c >> 32)) : 0ull;
    k = bitonic512_desc(k, buf);
    return k ? ((k << 32) | (k >> 32)) : 0ull;
}

// The winners among n <= kThreads * R gathered candidates, held R per thread
// in registers (thread t: candidates [R t, R t + R)), written as select_slots
// does. Returns the number of winners.
template <int R>
__device__ __forceinline__ uint32_t select_in_registers(const RegionSource& src, uint32_t n, Refine st,
                                                        uint32_t width, GatherSmem& sm, uint64_t* sel, int32_t* idx,
                                                        uint32_t first, uint32_t* status) {
    const int t = threadIdx.x;
    uint64_t x[R];
#pragma unroll
    for (int k = 0; k < R; ++k) {
        const uint32_t i = (uint32_t)(R * t + k);
        x[k] = 0;
        if (i < n) src.get(i, x[k]);
    }
    const uint64_t T = refine_threshold(x, st, sm, status);
    int32_t slot[R];
    uint32_t nsel = winner_slots(x, T, slot, sm.scan[0]);
    if (nsel > width) {
        if (t == 0) atomicOr(status, kStatusCandOverflow);
        nsel = width;
    }
#pragma unroll
    for (int k = 0; k < R; ++k)
        if (slot[k] >= 0 && (uint32_t)slot[k] < nsel) {
            sel[slot[k]] = x[k];
            if ((uint32_t)slot[k] - first < kChunkSlotsSel) idx[slot[k] - first] = (int32_t)(~(uint32_t)x[k]);
        }
    return nsel;
}

// The row's winners from the gathered candidates after the collection and a
// cluster barrier: sel[s] receives the composite of the winner of slot s
// (index order), zero past the last, and idx[s - first] the index of each
// winner whose slot is in [first, first + 128). sel is zero and idx -1 on
// entry. When some CTA had more than kCandCap candidates, or they are more
// than the registers hold, the row is refined from its gathered candidates or
// its full score array instead, and its winners sorted by index. Returns the
// number of winners. Every CTA that calls this computes the same result.
__device__ __forceinline__ uint32_t select_slots(const Gathered& g, const float* s, uint32_t L, uint32_t width,
                                                 GatherSmem& sm, const uint64_t* regions, uint64_t* sel,
                                                 int32_t* idx, uint32_t first, uint32_t* status) {
    const int t = threadIdx.x;
    RegionSource src;
    src.c = regions;
    uint32_t n = 0;
    bool fits = g.fast;
#pragma unroll
    for (int r = 0; r < kCluster; ++r) {
        src.b[r] = n;
        const uint32_t k = sm.count[r];
        fits = fits && k <= kCandCap;
        n += k;
    }
    src.b[kCluster] = n;
    BinPick l0f = g.l0;
    l0f.bin = (int)g.b0;
    if (fits) {
        const uint32_t expect = g.take_all ? g.l0.total : g.l0.gt + g.l0.eq;
        if (n != expect && t == 0) atomicOr(status, kStatusCandOverflow);
    }
    if (fits && n <= (uint32_t)kThreads * kRegCandSmall)
        return select_in_registers<kRegCandSmall>(src, n, refine_from_level0(l0f, width), width, sm, sel, idx, first,
                                                  status);
    if (fits && n <= (uint32_t)kThreads * kRegCandMid)
        return select_in_registers<kRegCandMid>(src, n, refine_from_level0(l0f, width), width, sm, sel, idx, first,
                                                status);
    if (fits && n <= (uint32_t)kThreads * kRegCandLarge)
        return select_in_registers<kRegCandLarge>(src, n, refine_from_level0(l0f, width), width, sm, sel, idx, first,
                                                  status);
    if (fits && n <= (uint32_t)kThreads * kRegCand)
        return select_in_registers<kRegCand>(src, n, refine_from_level0(l0f, width), width, sm, sel, idx, first,
                                             status);
    // The general path: refine (gathered candidates or the full row), then
    // order the winners by index.
    const uint32_t nsel = fits ? finish_row(src, refine_from_level0(l0f, width), width, sm, sel, status)
                               : finish_row(RowSource{s, L}, refine_from_level0(g.l0, width), width, sm, sel, status);
    const uint64_t c = winner_by_index(sel, reinterpret_cast<uint64_t*>(sm.h));
    __syncthreads();  // every thread has read its entry of sel
    sel[t] = c;
    if (c != 0 && (uint32_t)t - first < kChunkSlotsSel) idx[t - first] = (int32_t)(~(uint32_t)c);
    return nsel;
}

}  // namespace rowsel
}  // namespace dsrows
