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

struct LevelSpec {
    int shift;
    int bits;
};
// Digits of the composite, most significant first.
static __constant__ LevelSpec kLevels[6] = {{53, 11}, {42, 11}, {32, 10}, {21, 11}, {10, 11}, {0, 10}};

struct BinPick {
    int bin;        // -1 when the histogram holds fewer than `need` elements
    uint32_t gt;    // elements in bins above `bin`
    uint32_t eq;    // elements in `bin`
    uint32_t total; // elements in all bins
};

// Block-wide (512 threads, 4 bins each): the bin b with
//   count(bins >= b) >= need > count(bins > b).
// `scratch` is >= 24 words of shared memory.
__device__ inline BinPick pick_bin(const uint32_t* h, uint32_t need, uint32_t* scratch) {
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
    __syncthreads();
    return r;
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
constexpr int kLeaderCap = 8192;   // candidates the leader CTA holds in shared memory

constexpr uint32_t kRankDirect = 128;  // a threshold bin this small is ranked element by element

struct SelectSmem {
    uint32_t h[kHistBins];   // level-0 histogram (each CTA), then refinement levels (leader),
                             // then the threshold bin's elements when they are ranked directly
    uint32_t scratch[32];
    uint64_t cand[kLeaderCap];
    uint32_t ncand;
    uint32_t nsel;
    uint32_t nres;
};

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

// Refine digit by digit until the threshold bin is taken whole or holds at
// most kRankDirect elements, then keep the winners' composites in sel[0, 512)
// (zero past the last): every element above the bin, and the `need` best of
// the bin's elements, found by counting for each how many of them are better.
// Writes their indices to out (unless out is null). Returns the number of winners.
template <class Src>
__device__ inline uint32_t finish_row(const Src& src, Refine st, uint32_t width, uint32_t L, int32_t* out,
                                      SelectSmem& sm, uint64_t* sel, uint32_t* status, int32_t offset = 0) {
    const int t = threadIdx.x, lane = t & 31;
    const bool take_all = st.take_all;
    int level = st.level;
    uint64_t prefix = st.prefix;
    uint32_t need = st.need;
    uint32_t eq = st.eq;
    bool done = st.done;
    for (int lv = level + 1; lv < 6 && !done && eq > kRankDirect; ++lv) {
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
            done = true;
            break;
        }
        need -= pk.gt;
        prefix = (prefix << cur.bits) | (uint64_t)pk.bin;
        level = lv;
        eq = pk.eq;
        done = pk.eq == need;
    }
    const bool direct = !done;  // the bin's eq (<= kRankDirect) elements are ranked below
    const int shift = kLevels[level].shift;
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
        for (uint32_t k = t; k < nr; k += kThreads) {
            const uint64_t ck = bin_el[k];
            uint32_t better = 0;
            for (uint32_t j = 0; j < nr; ++j) better += bin_el[j] > ck ? 1u : 0u;
            if (better < need) {
                const uint32_t pos = atomicAdd(&sm.nsel, 1u);
                if (pos < (uint32_t)kTopK) sel[pos] = ck;
            }
        }
        __syncthreads();
    }
    const uint32_t got = sm.nsel;
    const uint32_t nsel = got < width ? got : width;
    if (got > width && t == 0) atomicOr(status, kStatusCandOverflow);
    if (out) write_winners(sm, sel, nsel, width, out, offset);
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
    r.l0 = pick_bin(sm.h, width, sm.scratch);
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
        return finish_row(SmemCandSource{sm.cand, got < (uint32_t)kLeaderCap ? got : (uint32_t)kLeaderCap}, st, width,
                          L, out, sm, sel, status, offset);
    }
    return finish_row(RowSource{s, L}, refine_from_level0(c.l0, width), width, L, out, sm, sel, status,
                      offset);
}

}  // namespace rowsel
}  // namespace dsrows
