// C-ABI entry points of libdsrows: validation, workspace layout, launches.
//
// Validation mirrors the row checks of mlx-native src/ops/deepseek_rows.rs
// (check_rows, sparse_params, sparse_io_checks, the indexer's per-row
// checks and `disjoint`), adapted to raw pointers: rows 1..8, kv_len and
// width nonzero, scale finite and positive, q_row unique for outputs,
// indices ranges disjoint for outputs, 32-bit ranges, plus pointer presence
// and alignment. Everything is checked before anything is enqueued.

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "kernels.h"

using namespace dsrows;

namespace {

thread_local std::string g_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_error = std::string("dsrows: ") + buf;
    return code;
}

int cuda_fail(cudaError_t err, const char* what) {
    return fail(DS_ECUDA, "%s failed: %s", what, cudaGetErrorString(err));
}

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// An NVTX range over the host-side enqueue of one stage ("dsrows.<stage>"), so
// a profiler can attribute each launch to its stage; free without a tool.
struct StageRange {
    explicit StageRange(const char* name) { nvtxRangePushA(name); }
    ~StageRange() { nvtxRangePop(); }
    StageRange(const StageRange&) = delete;
    StageRange& operator=(const StageRange&) = delete;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ---- workspace layout ------------------------------------------------------
struct Layout {
    size_t status = 0;  // u32 status word at offset 0
    size_t hist = 0, flags = 0, ctl_end = 0;
    size_t pub = 0, part = 0, scores = 0, total = 0;
    uint32_t attn_chunks = 0;
    uint64_t score_stride = 0;  // floats per row of the decode scores
};

// `rows` table entries (up to kVRowsMax virtual rows for the multi-query
// indexer): one histogram and one score row each.
Layout make_layout(int rows, const ds_row_t* table, bool attention = true) {
    Layout L;
    L.hist = 256;
    L.flags = align256(L.hist + (size_t)(rows > kRowsMax ? rows : kRowsMax) * kHistBins * 4);
    // flags: [8][64] head bits, [8] row bits, [8] "winners published" flags
    L.ctl_end = align256(L.flags + ((size_t)kRowsMax * kHeads + 2 * kRowsMax) * 4);
    L.pub = L.ctl_end;  // [8][512] u64 published winners + [8] u32 their number
    L.part = align256(L.pub + (size_t)kRowsMax * kTopK * 8 + kRowsMax * 4);
    uint32_t chunks = 0, max_len = 0;
    for (int e = 0; e < rows; ++e) {
        chunks += (table[e].width + kTailChunkSlots - 1) / kTailChunkSlots;
        if (table[e].kv_len > max_len) max_len = table[e].kv_len;
    }
    if (!attention) chunks = 0;
    L.attn_chunks = chunks;
    L.scores = align256(L.part + 2 * (size_t)chunks * kPartFloats * 4);  // two head halves per chunk
    L.score_stride = ((uint64_t)max_len + 63) & ~uint64_t(63);
    L.total = align256(L.scores + (size_t)rows * L.score_stride * 4);
    return L;
}

// ---- device facts and the tensor-map encoder --------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int num_sms() {
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode ? DS_OK : fail(DS_ECUDA, "cuTensorMapEncodeTiled is unavailable");
}

// 2D bf16 row-major [rows, 128] with a {64, box_rows} box and 128-byte swizzle.
int encode_rows128(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows, const char* what) {
    const cuuint64_t dims[2] = {128, rows};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DS_ECUDA, "tensor map for %s failed (CUresult %d)", what, (int)r);
    return DS_OK;
}

// ---- validation ----------------------------------------------------------------
enum Needs : unsigned { kNeedKeys = 1, kNeedKv = 2, kUniqueQ = 4, kDisjointOut = 8, kFullWidth = 16 };

int check_table(int rows, const ds_row_t* table) {
    if (rows < 1 || rows > DS_ROWS_MAX) return fail(DS_EINVAL, "rows must be 1..=%d, got %d", DS_ROWS_MAX, rows);
    if (!table) return fail(DS_EINVAL, "row table is NULL");
    for (int e = 0; e < rows; ++e) {
        const ds_row_t& r = table[e];
        if (r.kv_len == 0 || r.width == 0) return fail(DS_EINVAL, "row %d: kv_len and width must be nonzero", e);
        if (r.width > DS_TOPK) return fail(DS_EINVAL, "row %d: width %u exceeds %d", e, r.width, DS_TOPK);
        if (r.width > r.kv_len) return fail(DS_EINVAL, "row %d: width %u exceeds kv_len %u", e, r.width, r.kv_len);
        if ((uint64_t)r.index_offset + r.width > 0xFFFFFFFFull)
            return fail(DS_ESIZE, "row %d: index range exceeds u32", e);
        if ((uint64_t)r.q_row * DS_HEADS * DS_DIM > 0xFFFFFFFFFFull)
            return fail(DS_ESIZE, "row %d: q_row %u is out of range", e, r.q_row);
    }
    return DS_OK;
}

int check_set(const ds_row_set_t* set, unsigned needs) {
    if (!set) return fail(DS_EINVAL, "row set is NULL");
    int rc = check_table(set->rows, set->table);
    if (rc) return rc;
    const int rows = set->rows;
    for (int e = 0; e < rows; ++e) {
        if (needs & kFullWidth) {
            const ds_row_t& r = set->table[e];
            const uint32_t full = r.kv_len < (uint32_t)DS_TOPK ? r.kv_len : (uint32_t)DS_TOPK;
            if (r.width != full)
                return fail(DS_EINVAL, "row %d: width %u must be min(%d, kv_len) = %u", e, r.width, DS_TOPK, full);
        }
        if (needs & kNeedKeys) {
            if (!set->index_keys || !set->index_keys[e]) return fail(DS_EINVAL, "row %d: indexer keys are NULL", e);
            if (!aligned16(set->index_keys[e])) return fail(DS_EALIGN, "row %d: indexer keys not 16-B aligned", e);
        }
        if (needs & kNeedKv) {
            if (!set->kv || !set->kv[e]) return fail(DS_EINVAL, "row %d: kv cache is NULL", e);
            if (!aligned16(set->kv[e])) return fail(DS_EALIGN, "row %d: kv cache not 16-B aligned", e);
        }
        if (needs & kUniqueQ)
            for (int o = 0; o < e; ++o)
                if (set->table[o].q_row == set->table[e].q_row)
                    return fail(DS_EINVAL, "row %d: q_row %u is used twice", e, set->table[e].q_row);
        if (needs & kDisjointOut)
            for (int o = 0; o < e; ++o) {
                const uint64_t a0 = set->table[e].index_offset, a1 = a0 + set->table[e].width;
                const uint64_t b0 = set->table[o].index_offset, b1 = b0 + set->table[o].width;
                if (a0 < b1 && b0 < a1) return fail(DS_EINVAL, "index outputs of rows %d and %d overlap", o, e);
            }
    }
    return DS_OK;
}

// Positioned indexer rows (`dispatch_deepseek_indexer_rows`), each with
// query_len consecutive queries (query j at position start_pos + j): kv_len
// nonzero and not shorter than the last query's causal count
// (start_pos + query_len) / 4; offset nonnegative and offset + count - 1
// within int32; the rows' query_len x 512 output slots disjoint.
int check_indexer_rows(int rows, const ds_indexer_row_t* table, const ds_bf16* const* keys, bool need_keys,
                       uint32_t query_len = 1) {
    if (rows < 1 || rows > DS_ROWS_MAX) return fail(DS_EINVAL, "rows must be 1..=%d, got %d", DS_ROWS_MAX, rows);
    if (!table) return fail(DS_EINVAL, "indexer row table is NULL");
    if (query_len < 1 || (uint64_t)rows * query_len > DS_INDEX_VROWS_MAX)
        return fail(DS_EINVAL, "rows x query_len must be 1..=%d, got %d x %u", DS_INDEX_VROWS_MAX, rows, query_len);
    if (need_keys && !keys) return fail(DS_EINVAL, "index_keys is NULL");
    const uint64_t span = (uint64_t)DS_TOPK * query_len;
    for (int e = 0; e < rows; ++e) {
        const ds_indexer_row_t& r = table[e];
        if (r.kv_len == 0) return fail(DS_EINVAL, "indexer row %d: kv_len must be nonzero", e);
        if ((uint64_t)r.start_pos + query_len > 0xFFFFFFFFull)
            return fail(DS_EINVAL, "indexer row %d: position overflows", e);
        const uint32_t causal = (r.start_pos + query_len) / 4;  // the last query's count
        if (r.kv_len < causal)
            return fail(DS_EINVAL, "indexer row %d: kv_len %u is shorter than %u causal compressed entries", e,
                        r.kv_len, causal);
        if (r.offset < 0)
            return fail(DS_EINVAL, "indexer row %d: offset must be nonnegative; -1 is reserved for the sentinel", e);
        if (causal > 0 && (int64_t)r.offset + (int64_t)causal - 1 > (int64_t)INT32_MAX)
            return fail(DS_EINVAL, "indexer row %d: offset plus compressed index exceeds i32", e);
        if ((uint64_t)r.output_offset + span > 0xFFFFFFFFull)
            return fail(DS_ESIZE, "indexer row %d: output range exceeds u32", e);
        if (((uint64_t)r.q_row + query_len) * DS_INDEX_HEADS * DS_INDEX_DIM > 0xFFFFFFFFFFull)
            return fail(DS_ESIZE, "indexer row %d: q_row %u is out of range", e, r.q_row);
        if (need_keys) {
            if (!keys[e]) return fail(DS_EINVAL, "indexer row %d: keys are NULL", e);
            if (!aligned16(keys[e])) return fail(DS_EALIGN, "indexer row %d: keys not 16-B aligned", e);
        }
        for (int o = 0; o < e; ++o) {
            const uint64_t a0 = r.output_offset, a1 = a0 + span;
            const uint64_t b0 = table[o].output_offset, b1 = b0 + span;
            if (a0 < b1 && b0 < a1) return fail(DS_EINVAL, "indexer outputs of rows %d and %d overlap", o, e);
        }
    }
    return DS_OK;
}

// The selection table of positioned rows, one entry per (row e, query j) at
// v = e * query_len + j: kv_len = that query's causal count, 512 slots at
// output_offset + 512 j, query row q_row + j.
void indexer_selection_table(int rows, const ds_indexer_row_t* table, uint32_t query_len, ds_row_t* sel) {
    for (int e = 0; e < rows; ++e)
        for (uint32_t j = 0; j < query_len; ++j) {
            ds_row_t& v = sel[e * query_len + j];
            v.kv_len = (table[e].start_pos + j + 1) / 4;
            v.width = DS_TOPK;
            v.index_offset = table[e].output_offset + DS_TOPK * j;
            v.q_row = table[e].q_row + j;
        }
}

int check_workspace(const ds_row_set_t* set, void* ws, size_t bytes, const Layout& L) {
    (void)set;
    if (!ws) return fail(DS_EINVAL, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) & 255) return fail(DS_EALIGN, "workspace must be 256-byte aligned");
    if (bytes < L.total) return fail(DS_ESIZE, "workspace holds %zu bytes, needs %zu", bytes, L.total);
    return DS_OK;
}

// ---- stage launchers ---------------------------------------------------------------
cudaError_t launch_clear_stage(uint32_t* p, uint32_t words, cudaStream_t stream) {
    StageRange range("dsrows.clear");
    return launch_clear(p, words, stream);
}

// Entry e of `set` has query_len consecutive queries, virtual rows
// v = e * query_len + j with query row q_row + j; with `valid`, virtual row v
// scores only its keys j < valid[v] (the tensor map still spans the entry's
// kv_len keys), else every key. One query per entry runs the one-query kernel;
// more run the grouped kernel, up to kIndexerGroup queries per key tile.
// `inputs_ready` (see IndexerParams): 1 when the launch follows an ordinary
// launch (the clear kernel), so every input is complete and the key stream may
// start before the programmatic wait; 2 when the previous kernel writes the
// query and weights; 0 when it may write anything.
// Split `grid` CTAs over `segs` segments of tiles (segment s: tiles
// [tile_begin[s], tile_begin[s+1]), the last one up to `tiles`) in proportion to
// their tiles, every nonempty segment at least one CTA and none more CTAs than
// tiles; cta_begin[s] is the first CTA of segment s, cta_begin[segs] = grid.
// grid <= tiles, and grid >= the nonempty segments (grid = min(tiles, SMs)).
void split_ctas(const uint32_t* tile_begin, uint32_t* cta_begin, uint32_t segs, uint32_t tiles, uint32_t grid) {
    uint32_t ts[kSegMax], n[kSegMax];
    double rem[kSegMax];
    uint32_t used = 0;
    for (uint32_t s = 0; s < segs; ++s) {
        ts[s] = (s + 1 < segs ? tile_begin[s + 1] : tiles) - tile_begin[s];
        const double want = tiles ? (double)grid * ts[s] / tiles : 0.0;
        n[s] = (uint32_t)want;
        if (ts[s] > 0 && n[s] == 0) n[s] = 1;
        if (n[s] > ts[s]) n[s] = ts[s];
        rem[s] = want - n[s];
        used += n[s];
    }
    while (used > grid) {  // the minimum of one CTA took too many: shrink the largest
        uint32_t best = 0;
        for (uint32_t s = 1; s < segs; ++s)
            if (n[s] > n[best]) best = s;
        --n[best];
        rem[best] += 1.0;
        --used;
    }
    while (used < grid) {  // largest remainders first
        int best = -1;
        for (uint32_t s = 0; s < segs; ++s)
            if (n[s] < ts[s] && (best < 0 || rem[s] > rem[best])) best = (int)s;
        if (best < 0) break;
        ++n[best];
        rem[best] -= 1.0;
        ++used;
    }
    uint32_t c = 0;
    for (uint32_t s = 0; s < segs; ++s) {
        cta_begin[s] = c;
        c += n[s];
    }
    cta_begin[segs] = c;
}

template <class P>
int fill_and_launch_indexer(P& p, int group, const ds_row_set_t* set, uint32_t query_len, const ds_bf16* q_index,
                            const float* w_index, float* scores, uint64_t stride, uint32_t* hist, uint32_t* status,
                            cudaStream_t stream, uint32_t inputs_ready, const uint32_t* valid, const void* side_src,
                            void* side_dst, size_t side_bytes) {
    int rc = get_encoder();
    if (rc) return rc;
    std::memset(&p, 0, sizeof(p));
    const uint32_t tile = indexer_tile_keys();
    constexpr uint32_t kSegs = sizeof(p.tile_begin) / sizeof(p.tile_begin[0]);
    constexpr uint32_t kVRows = sizeof(p.valid) / sizeof(p.valid[0]);
    if ((uint64_t)set->rows * query_len > kVRows) return fail(DS_EINVAL, "too many indexer rows");
    uint32_t tiles = 0, segs = 0, max_q = 0;
    for (int e = 0; e < set->rows; ++e) {
        const ds_row_t& r = set->table[e];
        for (uint32_t j0 = 0; j0 < query_len; j0 += group) {
            const uint32_t nq = query_len - j0 < (uint32_t)group ? query_len - j0 : (uint32_t)group;
            const uint32_t v0 = e * query_len + j0;
            uint32_t cover = 0;
            for (uint32_t i = 0; i < nq; ++i) {
                const uint32_t n = valid ? valid[v0 + i] : r.kv_len;
                p.valid[v0 + i] = n;
                p.q_row[v0 + i] = r.q_row + j0 + i;
                cover = n > cover ? n : cover;
            }
            if (segs >= kSegs) return fail(DS_EINVAL, "too many indexer segments");
            p.tile_begin[segs] = tiles;
            p.seg_entry[segs] = (uint8_t)e;
            p.seg_vrow[segs] = (uint8_t)v0;
            p.seg_queries[segs] = (uint8_t)nq;
            ++segs;
            tiles += (cover + tile - 1) / tile;
        }
        if (r.q_row + query_len > max_q) max_q = r.q_row + query_len;
        rc = encode_rows128(&p.kmap[e], set->index_keys[e], r.kv_len, 128, "indexer keys");
        if (rc) return rc;
    }
    rc = encode_rows128(&p.qmap, q_index, (uint64_t)max_q * DS_INDEX_HEADS, 64, "indexer q");
    if (rc) return rc;
    p.w = w_index;
    p.scores = scores;
    p.hist = hist;
    p.status = status;
    p.score_stride = stride;
    p.inputs_ready = inputs_ready;
    p.side_src = static_cast<const uint4*>(side_src);
    p.side_dst = static_cast<uint4*>(side_dst);
    p.side_n16 = (uint32_t)(side_bytes / 16);
    p.rows = (uint32_t)set->rows;
    p.segs = segs;
    p.vrows = (uint32_t)set->rows * query_len;
    p.total_tiles = tiles;
    const int sms = num_sms();
    if (sms <= 0) return fail(DS_ECUDA, "no CUDA device");
    if (group == 1) split_ctas(p.tile_begin, p.cta_begin, segs, tiles, tiles < (uint32_t)sms ? tiles : (uint32_t)sms);
    cudaError_t err = launch_indexer(p, sms, stream, true);
    return err == cudaSuccess ? DS_OK : cuda_fail(err, "indexer launch");
}

// `side_*`: an optional copy the indexer makes for the attention (see IndexerParamsT).
int run_indexer(const ds_row_set_t* set, uint32_t query_len, const ds_bf16* q_index, const float* w_index,
                float* scores, uint64_t stride, uint32_t* hist, uint32_t* status, cudaStream_t stream,
                uint32_t inputs_ready, const uint32_t* valid = nullptr, const void* side_src = nullptr,
                void* side_dst = nullptr, size_t side_bytes = 0) {
    StageRange range("dsrows.indexer");
    // The tables hold CUtensorMaps (~1.3-2.2 KB); built per call on the host.
    if (query_len == 1) {
        IndexerParams1 p;
        return fill_and_launch_indexer(p, 1, set, query_len, q_index, w_index, scores, stride, hist, status, stream,
                                       inputs_ready, valid, side_src, side_dst, side_bytes);
    }
    IndexerParamsG p;
    return fill_and_launch_indexer(p, kIndexerGroup, set, query_len, q_index, w_index, scores, stride, hist, status,
                                   stream, inputs_ready, valid, side_src, side_dst, side_bytes);
}

// The level-0 histogram (with_hist) and the top-k kernel's selection
// (select), one 8-CTA cluster per row.
int run_topk(const ds_row_set_t* set, const float* scores, uint64_t stride, int32_t* out, const uint32_t* out_offset,
             uint8_t* ws, const Layout& L, bool with_hist, cudaStream_t stream,
             const int32_t* offsets = nullptr, bool select = true) {
    if (set->rows > kVRowsMax) return fail(DS_EINVAL, "too many top-k rows");
    StageRange range("dsrows.topk");
    TopkParams p;
    std::memset(&p, 0, sizeof(p));
    const uint32_t chunk = topk_chunk();
    uint32_t chunks = 0;
    for (int e = 0; e < set->rows; ++e) {
        p.kv_len[e] = set->table[e].kv_len;
        p.width[e] = set->table[e].width;
        p.out_offset[e] = out_offset[e];
        p.offset[e] = offsets ? offsets[e] : 0;
        p.chunk_begin[e] = chunks;
        chunks += (set->table[e].kv_len + chunk - 1) / chunk;
    }
    p.scores = scores;
    p.score_stride = stride;
    p.out = out;
    p.hist = reinterpret_cast<uint32_t*>(ws + L.hist);
    p.status = reinterpret_cast<uint32_t*>(ws + L.status);
    p.rows = (uint32_t)set->rows;
    p.total_chunks = chunks;
    cudaError_t err = cudaSuccess;
    if (with_hist) {
        err = launch_topk_hist(p, stream, true);
        if (err != cudaSuccess) return cuda_fail(err, "top-k histogram launch");
    }
    if (!select) return DS_OK;
    err = launch_topk_select(p, stream, true);
    return err == cudaSuccess ? DS_OK : cuda_fail(err, "top-k select launch");
}

// Selection (decode: `given` null) or the caller's indices (`given`), then the
// attention: one 8-CTA cluster per row.
int run_tail(const ds_row_set_t* set, const ds_bf16* q_attn, const float* sinks, size_t sinks_row_stride,
             float scale, ds_bf16* out, uint32_t* invalid, const float* scores, uint64_t score_stride,
             const int32_t* given, int32_t* indices, uint8_t* ws, const Layout& L, cudaStream_t stream,
             bool q_after_wait = false, bool attend = true, const int32_t* offsets = nullptr) {
    StageRange range(attend ? (given ? "dsrows.attention" : "dsrows.select+attention") : "dsrows.select");
    TailParams tp;
    std::memset(&tp, 0, sizeof(tp));
    uint32_t chunks = 0;
    for (int e = 0; e < set->rows; ++e) {
        const ds_row_t& r = set->table[e];
        tp.kv[e] = set->kv ? reinterpret_cast<const __nv_bfloat16*>(set->kv[e]) : nullptr;
        tp.kv_len[e] = r.kv_len;
        tp.width[e] = r.width;
        tp.index_offset[e] = r.index_offset;
        tp.q_row[e] = r.q_row;
        tp.chunk_begin[e] = chunks;
        chunks += (r.width + kTailChunkSlots - 1) / kTailChunkSlots;
    }
    tp.scores = scores;
    tp.score_stride = score_stride;
    tp.hist = reinterpret_cast<const uint32_t*>(ws + L.hist);
    tp.status = reinterpret_cast<uint32_t*>(ws + L.status);
    tp.q = reinterpret_cast<const __nv_bfloat16*>(q_attn);
    tp.q_after_wait = q_after_wait ? 1u : 0u;
    tp.attend = attend ? 1u : 0u;
    for (int e = 0; e < set->rows; ++e) tp.offset[e] = offsets ? offsets[e] : 0;
    tp.sinks = sinks;
    tp.sinks_row_stride = sinks_row_stride;
    // Selection only: no partials, flags or published winners are touched.
    tp.part = attend ? reinterpret_cast<float*>(ws + L.part) : nullptr;
    tp.flags = attend ? reinterpret_cast<uint32_t*>(ws + L.flags) : nullptr;
    // With attention, the best-first index list is ranked by one more cluster
    // from the winners each row publishes in the workspace.
    tp.ranker = attend && indices && given == nullptr && L.pub ? 1u : 0u;
    tp.pub = attend && L.pub ? reinterpret_cast<uint64_t*>(ws + L.pub) : nullptr;
    tp.out = reinterpret_cast<__nv_bfloat16*>(out);
    tp.invalid = invalid;
    tp.given = given;
    tp.indices = indices;
    tp.scale = scale;
    tp.rows = (uint32_t)set->rows;
    cudaError_t err = launch_decode_tail(tp, stream, true);
    return err == cudaSuccess ? DS_OK : cuda_fail(err, given ? "attention launch" : "decode select + attention launch");
}

// Best-first top-k of the set's rows into indices (+ offsets), after the
// level-0 histogram (built here with with_hist, else already in the
// workspace). Up to 8 rows: the decode's tail kernel in selection-only mode
// (its placement by distributed ranking is faster than the top-k kernel's
// leader-only sort); more: the top-k kernel.
int run_select(const ds_row_set_t* set, const float* scores, uint64_t stride, int32_t* indices, uint8_t* ws,
               const Layout& L, bool with_hist, cudaStream_t s, const int32_t* offsets = nullptr) {
    uint32_t off[kVRowsMax];
    for (int e = 0; e < set->rows; ++e) off[e] = set->table[e].index_offset;
    if (set->rows > kRowsMax) return run_topk(set, scores, stride, indices, off, ws, L, with_hist, s, offsets);
    if (with_hist) {
        const int rc = run_topk(set, scores, stride, indices, off, ws, L, true, s, offsets, false);
        if (rc) return rc;
    }
    return run_tail(set, nullptr, nullptr, 0, 1.0f, nullptr, nullptr, scores, stride, nullptr, indices, ws, L, s,
                    false, false, offsets);
}

int check_attn_args(const ds_bf16* q_attn, const float* sinks, size_t sinks_row_stride, float scale, ds_bf16* out) {
    if (!q_attn || !sinks || !out) return fail(DS_EINVAL, "q_attn, sinks and out must be non-NULL");
    if (!aligned16(q_attn) || !aligned16(out)) return fail(DS_EALIGN, "q_attn and out must be 16-B aligned");
    if (sinks_row_stride != 0 && sinks_row_stride < DS_HEADS)
        return fail(DS_EINVAL, "sinks_row_stride must be 0 or >= %d, got %zu", DS_HEADS, sinks_row_stride);
    if (!(scale > 0.0f) || !(scale < __builtin_huge_valf())) return fail(DS_EINVAL, "scale must be finite and positive");
    return DS_OK;
}

int check_indexer_args(const ds_bf16* q_index, const float* w_index) {
    if (!q_index || !w_index) return fail(DS_EINVAL, "q_index and w_index must be non-NULL");
    if (!aligned16(q_index)) return fail(DS_EALIGN, "q_index must be 16-B aligned");
    return DS_OK;
}

}  // namespace

// ---- top-k with scratch held by the library ------------------------------------
// Some callers cannot allocate device memory at the point where they call the
// top-k stage (a CUDA-graph or real-time caller that forbids allocation, or an
// embedder whose allocator is not reachable from the calling code). For them
// ds_rows_topk_static keeps the stage's scratch (status word and the per-row
// score histograms) in this one file-scope device array, sized for
// DS_ROWS_MAX rows; every GPU that loads the library holds it until the
// process exits.
namespace {

constexpr size_t kStaticHist = 256;
constexpr size_t kStaticBytes = kStaticHist + (size_t)kRowsMax * kHistBins * 4;
static_assert(kStaticBytes == DS_TOPK_STATIC_SCRATCH_BYTES, "header size must match the scratch layout");

}  // namespace

static __device__ __align__(256) uint8_t g_topk_scratch[kStaticBytes];

namespace {

std::mutex g_scratch_mu;
uint8_t* g_scratch_ptr[64] = {};

// The scratch's device address on the current device, looked up once per
// device. In host code `g_topk_scratch` names a host-side stand-in, never
// the device memory, so only this address may be passed to a kernel.
int topk_scratch(uint8_t** out) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(DS_ECUDA, "device %d is out of range", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* addr = nullptr;
        err = cudaGetSymbolAddress(&addr, g_topk_scratch);
        if (err != cudaSuccess) return cuda_fail(err, "cudaGetSymbolAddress of the top-k scratch");
        g_scratch_ptr[dev] = static_cast<uint8_t*>(addr);
    }
    *out = g_scratch_ptr[dev];
    return DS_OK;
}

// ---- the host-buffer decode ----------------------------------------------------
// Device staging of the step's inputs and outputs, after the decode workspace.
struct Staging {
    size_t q_index, w_index, q_attn, sinks, out, indices, invalid, total;
    uint32_t nq;          // query rows: max q_row + 1
    size_t sinks_floats;  // floats of sinks the entries read
    uint64_t index_elems; // max index_offset + width
};

Staging make_staging(const ds_row_set_t* set, size_t base, size_t sinks_row_stride) {
    Staging S{};
    uint32_t nq = 0;
    uint64_t ie = 0;
    for (int e = 0; e < set->rows; ++e) {
        const ds_row_t& r = set->table[e];
        nq = r.q_row + 1 > nq ? r.q_row + 1 : nq;
        const uint64_t end = (uint64_t)r.index_offset + r.width;
        ie = end > ie ? end : ie;
    }
    S.nq = nq;
    S.index_elems = ie;
    S.sinks_floats = sinks_row_stride ? (size_t)(nq - 1) * sinks_row_stride + DS_HEADS : DS_HEADS;
    S.q_index = align256(base);
    S.w_index = align256(S.q_index + (size_t)nq * DS_INDEX_HEADS * DS_INDEX_DIM * 2);
    S.q_attn = align256(S.w_index + (size_t)nq * DS_INDEX_HEADS * 4);
    S.sinks = align256(S.q_attn + (size_t)nq * DS_HEADS * DS_DIM * 2);
    S.out = align256(S.sinks + S.sinks_floats * 4);
    S.indices = align256(S.out + (size_t)nq * DS_HEADS * DS_DIM * 2);
    S.invalid = align256(S.indices + (size_t)ie * 4);
    S.total = align256(S.invalid + (size_t)nq * DS_HEADS * 4);
    return S;
}

// The device address of pinned (page-locked) host memory, which kernels may
// read and write directly; null for any other memory (pageable or device).
template <class T>
T* mapped_host(T* p) {
    if (!p) return nullptr;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost && a.devicePointer ? static_cast<T*>(a.devicePointer) : nullptr;
}

int copy_async(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s, const char* what) {
    if (bytes == 0) return DS_OK;
    cudaError_t err = cudaMemcpyAsync(dst, src, bytes, kind, s);
    return err == cudaSuccess ? DS_OK : cuda_fail(err, what);
}

}  // namespace

extern "C" {

size_t ds_rows_workspace_bytes(int rows, const ds_row_t* table) {
    if (check_table(rows, table)) return 0;
    return make_layout(rows, table).total;
}

int ds_rows_indexer_score(const ds_row_set_t* set, const ds_bf16* q_index, const float* w_index, float* scores,
                          size_t score_stride, void* stream) {
    int rc = check_set(set, kNeedKeys);
    if (rc) return rc;
    rc = check_indexer_args(q_index, w_index);
    if (rc) return rc;
    if (!scores) return fail(DS_EINVAL, "scores is NULL");
    for (int e = 0; e < set->rows; ++e)
        if (score_stride < set->table[e].kv_len)
            return fail(DS_EINVAL, "score_stride %zu is shorter than row %d (kv_len %u)", score_stride, e,
                        set->table[e].kv_len);
    return run_indexer(set, 1, q_index, w_index, scores, score_stride, nullptr, nullptr, (cudaStream_t)stream, 0);
}

int ds_rows_topk(const ds_row_set_t* set, const float* scores, size_t score_stride, int32_t* indices,
                 void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_set(set, kDisjointOut | kFullWidth);
    if (rc) return rc;
    if (!scores || !indices) return fail(DS_EINVAL, "scores and indices must be non-NULL");
    for (int e = 0; e < set->rows; ++e)
        if (score_stride < set->table[e].kv_len)
            return fail(DS_EINVAL, "score_stride %zu is shorter than row %d (kv_len %u)", score_stride, e,
                        set->table[e].kv_len);
    const Layout L = make_layout(set->rows, set->table);
    rc = check_workspace(set, workspace, workspace_bytes, L);
    if (rc) return rc;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t err = launch_clear_stage(reinterpret_cast<uint32_t*>(ws), (uint32_t)(L.ctl_end / 4), s);
    if (err != cudaSuccess) return cuda_fail(err, "workspace clear");
    return run_select(set, scores, score_stride, indices, ws, L, true, s);
}

int ds_rows_sparse_attn(const ds_row_set_t* set, const ds_bf16* q_attn, const float* sinks,
                        size_t sinks_row_stride, const int32_t* indices, float scale, ds_bf16* out,
                        uint32_t* invalid, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_set(set, kNeedKv | kUniqueQ);
    if (rc) return rc;
    rc = check_attn_args(q_attn, sinks, sinks_row_stride, scale, out);
    if (rc) return rc;
    if (!indices) return fail(DS_EINVAL, "indices is NULL");
    const Layout L = make_layout(set->rows, set->table);
    rc = check_workspace(set, workspace, workspace_bytes, L);
    if (rc) return rc;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t err = launch_clear_stage(reinterpret_cast<uint32_t*>(ws), (uint32_t)(L.ctl_end / 4), s);
    if (err != cudaSuccess) return cuda_fail(err, "workspace clear");
    return run_tail(set, q_attn, sinks, sinks_row_stride, scale, out, invalid, nullptr, 0, indices, nullptr, ws, L, s);
}

int ds_rows_decode(const ds_row_set_t* set, const ds_bf16* q_index, const float* w_index, const ds_bf16* q_attn,
                   const float* sinks, size_t sinks_row_stride, float scale, ds_bf16* out, int32_t* indices,
                   uint32_t* invalid, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_set(set, kNeedKeys | kNeedKv | kUniqueQ | kFullWidth | (indices ? kDisjointOut : 0u));
    if (rc) return rc;
    rc = check_indexer_args(q_index, w_index);
    if (rc) return rc;
    rc = check_attn_args(q_attn, sinks, sinks_row_stride, scale, out);
    if (rc) return rc;
    const Layout L = make_layout(set->rows, set->table);
    rc = check_workspace(set, workspace, workspace_bytes, L);
    if (rc) return rc;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t err = launch_clear_stage(reinterpret_cast<uint32_t*>(ws), (uint32_t)(L.ctl_end / 4), s);
    if (err != cudaSuccess) return cuda_fail(err, "workspace clear");
    float* scores = reinterpret_cast<float*>(ws + L.scores);
    uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
    uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
    rc = run_indexer(set, 1, q_index, w_index, scores, L.score_stride, hist, status, s, 1);
    if (rc) return rc;
    // Selection and attention in one kernel: one 8-CTA cluster per row keeps the
    // selection on chip and attends over it in best-first order, the order of
    // the indices it writes for the caller.
    return run_tail(set, q_attn, sinks, sinks_row_stride, scale, out, invalid, scores, L.score_stride, nullptr,
                    indices, ws, L, s);
}

size_t ds_rows_decode_host_workspace_bytes(int rows, const ds_row_t* table, size_t sinks_row_stride) {
    if (check_table(rows, table)) return 0;
    if (sinks_row_stride != 0 && sinks_row_stride < DS_HEADS) return 0;
    const ds_row_set_t set = {rows, table, nullptr, nullptr};
    return make_staging(&set, make_layout(rows, table).total, sinks_row_stride).total;
}

int ds_rows_decode_host(const ds_row_set_t* set, const ds_bf16* h_q_index, const float* h_w_index,
                        const ds_bf16* h_q_attn, const float* h_sinks, size_t sinks_row_stride, float scale,
                        ds_bf16* h_out, int32_t* h_indices, uint32_t* h_invalid, void* workspace,
                        size_t workspace_bytes, void* stream) {
    int rc = check_set(set, kNeedKeys | kNeedKv | kUniqueQ | kFullWidth | (h_indices ? kDisjointOut : 0u));
    if (rc) return rc;
    if (!h_q_index || !h_w_index || !h_q_attn || !h_sinks || !h_out)
        return fail(DS_EINVAL, "host q_index, w_index, q_attn, sinks and out must be non-NULL");
    if (!aligned16(h_q_index) || !aligned16(h_q_attn) || !aligned16(h_out))
        return fail(DS_EALIGN, "host q_index, q_attn and out must be 16-B aligned");
    if (sinks_row_stride != 0 && sinks_row_stride < DS_HEADS)
        return fail(DS_EINVAL, "sinks_row_stride must be 0 or >= %d, got %zu", DS_HEADS, sinks_row_stride);
    if (!(scale > 0.0f) || !(scale < __builtin_huge_valf())) return fail(DS_EINVAL, "scale must be finite and positive");
    const Layout L = make_layout(set->rows, set->table);
    const Staging S = make_staging(set, L.total, sinks_row_stride);
    if (!workspace) return fail(DS_EINVAL, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(DS_EALIGN, "workspace must be 256-byte aligned");
    if (workspace_bytes < S.total)
        return fail(DS_ESIZE, "workspace holds %zu bytes, needs %zu", workspace_bytes, S.total);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    const uint32_t nq = S.nq;
    const bool dense = nq == (uint32_t)set->rows;  // every query row 0..nq-1 is an entry's
    const size_t qI_row = (size_t)DS_INDEX_HEADS * DS_INDEX_DIM, wI_row = DS_INDEX_HEADS;
    const size_t qA_row = (size_t)DS_HEADS * DS_DIM;
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;

    // The indexer's query and weights go to device staging (its query is a
    // TMA operand). Pinned and dense: the workspace-clear kernel copies them
    // (no copy engine round trip); else copies, whole arrays or entry by entry.
    auto* d_qI = reinterpret_cast<ds_bf16*>(ws + S.q_index);
    auto* d_wI = reinterpret_cast<float*>(ws + S.w_index);
    const ds_bf16* m_qI = dense ? mapped_host(h_q_index) : nullptr;
    const float* m_wI = dense && aligned16(h_w_index) ? mapped_host(h_w_index) : nullptr;
    const bool kernel_copy = m_qI && m_wI;
    if (!kernel_copy && dense) {
        rc = copy_async(d_qI, h_q_index, nq * qI_row * 2, h2d, s, "q_index copy");
        if (!rc) rc = copy_async(d_wI, h_w_index, nq * wI_row * 4, h2d, s, "w_index copy");
    } else if (!kernel_copy) {
        for (int e = 0; e < set->rows && !rc; ++e) {
            const size_t r = set->table[e].q_row;
            rc = copy_async(d_qI + r * qI_row, h_q_index + r * qI_row, qI_row * 2, h2d, s, "q_index copy");
            if (!rc) rc = copy_async(d_wI + r * wI_row, h_w_index + r * wI_row, wI_row * 4, h2d, s, "w_index copy");
        }
    }
    if (rc) return rc;
    // The attention reads q_attn and the sinks, and writes its outputs, in
    // pinned host memory directly; other host memory goes through staging.
    // A pinned q_attn is copied into staging by the indexer's epilogue warps
    // while they wait for the first scores (the attention would otherwise
    // fetch it from host memory on its critical path); the attention then
    // fetches it after its wait.
    const ds_bf16* m_qA = mapped_host(h_q_attn);
    const ds_bf16* d_qA = m_qA ? reinterpret_cast<const ds_bf16*>(ws + S.q_attn) : nullptr;
    const float* d_sk = mapped_host(h_sinks);
    ds_bf16* d_out = mapped_host(h_out);
    int32_t* d_idx = h_indices ? mapped_host(h_indices) : nullptr;
    uint32_t* d_inv = h_invalid ? mapped_host(h_invalid) : nullptr;
    const bool stage_out = !d_out, stage_idx = h_indices && !d_idx, stage_inv = h_invalid && !d_inv;
    if (!d_qA) {
        auto* st = reinterpret_cast<ds_bf16*>(ws + S.q_attn);
        if (dense) {
            rc = copy_async(st, h_q_attn, nq * qA_row * 2, h2d, s, "q_attn copy");
        } else {
            for (int e = 0; e < set->rows && !rc; ++e) {
                const size_t o = (size_t)set->table[e].q_row * qA_row;
                rc = copy_async(st + o, h_q_attn + o, qA_row * 2, h2d, s, "q_attn copy");
            }
        }
        d_qA = st;
    }
    if (!rc && !d_sk) {
        auto* st = reinterpret_cast<float*>(ws + S.sinks);
        rc = copy_async(st, h_sinks, S.sinks_floats * 4, h2d, s, "sinks copy");
        d_sk = st;
    }
    if (rc) return rc;
    if (stage_out) d_out = reinterpret_cast<ds_bf16*>(ws + S.out);
    if (stage_idx) d_idx = reinterpret_cast<int32_t*>(ws + S.indices);
    if (stage_inv) d_inv = reinterpret_cast<uint32_t*>(ws + S.invalid);

    cudaError_t err =
        kernel_copy ? launch_clear_copy(reinterpret_cast<uint32_t*>(ws), (uint32_t)(L.ctl_end / 4), m_qI, d_qI,
                                        nq * qI_row * 2, m_wI, d_wI, nq * wI_row * 4, s)
                    : launch_clear(reinterpret_cast<uint32_t*>(ws), (uint32_t)(L.ctl_end / 4), s);
    if (err != cudaSuccess) return cuda_fail(err, "workspace clear");
    float* scores = reinterpret_cast<float*>(ws + L.scores);
    // With the kernel copy the indexer launches early (programmatic dependent
    // launch) and waits for that kernel (griddepcontrol.wait) before its first
    // query and key loads and before it reads the head weights.
    rc = run_indexer(set, 1, d_qI, d_wI, scores, L.score_stride, reinterpret_cast<uint32_t*>(ws + L.hist),
                     reinterpret_cast<uint32_t*>(ws + L.status), s, kernel_copy ? 2u : 1u, nullptr, m_qA,
                     ws + S.q_attn, m_qA ? nq * qA_row * 2 : 0);
    if (rc) return rc;
    rc = run_tail(set, d_qA, d_sk, sinks_row_stride, scale, d_out, d_inv, scores, L.score_stride, nullptr, d_idx, ws,
                  L, s, m_qA != nullptr);
    if (rc) return rc;

    // Staged outputs come back by copy.
    for (int e = 0; e < set->rows && !rc; ++e) {
        const ds_row_t& r = set->table[e];
        const size_t q = r.q_row;
        if (stage_out && (!dense || e == 0))
            rc = dense ? copy_async(h_out, d_out, nq * qA_row * 2, d2h, s, "out copy")
                       : copy_async(h_out + q * qA_row, d_out + q * qA_row, qA_row * 2, d2h, s, "out copy");
        if (!rc && stage_inv)
            rc = copy_async(h_invalid + q * DS_HEADS, d_inv + q * DS_HEADS, DS_HEADS * 4, d2h, s, "invalid copy");
        if (!rc && stage_idx)
            rc = copy_async(h_indices + r.index_offset, d_idx + r.index_offset, (size_t)r.width * 4, d2h, s,
                            "indices copy");
    }
    return rc;
}

int ds_rows_topk_static(const ds_row_set_t* set, const float* scores, size_t score_stride, int32_t* indices,
                        void* stream) {
    int rc = check_set(set, kDisjointOut | kFullWidth);
    if (rc) return rc;
    if (!scores || !indices) return fail(DS_EINVAL, "scores and indices must be non-NULL");
    for (int e = 0; e < set->rows; ++e)
        if (score_stride < set->table[e].kv_len)
            return fail(DS_EINVAL, "score_stride %zu is shorter than row %d (kv_len %u)", score_stride, e,
                        set->table[e].kv_len);
    const size_t need = kStaticHist + (size_t)set->rows * kHistBins * 4;
    if (need > kStaticBytes)
        return fail(DS_ESIZE, "top-k needs %zu bytes of scratch, the library holds %zu", need, kStaticBytes);
    uint8_t* ws = nullptr;
    rc = topk_scratch(&ws);
    if (rc) return rc;
    // The array holds only the status word and the histograms (no partials,
    // flags or scores: the selection-only path touches neither).
    Layout L{};
    L.hist = kStaticHist;
    cudaStream_t s = (cudaStream_t)stream;
    // The array keeps the previous call's contents: zero the status word and
    // the histograms before they are rebuilt.
    cudaError_t err = launch_clear(reinterpret_cast<uint32_t*>(ws), (uint32_t)(kStaticBytes / 4), s);
    if (err != cudaSuccess) return cuda_fail(err, "scratch clear");
    return run_select(set, scores, score_stride, indices, ws, L, true, s);
}

size_t ds_rows_indexer_topk_queries_workspace_bytes(int rows, const ds_indexer_row_t* table, uint32_t query_len) {
    if (check_indexer_rows(rows, table, nullptr, false, query_len)) return 0;
    ds_row_t sel[DS_INDEX_VROWS_MAX];
    indexer_selection_table(rows, table, query_len, sel);
    return make_layout(rows * (int)query_len, sel, false).total;
}

size_t ds_rows_indexer_topk_workspace_bytes(int rows, const ds_indexer_row_t* table) {
    return ds_rows_indexer_topk_queries_workspace_bytes(rows, table, 1);
}

int ds_rows_indexer_topk_queries(int rows, const ds_indexer_row_t* table, uint32_t query_len,
                                 const ds_bf16* const* index_keys, const ds_bf16* q_index, const float* w_index,
                                 int32_t* indices, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_indexer_rows(rows, table, index_keys, true, query_len);
    if (rc) return rc;
    rc = check_indexer_args(q_index, w_index);
    if (rc) return rc;
    if (!indices) return fail(DS_EINVAL, "indices is NULL");
    const int vrows = rows * (int)query_len;
    ds_row_t keys_tab[DS_ROWS_MAX], sel_tab[DS_INDEX_VROWS_MAX];
    uint32_t valid[DS_INDEX_VROWS_MAX];
    int32_t offsets[DS_INDEX_VROWS_MAX];
    indexer_selection_table(rows, table, query_len, sel_tab);
    for (int e = 0; e < rows; ++e) {
        keys_tab[e] = sel_tab[e * query_len];
        keys_tab[e].kv_len = table[e].kv_len;  // the tensor map spans the whole cache
        keys_tab[e].q_row = table[e].q_row;
    }
    for (int v = 0; v < vrows; ++v) {
        valid[v] = sel_tab[v].kv_len;
        offsets[v] = table[v / query_len].offset;
    }
    const Layout L = make_layout(vrows, sel_tab, false);
    const ds_row_set_t kset = {rows, keys_tab, index_keys, nullptr};
    const ds_row_set_t sset = {vrows, sel_tab, nullptr, nullptr};
    rc = check_workspace(&sset, workspace, workspace_bytes, L);
    if (rc) return rc;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t err = launch_clear_stage(reinterpret_cast<uint32_t*>(ws), (uint32_t)(L.ctl_end / 4), s);
    if (err != cudaSuccess) return cuda_fail(err, "workspace clear");
    float* scores = reinterpret_cast<float*>(ws + L.scores);
    rc = run_indexer(&kset, query_len, q_index, w_index, scores, L.score_stride,
                     reinterpret_cast<uint32_t*>(ws + L.hist), reinterpret_cast<uint32_t*>(ws + L.status), s, 1,
                     valid);
    if (rc) return rc;
    // The indexer built the level-0 histogram of each query's valid scores.
    return run_select(&sset, scores, L.score_stride, indices, ws, L, false, s, offsets);
}

int ds_rows_indexer_topk(int rows, const ds_indexer_row_t* table, const ds_bf16* const* index_keys,
                         const ds_bf16* q_index, const float* w_index, int32_t* indices, void* workspace,
                         size_t workspace_bytes, void* stream) {
    return ds_rows_indexer_topk_queries(rows, table, 1, index_keys, q_index, w_index, indices, workspace,
                                        workspace_bytes, stream);
}

int ds_rows_compress_kv(int rows, const ds_compressor_row_t* table, const float* kv, const float* score,
                        const float* ape, const float* norm, uint32_t ratio, uint32_t head_dim, float epsilon,
                        ds_bf16* out, void* stream) {
    if (rows < 1 || rows > DS_ROWS_MAX) return fail(DS_EINVAL, "rows must be 1..=%d, got %d", DS_ROWS_MAX, rows);
    if (!table) return fail(DS_EINVAL, "compressor row table is NULL");
    const bool supported = (ratio == 4 && (head_dim == 128 || head_dim == 512)) || (ratio == 128 && head_dim == 512);
    if (!supported)
        return fail(DS_EINVAL, "compressor (ratio, head_dim) must be (4,128), (4,512) or (128,512), got (%u,%u)",
                    ratio, head_dim);
    if (!(epsilon > 0.0f) || !(epsilon < __builtin_huge_valf()))
        return fail(DS_EINVAL, "compressor epsilon must be finite and positive");
    if (!kv || !score || !ape || !norm || !out) return fail(DS_EINVAL, "kv, score, ape, norm and out must be non-NULL");
    if (!aligned16(kv) || !aligned16(score) || !aligned16(ape) || !aligned16(norm) || !aligned16(out))
        return fail(DS_EALIGN, "kv, score, ape, norm and out must be 16-B aligned");
    const uint32_t coff = ratio == 4 ? 2 : 1;
    const size_t state_bytes = (size_t)coff * ratio * coff * head_dim * sizeof(float);
    CompressorParams p;
    std::memset(&p, 0, sizeof(p));
    for (int e = 0; e < rows; ++e) {
        const ds_compressor_row_t& r = table[e];
        if (r.start_pos == 0 || r.start_pos == 0xFFFFFFFFu)
            return fail(DS_EINVAL, "compressor row %d: position must be in 1..u32::MAX, got %u", e, r.start_pos);
        if (!r.kv_state || !r.score_state) return fail(DS_EINVAL, "compressor row %d: state is NULL", e);
        if (!aligned16(r.kv_state) || !aligned16(r.score_state))
            return fail(DS_EALIGN, "compressor row %d: state not 16-B aligned", e);
        const uintptr_t mine[2] = {reinterpret_cast<uintptr_t>(r.kv_state), reinterpret_cast<uintptr_t>(r.score_state)};
        if (mine[0] < mine[1] + state_bytes && mine[1] < mine[0] + state_bytes)
            return fail(DS_EINVAL, "compressor row %d: kv_state and score_state overlap", e);
        for (int o = 0; o < e; ++o) {
            const uintptr_t other[2] = {reinterpret_cast<uintptr_t>(table[o].kv_state),
                                        reinterpret_cast<uintptr_t>(table[o].score_state)};
            for (uintptr_t a : mine)
                for (uintptr_t b : other)
                    if (a < b + state_bytes && b < a + state_bytes)
                        return fail(DS_EINVAL, "compressor states of rows %d and %d overlap", o, e);
        }
        p.kv_state[e] = r.kv_state;
        p.score_state[e] = r.score_state;
        p.start_pos[e] = r.start_pos;
    }
    p.kv = kv;
    p.score = score;
    p.ape = ape;
    p.norm = norm;
    p.out = reinterpret_cast<__nv_bfloat16*>(out);
    p.rows = (uint32_t)rows;
    p.ratio = ratio;
    p.head_dim = head_dim;
    p.eps = epsilon;
    cudaError_t err = launch_compressor(p, (cudaStream_t)stream, true);
    return err == cudaSuccess ? DS_OK : cuda_fail(err, "compressor launch");
}

int ds_rows_selftest_bounded_wait(uint32_t* status, uint32_t* result, uint64_t budget_ns, void* stream) {
    if (!status || !result) return fail(DS_EINVAL, "status and result must be non-NULL");
    if (budget_ns < 1000ull || budget_ns > 10000000000ull)
        return fail(DS_EINVAL, "budget_ns must be 1e3..1e10, got %llu", (unsigned long long)budget_ns);
    const cudaError_t err = launch_wait_selftest(status, result, budget_ns, (cudaStream_t)stream);
    return err == cudaSuccess ? DS_OK : cuda_fail(err, "bounded-wait self-test launch");
}

int ds_rows_topk_static_status(uint32_t* status, void* stream) {
    if (!status) return fail(DS_EINVAL, "status is NULL");
    if (reinterpret_cast<uintptr_t>(status) & 3) return fail(DS_EALIGN, "status must be 4-byte aligned");
    uint8_t* ws = nullptr;
    const int rc = topk_scratch(&ws);
    if (rc) return rc;
    const cudaError_t err = cudaMemcpyAsync(status, ws, sizeof(uint32_t), cudaMemcpyDefault, (cudaStream_t)stream);
    return err == cudaSuccess ? DS_OK : cuda_fail(err, "status copy");
}

const char* ds_rows_last_error(void) { return g_error.c_str(); }

const char* ds_rows_version(void) { return "dsrows 0.1.0 (sm_103a)"; }

}  // extern "C"
