// Launch tables and launchers of the dsrows kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dsrows.h"

namespace dsrows {

// Indexer score. A virtual row is one (entry, query) pair with its own query
// row and number of scored keys; a segment is one entry with a run of up to
// kIndexerGroup consecutive virtual rows that share each key tile.
constexpr int kSegMax = 32;
constexpr int kVRowsMax = DS_INDEX_VROWS_MAX;
constexpr int kIndexerGroup = 4;  // queries per key tile in the multi-query kernel

// Arrays sized for the kernel that takes them: SEGS segments, VROWS virtual
// rows (the one-query kernel takes the smaller table: a shorter launch).
template <int SEGS, int VROWS>
struct IndexerParamsT {
    CUtensorMap kmap[DS_ROWS_MAX];  // bf16 [kv_len, 128], box {64, 128}, 128-B swizzle
    CUtensorMap qmap;               // bf16 [Q*64, 128], box {64, 64}, 128-B swizzle
    const float* w;                 // [Q, 64]
    float* scores;                  // virtual row v at v * score_stride
    uint32_t* hist;                 // optional [vrows][2048] score-key histogram
    uint32_t* status;               // device status word
    uint32_t inputs_ready;          // 1: every input was complete when the launch began (it follows an
                                    // ordinary launch), so loads may start before griddepcontrol.wait;
                                    // 2: the keys were, the query and head weights come from the
                                    // previous kernel; 0: nothing is read before the wait
    uint64_t score_stride;
    uint32_t rows;                  // entries (key caches)
    uint32_t segs;
    uint32_t vrows;
    uint32_t total_tiles;
    uint32_t tile_begin[SEGS];      // first 128-key tile of each segment
    uint32_t cta_begin[SEGS + 1];   // one query per entry: the first CTA of each segment
    uint8_t seg_entry[SEGS];
    uint8_t seg_vrow[SEGS];         // the segment's first virtual row
    uint8_t seg_queries[SEGS];      // its virtual rows: 1..group
    uint32_t valid[VROWS];          // keys j < valid[v] are scored
    uint32_t q_row[VROWS];          // query and head-weight row of each virtual row
    // Optional copy for the next kernel, done by the epilogue warps while they
    // wait for the first scores: side_n16 16-byte words from side_src (pinned
    // host memory) to side_dst.
    const uint4* side_src;
    uint4* side_dst;
    uint32_t side_n16;
};
using IndexerParams1 = IndexerParamsT<DS_ROWS_MAX, DS_ROWS_MAX>;  // one query per entry
using IndexerParamsG = IndexerParamsT<kSegMax, kVRowsMax>;        // up to kIndexerGroup per segment

// Top-k: level-0 histogram, then one 8-CTA cluster per row for the selection.
struct TopkParams {
    const float* scores;
    uint64_t score_stride;
    int32_t* out;          // indices; entry e at out_offset[e]
    uint32_t* hist;        // [8][2048] level 0 (top 11 key bits), zero before it is built
    uint32_t* status;
    uint32_t rows;
    uint32_t total_chunks;    // histogram CTAs (chunks of topk_chunk() scores)
    uint32_t kv_len[kVRowsMax];
    uint32_t width[kVRowsMax];
    uint32_t out_offset[kVRowsMax];
    uint32_t chunk_begin[kVRowsMax];
    int32_t offset[kVRowsMax];   // added to every emitted index (positioned indexer)
};

// Selection (decode) and attention, one 8-CTA cluster per row; with `given`,
// the attention of the caller's indices.
constexpr uint32_t kTailChunkSlots = 128;  // slots per attention chunk

struct TailParams {
    const float* scores;          // indexer scores, entry e at e * score_stride
    uint64_t score_stride;
    const uint32_t* hist;         // [8][2048] level-0 histogram built by the indexer
    uint32_t* status;
    const __nv_bfloat16* kv[DS_ROWS_MAX];
    const __nv_bfloat16* q;       // [Q, 64, 512]
    uint32_t q_after_wait;        // 1: q is written by the previous kernel (fetch it after the wait)
    uint32_t attend;              // 0: selection only (decode mode): write the indices and stop
    const float* sinks;
    uint64_t sinks_row_stride;
    float* part;                  // partials: m[32], l[32], acc[32][512] per (chunk, head half)
    uint32_t* flags;              // [8][64] head flags, [8] row flags, [8] publish flags; zero on entry
    uint64_t* pub;                // [8][512] published winners (index order), then [8] u32 their number
    uint32_t ranker;              // 1: one more cluster ranks the published winners (best-first list)
    __nv_bfloat16* out;           // [Q, 64, 512]
    uint32_t* invalid;            // optional [Q, 64]
    const int32_t* given;         // the caller's indices (attention only), entry e at index_offset[e]
    int32_t* indices;             // optional best-first selection (decode), entry e at index_offset[e]
    float scale;
    uint32_t rows;
    uint32_t kv_len[DS_ROWS_MAX];
    uint32_t width[DS_ROWS_MAX];
    uint32_t index_offset[DS_ROWS_MAX];
    uint32_t q_row[DS_ROWS_MAX];
    uint32_t chunk_begin[DS_ROWS_MAX];  // first 128-slot chunk of each row
    int32_t offset[DS_ROWS_MAX];        // added to the selected indices written out
};

// Learned KV compressor, one decode token per row: one 8-CTA cluster per row.
struct CompressorParams {
    float* kv_state[DS_ROWS_MAX];     // fp32 [coff * ratio, coff * head_dim], updated in place
    float* score_state[DS_ROWS_MAX];
    const float* kv;                  // fp32 [rows, coff * head_dim]
    const float* score;               // fp32 [rows, coff * head_dim]
    const float* ape;                 // fp32 [ratio, coff * head_dim]
    const float* norm;                // fp32 [head_dim]
    __nv_bfloat16* out;               // bf16 [rows, head_dim]
    uint32_t start_pos[DS_ROWS_MAX];
    uint32_t rows;
    uint32_t ratio;
    uint32_t head_dim;
    float eps;
};

cudaError_t launch_compressor(const CompressorParams& p, cudaStream_t stream, bool pdl);

uint32_t indexer_tile_keys();
// One query per key tile (decode), or up to kIndexerGroup.
cudaError_t launch_indexer(const IndexerParams1& p, int num_sms, cudaStream_t stream, bool pdl);
cudaError_t launch_indexer(const IndexerParamsG& p, int num_sms, cudaStream_t stream, bool pdl);

uint32_t topk_chunk();  // scores per histogram / collection CTA
cudaError_t launch_topk_hist(const TopkParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_topk_select(const TopkParams& p, cudaStream_t stream, bool pdl);

// Zero `words` 32-bit words (the workspace control region); an ordinary launch.
cudaError_t launch_clear(uint32_t* p, uint32_t words, cudaStream_t stream);

// The bounded-wait self-test (one CTA): result[0] = a completed wait succeeded,
// result[1] = a wait on a phase nothing completes gave up after budget_ns.
cudaError_t launch_wait_selftest(uint32_t* status, uint32_t* result, uint64_t budget_ns, cudaStream_t stream);
// The same, and copies a_bytes and b_bytes (multiples of 16; 16-byte aligned)
// from a_src and b_src to a_dst and b_dst before it completes.
cudaError_t launch_clear_copy(uint32_t* p, uint32_t words, const void* a_src, void* a_dst, size_t a_bytes,
                              const void* b_src, void* b_dst, size_t b_bytes, cudaStream_t stream);

size_t decode_tail_smem_bytes();
cudaError_t launch_decode_tail(const TailParams& p, cudaStream_t stream, bool pdl);

}  // namespace dsrows
