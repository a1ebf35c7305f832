// Launch tables and launchers of the dsrows kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dsrows.h"

namespace dsrows {

// Indexer score: one TMA tensor map per row's key cache, one for the queries.
struct IndexerParams {
    CUtensorMap kmap[DS_ROWS_MAX];  // bf16 [kv_len, 128], box {64, 128}, 128-B swizzle
    CUtensorMap qmap;               // bf16 [Q*64, 128], box {64, 64}, 128-B swizzle
    const float* w;                 // [Q, 64]
    float* scores;                  // entry e at e * score_stride
    uint32_t* hist;                 // optional [8][2048] score-key histogram
    uint32_t* status;               // device status word
    uint32_t inputs_ready;          // 1: every input was complete when the launch began (it follows an
                                    // ordinary launch), so loads may start before griddepcontrol.wait
    uint64_t score_stride;
    uint32_t rows;
    uint32_t total_tiles;
    uint32_t kv_len[DS_ROWS_MAX];
    uint32_t q_row[DS_ROWS_MAX];
    uint32_t tile_begin[DS_ROWS_MAX];
};

// Top-k: level-0 histogram, then one 8-CTA cluster per row for the selection.
struct TopkParams {
    const float* scores;
    uint64_t score_stride;
    int32_t* out;          // indices; entry e at out_offset[e]
    uint32_t* hist;        // [8][2048] level 0 (top 11 key bits), zero before it is built
    uint32_t* status;
    uint32_t rows;
    uint32_t order_by_index;  // 0: best first; 1: ascending index (the decode's canonical order)
    uint32_t total_chunks;    // histogram CTAs (chunks of topk_chunk() scores)
    uint32_t kv_len[DS_ROWS_MAX];
    uint32_t width[DS_ROWS_MAX];
    uint32_t out_offset[DS_ROWS_MAX];
    uint32_t chunk_begin[DS_ROWS_MAX];
    int32_t offset[DS_ROWS_MAX];   // added to every emitted index (positioned indexer)
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
    const float* sinks;
    uint64_t sinks_row_stride;
    float* part;                  // partials: m[32], l[32], acc[32][512] per (chunk, head half)
    uint32_t* flags;              // [8][64] head flags, zero on entry
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

size_t indexer_smem_bytes();
uint32_t indexer_tile_keys();
cudaError_t launch_indexer(const IndexerParams& p, int num_sms, cudaStream_t stream, bool pdl);

uint32_t topk_chunk();  // scores per histogram / collection CTA
cudaError_t launch_topk_hist(const TopkParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_topk_select(const TopkParams& p, cudaStream_t stream, bool pdl);

// Zero `words` 32-bit words (the workspace control region); an ordinary launch.
cudaError_t launch_clear(uint32_t* p, uint32_t words, cudaStream_t stream);

size_t decode_tail_smem_bytes();
cudaError_t launch_decode_tail(const TailParams& p, cudaStream_t stream, bool pdl);

}  // namespace dsrows
