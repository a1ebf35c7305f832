/*
 * dsrows: one decode step of DeepSeek-style sparse attention over up to eight
 * independent rows (requests), each with its own caches and its own length,
 * on one NVIDIA GB300 (sm_103a).
 *
 * The operations follow the DeepSeek-V4 joint-decode kernels of the mlx-native
 * crate: `src/shaders/deepseek_rows.metal` (sections "Lightning indexer score
 * and deterministic top-512" and "Sparse attention (selected shared-KV rows
 * with learned sinks)") and their dispatch in `src/ops/deepseek_rows.rs`
 * (`dispatch_deepseek_indexer_rows`, `dispatch_deepseek_sparse_attention_rows`,
 * row structs `DeepSeekIndexerRow` / `DeepSeekSparseAttentionRow`).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers, owned by the caller, which also
 *   guarantees their sizes (stated per argument). The library allocates no
 *   memory and never synchronises the host; every entry point only enqueues
 *   work on `stream` (a cudaStream_t; NULL is the legacy default stream).
 * - bf16 tensors are passed as `ds_bf16` (uint16_t bit patterns).
 * - Arguments are validated on the host before anything is enqueued. On a
 *   bad argument the call enqueues nothing, returns a negative `DS_E*` code
 *   and sets a message readable with ds_rows_last_error() (per host thread).
 *   A CUDA launch failure returns DS_ECUDA.
 * - Bad DATA (NaN/Inf inputs, an out-of-range index) is not a call error: it
 *   zeroes the affected attention heads ("fail closed") and is reported in
 *   the optional `invalid` output.
 * - Row `r` of a joint call is bitwise equal to a call with only row `r`: all
 *   tiling, split counts and reduction orders depend on that row's kv_len and
 *   width alone.
 * - Calls that share a workspace or an output must not overlap in time
 *   (order them on one stream).
 * - A call's kernels are chained with programmatic dependent launch. Its first
 *   kernel may become resident while the stream's previous kernel still runs,
 *   but it waits for that kernel to complete before it reads or writes
 *   anything. Its last kernel lets the stream's next kernel launch early: a
 *   kernel the caller launches next with programmatic stream serialization
 *   must wait (griddepcontrol.wait, cudaGridDependencySynchronize) before it
 *   touches this call's outputs. Ordinary launches need nothing.
 */
#ifndef DSROWS_H
#define DSROWS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS_ROWS_MAX 8     /* rows per call (binding slots per cache family) */
#define DS_INDEX_HEADS 64 /* indexer query heads */
#define DS_INDEX_DIM 128  /* indexer key / query width */
#define DS_INDEX_VROWS_MAX 64 /* rows x queries of one multi-query indexer call */
#define DS_TOPK 512       /* most selected KV rows per row */
#define DS_HEADS 64       /* attention heads */
#define DS_DIM 512        /* shared-KV row width (K and V) */

/* Status codes. */
#define DS_OK 0
#define DS_EINVAL (-1) /* a bad argument (message says which) */
#define DS_ESIZE (-2)  /* workspace too small, or a size overflows 32 bits */
#define DS_EALIGN (-3) /* a pointer is not aligned as required */
#define DS_ECUDA (-4)  /* a CUDA call failed while enqueueing */

typedef uint16_t ds_bf16;

/*
 * One row of a call (`DeepSeekSparseAttentionRow` plus the indexer's fields).
 *   kv_len       keys / KV rows in the row's caches (> 0).
 *   width        selected slots of the row: 1 <= width <= min(512, kv_len).
 *                The top-k stage and the decode step select exactly
 *                min(512, kv_len) (DS_EINVAL otherwise) and write that many
 *                indices, -1 in slots past the row's finite scores; the
 *                attention stage takes any width in that range (the caller's
 *                index list).
 *   index_offset element offset of the row's `width` int32 indices in the
 *                indices buffer.
 *   q_row        row of the [*, 64, 128] / [*, 64, 512] queries, the [*, 64]
 *                head weights, per-row sinks, outputs and invalid flags.
 */
typedef struct {
    uint32_t kv_len;
    uint32_t width;
    uint32_t index_offset;
    uint32_t q_row;
} ds_row_t;

/*
 * The rows of a call: `rows` entries of `table` (host memory), and per entry
 * a device pointer to its caches (host arrays of `rows` pointers):
 *   index_keys[e]  bf16 [kv_len, 128] row-major indexer keys   (16-B aligned)
 *   kv[e]          bf16 [kv_len, 512] row-major shared K/V rows (16-B aligned)
 * A call reads only the cache family it needs; the other may be NULL.
 */
typedef struct {
    int rows;
    const ds_row_t* table;
    const ds_bf16* const* index_keys;
    const ds_bf16* const* kv;
} ds_row_set_t;

/*
 * Device status. The first 4 bytes of a workspace hold a uint32 status word.
 * Every call that takes a workspace zeroes it when it starts, and its kernels
 * OR these bits into it:
 *   DS_STATUS_WAIT_TIMEOUT  a bounded device-side wait (2 s of %globaltimer)
 *                           gave up; the kernel unwound without finishing and
 *                           the call's outputs are not valid.
 *   DS_STATUS_OVERFLOW      an internal consistency check of the selection
 *                           failed (candidate counts disagreed); its indices
 *                           may be incomplete. Not expected in any input.
 * Read the word once the call has completed (for example a 4-byte
 * cudaMemcpyAsync on the same stream); the next call on the workspace clears
 * it. 0: neither happened. ds_rows_topk_static keeps its word in the
 * library (ds_rows_topk_static_status reads it).
 */
#define DS_STATUS_WAIT_TIMEOUT 1u
#define DS_STATUS_OVERFLOW 2u

/*
 * Workspace bytes that every entry point below needs for this row table
 * (the largest need over the entry points). 0 when the table is invalid
 * (see ds_rows_last_error). The workspace must be 256-byte aligned; its
 * contents need no initialisation and are scratch between calls.
 */
size_t ds_rows_workspace_bytes(int rows, const ds_row_t* table);

/*
 * (1) Lightning-indexer score (`deepseek_indexer_score_mma_rows_bf16`):
 *   scores[e * score_stride + j] =
 *       sum_{h<64} w_index[q_row, h] * max(0, sum_{d<128} q_index[q_row, h, d] * K_e[j, d])
 * for j < kv_len of entry e; a non-finite score is stored as -inf. Every key
 * is valid (no causal cut).
 *   q_index     bf16 [Q, 64, 128]                              (16-B aligned)
 *   w_index     fp32 [Q, 64]
 *   scores      fp32, entry e at e * score_stride; score_stride >= max kv_len.
 *               Elements j >= kv_len of a row are not written.
 */
int ds_rows_indexer_score(const ds_row_set_t* set, const ds_bf16* q_index, const float* w_index,
                          float* scores, size_t score_stride, void* stream);

/*
 * (2) Deterministic top-k (`deepseek_indexer_topk_block/merge/finalize_rows_i32`):
 * for each entry e, the first `width` indices j < kv_len ordered best first by
 * (score descending, then lower index), over the finite scores only; slots past
 * the number of finite scores hold -1. -0.0 and +0.0 tie.
 *   scores      fp32, entry e at e * score_stride (as ds_rows_indexer_score).
 *   indices     int32, entry e writes [index_offset, index_offset + width);
 *               these ranges must not overlap.
 *   workspace   at least ds_rows_workspace_bytes(...) bytes.
 */
int ds_rows_topk(const ds_row_set_t* set, const float* scores, size_t score_stride,
                 int32_t* indices, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Top-k without a workspace. There is no counterpart on the prior-art pages:
 * this entry point exists for callers that cannot allocate device memory when
 * they run the top-k stage, for example code running under a CUDA graph or a
 * real-time loop that forbids allocation, or an embedding whose device
 * allocator is not reachable from the calling code. It computes exactly what
 * ds_rows_topk computes (same arguments, bitwise the same indices) but keeps
 * its scratch in one fixed array inside the library instead of a
 * caller-provided workspace, and allocates nothing.
 *   - Size: the array holds DS_TOPK_STATIC_SCRATCH_BYTES bytes (about 64 KiB),
 *     enough for DS_ROWS_MAX rows of any kv_len; every GPU that loads the
 *     library keeps it until the process exits. A table needing more is
 *     rejected with DS_ESIZE (more than DS_ROWS_MAX rows is DS_EINVAL).
 *   - Set-up: the first call on each device looks up the array's device
 *     address (with that device current). Make that first call before any
 *     stream capture.
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     previous call's contents; each call clears what must start at zero.
 *     Calls that overlap on the GPU (different streams, no ordering between
 *     them) race on the array and give wrong results: order them.
 */
#define DS_TOPK_STATIC_SCRATCH_BYTES 65792
int ds_rows_topk_static(const ds_row_set_t* set, const float* scores, size_t score_stride,
                        int32_t* indices, void* stream);

/*
 * The status word of ds_rows_topk_static on the current device (DS_STATUS_*
 * bits, as in a workspace's first word; each ds_rows_topk_static call clears
 * it when it starts). Enqueues a 4-byte copy of the word on `stream` into
 * `status` (device or page-locked host memory, 4-byte aligned); read it once
 * the stream has passed this point. Allocates nothing; like the top-k call it
 * shares the library's array, so a call on another stream that overlaps it
 * races. DS_EINVAL for a NULL `status`, DS_ECUDA when the copy cannot be
 * enqueued.
 */
int ds_rows_topk_static_status(uint32_t* status, void* stream);

/*
 * (3)+(4) Gather and sink-softmax sparse attention
 * (`deepseek_sparse_attention_score_rows_bf16` + `..._reduce_rows_bf16`):
 * for each entry e and head h, over the slots t < width with index
 * i_t = indices[index_offset + t]:
 *   i_t == -1 is skipped; i_t < -1 or i_t >= kv_len zeroes every head of e;
 *   l_t = scale * q_attn[q_row, h, :] . KV_e[i_t, :]
 *   m = max(sink_h, max_t l_t), den = exp(sink_h - m) + sum_t exp(l_t - m)
 *   out[q_row, h, :] = bf16( sum_t exp(l_t - m) * KV_e[i_t, :] / den )
 * The sink has no value row. A non-finite sink, q element or selected KV
 * element, an overflowed logit or den <= 0 zeroes the head (fail closed).
 * The sums run over the row's valid indices in ascending order (duplicates
 * kept), so the result does not depend on the order of the indices within
 * [index_offset, index_offset + width): it is a function of their multiset.
 *   q_attn      bf16 [Q, 64, 512]                              (16-B aligned)
 *   sinks       fp32; head h of entry e at sinks[q_row * sinks_row_stride + h];
 *               sinks_row_stride 0 shares one [64] vector, else >= 64.
 *   indices     int32 (as written by ds_rows_topk).
 *   scale       finite and > 0 (1/sqrt(512) for the DeepSeek shapes).
 *   out         bf16 [Q, 64, 512]; q_row must be unique across the entries.
 *   invalid     optional uint32 [Q, 64]: 1 where the head was zeroed, else 0.
 *   workspace   at least ds_rows_workspace_bytes(...) bytes.
 */
int ds_rows_sparse_attn(const ds_row_set_t* set, const ds_bf16* q_attn, const float* sinks,
                        size_t sinks_row_stride, const int32_t* indices, float scale,
                        ds_bf16* out, uint32_t* invalid, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * The whole decode step: (1) indexer score -> (2) top-`width` -> (3)+(4)
 * gather and sink attention, on one stream. Scores and the selection stay in
 * the workspace. Arguments as in the stages above; `indices` is optional
 * (NULL: the selection is not written out) and, when given, receives the
 * selected indices best first at each entry's index_offset (ranges must not
 * overlap). The attention sums over the selected rows in ascending index
 * order, as ds_rows_sparse_attn does, so `out` is bitwise what
 * ds_rows_sparse_attn gives on those indices.
 */
int ds_rows_decode(const ds_row_set_t* set, const ds_bf16* q_index, const float* w_index,
                   const ds_bf16* q_attn, const float* sinks, size_t sinks_row_stride,
                   float scale, ds_bf16* out, int32_t* indices, uint32_t* invalid,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes for ds_rows_decode_host: the decode workspace plus device
 * staging for the step's inputs and outputs; 0 when the table is invalid. */
size_t ds_rows_decode_host_workspace_bytes(int rows, const ds_row_t* table, size_t sinks_row_stride);

/*
 * ds_rows_decode with the step's inputs and outputs in HOST memory. The
 * caches stay on the device (`set`). Everything is ordered on `stream`, and
 * the call returns before the step completes: synchronise `stream` before
 * reading h_out. Results are bitwise those of ds_rows_decode.
 *   - h_q_index and h_w_index are copied into device staging inside the
 *     workspace (the indexer's query is a tensor-core operand); when pinned,
 *     by the workspace-clear kernel itself.
 *   - A pinned h_q_attn is copied into staging by the indexer while it waits
 *     for its first scores; the attention reads h_sinks, and writes h_out,
 *     h_indices and h_invalid, in place when they are pinned (page-locked)
 *     host memory. Any other host memory goes through staging, with
 *     cudaMemcpyAsync before and after the kernels.
 * The call may be captured in a CUDA graph.
 *   h_q_index   bf16 [Q, 64, 128] (16-B aligned); h_w_index fp32 [Q, 64]
 *   h_q_attn    bf16 [Q, 64, 512] (16-B aligned); h_sinks as for ds_rows_decode
 *   h_out       bf16 [Q, 64, 512] (16-B aligned): the entries' q_rows are
 *               written, no others.
 *   h_indices   optional int32 (as ds_rows_decode's indices).
 *   h_invalid   optional uint32 [Q, 64]: the entries' q_rows are written.
 *   Q = max q_row + 1. When the entries use every q_row 0..Q-1, a staged array
 *   travels as one copy, else one copy per entry.
 *   workspace   at least ds_rows_decode_host_workspace_bytes(...) bytes.
 * Errors as ds_rows_decode, plus DS_EINVAL for a NULL host array.
 */
int ds_rows_decode_host(const ds_row_set_t* set, const ds_bf16* h_q_index, const float* h_w_index,
                        const ds_bf16* h_q_attn, const float* h_sinks, size_t sinks_row_stride, float scale,
                        ds_bf16* h_out, int32_t* h_indices, uint32_t* h_invalid, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * One row of a positioned indexer call (`DeepSeekIndexerRow`; compression
 * ratio 4, one query per row):
 *   kv_len        compressed keys in the row's indexer cache (> 0).
 *   start_pos     the query's absolute position. The row's valid keys are
 *                 j < valid_count = (start_pos + 1) / 4; kv_len must be at
 *                 least valid_count (start_pos < 2^32 - 1).
 *   offset        added to every emitted index: >= 0, and
 *                 offset + valid_count - 1 must fit int32 (-1 is the sentinel).
 *   q_row         row of the [*, 64, 128] queries and [*, 64] head weights.
 *   output_offset element offset of the row's 512 output indices; the ranges
 *                 [output_offset, output_offset + 512) must not overlap.
 */
typedef struct {
    uint32_t kv_len;
    uint32_t start_pos;
    int32_t offset;
    uint32_t q_row;
    uint32_t output_offset;
} ds_indexer_row_t;

/* Workspace bytes for ds_rows_indexer_topk with this table; 0 when the table
 * is invalid (see ds_rows_last_error). 256-byte aligned, scratch between calls. */
size_t ds_rows_indexer_topk_workspace_bytes(int rows, const ds_indexer_row_t* table);

/*
 * (1)+(2) Positioned indexer and causal top-512 (`dispatch_deepseek_indexer_rows`:
 * `deepseek_indexer_score_mma_rows_bf16` with its valid_count, then
 * `deepseek_indexer_topk_block/merge/finalize_rows_i32`). For each entry e, with
 * valid_count = min(kv_len, (start_pos + 1) / 4):
 *   s[j] = sum_{h<64} w_index[q_row, h] * max(0, q_index[q_row, h, :] . K_e[j, :])
 * for j < valid_count (keys at or past valid_count take no part), and
 *   indices[output_offset + t], t < 512 = the t-th best j (score descending,
 *   then lower index, finite scores only) plus offset, for t < valid_count when
 *   such a j exists; every other slot is -1.
 *   index_keys  host array of `rows` device pointers: bf16 [kv_len, 128] (16-B aligned).
 *   q_index     bf16 [Q, 64, 128] (16-B aligned); w_index fp32 [Q, 64].
 *   indices     int32, 512 per entry at output_offset.
 *   workspace   at least ds_rows_indexer_topk_workspace_bytes(...) bytes.
 */
int ds_rows_indexer_topk(int rows, const ds_indexer_row_t* table, const ds_bf16* const* index_keys,
                         const ds_bf16* q_index, const float* w_index, int32_t* indices,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes for ds_rows_indexer_topk_queries; 0 when the arguments are
 * invalid. ds_rows_indexer_topk_workspace_bytes(r, t) equals this with
 * query_len 1. */
size_t ds_rows_indexer_topk_queries_workspace_bytes(int rows, const ds_indexer_row_t* table, uint32_t query_len);

/*
 * (1)+(2) with query_len consecutive queries per entry (the query loop of
 * `deepseek_indexer_score_mma_rows_bf16`, whose query j sits at position
 * start_pos + j; its valid_count = min(kv_len, (start_pos + j + 1) / 4)). For
 * each entry e and query j < query_len, exactly ds_rows_indexer_topk of the
 * entry with start_pos + j, q_row + j and output_offset + 512 j. (The pages'
 * top-k kernels take the first query only; each query's own list is the
 * reading taken here.)
 *   query_len   1 .. 64 with rows * query_len <= DS_INDEX_VROWS_MAX.
 *   table       as for ds_rows_indexer_topk, except: kv_len must be at least
 *               the last query's count (start_pos + query_len) / 4,
 *               start_pos + query_len must fit u32, offset + that count - 1
 *               must fit int32, q_row .. q_row + query_len - 1 are the
 *               entry's query rows, and the output ranges are
 *               [output_offset, output_offset + 512 query_len).
 *   indices     int32, 512 per (entry, query) at output_offset + 512 j.
 *   workspace   at least ds_rows_indexer_topk_queries_workspace_bytes(...) bytes.
 * Up to four queries of an entry share each key tile on the tensor cores, so
 * the keys are read once for them. Errors as ds_rows_indexer_topk.
 */
int ds_rows_indexer_topk_queries(int rows, const ds_indexer_row_t* table, uint32_t query_len,
                                 const ds_bf16* const* index_keys, const ds_bf16* q_index, const float* w_index,
                                 int32_t* indices, void* workspace, size_t workspace_bytes, void* stream);

/*
 * One row of a KV compressor call (`DeepSeekCompressorRow`): the row's
 * recurrent window (device fp32, updated in place) and its token's position.
 *   kv_state     fp32 [coff * ratio, coff * head_dim]     (16-B aligned)
 *   score_state  fp32, same shape                          (16-B aligned)
 *   start_pos    the decode token's absolute position, 1 .. 2^32 - 2.
 * coff is 2 for ratio 4 (overlapping windows) and 1 for ratio 128. The state
 * buffers of a call must not overlap.
 */
typedef struct {
    float* kv_state;
    float* score_state;
    uint32_t start_pos;
} ds_compressor_row_t;

/*
 * (5) Learned KV compressor, one decode token per row
 * (`deepseek_compressor_rows_bf16`, `dispatch_deepseek_compressor_rows`), for
 * (ratio, head_dim) in {(4, 128), (4, 512), (128, 512)}. With P = coff * head_dim:
 *   1. the token (t = start_pos mod ratio) is written to state row
 *      (ratio if coff == 2 else 0) + t: kv (0 where not finite) and
 *      score + ape[t] (NaN where either is not finite);
 *   2. when start_pos + 1 is a multiple of ratio, each feature f softmax-pools
 *      the window's values with its scores (coff * ratio rows; with coff == 2
 *      the first ratio rows read feature f, the others head_dim + f), rounds
 *      to bf16 (c) and writes out = bf16(c * norm / sqrt(mean(c^2) + epsilon)),
 *      or zeros when a score is NaN or +inf, or a value, pooled value, norm,
 *      sum or result is not finite; with coff == 2 the window then shifts the
 *      current block into the previous rows. Otherwise out is zero.
 *   kv, score  fp32 [rows, P]; ape fp32 [ratio, P]; norm fp32 [head_dim]
 *              (all 16-B aligned); epsilon finite and > 0.
 *   out        bf16 [rows, head_dim]                       (16-B aligned)
 */
int ds_rows_compress_kv(int rows, const ds_compressor_row_t* table, const float* kv, const float* score,
                        const float* ape, const float* norm, uint32_t ratio, uint32_t head_dim,
                        float epsilon, ds_bf16* out, void* stream);

/*
 * Self-test of the device-side failure detection, on the current device. One
 * CTA runs the library's bounded mbarrier wait twice on a shared-memory
 * barrier: on a phase that completes, and on a phase that nothing completes,
 * each with a budget of `budget_ns` nanoseconds of %globaltimer (1,000 to
 * 10,000,000,000). It writes result[0] = 1 if the first wait succeeded and
 * result[1] = 1 if the second gave up, and ORs DS_STATUS_WAIT_TIMEOUT into
 * *status when it gives up, as the library's kernels do. Nothing faults and
 * the device stays usable. Takes about budget_ns on the GPU.
 *   status   device uint32 (zeroed by the caller beforehand)
 *   result   device uint32 [2]
 */
int ds_rows_selftest_bounded_wait(uint32_t* status, uint32_t* result, uint64_t budget_ns, void* stream);

/* Message of the last failed call on this host thread ("" if none). */
const char* ds_rows_last_error(void);

/* Library version string. */
const char* ds_rows_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSROWS_H */
