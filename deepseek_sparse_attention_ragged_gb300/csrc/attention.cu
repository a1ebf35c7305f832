// Gather + sink-softmax sparse attention (mlx-native deepseek_rows.metal, kernels
// deepseek_sparse_attention_score_rows_bf16 and deepseek_sparse_attention_reduce_rows_bf16;
// gather semantics of deepseek_sparse_attention_gather_rows_bf16).
//
// Per row e and head h over the selected slots t (index i_t):
//   l_t = scale * q_h . KV[i_t],  m = max(sink_h, max l_t),
//   den = exp(sink_h - m) + sum exp(l_t - m),  out_h = sum exp(l_t - m) KV[i_t] / den.
//
// GB300 design. A row's `width` slots are split into chunks of 64; one CTA per
// (row, half of the 64 heads, chunk) gathers its 64 KV rows (1 KiB each,
// 16-byte cp.async, read once for the CTA's 32 heads), computes the 32x64
// logits S = Q G^T and the 32x512 partial P G on tensor cores (mma.sync
// m16n8k16 bf16, fp32 accumulate), with a chunk-local softmax (m_c, l_c)
// whose warp reductions run for four heads side by side. P enters the second
// product as a bf16 hi + lo pair, which keeps ~16 bits of each weight. A
// second kernel combines the chunks of a (row, half) in chunk order with the sink:
//   m = max(sink, m_c), den = exp(sink - m) + sum_c l_c exp(m_c - m),
//   out = sum_c acc_c exp(m_c - m) / den,
// so every reduction order depends on the row's width alone.
//
// Fail-closed rules: an index < -1 or >= kv_len flags the whole row; a
// non-finite logit (non-finite q or KV element, or overflow) flags its head;
// a non-finite sink or denominator flags the head; a flagged head is written
// as zeros, and any non-finite output element is written as zero.

#include "attend.cuh"
#include "common.cuh"
#include "kernels.h"

namespace dsrows {

using namespace attend;

namespace {

constexpr int kThreads = 256;
constexpr int kHalf = kHeads / 2;         // 32 heads per CTA

struct SmemLayout {
    static constexpr size_t q = 0;
    static constexpr size_t g = q + (size_t)kHalf * kQStride * 2;
    static constexpr size_t p_hi = g + (size_t)kSlots * kQStride * 2;
    static constexpr size_t p_lo = p_hi + (size_t)kHalf * kPStride * 2;
    static constexpr size_t lg = p_lo + (size_t)kHalf * kPStride * 2;
    static constexpr size_t idx = lg + (size_t)kHalf * kLgStride * 4;
    static constexpr size_t total = idx + kSlots * 4;
};
constexpr size_t kSmemBytes = SmemLayout::total;

// CTA b -> (entry, head half, chunk): entry e owns CTAs [2 chunk_begin[e], 2 chunk_begin[e+1]).
__device__ __forceinline__ int entry_of_cta(const AttnParams& p, uint32_t b) {
    int e = 0;
#pragma unroll
    for (int i = 1; i < kRowsMax; ++i)
        if (i < (int)p.rows && b >= 2 * p.chunk_begin[i]) e = i;
    return e;
}

}  // namespace

// One CTA per (row, head half, 64-slot chunk): blockIdx = 2 * chunk_begin[e] + 2 * c + half... laid out as
// [entry][half][chunk] so a row's two halves are adjacent ranges.
__global__ void __launch_bounds__(kThreads, 1) attn_partial_kernel(const AttnParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __nv_bfloat16* q_s = reinterpret_cast<__nv_bfloat16*>(smem + SmemLayout::q);
    __nv_bfloat16* g_s = reinterpret_cast<__nv_bfloat16*>(smem + SmemLayout::g);
    __nv_bfloat16* ph_s = reinterpret_cast<__nv_bfloat16*>(smem + SmemLayout::p_hi);
    __nv_bfloat16* pl_s = reinterpret_cast<__nv_bfloat16*>(smem + SmemLayout::p_lo);
    float* lg_s = reinterpret_cast<float*>(smem + SmemLayout::lg);
    int* idx_s = reinterpret_cast<int*>(smem + SmemLayout::idx);

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int e = entry_of_cta(p, blockIdx.x);
    const uint32_t W = p.width[e];
    const uint32_t nchunks = (W + kSlots - 1) / kSlots;
    const uint32_t local = blockIdx.x - 2 * p.chunk_begin[e];
    const int half = (int)(local / nchunks);
    const uint32_t c = local % nchunks;
    const int head0 = half * kHalf;
    const int L = (int)p.kv_len[e];
    const __nv_bfloat16* kv = p.kv[e];

    pdl_trigger();
    // The query is an input of the call: fetch it while the previous kernel finishes.
    load_q<kHalf, kThreads>(q_s, p.q + ((size_t)p.q_row[e] * kHeads + head0) * kDim, t);
    cp_async_commit();
    pdl_wait();  // the indices come from the previous kernel

    // Selected indices of this chunk: -1 for sentinels, bad indices and slots past the width.
    if (t < kSlots) {
        const uint32_t slot = c * kSlots + t;
        int i = -1;
        if (slot < W) {
            const int v = __ldcg(p.indices + p.index_offset[e] + slot);
            if (v < -1 || v >= L) atomicOr(&p.flags[kRowsMax * kHeads + e], 1u);
            else i = v;
        }
        idx_s[t] = i;
    }
    __syncthreads();

    // Gather the chunk's selected KV rows (1 KiB each, once for the CTA's 32 heads).
    gather_kv<kThreads>(g_s, idx_s, kv, t);
    cp_async_wait_all();
    __syncthreads();

    logits<kHalf>(q_s, g_s, lg_s, p.scale, warp, lane);
    __syncthreads();

    float* part = p.part + (size_t)blockIdx.x * kPartFloats;
    softmax<4>(lg_s, idx_s, ph_s, pl_s, warp, lane, [&](int h, float m, float l, bool bad) {
        if (bad) atomicOr(&p.flags[e * kHeads + head0 + h], 1u);
        part[h] = m;
        part[kHalf + h] = l;
    });
    __syncthreads();

    float acc[16][4];
    pv<128>(ph_s, pl_s, g_s, warp, lane, acc);
    float* pacc = part + 2 * kHalf;
    const int h0 = 16 * (warp >> 2) + (lane >> 2);
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
        const int f = (warp & 3) * 128 + nt * 8 + 2 * (lane & 3);
        *reinterpret_cast<float2*>(pacc + (size_t)h0 * kDim + f) = make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2*>(pacc + (size_t)(h0 + 8) * kDim + f) = make_float2(acc[nt][2], acc[nt][3]);
    }
}

// Combine the chunks of a (row, head half): CTA = (row, half, 64 features), thread = (head, 8 features).
constexpr int kCombineFeatures = 64;
constexpr int kCombineBlocks = kDim / kCombineFeatures;  // 8 per (row, half)

__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnParams p) {
    __shared__ CombineSmem<kHalf> cs;
    const int e = blockIdx.x / (2 * kCombineBlocks);
    const int half = (blockIdx.x / kCombineBlocks) & 1;
    const int fb = blockIdx.x % kCombineBlocks;
    const int head0 = half * kHalf;
    const uint32_t W = p.width[e];
    const int nchunks = (int)((W + kSlots - 1) / kSlots);
    const float* part0 = p.part + ((size_t)2 * p.chunk_begin[e] + (size_t)half * nchunks) * kPartFloats;
    const uint32_t q_row = p.q_row[e];
    pdl_trigger();
    pdl_wait();  // partials and flags come from the partial kernel
    const bool row_bad = __ldcg(p.flags + kRowsMax * kHeads + e) != 0;
    combine_slice<kHalf, 256>(part0, kPartFloats, nchunks, fb * kCombineFeatures, p.sinks + (size_t)q_row * p.sinks_row_stride + head0,
                      row_bad, p.flags + e * kHeads + head0, p.out + ((size_t)q_row * kHeads + head0) * kDim,
                      p.invalid && fb == 0 ? p.invalid + (size_t)q_row * kHeads + head0 : nullptr, cs);
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream, bool pdl) {
    static bool configured = false;
    if (!configured) {
        cudaError_t err = cudaFuncSetAttribute(attn_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kSmemBytes);
        if (err != cudaSuccess) return err;
        configured = true;
    }
    if (p.total_chunks == 0) return cudaSuccess;
    cudaError_t err = launch_kernel(attn_partial_kernel, dim3(2 * p.total_chunks), dim3(kThreads),
                                    kSmemBytes, stream, pdl, p);
    if (err != cudaSuccess) return err;
    return launch_kernel(attn_combine_kernel, dim3(p.rows * 2 * kCombineBlocks), dim3(256), 0, stream, true, p);
}

}  // namespace dsrows
