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

#include "common.cuh"
#include "kernels.h"

namespace dsrows {

namespace {

constexpr int kThreads = 256;
constexpr int kSlots = kAttnSlots;        // 64 selected slots per CTA
constexpr int kHalf = kHeads / 2;         // 32 heads per CTA
constexpr int kQStride = kDim + 8;        // bf16 per smem row: 1040 B, conflict-free ldmatrix
constexpr int kPStride = kSlots + 8;      // 144 B rows, conflict-free ldmatrix
constexpr int kLgStride = kSlots + 1;

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

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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
    if (blockIdx.x >= 2 * p.total_chunks) {
        // Best-first indices for the caller, off the critical path: this CTA
        // orders row e's selection (ascending index) by (score desc, index asc).
        const int e = (int)(blockIdx.x - 2 * p.total_chunks);
        const uint32_t W = p.width[e];
        pdl_trigger();
        pdl_wait();  // the selection and the scores come from the previous kernels
        const float* sc = p.scores + (size_t)e * p.score_stride;
        uint64_t x[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint32_t slot = t + q * kThreads;
            const int j = slot < W ? __ldcg(p.indices + p.index_offset[e] + slot) : -1;
            x[q] = j >= 0 ? composite(score_key(__ldcg(sc + j)), (uint32_t)j) : 0ull;
        }
        sort512_desc<kThreads>(x, reinterpret_cast<uint64_t*>(smem));
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint32_t slot = t + q * kThreads;
            if (slot < W) p.sorted_out[p.sorted_offset[e] + slot] = x[q] ? (int32_t)(~(uint32_t)x[q]) : -1;
        }
        return;
    }
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
    const __nv_bfloat16* q = p.q + ((size_t)p.q_row[e] * kHeads + head0) * kDim;
    for (int k = t; k < kHalf * (kDim / 8); k += kThreads) {
        const int row = k >> 6, col = (k & 63) * 8;
        cp_async16(q_s + row * kQStride + col, q + (size_t)row * kDim + col);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
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
    for (int k = t; k < kSlots * (kDim / 8); k += kThreads) {
        const int row = k >> 6, col = (k & 63) * 8;
        const int i = idx_s[row];
        __nv_bfloat16* dst = g_s + row * kQStride + col;
        if (i >= 0) cp_async16(dst, kv + (size_t)i * kDim + col);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- S = Q G^T : warp -> 16 heads x 16 slots ----------------------------
    const int mt = warp >> 2;  // head tile (16 heads)
    {
        const int nq = warp & 3;  // slot quarter (16 slots)
        float acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
        const uint32_t a_addr = smem_u32(q_s + (16 * mt + (lane & 15)) * kQStride + (lane >> 4) * 8);
        const uint32_t b_addr =
            smem_u32(g_s + (16 * nq + (lane >> 4) * 8 + (lane & 7)) * kQStride + ((lane >> 3) & 1) * 8);
#pragma unroll 8
        for (int k0 = 0; k0 < kDim; k0 += 16) {
            uint32_t a[4], b[4];
            ldsm_x4(a_addr + k0 * 2, a[0], a[1], a[2], a[3]);
            ldsm_x4(b_addr + k0 * 2, b[0], b[1], b[2], b[3]);
            mma_bf16(acc[0], a, b[0], b[1]);
            mma_bf16(acc[1], a, b[2], b[3]);
        }
        const int h0 = 16 * mt + (lane >> 2);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int s0 = 16 * nq + nt * 8 + 2 * (lane & 3);
            lg_s[h0 * kLgStride + s0] = acc[nt][0] * p.scale;
            lg_s[h0 * kLgStride + s0 + 1] = acc[nt][1] * p.scale;
            lg_s[(h0 + 8) * kLgStride + s0] = acc[nt][2] * p.scale;
            lg_s[(h0 + 8) * kLgStride + s0 + 1] = acc[nt][3] * p.scale;
        }
    }
    __syncthreads();

    // ---- chunk softmax: warp -> 4 heads (reduced side by side), lane -> 2 slots
    float* part = p.part + (size_t)blockIdx.x * kPartFloats;
    {
        constexpr int kH = kHalf / 8;  // 4 heads per warp
        const bool live0 = idx_s[lane] >= 0, live1 = idx_s[lane + 32] >= 0;
        float l0[kH], l1[kH], m[kH], w0[kH], w1[kH], sum[kH];
        bool bad[kH];
#pragma unroll
        for (int i = 0; i < kH; ++i) {
            const int h = warp * kH + i;
            l0[i] = lg_s[h * kLgStride + lane];
            l1[i] = lg_s[h * kLgStride + lane + 32];
            const bool ok0 = live0 && finite_f(l0[i]), ok1 = live1 && finite_f(l1[i]);
            bad[i] = (live0 && !ok0) || (live1 && !ok1);
            if (!ok0) l0[i] = -INFINITY;
            if (!ok1) l1[i] = -INFINITY;
            m[i] = fmaxf(l0[i], l1[i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < kH; ++i) m[i] = fmaxf(m[i], __shfl_xor_sync(0xFFFFFFFFu, m[i], o));
#pragma unroll
        for (int i = 0; i < kH; ++i) {
            w0[i] = l0[i] == -INFINITY ? 0.0f : expf(l0[i] - m[i]);
            w1[i] = l1[i] == -INFINITY ? 0.0f : expf(l1[i] - m[i]);
            sum[i] = w0[i] + w1[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < kH; ++i) sum[i] += __shfl_xor_sync(0xFFFFFFFFu, sum[i], o);
#pragma unroll
        for (int i = 0; i < kH; ++i) {
            const int h = warp * kH + i;
            if (__any_sync(0xFFFFFFFFu, bad[i]) && lane == 0) atomicOr(&p.flags[e * kHeads + head0 + h], 1u);
            const __nv_bfloat16 hi0 = __float2bfloat16_rn(w0[i]), hi1 = __float2bfloat16_rn(w1[i]);
            ph_s[h * kPStride + lane] = hi0;
            ph_s[h * kPStride + lane + 32] = hi1;
            pl_s[h * kPStride + lane] = __float2bfloat16_rn(w0[i] - __bfloat162float(hi0));
            pl_s[h * kPStride + lane + 32] = __float2bfloat16_rn(w1[i] - __bfloat162float(hi1));
            if (lane == 0) {
                part[h] = m[i];
                part[kHalf + h] = sum[i];
            }
        }
    }
    __syncthreads();

    // ---- acc = P G : warp -> 16 heads x 128 features ------------------------
    {
        const int fq = warp & 3;
        float acc[16][4];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
        // ldmatrix.trans lane address: row (slot) = k0 + (mi % 2) * 8 + lane % 8, col = n0 + (mi / 2) * 8.
        const int mi = lane >> 3;
        const uint32_t b_base =
            smem_u32(g_s + ((mi & 1) * 8 + (lane & 7)) * kQStride + fq * 128 + (mi >> 1) * 8);
#pragma unroll
        for (int ks = 0; ks < kSlots / 16; ++ks) {
            uint32_t ah[4], al[4];
            const int off = (16 * mt + (lane & 15)) * kPStride + 16 * ks + (lane >> 4) * 8;
            ldsm_x4(smem_u32(ph_s + off), ah[0], ah[1], ah[2], ah[3]);
            ldsm_x4(smem_u32(pl_s + off), al[0], al[1], al[2], al[3]);
#pragma unroll
            for (int pr = 0; pr < 8; ++pr) {
                uint32_t b[4];
                ldsm_x4_t(b_base + (16 * ks * kQStride + 16 * pr) * 2, b[0], b[1], b[2], b[3]);
                mma_bf16(acc[2 * pr], ah, b[0], b[1]);
                mma_bf16(acc[2 * pr], al, b[0], b[1]);
                mma_bf16(acc[2 * pr + 1], ah, b[2], b[3]);
                mma_bf16(acc[2 * pr + 1], al, b[2], b[3]);
            }
        }
        float* pacc = part + 2 * kHalf;
        const int h0 = 16 * mt + (lane >> 2);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int f = fq * 128 + nt * 8 + 2 * (lane & 3);
            *reinterpret_cast<float2*>(pacc + (size_t)h0 * kDim + f) = make_float2(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<float2*>(pacc + (size_t)(h0 + 8) * kDim + f) = make_float2(acc[nt][2], acc[nt][3]);
        }
    }
}

// Combine the chunks of a (row, head half): CTA = (row, half, 64 features), thread = (head, 8 features).
constexpr int kCombineFeatures = 64;
constexpr int kCombineBlocks = kDim / kCombineFeatures;  // 8 per (row, half)

__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnParams p) {
    __shared__ float mc_s[kAttnChunksMax][kHalf];
    __shared__ float lc_s[kAttnChunksMax][kHalf];
    __shared__ float fac[kHalf][kAttnChunksMax + 1];
    __shared__ float inv_den[kHalf];
    __shared__ uint32_t bad[kHalf];
    const int e = blockIdx.x / (2 * kCombineBlocks);
    const int half = (blockIdx.x / kCombineBlocks) & 1;
    const int fb = blockIdx.x % kCombineBlocks;
    const int head0 = half * kHalf;
    const int t = threadIdx.x;
    const uint32_t W = p.width[e];
    const int nchunks = (int)((W + kSlots - 1) / kSlots);
    const float* part0 = p.part + ((size_t)2 * p.chunk_begin[e] + (size_t)half * nchunks) * kPartFloats;
    pdl_trigger();
    pdl_wait();  // partials and flags come from the partial kernel

    // Issue every load of this thread before using any.
    const int h = t >> 3;
    const int f = fb * kCombineFeatures + (t & 7) * 8;
    float4 v[kAttnChunksMax][2];
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c)
        if (c < nchunks) {
            const float* src = part0 + (size_t)c * kPartFloats + 2 * kHalf + (size_t)h * kDim + f;
            v[c][0] = __ldcg(reinterpret_cast<const float4*>(src));
            v[c][1] = __ldcg(reinterpret_cast<const float4*>(src + 4));
        }
    if (t < nchunks * kHalf) {
        const int c = t / kHalf, hh = t % kHalf;
        mc_s[c][hh] = __ldcg(part0 + (size_t)c * kPartFloats + hh);
        lc_s[c][hh] = __ldcg(part0 + (size_t)c * kPartFloats + kHalf + hh);
    }
    __syncthreads();
    if (t < kHalf) {
        const int hd = head0 + t;
        const bool row_bad = __ldcg(p.flags + kRowsMax * kHeads + e) != 0;
        const float sink = p.sinks[(size_t)p.q_row[e] * p.sinks_row_stride + hd];
        uint32_t inv = row_bad || __ldcg(p.flags + e * kHeads + hd) != 0 || !finite_f(sink);
        float m = sink;
        for (int c = 0; c < nchunks; ++c) m = fmaxf(m, mc_s[c][t]);
        float den = finite_f(sink) ? expf(sink - m) : 0.0f;
        for (int c = 0; c < nchunks; ++c) {
            const float mc = mc_s[c][t];
            const float fc = mc == -INFINITY ? 0.0f : expf(mc - m);
            fac[t][c] = fc;
            den = fmaf(lc_s[c][t], fc, den);
        }
        if (!finite_f(den) || !(den > 0.0f) || !finite_f(m)) inv = 1;
        inv_den[t] = 1.0f / den;
        bad[t] = inv;
        if (p.invalid && fb == 0) p.invalid[(size_t)p.q_row[e] * kHeads + hd] = inv;
    }
    __syncthreads();

    float r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c) {
        if (c < nchunks) {
            const float w = fac[h][c];
            r[0] = fmaf(v[c][0].x, w, r[0]); r[1] = fmaf(v[c][0].y, w, r[1]);
            r[2] = fmaf(v[c][0].z, w, r[2]); r[3] = fmaf(v[c][0].w, w, r[3]);
            r[4] = fmaf(v[c][1].x, w, r[4]); r[5] = fmaf(v[c][1].y, w, r[5]);
            r[6] = fmaf(v[c][1].z, w, r[6]); r[7] = fmaf(v[c][1].w, w, r[7]);
        }
    }
    const float sc = inv_den[h];
    const bool zero = bad[h] != 0;
    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float x = r[i] * sc;
        o[i] = __float2bfloat16_rn(!zero && finite_f(x) ? x : 0.0f);
    }
    __nv_bfloat16* out = p.out + ((size_t)p.q_row[e] * kHeads + head0 + h) * kDim + f;
    *reinterpret_cast<uint4*>(out) = *reinterpret_cast<const uint4*>(o);
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
    const uint32_t sort_ctas = p.sorted_out ? p.rows : 0u;
    cudaError_t err = launch_kernel(attn_partial_kernel, dim3(2 * p.total_chunks + sort_ctas), dim3(kThreads),
                                    kSmemBytes, stream, pdl, p);
    if (err != cudaSuccess) return err;
    return launch_kernel(attn_combine_kernel, dim3(p.rows * 2 * kCombineBlocks), dim3(256), 0, stream, true, p);
}

}  // namespace dsrows
