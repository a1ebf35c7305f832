// Gather + sink-softmax sparse attention (mlx-native deepseek_rows.metal, kernels
// deepseek_sparse_attention_score_rows_bf16 and deepseek_sparse_attention_reduce_rows_bf16;
// gather semantics of deepseek_sparse_attention_gather_rows_bf16).
//
// Per row e and head h over the selected slots t (index i_t):
//   l_t = scale * q_h . KV[i_t],  m = max(sink_h, max l_t),
//   den = exp(sink_h - m) + sum exp(l_t - m),  out_h = sum exp(l_t - m) KV[i_t] / den.
//
// GB300 design. A row's `width` slots are split into chunks of 32; one CTA per
// (row, chunk) gathers its 32 KV rows (1 KiB each, 16-byte cp.async, read once
// for all 64 heads), computes the 64x32 logits S = Q G^T and the 64x512
// partial P G on tensor cores (mma.sync m16n8k16 bf16, fp32 accumulate), with
// a chunk-local softmax (m_c, l_c). P enters the second product as a bf16
// hi + lo pair, which keeps ~16 bits of each weight. A second kernel combines
// the chunks of a row in chunk order with the sink:
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
constexpr int kSlots = kAttnSlots;  // 32
constexpr int kQStride = kDim + 8;  // bf16 per smem row: 1040 B, conflict-free ldmatrix
constexpr int kPStride = kSlots + 8;
constexpr int kLgStride = kSlots + 1;

struct SmemLayout {
    static constexpr size_t q = 0;
    static constexpr size_t g = q + (size_t)kHeads * kQStride * 2;
    static constexpr size_t p_hi = g + (size_t)kSlots * kQStride * 2;
    static constexpr size_t p_lo = p_hi + (size_t)kHeads * kPStride * 2;
    static constexpr size_t lg = p_lo + (size_t)kHeads * kPStride * 2;
    static constexpr size_t idx = lg + (size_t)kHeads * kLgStride * 4;
    static constexpr size_t total = idx + kSlots * 4;
};
constexpr size_t kSmemBytes = SmemLayout::total;

__device__ __forceinline__ int entry_of_chunk(const AttnParams& p, uint32_t c) {
    int e = 0;
#pragma unroll
    for (int i = 1; i < kRowsMax; ++i)
        if (i < (int)p.rows && c >= p.chunk_begin[i]) e = i;
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

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) attn_partial_kernel(const AttnParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __nv_bfloat16* q_s = reinterpret_cast<__nv_bfloat16*>(smem + SmemLayout::q);
    __nv_bfloat16* g_s = reinterpret_cast<__nv_bfloat16*>(smem + SmemLayout::g);
    __nv_bfloat16* ph_s = reinterpret_cast<__nv_bfloat16*>(smem + SmemLayout::p_hi);
    __nv_bfloat16* pl_s = reinterpret_cast<__nv_bfloat16*>(smem + SmemLayout::p_lo);
    float* lg_s = reinterpret_cast<float*>(smem + SmemLayout::lg);
    int* idx_s = reinterpret_cast<int*>(smem + SmemLayout::idx);

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int e = entry_of_chunk(p, blockIdx.x);
    const uint32_t c = blockIdx.x - p.chunk_begin[e];
    const uint32_t W = p.width[e];
    const int L = (int)p.kv_len[e];
    const __nv_bfloat16* kv = p.kv[e];

    pdl_trigger();
    // The query is an input of the call: fetch it while the previous kernel finishes.
    const __nv_bfloat16* q = p.q + (size_t)p.q_row[e] * kHeads * kDim;
    for (int k = t; k < kHeads * (kDim / 8); k += kThreads) {
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

    // Gather the chunk's selected KV rows (1 KiB each, once for all heads).
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
    const int mt = warp >> 1;       // head tile (16 heads)
    {
        const int nh = warp & 1;    // slot half (16 slots)
        float acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
        const uint32_t a_addr = smem_u32(q_s + (16 * mt + (lane & 15)) * kQStride + (lane >> 4) * 8);
        const uint32_t b_addr =
            smem_u32(g_s + (16 * nh + (lane >> 4) * 8 + (lane & 7)) * kQStride + ((lane >> 3) & 1) * 8);
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
            const int s0 = 16 * nh + nt * 8 + 2 * (lane & 3);
            lg_s[h0 * kLgStride + s0] = acc[nt][0] * p.scale;
            lg_s[h0 * kLgStride + s0 + 1] = acc[nt][1] * p.scale;
            lg_s[(h0 + 8) * kLgStride + s0] = acc[nt][2] * p.scale;
            lg_s[(h0 + 8) * kLgStride + s0 + 1] = acc[nt][3] * p.scale;
        }
    }
    __syncthreads();

    // ---- chunk softmax: warp -> 8 heads, lane -> slot -----------------------
    float* part = p.part + (size_t)blockIdx.x * kPartFloats;
    {
        const bool live = idx_s[lane] >= 0;
        for (int hh = 0; hh < 8; ++hh) {
            const int h = warp * 8 + hh;
            const float l = lg_s[h * kLgStride + lane];
            const bool ok = live && finite_f(l);
            if (__any_sync(0xFFFFFFFFu, live && !ok) && lane == 0) atomicOr(&p.flags[e * kHeads + h], 1u);
            const float m = warp_max(ok ? l : -INFINITY);
            const float w = ok ? expf(l - m) : 0.0f;
            const float sum = warp_sum(w);
            const __nv_bfloat16 hi = __float2bfloat16_rn(w);
            const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
            ph_s[h * kPStride + lane] = hi;
            pl_s[h * kPStride + lane] = lo;
            if (lane == 0) {
                part[h] = m;
                part[kHeads + h] = sum;
            }
        }
    }
    __syncthreads();

    // ---- acc = P G : warp -> 16 heads x 256 features ------------------------
    {
        const int fh = warp & 1;
        float acc[32][4];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
        uint32_t ah[2][4], al[2][4];
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int off = (16 * mt + (lane & 15)) * kPStride + 16 * ks + (lane >> 4) * 8;
            ldsm_x4(smem_u32(ph_s + off), ah[ks][0], ah[ks][1], ah[ks][2], ah[ks][3]);
            ldsm_x4(smem_u32(pl_s + off), al[ks][0], al[ks][1], al[ks][2], al[ks][3]);
        }
        // ldmatrix.trans lane address: row (slot) = k0 + (mi % 2) * 8 + lane % 8, col = n0 + (mi / 2) * 8.
        const int mi = lane >> 3;
        const uint32_t b_base =
            smem_u32(g_s + ((mi & 1) * 8 + (lane & 7)) * kQStride + fh * 256 + (mi >> 1) * 8);
#pragma unroll
        for (int pr = 0; pr < 16; ++pr) {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t b[4];
                ldsm_x4_t(b_base + (16 * ks * kQStride + 16 * pr) * 2, b[0], b[1], b[2], b[3]);
                mma_bf16(acc[2 * pr], ah[ks], b[0], b[1]);
                mma_bf16(acc[2 * pr], al[ks], b[0], b[1]);
                mma_bf16(acc[2 * pr + 1], ah[ks], b[2], b[3]);
                mma_bf16(acc[2 * pr + 1], al[ks], b[2], b[3]);
            }
        }
        float* pacc = part + 2 * kHeads;
        const int h0 = 16 * mt + (lane >> 2);
#pragma unroll
        for (int nt = 0; nt < 32; ++nt) {
            const int f = fh * 256 + nt * 8 + 2 * (lane & 3);
            *reinterpret_cast<float2*>(pacc + (size_t)h0 * kDim + f) = make_float2(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<float2*>(pacc + (size_t)(h0 + 8) * kDim + f) = make_float2(acc[nt][2], acc[nt][3]);
        }
    }
}

// Combine the chunks of a row: CTA = (row, 16 features), thread = (head, 4 features).
constexpr int kCombineFeatures = 16;
constexpr int kCombineBlocks = kDim / kCombineFeatures;  // 32 per row

__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnParams p) {
    __shared__ float mc_s[kAttnChunksMax][kHeads];
    __shared__ float lc_s[kAttnChunksMax][kHeads];
    __shared__ float fac[kHeads][kAttnChunksMax + 1];
    __shared__ float inv_den[kHeads];
    __shared__ uint32_t bad[kHeads];
    const int e = blockIdx.x / kCombineBlocks;
    const int fb = blockIdx.x % kCombineBlocks;
    const int t = threadIdx.x;
    const uint32_t W = p.width[e];
    const int nchunks = (int)((W + kSlots - 1) / kSlots);
    const float* part0 = p.part + (size_t)p.chunk_begin[e] * kPartFloats;
    pdl_trigger();
    pdl_wait();  // partials and flags come from the partial kernel

    // Issue every load of this thread before using any.
    const int h = t >> 2;
    const int f = fb * kCombineFeatures + (t & 3) * 4;
    float4 v[kAttnChunksMax];
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c)
        if (c < nchunks)
            v[c] = __ldcg(reinterpret_cast<const float4*>(part0 + (size_t)c * kPartFloats + 2 * kHeads +
                                                          (size_t)h * kDim + f));
    for (int i = t; i < nchunks * kHeads; i += 256) {
        const int c = i / kHeads, hh = i % kHeads;
        mc_s[c][hh] = __ldcg(part0 + (size_t)c * kPartFloats + hh);
        lc_s[c][hh] = __ldcg(part0 + (size_t)c * kPartFloats + kHeads + hh);
    }
    __syncthreads();
    if (t < kHeads) {
        const bool row_bad = __ldcg(p.flags + kRowsMax * kHeads + e) != 0;
        const float sink = p.sinks[(size_t)p.q_row[e] * p.sinks_row_stride + t];
        uint32_t inv = row_bad || __ldcg(p.flags + e * kHeads + t) != 0 || !finite_f(sink);
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
        if (p.invalid && fb == 0) p.invalid[(size_t)p.q_row[e] * kHeads + t] = inv;
    }
    __syncthreads();

    float4 acc = make_float4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c) {
        if (c < nchunks) {
            const float w = fac[h][c];
            acc.x = fmaf(v[c].x, w, acc.x);
            acc.y = fmaf(v[c].y, w, acc.y);
            acc.z = fmaf(v[c].z, w, acc.z);
            acc.w = fmaf(v[c].w, w, acc.w);
        }
    }
    const float sc = inv_den[h];
    const bool zero = bad[h] != 0;
    const float r[4] = {acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc};
    __nv_bfloat16 o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = __float2bfloat16_rn(!zero && finite_f(r[i]) ? r[i] : 0.0f);
    __nv_bfloat16* out = p.out + ((size_t)p.q_row[e] * kHeads + h) * kDim + f;
    *reinterpret_cast<uint2*>(out) = *reinterpret_cast<const uint2*>(o);
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
    cudaError_t err = launch_kernel(attn_partial_kernel, dim3(p.total_chunks), dim3(kThreads), kSmemBytes, stream,
                                    pdl, p);
    if (err != cudaSuccess) return err;
    return launch_kernel(attn_combine_kernel, dim3(p.rows * kCombineBlocks), dim3(256), 0, stream, true, p);
}

}  // namespace dsrows
