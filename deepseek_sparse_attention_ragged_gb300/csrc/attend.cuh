// Attention building blocks: 16-byte asynchronous copies and the combine of a
// row's chunk partials with the sink (fixed chunk order), shared by the
// selection + attention kernel's paths.
#pragma once

#include "common.cuh"

namespace dsrows {
namespace attend {

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Combine feature columns [f0, f0 + F) of H heads over the n chunk partials of
// one row (or head half) with NT threads: thread -> one head and F H / NT
// consecutive features. A partial is m[H], l[H], acc[H][512] (fp32), `stride`
// floats apart from part0, except that chunk own_c's accumulators of these
// columns are read from `own` ([H][F] in shared memory; own_c < 0: none);
// flags[h] marks a head with a non-finite logit,
// *row_flag the whole row; the heads' outputs start at out (rows of 512 bf16),
// and invalid (optional) receives each head's flag. Per head, in chunk order
// (the order depends on the number of chunks alone):
//   m = max(sink, m_c), den = exp(sink - m) + sum_c l_c exp(m_c - m),
//   out = (sum_c exp(m_c - m) acc_c) / den.
// The head is written as zeros when it is flagged or its sink, maximum or
// denominator is not finite (or den <= 0); any non-finite element as zero.
// Every thread of a head computes the head's factors itself: no block barrier.
template <int H, int NT, int F>
__device__ __forceinline__ void combine_slice(const float* part0, size_t stride, int n, int f0, const float* own,
                                              int own_c, const float* sinks,
                                              const uint32_t* row_flag, const uint32_t* flags, __nv_bfloat16* out,
                                              uint32_t* invalid) {
    constexpr int FPT = F * H / NT;  // features per thread
    constexpr int TPH = F / FPT;     // threads per head
    static_assert(FPT == 4 || FPT == 8, "4 or 8 features per thread");
    const int t = threadIdx.x;
    const int h = t / TPH;
    const int f = f0 + (t % TPH) * FPT;
    // Issue every load of this thread before using any: the partial's features,
    // its statistics and the flags travel in one round trip to L2.
    float4 v[kAttnChunksMax][FPT / 4];
    float mc[kAttnChunksMax], lc[kAttnChunksMax];
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c)
        if (c < n) {
            const float* pc = part0 + (size_t)c * stride;
            if (c == own_c) {
                const float* src = own + h * F + (f - f0);
#pragma unroll
                for (int u = 0; u < FPT / 4; ++u) v[c][u] = *reinterpret_cast<const float4*>(src + 4 * u);
            } else {
                const float* src = pc + 2 * H + (size_t)h * kDim + f;
#pragma unroll
                for (int u = 0; u < FPT / 4; ++u) v[c][u] = __ldcg(reinterpret_cast<const float4*>(src + 4 * u));
            }
            mc[c] = __ldcg(pc + h);
            lc[c] = __ldcg(pc + H + h);
        }
    const uint32_t flagged = __ldcg(flags + h) | __ldcg(row_flag);
    const float sink = sinks[h];
    float m = sink;
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c)
        if (c < n) m = fmaxf(m, mc[c]);
    float den = finite_f(sink) ? expf(sink - m) : 0.0f;
    float fac[kAttnChunksMax];
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c)
        if (c < n) {
            fac[c] = mc[c] == -INFINITY ? 0.0f : expf(mc[c] - m);
            den = fmaf(lc[c], fac[c], den);
        }
    const bool zero = flagged != 0 || !finite_f(sink) || !finite_f(den) || !(den > 0.0f) || !finite_f(m);
    if (invalid && t % TPH == 0) invalid[h] = zero ? 1u : 0u;
    const float inv_den = 1.0f / den;
    float r[FPT];
#pragma unroll
    for (int i = 0; i < FPT; ++i) r[i] = 0.0f;
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c) {
        if (c < n) {
            const float w = fac[c];
#pragma unroll
            for (int u = 0; u < FPT / 4; ++u) {
                r[4 * u] = fmaf(v[c][u].x, w, r[4 * u]);
                r[4 * u + 1] = fmaf(v[c][u].y, w, r[4 * u + 1]);
                r[4 * u + 2] = fmaf(v[c][u].z, w, r[4 * u + 2]);
                r[4 * u + 3] = fmaf(v[c][u].w, w, r[4 * u + 3]);
            }
        }
    }
    __align__(16) __nv_bfloat16 o[FPT];
#pragma unroll
    for (int i = 0; i < FPT; ++i) {
        const float x = r[i] * inv_den;
        o[i] = __float2bfloat16_rn(!zero && finite_f(x) ? x : 0.0f);
    }
    __nv_bfloat16* dst = out + (size_t)h * kDim + f;
    if (FPT == 8) *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(o);
    else *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(o);
}

}  // namespace attend
}  // namespace dsrows
