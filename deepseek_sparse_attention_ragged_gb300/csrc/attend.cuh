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

// Per-head combine of a row's chunks with the sink (the reduction order
// depends on the number of chunks alone):
//   m = max(sink, m_c), den = exp(sink - m) + sum_c l_c exp(m_c - m),
//   fac_c = exp(m_c - m), out = (sum_c fac_c acc_c) / den.
// Writes fac[0, n) and returns 1/den; `bad` is set when the head must be
// written as zeros (non-finite sink, max or denominator).
template <class MC, class LC>
__device__ __forceinline__ float combine_factors(float sink, int n, MC mc, LC lc, float* fac, bool& bad) {
    float m = sink;
    for (int c = 0; c < n; ++c) m = fmaxf(m, mc(c));
    float den = finite_f(sink) ? expf(sink - m) : 0.0f;
    for (int c = 0; c < n; ++c) {
        const float mcc = mc(c);
        const float fc = mcc == -INFINITY ? 0.0f : expf(mcc - m);
        fac[c] = fc;
        den = fmaf(lc(c), fc, den);
    }
    if (!finite_f(sink) || !finite_f(den) || !(den > 0.0f) || !finite_f(m)) bad = true;
    return 1.0f / den;
}

// Shared memory of combine_slice for H heads.
template <int H>
struct CombineSmem {
    float mc[kAttnChunksMax][H];
    float lc[kAttnChunksMax][H];
    float fac[H][kAttnChunksMax + 1];
    float inv_den[H];
    uint32_t bad[H];
};

// Combine feature columns [f0, f0 + F) of H heads over the n chunk partials of
// one row (or head half) with NT threads (thread -> one head, F H / NT
// features). A partial is m[H], l[H], acc[H][512] (fp32), `stride` floats apart
// from part0; flags[h] marks a head with a non-finite logit, *row_flag the
// whole row; the heads' outputs start at out (rows of 512 bf16), and invalid
// (optional) receives each head's flag.
template <int H, int NT, int F = 64>
__device__ __forceinline__ void combine_slice(const float* part0, size_t stride, int n, int f0, const float* sinks,
                                              const uint32_t* row_flag, const uint32_t* flags, __nv_bfloat16* out,
                                              uint32_t* invalid, CombineSmem<H>& cs) {
    constexpr int FPT = F * H / NT;  // features per thread
    static_assert(FPT == 4 || FPT == 8, "4 or 8 features per thread");
    static_assert(NT >= kAttnChunksMax * H, "one thread per (chunk, head) statistic");
    const int t = threadIdx.x;
    const int h = t / (F / FPT);
    const int f = f0 + (t % (F / FPT)) * FPT;
    // Issue every load of this thread before using any.
    float4 v[kAttnChunksMax][FPT / 4];
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c)
        if (c < n) {
            const float* src = part0 + (size_t)c * stride + 2 * H + (size_t)h * kDim + f;
#pragma unroll
            for (int u = 0; u < FPT / 4; ++u) v[c][u] = __ldcg(reinterpret_cast<const float4*>(src + 4 * u));
        }
    // The flags travel with the partials' statistics: one round trip to L2.
    uint32_t flagged = 0;
    if (t < H) flagged = __ldcg(flags + t) | __ldcg(row_flag);
    if (t < n * H) {
        const int c = t / H, hh = t % H;
        cs.mc[c][hh] = __ldcg(part0 + (size_t)c * stride + hh);
        cs.lc[c][hh] = __ldcg(part0 + (size_t)c * stride + H + hh);
    }
    __syncthreads();
    if (t < H) {
        bool b = flagged != 0;
        cs.inv_den[t] = combine_factors(
            sinks[t], n, [&](int c) { return cs.mc[c][t]; }, [&](int c) { return cs.lc[c][t]; }, cs.fac[t], b);
        cs.bad[t] = b ? 1u : 0u;
        if (invalid) invalid[t] = b ? 1u : 0u;
    }
    __syncthreads();
    float r[FPT];
#pragma unroll
    for (int i = 0; i < FPT; ++i) r[i] = 0.0f;
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c) {
        if (c < n) {
            const float w = cs.fac[h][c];
#pragma unroll
            for (int u = 0; u < FPT / 4; ++u) {
                r[4 * u] = fmaf(v[c][u].x, w, r[4 * u]);
                r[4 * u + 1] = fmaf(v[c][u].y, w, r[4 * u + 1]);
                r[4 * u + 2] = fmaf(v[c][u].z, w, r[4 * u + 2]);
                r[4 * u + 3] = fmaf(v[c][u].w, w, r[4 * u + 3]);
            }
        }
    }
    const float sc = cs.inv_den[h];
    const bool zero = cs.bad[h] != 0;
    __align__(16) __nv_bfloat16 o[FPT];
#pragma unroll
    for (int i = 0; i < FPT; ++i) {
        const float x = r[i] * sc;
        o[i] = __float2bfloat16_rn(!zero && finite_f(x) ? x : 0.0f);
    }
    __nv_bfloat16* dst = out + (size_t)h * kDim + f;
    if (FPT == 8) *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(o);
    else *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(o);
}

}  // namespace attend
}  // namespace dsrows
