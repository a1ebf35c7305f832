// Building blocks of one attention chunk: H query heads (32 or 64) against 64
// gathered KV rows, shared by the stand-alone attention kernels and the
// decode's fused select + attend kernel so that both compute every element
// with the same operations in the same order.
//
// Per head h of the chunk (slots t, index i_t, -1 = empty):
//   l_t = scale * q_h . KV[i_t]                     (tensor cores, fp32 accumulate)
//   m_c = max over live slots of l_t, l_c = sum exp(l_t - m_c)
//   acc_c = sum_t exp(l_t - m_c) KV[i_t]            (P as a bf16 hi + lo pair)
// Warp roles: the logits take warp -> (16 heads, 16 slots); the softmax takes
// warp -> HW heads, lane -> 2 slots; P G takes warp -> (16 heads, FW features).
// The roles only decide which warp computes an element, never how.
#pragma once

#include "common.cuh"

namespace dsrows {
namespace attend {

constexpr int kSlots = kAttnSlots;    // 64 selected slots per chunk
constexpr int kQStride = kDim + 8;    // bf16 per smem row: 1040 B, conflict-free ldmatrix
constexpr int kPStride = kSlots + 8;  // 144 B rows, conflict-free ldmatrix
constexpr int kLgStride = kSlots + 1;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
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

// Issue the copy of H query rows (512 bf16 each, contiguous) into q_s.
template <int H, int NT>
__device__ __forceinline__ void load_q(__nv_bfloat16* q_s, const __nv_bfloat16* q, int t) {
    for (int k = t; k < H * (kDim / 8); k += NT) {
        const int row = k >> 6, col = (k & 63) * 8;
        cp_async16(q_s + row * kQStride + col, q + (size_t)row * kDim + col);
    }
}

// Issue the gather of the chunk's 64 KV rows (1 KiB each); empty slots are zeros.
template <int NT>
__device__ __forceinline__ void gather_kv(__nv_bfloat16* g_s, const int* idx_s, const __nv_bfloat16* kv, int t) {
    for (int k = t; k < kSlots * (kDim / 8); k += NT) {
        const int row = k >> 6, col = (k & 63) * 8;
        const int i = idx_s[row];
        __nv_bfloat16* dst = g_s + row * kQStride + col;
        if (i >= 0) cp_async16(dst, kv + (size_t)i * kDim + col);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
}

// lg_s[h][t] = scale * (Q G^T)[h][t]: warp -> 16 heads x 16 slots.
template <int H>
__device__ __forceinline__ void logits(const __nv_bfloat16* q_s, const __nv_bfloat16* g_s, float* lg_s, float scale,
                                       int warp, int lane) {
    static_assert(H % 16 == 0, "heads come in tiles of 16");
    const int mt = warp >> 2;  // head tile (16 heads)
    const int nq = warp & 3;   // slot quarter (16 slots)
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
        lg_s[h0 * kLgStride + s0] = acc[nt][0] * scale;
        lg_s[h0 * kLgStride + s0 + 1] = acc[nt][1] * scale;
        lg_s[(h0 + 8) * kLgStride + s0] = acc[nt][2] * scale;
        lg_s[(h0 + 8) * kLgStride + s0 + 1] = acc[nt][3] * scale;
    }
}

// Chunk softmax over lg_s, heads [HW warp, HW warp + HW): writes P = exp(l - m_c)
// as bf16 hi + lo into ph_s / pl_s and, from lane 0, put(h, m_c, l_c, bad) per
// head, where bad marks a live slot with a non-finite logit. Empty slots weigh zero.
template <int HW, class Put>
__device__ __forceinline__ void softmax(const float* lg_s, const int* idx_s, __nv_bfloat16* ph_s,
                                        __nv_bfloat16* pl_s, int warp, int lane, Put put) {
    constexpr int kH = HW;  // heads per warp, reduced side by side
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
        const bool any_bad = __any_sync(0xFFFFFFFFu, bad[i]);
        const __nv_bfloat16 hi0 = __float2bfloat16_rn(w0[i]), hi1 = __float2bfloat16_rn(w1[i]);
        ph_s[h * kPStride + lane] = hi0;
        ph_s[h * kPStride + lane + 32] = hi1;
        pl_s[h * kPStride + lane] = __float2bfloat16_rn(w0[i] - __bfloat162float(hi0));
        pl_s[h * kPStride + lane + 32] = __float2bfloat16_rn(w1[i] - __bfloat162float(hi1));
        if (lane == 0) put(h, m[i], sum[i], any_bad);
    }
}

// acc = P G for warp -> 16 heads x FW features (FW = 64 or 128). Element
// acc[nt][k] is head 16 (warp / G) + lane / 4 (+ 8 for k >= 2), feature
// FW (warp % G) + 8 nt + 2 (lane % 4) + k % 2, with G = 512 / FW.
template <int FW>
__device__ __forceinline__ void pv(const __nv_bfloat16* ph_s, const __nv_bfloat16* pl_s, const __nv_bfloat16* g_s,
                                   int warp, int lane, float (&acc)[FW / 8][4]) {
    constexpr int G = kDim / FW;
    const int mt = warp / G, fq = warp % G;
#pragma unroll
    for (int i = 0; i < FW / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
    // ldmatrix.trans lane address: row (slot) = k0 + (mi % 2) * 8 + lane % 8, col = n0 + (mi / 2) * 8.
    const int mi = lane >> 3;
    const uint32_t b_base = smem_u32(g_s + ((mi & 1) * 8 + (lane & 7)) * kQStride + fq * FW + (mi >> 1) * 8);
#pragma unroll
    for (int ks = 0; ks < kSlots / 16; ++ks) {
        uint32_t ah[4], al[4];
        const int off = (16 * mt + (lane & 15)) * kPStride + 16 * ks + (lane >> 4) * 8;
        ldsm_x4(smem_u32(ph_s + off), ah[0], ah[1], ah[2], ah[3]);
        ldsm_x4(smem_u32(pl_s + off), al[0], al[1], al[2], al[3]);
#pragma unroll
        for (int pr = 0; pr < FW / 16; ++pr) {
            uint32_t b[4];
            ldsm_x4_t(b_base + (16 * ks * kQStride + 16 * pr) * 2, b[0], b[1], b[2], b[3]);
            mma_bf16(acc[2 * pr], ah, b[0], b[1]);
            mma_bf16(acc[2 * pr], al, b[0], b[1]);
            mma_bf16(acc[2 * pr + 1], ah, b[2], b[3]);
            mma_bf16(acc[2 * pr + 1], al, b[2], b[3]);
        }
    }
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

// Combine feature columns [f0, f0 + 64) of H heads over the n chunk partials of
// one row (or head half) with NT threads (thread -> one head, 64 H / NT
// features). A partial is m[H], l[H], acc[H][512] (fp32), `stride` floats apart
// from part0; flags[h] marks a head with a non-finite logit, row_bad the whole
// row; the heads' outputs start at out (rows of 512 bf16), and invalid
// (optional) receives each head's flag.
template <int H, int NT>
__device__ __forceinline__ void combine_slice(const float* part0, size_t stride, int n, int f0, const float* sinks,
                                              bool row_bad, const uint32_t* flags, __nv_bfloat16* out,
                                              uint32_t* invalid, CombineSmem<H>& cs) {
    constexpr int FPT = 64 * H / NT;  // features per thread
    static_assert(FPT == 4 || FPT == 8, "4 or 8 features per thread");
    static_assert(NT >= kAttnChunksMax * H, "one thread per (chunk, head) statistic");
    const int t = threadIdx.x;
    const int h = t / (64 / FPT);
    const int f = f0 + (t % (64 / FPT)) * FPT;
    // Issue every load of this thread before using any.
    float4 v[kAttnChunksMax][FPT / 4];
#pragma unroll
    for (int c = 0; c < kAttnChunksMax; ++c)
        if (c < n) {
            const float* src = part0 + (size_t)c * stride + 2 * H + (size_t)h * kDim + f;
#pragma unroll
            for (int u = 0; u < FPT / 4; ++u) v[c][u] = __ldcg(reinterpret_cast<const float4*>(src + 4 * u));
        }
    if (t < n * H) {
        const int c = t / H, hh = t % H;
        cs.mc[c][hh] = __ldcg(part0 + (size_t)c * stride + hh);
        cs.lc[c][hh] = __ldcg(part0 + (size_t)c * stride + H + hh);
    }
    __syncthreads();
    if (t < H) {
        bool b = row_bad || __ldcg(flags + t) != 0;
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
