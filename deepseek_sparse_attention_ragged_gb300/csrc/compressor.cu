// Learned KV compressor, one decode token per row (mlx-native deepseek_rows.metal,
// kernel deepseek_compressor_rows_bf16; dispatch_deepseek_compressor_rows).
//
// With coff = 2 for ratio 4 (overlapping windows) and 1 for ratio 128, and
// P = coff * head_dim features per token, per row:
//   1. the token (token = start_pos mod ratio) is written to state row
//      (ratio if overlapping else 0) + token: its kv (0 where not finite) and
//      score + ape[token] (NaN where either is not finite);
//   2. when start_pos + 1 is a multiple of ratio, each feature f softmax-pools
//      the window's values with its scores (2 ratio rows when overlapping: the
//      first ratio rows read feature f, the rest feature head_dim + f), the
//      pooled value is rounded to bf16, and the row is RMS-normalised:
//        out = bf16(c * norm / sqrt(mean(c^2) + eps)),
//      all zero when any score is NaN or +inf, any value, pooled value, norm,
//      sum or result is not finite; overlapping windows then shift the current
//      block into the previous rows. Otherwise the output row is zero.
//
// GB300 design: one 8-CTA cluster per row; CTA r owns output features
// [r D/8, (r+1) D/8) in float4 columns, and a CTA keeps its whole share of the
// window in flight: every window row it pools is loaded before any is used,
// and the token's own row comes from the thread that computes it, so the loads
// do not wait for the token's write.
//   - ratio 4: 16 threads per column split the window's rows, combined by a
//     fixed-order shuffle tree; the token's row arrives by a shuffle;
//   - ratio 128 (head_dim 512): lane l of warp w takes column l mod 16 of
//     window rows 16 q + 2 w + l / 16, so each load of a warp reads two rows'
//     256 bytes contiguously; the max and the exponential sums combine over the
//     lane pair by shuffle and over the 8 warps through shared memory, in warp
//     order. Each thread owns its features in every state row, so
// the token write, the pooling and the shift need no barrier beyond the
// block's; the RMS sum and the fail-closed flags cross the
// cluster as st.async pushes into every CTA (counted on mbarriers) and are
// added in rank order.

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace dsrows {

namespace cg = cooperative_groups;

namespace {

constexpr int kCompCluster = 8;
constexpr int kCompThreads = 256;
constexpr int kSplit = 16;        // threads per float4 column
// No output can overflow while every norm is at most this: |output| <= sqrt(512) |norm|.
constexpr float kNormSafe = 1e37f;
// Window rows per thread: 128 / 16 with ratio 128, one (2 * 4 rows over 16 threads) with ratio 4.
constexpr int kRowsRatio128 = 8;
constexpr int kRowsRatio4 = 1;

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float comp(const float4& v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

struct __align__(8) CompSmem {
    uint64_t bar_sq;           // the cluster's shares arrive here (st.async)
    uint64_t bar_yb;           // ... and their output flags
    float col_sq[kSplit];      // per float4 column: sum of c^2
    uint32_t col_bad[kSplit];
    uint32_t cta_ybad;
    uint32_t sq_all[kCompCluster];   // every CTA's sum of c^2 (fp32 bits), by rank
    uint32_t bad_all[kCompCluster];  // every CTA's bad flag, by rank
    uint32_t yb_all[kCompCluster];   // every CTA's output flag, by rank
    // Ratio 128: per warp and column, the window's max, its flags, and the
    // exponential sums of the warp's rows.
    float red_m[kCompThreads / 32][kSplit][4];
    uint32_t red_b[kCompThreads / 32][kSplit];
    float red_d[kCompThreads / 32][kSplit][4];
    float red_n[kCompThreads / 32][kSplit][4];
};

}  // namespace

template <int kRowsPerThread>
__global__ void __cluster_dims__(kCompCluster, 1, 1) __launch_bounds__(kCompThreads)
    compressor_kernel(const CompressorParams p) {
    __shared__ CompSmem sm;
    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t rank = cluster.block_rank();
    const int row = blockIdx.x / kCompCluster;
    const int t = threadIdx.x;
    const int D = (int)p.head_dim, R = (int)p.ratio;
    const bool overlap = R == 4;
    const int coff = overlap ? 2 : 1;
    const int P = coff * D;
    const uint32_t pos = p.start_pos[row];
    const int token = (int)(pos % (uint32_t)R);
    const int slot = (overlap ? R : 0) + token;
    const int FB = D / kCompCluster;          // features of this CTA: 16 or 64
    const int ncol = FB / 4;
    const int col = t / kSplit, sub = t % kSplit;
    const bool active = col < ncol;
    const int f0 = FB * (int)rank + 4 * col;  // first of this column's four features
    float* kvs = p.kv_state[row];
    float* scs = p.score_state[row];

    // The exchange barriers, visible to the cluster before any CTA stores into
    // another (this overlaps the previous kernel).
    if (t == 0) {
        mbar_init(&sm.bar_sq, 1);
        mbar_init(&sm.bar_yb, 1);
        fence_barrier_init();
    }
    cluster.sync();
    pdl_wait();  // inputs and states may come from the previous kernel
    // The next kernel may start launching; it waits for this grid to complete
    // before it reads anything (griddepcontrol.wait).
    pdl_trigger();

    const bool complete = (pos + 1) % (uint32_t)R == 0;  // the same for the whole cluster
    const int items = coff * R;
    // After the pooling, the thread that writes column wcol (features wf0..wf0+3)
    // holds its softmax sums den/num and the column's flags in `bad`.
    bool writer;
    int wcol, wf0;
    float den[4] = {0, 0, 0, 0}, num[4] = {0, 0, 0, 0};
    uint32_t bad = 0;
    if constexpr (kRowsPerThread == kRowsRatio128) {
        // ---- ratio 128 (head_dim 512, 16 columns per CTA): lane l of warp w takes
        // column l % 16 of window rows 16 q + 2 w + l / 16, so a warp's load covers
        // two rows' 256 bytes each, contiguously. The thread that owns the token's
        // row computes and writes it instead of loading it.
        const int lane = t & 31, w = t >> 5;
        const int ch = lane & (kSplit - 1), par = lane >> 4;
        const int fc = FB * (int)rank + 4 * ch;
        float4 sw[kRowsPerThread], vw[kRowsPerThread];
#pragma unroll
        for (int q = 0; q < kRowsPerThread; ++q) {
            const int i = kSplit * q + 2 * w + par;  // the token's row (old contents) is replaced below
            sw[q] = ld4(scs + (size_t)i * P + fc);
            vw[q] = ld4(kvs + (size_t)i * P + fc);
        }
        const int qs = slot - 2 * w - par;
        const bool has_token = qs >= 0 && qs % kSplit == 0;  // this thread's rows include the token's
        float4 vk = make_float4(0.f, 0.f, 0.f, 0.f), sk = vk;
        if (has_token) {
            const float4 v = ld4(p.kv + (size_t)row * P + fc);
            const float4 s0 = ld4(p.score + (size_t)row * P + fc);
            const float4 a = ld4(p.ape + (size_t)token * P + fc);
            float* vo = &vk.x;
            float* so = &sk.x;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float vv = comp(v, k);
                const float ss = comp(s0, k) + comp(a, k);
                const bool ok = finite_f(vv);
                vo[k] = ok ? vv : 0.0f;
                so[k] = ok && finite_f(ss) ? ss : __int_as_float(0x7FC00000);
            }
            st4(kvs + (size_t)slot * P + fc, vk);
            st4(scs + (size_t)slot * P + fc, sk);
        }
#pragma unroll
        for (int q = 0; q < kRowsPerThread; ++q)
            if (kSplit * q + 2 * w + par == slot) {
                sw[q] = sk;
                vw[q] = vk;
            }
        writer = w == 0 && par == 0;
        wcol = ch;
        wf0 = fc;
        if (!complete) {
            if (writer) *reinterpret_cast<uint2*>(p.out + (size_t)row * D + wf0) = make_uint2(0u, 0u);
            return;
        }
        float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < kRowsPerThread; ++q)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float s = comp(sw[q], k);
                bad |= (s != s || s == INFINITY || !finite_f(comp(vw[q], k))) ? 1u : 0u;
                m[k] = fmaxf(m[k], s);
            }
#pragma unroll
        for (int k = 0; k < 4; ++k) m[k] = fmaxf(m[k], __shfl_xor_sync(0xFFFFFFFFu, m[k], kSplit));
        bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, kSplit);
        if (par == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) sm.red_m[w][ch][k] = m[k];
            sm.red_b[w][ch] = bad;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float mm = sm.red_m[0][ch][k];
            for (int w2 = 1; w2 < kCompThreads / 32; ++w2) mm = fmaxf(mm, sm.red_m[w2][ch][k]);
            m[k] = mm;
        }
#pragma unroll
        for (int q = 0; q < kRowsPerThread; ++q)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float e = expf(comp(sw[q], k) - m[k]);
                den[k] += e;
                num[k] = fmaf(e, comp(vw[q], k), num[k]);
            }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            den[k] += __shfl_xor_sync(0xFFFFFFFFu, den[k], kSplit);
            num[k] += __shfl_xor_sync(0xFFFFFFFFu, num[k], kSplit);
        }
        if (par == 0)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                sm.red_d[w][ch][k] = den[k];
                sm.red_n[w][ch][k] = num[k];
            }
        __syncthreads();
        if (writer) {
            bad = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) den[k] = num[k] = 0.0f;
            for (int w2 = 0; w2 < kCompThreads / 32; ++w2) {  // warp order
                bad |= sm.red_b[w2][ch];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    den[k] += sm.red_d[w2][ch][k];
                    num[k] += sm.red_n[w2][ch][k];
                }
            }
        }
    } else {
        // ---- ratio 4: the column's 16 threads split the window's rows.
        // 2a. pooling: this thread takes window rows sub, sub + 16, ...; all of
        // them but the token's own row are loaded before anything is used, so their
        // round trips overlap each other and the token's.
        float4 sw[kRowsPerThread], vw[kRowsPerThread];
        if (complete && active) {
#pragma unroll
            for (int q = 0; q < kRowsPerThread; ++q) {
                const int i = sub + q * kSplit;
                if (i < items && i != slot) {
                    const int sf = (overlap && i >= R) ? D + f0 : f0;
                    sw[q] = ld4(scs + (size_t)i * P + sf);
                    vw[q] = ld4(kvs + (size_t)i * P + sf);
                }
            }
        }

        // 1. the token's state row, for this column's features
        float4 vk = make_float4(0.f, 0.f, 0.f, 0.f), sk = vk;
        if (active && sub < coff) {
            const int sf = sub * D + f0;
            const float4 v = ld4(p.kv + (size_t)row * P + sf);
            const float4 s0 = ld4(p.score + (size_t)row * P + sf);
            const float4 a = ld4(p.ape + (size_t)token * P + sf);
            float* vo = &vk.x;
            float* so = &sk.x;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float vv = comp(v, k);
                const float ss = comp(s0, k) + comp(a, k);
                const bool ok = finite_f(vv);
                vo[k] = ok ? vv : 0.0f;
                so[k] = ok && finite_f(ss) ? ss : __int_as_float(0x7FC00000);
            }
            st4(kvs + (size_t)slot * P + sf, vk);
            st4(scs + (size_t)slot * P + sf, sk);
        }
        writer = active && sub == 0;
        wcol = col;
        wf0 = f0;
        if (!complete) {
            if (writer) *reinterpret_cast<uint2*>(p.out + (size_t)row * D + wf0) = make_uint2(0u, 0u);
            return;
        }

        // 2b. the token's row enters the window from the thread that wrote it:
        // the column's 16 threads are consecutive lanes of one warp, and the row's
        // features of this column belong to thread sub = 1 when the windows
        // overlap (the token's row reads features D + f0) and sub = 0 otherwise.
        {
            const int lane = t & 31;
            const int src = (lane & ~(kSplit - 1)) | (overlap ? 1 : 0);
            float4 vt, st;
            vt.x = __shfl_sync(0xFFFFFFFFu, vk.x, src);
            vt.y = __shfl_sync(0xFFFFFFFFu, vk.y, src);
            vt.z = __shfl_sync(0xFFFFFFFFu, vk.z, src);
            vt.w = __shfl_sync(0xFFFFFFFFu, vk.w, src);
            st.x = __shfl_sync(0xFFFFFFFFu, sk.x, src);
            st.y = __shfl_sync(0xFFFFFFFFu, sk.y, src);
            st.z = __shfl_sync(0xFFFFFFFFu, sk.z, src);
            st.w = __shfl_sync(0xFFFFFFFFu, sk.w, src);
#pragma unroll
            for (int q = 0; q < kRowsPerThread; ++q)
                if (sub + q * kSplit == slot) {
                    sw[q] = st;
                    vw[q] = vt;
                }
        }
        float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (active) {
#pragma unroll
            for (int q = 0; q < kRowsPerThread; ++q)
                if (sub + q * kSplit < items)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float s = comp(sw[q], k);
                        bad |= (s != s || s == INFINITY || !finite_f(comp(vw[q], k))) ? 1u : 0u;
                        m[k] = fmaxf(m[k], s);
                    }
        }
#pragma unroll
        for (int o = kSplit / 2; o > 0; o >>= 1) {
#pragma unroll
            for (int k = 0; k < 4; ++k) m[k] = fmaxf(m[k], __shfl_xor_sync(0xFFFFFFFFu, m[k], o));
            bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, o);
        }
        if (active) {
#pragma unroll
            for (int q = 0; q < kRowsPerThread; ++q)
                if (sub + q * kSplit < items)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float e = expf(comp(sw[q], k) - m[k]);
                        den[k] += e;
                        num[k] = fmaf(e, comp(vw[q], k), num[k]);
                    }
        }
#pragma unroll
        for (int o = kSplit / 2; o > 0; o >>= 1)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                den[k] += __shfl_xor_sync(0xFFFFFFFFu, den[k], o);
                num[k] += __shfl_xor_sync(0xFFFFFFFFu, num[k], o);
            }
    }
    float c[4];
    float sq = 0.0f;
    const float4 nrm = writer ? ld4(p.norm + wf0) : make_float4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float pooled = num[k] / den[k];
        const bool ok = finite_f(pooled);
        c[k] = bf16_round(ok ? pooled : 0.0f);
        bad |= (!ok || !finite_f(comp(nrm, k))) ? 1u : 0u;
        bad |= fabsf(comp(nrm, k)) > kNormSafe ? 2u : 0u;
        sq = fmaf(c[k], c[k], sq);
    }

    // ---- 3. RMS over the row: column -> CTA -> cluster, in fixed order ----------
    if (writer) {
        sm.col_sq[wcol] = sq;
        sm.col_bad[wcol] = bad;
    }
    __syncthreads();
    if (t == 0) {
        float s = 0.0f;
        uint32_t b = 0;
        for (int j = 0; j < ncol; ++j) {
            s += sm.col_sq[j];
            b |= sm.col_bad[j];
        }
        // Push this CTA's share into every CTA (itself too): 8 bytes each, counted
        // on the receiver's bar_sq, which expects 8 bytes from every rank.
        mbar_arrive_expect_tx(&sm.bar_sq, 8 * kCompCluster);
        for (int r = 0; r < kCompCluster; ++r) {
            st_async_remote(&sm.sq_all[rank], __float_as_uint(s), &sm.bar_sq, (uint32_t)r);
            st_async_remote(&sm.bad_all[rank], b, &sm.bar_sq, (uint32_t)r);
        }
    }
    mbar_wait_cluster(&sm.bar_sq, 0, nullptr);
    float total = 0.0f;
    uint32_t any_bad = 0;
    for (int r = 0; r < kCompCluster; ++r) {  // rank order
        total += __uint_as_float(sm.sq_all[r]);
        any_bad |= sm.bad_all[r];
    }
    bool invalid = (any_bad & 1u) != 0 || !finite_f(total);
    const float scale = invalid ? 0.0f : 1.0f / sqrtf(total / (float)D + p.eps);
    if (!finite_f(scale)) invalid = true;
    float y[4];
    uint32_t ybad = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        y[k] = c[k] * scale * comp(nrm, k);
        ybad |= finite_f(y[k]) ? 0u : 1u;
    }
    // |c scale| <= sqrt(D) (every c^2 is at most the total), so a non-finite
    // output needs a norm above kNormSafe somewhere in the row. Only then does
    // the cluster exchange the output flags; every CTA sees the same bits and
    // takes the same branch.
    if (any_bad & 2u) {
        if (t == 0) sm.cta_ybad = 0;
        __syncthreads();
        if (writer && ybad) atomicOr(&sm.cta_ybad, 1u);
        __syncthreads();
        if (t == 0) {
            mbar_arrive_expect_tx(&sm.bar_yb, 4 * kCompCluster);
            for (int r = 0; r < kCompCluster; ++r)
                st_async_remote(&sm.yb_all[rank], sm.cta_ybad, &sm.bar_yb, (uint32_t)r);
        }
        mbar_wait_cluster(&sm.bar_yb, 0, nullptr);
        for (int r = 0; r < kCompCluster; ++r) invalid = invalid || sm.yb_all[r];
    }

    if (writer) {
        __align__(8) __nv_bfloat16 o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = __float2bfloat16_rn(invalid ? 0.0f : y[k]);
        *reinterpret_cast<uint2*>(p.out + (size_t)row * D + wf0) = *reinterpret_cast<const uint2*>(o);
    }

    // ---- 4. overlapping windows: the current block becomes the previous one ---
    if (overlap && active && sub < 2 * R) {
        const int i = sub >> 1, h = sub & 1;  // previous row i, feature half h
        const size_t dst = (size_t)i * P + h * D + f0, src = (size_t)(R + i) * P + h * D + f0;
        st4(kvs + dst, ld4(kvs + src));
        st4(scs + dst, ld4(scs + src));
    }
    // No CTA reads another's shared memory, and every store into this CTA's
    // has landed (every barrier it waited on completed; all CTAs skip or run
    // the output-flag exchange together): the CTAs leave independently.
}

cudaError_t launch_compressor(const CompressorParams& p, cudaStream_t stream, bool pdl) {
    if (p.rows == 0) return cudaSuccess;
    if (p.ratio == 4)
        return launch_kernel(compressor_kernel<kRowsRatio4>, dim3(p.rows * kCompCluster), dim3(kCompThreads), 0,
                             stream, pdl, p);
    if (p.ratio == 128)
        return launch_kernel(compressor_kernel<kRowsRatio128>, dim3(p.rows * kCompCluster), dim3(kCompThreads), 0,
                             stream, pdl, p);
    return cudaErrorInvalidValue;  // the boundary admits ratios 4 and 128 only
}

}  // namespace dsrows
