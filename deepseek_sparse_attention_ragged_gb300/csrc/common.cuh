// Shared constants, launch tables and sm_103a PTX helpers for the dsrows kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "dsrows.h"

namespace dsrows {

constexpr int kRowsMax = DS_ROWS_MAX;
constexpr int kIdxHeads = DS_INDEX_HEADS;
constexpr int kIdxDim = DS_INDEX_DIM;
constexpr int kTopK = DS_TOPK;
constexpr int kHeads = DS_HEADS;
constexpr int kDim = DS_DIM;

// Device-side status bits written into the workspace control header.
constexpr uint32_t kStatusWaitTimeout = DS_STATUS_WAIT_TIMEOUT;  // a bounded wait gave up
constexpr uint32_t kStatusCandOverflow = DS_STATUS_OVERFLOW;      // internal: counts disagreed

// Time budget of every spin-wait on an mbarrier (nanoseconds of %globaltimer).
constexpr uint64_t kWaitBudgetNs = 2000000000ull;

// ---------------------------------------------------------------------------
// Workspace layout (bytes, all 256-aligned)
// ---------------------------------------------------------------------------
//   [0, 256)                 control: u32 status, pad
//   hist   [8][2048] u32     level-0 histogram of score keys per entry
//   flags  [8][64 + 1] u32   per-entry, per-head attention invalid bits, row bits
//   part   [chunks][2][...]  attention partials: m[32], l[32], acc[32][512] per
//                            (128-slot chunk, head half)
//   scores [8][stride] f32   indexer scores (decode only)
constexpr int kHistBins = 2048;
constexpr int kAttnChunksMax = 8;                    // bound on a row's attention chunks
// One attention partial (a chunk of one head half): m[32], l[32], acc[32][512] (fp32).
constexpr size_t kPartFloats = 32 + 32 + (size_t)(kHeads / 2) * kDim;

// ---------------------------------------------------------------------------
// PTX helpers (device)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same, acquiring at cluster scope: what the arrivals of other CTAs of the
// cluster released (their writes to this CTA's or global memory) is visible.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* status) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t start = global_timer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (global_timer_ns() - start > kWaitBudgetNs) {
            if (status) atomicOr(status, kStatusWaitTimeout);
            return false;
        }
    }
}

// The shared::cluster address of this CTA's shared-memory address `smem_addr`
// in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t smem_addr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_addr), "r"(rank));
    return d;
}

// A cluster barrier in two halves: arrive (releasing this thread's earlier
// writes to the cluster) and wait (acquiring the others'); every thread of the
// CTA executes both, and may do CTA-local work in between.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Global flag accesses at GPU scope: a release store after the data it
// announces, an acquire load before the data is read.
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Plain stores to distributed shared memory (a shared::cluster address); they
// become visible to the target CTA at the next cluster barrier.
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, uint64_t v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Store `v` to the word at the same offset as `dst` in CTA `rank` of the
// cluster, completing 4 bytes of transaction on that CTA's mbarrier at the same
// offset as `bar`.
__device__ __forceinline__ void st_async_remote(uint32_t* dst, uint32_t v, uint64_t* bar, uint32_t rank) {
    uint32_t d, b;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_u32(dst)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(b) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(d), "r"(v), "r"(b)
                 : "memory");
}

// The same for an 8-byte value.
__device__ __forceinline__ void st_async_remote_u64(uint64_t* dst, uint64_t v, uint64_t* bar, uint32_t rank) {
    uint32_t d, b;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_u32(dst)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(b) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(d), "l"(v), "r"(b)
                 : "memory");
}

// Wait for the phase of `parity` to complete, for at most `budget_ns`.
// Returns false (and records kStatusWaitTimeout) when the budget runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status,
                                          uint64_t budget_ns = kWaitBudgetNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - start > budget_ns) {
            if (status) atomicOr(status, kStatusWaitTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

// Order this thread's earlier generic-proxy accesses of shared memory before
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global to this CTA's shared memory, completing on `bar` (complete_tx).
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Store with an L2 cache-eviction policy (createpolicy).
__device__ __forceinline__ void st_global_hint(float* p, float v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy) : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2D tiled TMA load into shared memory, completing on `bar` (complete_tx).
// x (innermost, elements) must be a multiple of 16 bytes / element size.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// ---- tcgen05 (5th-generation tensor cores, accumulators in TMEM) ----------

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp gets lane (base + i).
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 32 bits, 8 consecutive columns.
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}

// 32 lanes x 32 bits, 32 consecutive columns.
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): K-major, 128-byte swizzle.
// Rows of 128 B, 8-row groups 1024 B apart (SBO); LBO unused for this layout.
__device__ __forceinline__ uint64_t smem_desc_sw128_kmajor(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);         // start address, bits [0,14)
    d |= (uint64_t)(16 >> 4) << 16;                       // leading byte offset (ignored)
    d |= (uint64_t)(1024 >> 4) << 32;                     // stride byte offset
    d |= (uint64_t)1 << 46;                               // descriptor version (tcgen05)
    d |= (uint64_t)2 << 61;                               // layout: SWIZZLE_128B
    return d;
}

// Shared-memory matrix descriptor: MN-major, 128-byte swizzle. Atoms of 64
// MN-elements (128 B) x 8 K-rows (1024 B); LBO = bytes between atoms along
// MN, SBO = bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t smem_desc_sw128_mnmajor(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);         // start address, bits [0,14)
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;           // leading byte offset
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;           // stride byte offset
    d |= (uint64_t)1 << 46;                               // descriptor version (tcgen05)
    d |= (uint64_t)2 << 61;                               // layout: SWIZZLE_128B
    return d;
}

// Instruction descriptor bit: A is MN-major (transposed) instead of K-major.
constexpr uint32_t kIdescAMnMajor = 1u << 15;

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// Launch `kernel` on `stream`; with `pdl` the launch may begin before the previous
// kernel in the stream completes (programmatic dependent launch): the kernel
// must execute pdl_wait() before it reads anything that kernel produced.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device. The attribute belongs to the device's context, so it is set once per
// device (bit d of `done`); threads that race here only repeat the same call.
template <typename... KArgs>
inline cudaError_t set_smem_limit_once(void (*kernel)(KArgs...), size_t bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t)1 << dev : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return err;
}

// Programmatic dependent launch controls (no-ops for a launch without PDL).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Sort 512 64-bit values in descending order with NT = 256 or 512 threads;
// thread t holds the values of positions t + k NT in x[k]; `buf` is 512 words
// of shared memory. Zero may repeat (padding); other values must be distinct.
// Each warp sorts 32-value runs with a shuffle bitonic network; four merge
// rounds then pair the sorted runs (32 -> 64 -> 128 -> 256 -> 512): a value's
// place in the merged run is its place in its own run plus the partner run's
// values that go before it (a binary search). On return x[k] is the value of
// rank t + k NT.
template <int NT>
__device__ __forceinline__ void sort512_desc(uint64_t (&x)[512 / NT], uint64_t* buf) {
    constexpr int PER = 512 / NT;
    const int t = threadIdx.x, lane = t & 31;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
#pragma unroll
        for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
            for (int j = k >> 1; j > 0; j >>= 1) {
                const uint64_t y = __shfl_xor_sync(0xFFFFFFFFu, x[q], j);
                const bool desc = (lane & k) == 0;
                const bool lower = (lane & j) == 0;
                const uint64_t hi = x[q] > y ? x[q] : y, lo = x[q] > y ? y : x[q];
                x[q] = (lower == desc) ? hi : lo;
            }
        }
    }
    uint32_t pos[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) pos[q] = lane;  // place inside the current run
#pragma unroll
    for (int run = 32; run < 512; run <<= 1) {
        __syncthreads();
#pragma unroll
        for (int q = 0; q < PER; ++q) buf[t + q * NT] = x[q];
        __syncthreads();
        uint32_t dst[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const uint32_t p = (uint32_t)(t + q * NT);
            const uint32_t base = p & ~(uint32_t)(2 * run - 1);
            const bool first = (p & run) == 0;
            const uint64_t* partner = buf + base + (first ? run : 0);
            // Partner values that go before x: the larger ones, and for the second
            // run of the pair also the equal ones, so equal values keep distinct places.
            uint32_t c = 0;
#pragma unroll
            for (int step = 512; step > 0; step >>= 1) {
                if (step <= run && c + step <= (uint32_t)run) {
                    const uint64_t y = partner[c + step - 1];
                    if (y > x[q] || (!first && y == x[q])) c += step;
                }
            }
            dst[q] = base + pos[q] + c;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < PER; ++q) buf[dst[q]] = x[q];
        __syncthreads();
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            x[q] = buf[t + q * NT];
            pos[q] = (uint32_t)(t + q * NT) & (uint32_t)(2 * run - 1);
        }
    }
}

// Order-preserving map of a finite fp32 score to u32 (larger score -> larger key);
// -0.0 maps like +0.0 so that the two tie.
__device__ __forceinline__ uint32_t score_key(float s) {
    uint32_t u = __float_as_uint(s);
    if ((u & 0x7FFFFFFFu) == 0) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ bool finite_f(float x) { return (__float_as_uint(x) & 0x7F800000u) != 0x7F800000u; }

// The composite that orders (score desc, index asc) as one descending u64.
__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t index) {
    return ((uint64_t)key << 32) | (uint64_t)(~index);
}

}  // namespace dsrows
