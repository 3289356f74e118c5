// Device helpers for sm_103a: mbarriers, bulk (TMA 1-D) copies global -> shared, thread-block
// cluster barriers and distributed shared memory, warp reductions and scans.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace spec {

constexpr int kWarp = 32;

// ---------------------------------------------------------------- special registers

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

// Waits for the phase to complete, for at most `limit_ns` nanoseconds. Returns false on
// timeout: the caller records an error and carries on along its normal control flow (it
// still reaches every block and cluster barrier, so no other thread is left waiting).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t phase,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, phase)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, phase)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// try_wait that lets the hardware suspend the thread for up to `hint_ns` while the phase is
// incomplete (the thread resumes as soon as it completes), so waiting warps do not spin.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t phase, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(phase), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Waits for the phase, suspended between attempts; gives up after `max_tries` attempts of up to
// `hint_ns` each (seconds in total) and returns false. The caller records the error and still
// reaches every block and cluster barrier, so no peer is left waiting.
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint64_t *bar, uint32_t phase, uint32_t hint_ns,
                                                        int max_tries) {
    for (int t = 0; t < max_tries; ++t)
        if (mbar_try_wait_sleep(bar, phase, hint_ns)) return true;
    return false;
}

// try_wait with acquire at cluster scope: the waiter sees what other CTAs of the cluster wrote
// before their (release) arrivals. Suspends for up to `hint_ns` while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t phase, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(phase), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t phase, uint32_t hint_ns,
                                                          int max_tries) {
    for (int t = 0; t < max_tries; ++t)
        if (mbar_try_wait_cluster(bar, phase, hint_ns)) return true;
    return false;
}

// Arrive on the mbarrier at a shared::cluster address (this CTA's or another's), releasing this
// thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 16-byte store into another CTA's shared memory (a shared::cluster address) that completes its
// bytes on that CTA's mbarrier (also a shared::cluster address). Asynchronous: the receiver sees
// the data once the barrier's phase completes.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, uint4 v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote_addr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
                 : "memory");
}

// ---------------------------------------------------------------- named barriers
// Barrier `id` (1..15) completes when `count` threads (a multiple of 32) have arrived: bar_sync
// arrives and waits, bar_arrive only arrives. What a thread wrote before arriving is visible to
// the threads that waited. The non-aligned forms: the threads of a warp may arrive apart.
__device__ __forceinline__ void bar_sync(int id, int count) {
    asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int count) {
    asm volatile("barrier.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar` with a byte count.
// dst, src and bytes must be multiples of 16. The policy evicts the streamed lines first.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Prefetch `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// A plain arrival (release, CTA scope) on a local mbarrier.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialisation may start before the kernel ahead
// of it in the stream finishes; it must call griddep_wait() before it reads anything that
// kernel writes. griddep_launch_dependents() lets the kernel behind this one start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- cluster

// The two halves of a cluster barrier: every thread of the cluster arrives once, then waits once
// (possibly much later) before it arrives again.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_map(const void *local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
    return r;
}
__device__ __forceinline__ double dsmem_ld_f64(uint32_t addr) {
    double v;
    asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ int32_t dsmem_ld_s32(uint32_t addr) {
    int32_t v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// ---------------------------------------------------------------- warp collectives

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_min_i32(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// Inclusive scan over the lanes, in lane order.
__device__ __forceinline__ double warp_inclusive_scan_f64(double v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        double n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Elementwise max of two packed bfloat16 pairs; a NaN operand yields the other operand.
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// the same with a NaN operand giving NaN
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// ---- the debug build (-DSPEC_DEBUG): index checks that record instead of trapping
// SPEC_IN(i, n, code) is true when 0 <= i < n. In the debug build a failed check records, in this
// translation unit's words, the first failure's code (which array), source line and index, counts
// every failure, and the caller skips the access; spec_debug_fetch() reads and clears the words.
// In the release build it is the constant true and costs nothing.
enum : int {
    DBG_LOGITS = 1,     // a target or draft row, or a vector beyond a row
    DBG_RECORDS = 2,    // per-chunk workspace (statistics records, alpha and residual shares)
    DBG_ROWS = 3,       // per-row workspace (values, decisions, draft-token records, item results)
    DBG_OUT_ROWS = 4,   // per-row outputs (out_tokens, alpha_rows, rho_rows, resid_rows)
    DBG_OUT_REQS = 5,   // per-request outputs and counters
    DBG_PACKED = 6,     // the compaction's packed outputs
    DBG_CUT = 7,        // the truncation kernel's rows and cuts
};
#ifdef SPEC_DEBUG
static __device__ unsigned int g_spec_dbg[4];  // first code, its line, its index, failures
static __device__ __noinline__ bool spec_dbg_fail(int code, int line, long long idx) {
    if (atomicCAS(&g_spec_dbg[0], 0u, static_cast<unsigned>(code)) == 0u) {
        g_spec_dbg[1] = static_cast<unsigned>(line);
        g_spec_dbg[2] = static_cast<unsigned>(idx);
    }
    atomicAdd(&g_spec_dbg[3], 1u);
    return false;
}
#define SPEC_IN(i, n, code)                                                                          \
    ((static_cast<long long>(i) >= 0 && static_cast<long long>(i) < static_cast<long long>(n))      \
         ? true                                                                                      \
         : ::spec::spec_dbg_fail((code), __LINE__, static_cast<long long>(i)))
// reads and clears this translation unit's words (host)
static inline cudaError_t spec_dbg_take(unsigned int out[4]) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_spec_dbg, sizeof(unsigned int) * 4);
    if (e != cudaSuccess) return e;
    const unsigned int zero[4] = {0u, 0u, 0u, 0u};
    return cudaMemcpyToSymbol(g_spec_dbg, zero, sizeof(zero));
}
#else
#define SPEC_IN(i, n, code) true
#endif

// base-2 exponential on the special-function unit (relative error about 2 ulp)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Host: launch `kernel` so that it may start while the kernel ahead of it in `stream` is still
// running (programmatic stream serialisation); the kernel must call griddep_wait() first thing
// before touching that kernel's outputs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace spec
