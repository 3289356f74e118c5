// Batched speculative-decoding verifier for GB300 (sm_103a): spec_verify.
//
// The rule is the one of "SOTA-227: Decode with a draft model and an accept-reject rule"
// ("What to do", steps 3-4) and SDCP Rules 1 and 2 ("Acceptance Rules"); the C ABI and its
// conventions are documented in include/spec_verify.h.
//
// Two kernels per call: the per-position kernel verifies every (request, position) on a
// persistent grid of thread-block clusters (spec_stream_kernel.cuh when a CTA's slice of a row
// fits its tiles, else spec_rows_kernel.cuh; both on spec_rows.cuh); the selection kernel walks
// each request's accept flags left to right (a warp ballot), picks the candidate of the first
// rejection or the bonus, applies stop-token / max_new truncation and reduces alpha for the
// gamma controller.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "spec_device.cuh"
#include "spec_verify.h"

#include "spec_rows_kernel.cuh"
#include "spec_stream_kernel.cuh"
#include "spec_trunc.cuh"
#include "spec_tail.cuh"

namespace spec {

// ------------------------------------------------------------------------------------------
// Per-request selection: the first rejection, the emitted tokens, stopping, alpha reduction.

__global__ void __launch_bounds__(kFinThreads) spec_select_kernel(const FinParams P) { (void)select_body(P); }

// ------------------------------------------------------------------------------------------
// Host side

struct WsLayout {
    size_t flag, tok, status, fb, prob, margin, alpha, cut, total;
};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static WsLayout ws_layout(int32_t B, int32_t total_rows) {
    WsLayout L;
    const size_t T = static_cast<size_t>(total_rows > 0 ? total_rows : 0);
    const size_t nd = total_rows > B ? static_cast<size_t>(total_rows - B) : 0;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    L.flag = take(T * 4);
    L.tok = take(T * 4);
    L.status = take(T * 4);
    L.fb = take(T * 4);
    L.prob = take(T * 4);
    L.margin = take(T * 4);
    L.alpha = take((nd > 0 ? nd : 1) * 4);
    L.cut = take(T * 8);  // top-k / top-p cut per target row
    L.total = off;
    return L;
}

using RowsKernel = void (*)(const RowsParams);

template <int DT>
static RowsKernel rows_kernel_for(int nvt) {
    switch (nvt) {
        case 2: return spec_rows_kernel<DT, 2>;
        case 4: return spec_rows_kernel<DT, 4>;
        default: return spec_rows_kernel<DT, kMaxNvt>;
    }
}

// One cluster size of the per-position kernel: its slices, registers per thread and the number
// of clusters that can be resident at once (occupancy API; one CTA per SM).
struct ClusterOption {
    int C = 0;
    int nvt = 0;
    int slice_vecs_max = 0;
    size_t smem = 0;
    int active = 0;
    int per_sm = 1;  // CTAs resident per SM
};

struct ShapeTable {
    int dev = -1, nvec_row = -1;
    ClusterOption opt[5];   // rows kernel, C = 1, 2, 4, 8, 16
    ClusterOption sopt[5];  // streaming kernel, C = 1, 2, 4, 8, 16
};

// Resident clusters of C CTAs of kernel k (`block` threads, `smem` bytes of dynamic shared memory).
static int clusters_resident(const void *k, int C, int block, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(C * 16, 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(block), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, k, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return active;
}

template <int DT>
static cudaError_t shape_table(int nvec_row, ShapeTable &out) {
    static std::mutex mu;
    static ShapeTable cached;
    static bool attrs_set[4] = {false, false, false, false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (cached.dev == dev && cached.nvec_row == nvec_row) {
        out = cached;
        return cudaSuccess;
    }
    int max_optin = 0;
    e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    ShapeTable t;
    t.dev = dev;
    t.nvec_row = nvec_row;
    for (int ci = 0; ci < 5; ++ci) {
        const int C = 1 << ci;
        ClusterOption &o = t.opt[ci];
        if (C > nvec_row) continue;
        const int slice = (nvec_row + C - 1) / C;
        // vectors per data thread: 2, 4 or 5 (the largest slice that fits the registers)
        const int nvt = (slice <= 2 * kThreads) ? 2 : (slice <= 4 * kThreads) ? 4 : kMaxNvt;
        if (nvt * kThreads < slice) continue;  // a slice must fit the registers of one CTA
        const RowsKernel k = rows_kernel_for<DT>(nvt);
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        // the row ring, then the exchange slots (kNMS exchanges x C records)
        const size_t smem = static_cast<size_t>(kRing) * slice * 16 + static_cast<size_t>(kNMS) * kMaxCluster * sizeof(Msg);
        if (smem + fa.sharedSizeBytes > static_cast<size_t>(max_optin)) continue;
        const int ki = (nvt == 2) ? 0 : (nvt == 4) ? 1 : 2;
        if (!attrs_set[ki]) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     max_optin - static_cast<int>(fa.sharedSizeBytes));
            if (e != cudaSuccess) return e;
            attrs_set[ki] = true;
        }
        const int active = clusters_resident(reinterpret_cast<const void *>(k), C, kBlock, smem);
        if (active <= 0) continue;
        o.C = C;
        o.nvt = nvt;
        o.slice_vecs_max = slice;
        o.smem = smem;
        o.active = active;
        o.per_sm = 2;
    }
    // the streaming kernel: one CTA per SM, a slice of at most Geo<DT>::kMaxTiles tiles
    static bool stream_attrs_set = false;
    for (int ci = 0; ci < 5; ++ci) {
        const int C = 1 << ci;
        ClusterOption &o = t.sopt[ci];
        if (C > nvec_row) continue;
        const int slice = (nvec_row + C - 1) / C;
        if (slice > Geo<DT>::kMaxTiles * Geo<DT>::kTileVecs) continue;
        const RowsKernel k = spec_stream_kernel<DT>;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        const size_t smem = Geo<DT>::kDynSmem;
        if (smem + fa.sharedSizeBytes > static_cast<size_t>(max_optin)) continue;
        if (!stream_attrs_set) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     max_optin - static_cast<int>(fa.sharedSizeBytes));
            if (e != cudaSuccess) return e;
            stream_attrs_set = true;
        }
        const int active = clusters_resident(reinterpret_cast<const void *>(k), C, kStreamBlock, smem);
        if (active <= 0) continue;
        o.C = C;
        o.nvt = 0;
        o.slice_vecs_max = slice;
        o.smem = smem;
        o.active = active;
        o.per_sm = 1;
    }
    cached = t;
    out = t;
    return cudaSuccess;
}

// The persistent grid. The kernel: the streaming kernel whenever a CTA's slice fits its tiles
// (pass 2 of an item overlaps the next item's pass 1; measured faster on all five workloads),
// else the rows kernel. The cluster size: the one that keeps the most SMs busy on this many
// target rows (a cluster lives in one GPC, so large clusters strand SMs; too few rows leave
// clusters idle); ties go to the smaller cluster (fewer barriers per logit).
// SPEC_VERIFY_KERNEL=rows or =stream in the environment restricts the choice to one kernel
// (read on every call).
struct Plan {
    ClusterOption opt;
    bool streaming = false;
    bool ok = false;
};

template <int DT>
static Plan choose_plan(int nvec_row, int total_rows, int B) {
    Plan plan;
    ShapeTable t;
    if (shape_table<DT>(nvec_row, t) != cudaSuccess) return plan;
    const char *force = std::getenv("SPEC_VERIFY_KERNEL");
    const bool only_rows = force && std::strcmp(force, "rows") == 0;
    const bool only_stream = force && std::strcmp(force, "stream") == 0;
    (void)B;
    for (int pass = 0; pass < 2 && !plan.ok; ++pass) {
        const bool streaming = pass == 0;
        if ((streaming && only_rows) || (!streaming && only_stream)) continue;
        long long best_score = 0;
        for (int ci = 0; ci < 5; ++ci) {
            const ClusterOption &o = streaming ? t.sopt[ci] : t.opt[ci];
            if (o.C == 0 || o.active <= 0) continue;
            // SMs covered, in units of 1/2 SM
            const long long score = static_cast<long long>(std::min(o.active, total_rows)) * o.C * 2 / o.per_sm;
            if (score > best_score) {
                best_score = score;
                plan.opt = o;
                plan.streaming = streaming;
                plan.ok = true;
            }
        }
    }
    return plan;
}

template <int DT>
static spec_status launch_rows(const RowsParams &P, cudaStream_t stream) {
    const Plan plan = choose_plan<DT>(P.nvec_row, P.total_rows, P.B);
    if (!plan.ok) return SPEC_ERR_UNSUPPORTED;
    const ClusterOption &o = plan.opt;
    RowsParams Q = P;
    Q.slice_vecs_max = o.slice_vecs_max;
    Q.nclusters = std::min(o.active, P.total_rows);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = o.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(Q.nclusters * o.C), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(plan.streaming ? kStreamBlock : kBlock), 1, 1);
    cfg.dynamicSmemBytes = o.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const RowsKernel k = plan.streaming ? spec_stream_kernel<DT> : rows_kernel_for<DT>(o.nvt);
    if (cudaLaunchKernelEx(&cfg, k, Q) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}

}  // namespace spec

using namespace spec;

extern "C" size_t spec_verify_workspace_size(int32_t B, int32_t V, int32_t total_rows, spec_dtype dtype) {
    (void)V;
    (void)dtype;
    return ws_layout(B, total_rows).total;
}

// The round's tail in one kernel: the selection, then (its outputs visible to the whole CTA) the
// compaction, then the gamma choice on one thread.
__global__ void __launch_bounds__(kFinThreads) spec_round_tail_kernel(const FinParams F, const CompactParams C,
                                                                      const GammaParams G) {
    const bool offsets_ok = select_body(F);
    __syncthreads();
    // the same offsets (same array, same B and total_rows) need no second check
    compact_body(C, false, (C.row_off == F.row_off && C.B == F.B && C.total_rows == F.total_rows) ? (offsets_ok ? 1 : 0) : -1);
    __syncthreads();
    if (threadIdx.x == 0) gamma_body(G);
}

// spec_verify's checks and launches; with C and G, the tail kernel of a round in place of the
// selection kernel. Nothing is enqueued when a check fails.
static spec_status verify_enqueue(const spec_verify_args *a, void *workspace, size_t workspace_bytes,
                                  cudaStream_t stream, const CompactParams *C, const GammaParams *G) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->B < 1 || a->V < 1 || a->K_max < 0 || a->K_max > 64 || a->total_rows < a->B) return SPEC_ERR_INVALID_ARG;
    if (static_cast<int64_t>(a->total_rows) > static_cast<int64_t>(a->B) * (a->K_max + 1)) return SPEC_ERR_INVALID_ARG;
    if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (!a->target_logits || !a->row_off || !a->uniforms || !a->accept_len || !a->out_tokens || !a->req_status)
        return SPEC_ERR_INVALID_ARG;
    const bool has_drafts = a->total_rows > a->B;
    if (has_drafts && (!a->draft_logits || !a->draft_tokens)) return SPEC_ERR_INVALID_ARG;
    const size_t eb = (a->dtype == SPEC_BF16) ? 2 : 4;
    const size_t row_bytes = eb * static_cast<size_t>(a->V);
    if (row_bytes % 16 != 0) return SPEC_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(a->target_logits) % 16 != 0) return SPEC_ERR_UNSUPPORTED;
    if (has_drafts && reinterpret_cast<uintptr_t>(a->draft_logits) % 16 != 0) return SPEC_ERR_UNSUPPORTED;
    if (row_bytes / 16 > static_cast<size_t>(INT_MAX)) return SPEC_ERR_UNSUPPORTED;
    if (!a->temperature && !(a->temperature_scalar >= 0.0f && std::isfinite(a->temperature_scalar)))
        return SPEC_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(a->B, a->total_rows);
    if (!workspace || workspace_bytes < L.total || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return SPEC_ERR_WORKSPACE;

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    RowsParams P = {};
    P.target = a->target_logits;
    P.draft = a->draft_logits;
    P.row_off = a->row_off;
    P.draft_tokens = a->draft_tokens;
    P.uniforms = a->uniforms;
    P.temperature = a->temperature;
    P.temperature_scalar = a->temperature_scalar;
    P.B = a->B;
    P.V = a->V;
    P.K_max = a->K_max;
    P.total_rows = a->total_rows;
    P.nvec_row = static_cast<int32_t>(row_bytes / 16);
    P.item_flag = reinterpret_cast<int32_t *>(ws + L.flag);
    P.item_tok = reinterpret_cast<int32_t *>(ws + L.tok);
    P.item_status = reinterpret_cast<int32_t *>(ws + L.status);
    P.item_fb = reinterpret_cast<int32_t *>(ws + L.fb);
    P.item_prob = reinterpret_cast<float *>(ws + L.prob);
    P.item_margin = reinterpret_cast<float *>(ws + L.margin);
    P.alpha_ws = reinterpret_cast<float *>(ws + L.alpha);
    P.alpha_rows = a->alpha_rows;
    P.rho_rows = a->rho_rows;
    P.resid_rows = a->resid_rows;
    P.top_p = a->top_p;
    P.trunc = nullptr;
    if (a->top_k || a->top_p) {
        // top-k / top-p: the cut of every target row, before the per-position kernel reads it
        TruncParams Tp = {};
        Tp.target = a->target_logits;
        Tp.row_off = a->row_off;
        Tp.temperature = a->temperature;
        Tp.temperature_scalar = a->temperature_scalar;
        Tp.top_k = a->top_k;
        Tp.top_p = a->top_p;
        Tp.B = a->B;
        Tp.V = a->V;
        Tp.total_rows = a->total_rows;
        Tp.cut = reinterpret_cast<int2 *>(ws + L.cut);
        if (a->dtype == SPEC_BF16)
            spec_trunc_kernel<SPEC_BF16><<<a->total_rows, kTruncThreads, 0, stream>>>(Tp);
        else
            spec_trunc_kernel<SPEC_F32><<<a->total_rows, kTruncThreads, 0, stream>>>(Tp);
        if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
        P.trunc = Tp.cut;
    }

    if (a->rows_event_begin && cudaEventRecord(a->rows_event_begin, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    const spec_status st = (a->dtype == SPEC_BF16) ? launch_rows<SPEC_BF16>(P, stream) : launch_rows<SPEC_F32>(P, stream);
    if (st != SPEC_OK) return st;
    if (a->rows_event_end && cudaEventRecord(a->rows_event_end, stream) != cudaSuccess) return SPEC_ERR_CUDA;

    FinParams F = {};
    F.row_off = a->row_off;
    F.draft_tokens = a->draft_tokens;
    F.stop_token = a->stop_token;
    F.max_new = a->max_new;
    F.B = a->B;
    F.K_max = a->K_max;
    F.total_rows = a->total_rows;
    F.item_flag = P.item_flag;
    F.item_tok = P.item_tok;
    F.item_status = P.item_status;
    F.item_fb = P.item_fb;
    F.item_prob = P.item_prob;
    F.item_margin = P.item_margin;
    F.alpha_ws = P.alpha_ws;
    F.accept_len = a->accept_len;
    F.n_emitted = a->n_emitted;
    F.out_tokens = a->out_tokens;
    F.req_status = a->req_status;
    F.fallback = a->fallback;
    F.alpha_count = a->alpha_count;
    F.frontier_prob = a->frontier_prob;
    F.frontier_margin = a->frontier_margin;
    F.alpha_sum = a->alpha_sum;
    F.depth_reached = a->depth_reached;
    F.depth_accepted = a->depth_accepted;
    const cudaError_t e = (C && G) ? launch_after(spec_round_tail_kernel, dim3(1), dim3(kFinThreads), stream, F, *C, *G)
                                   : launch_after(spec_select_kernel, dim3(1), dim3(kFinThreads), stream, F);
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" spec_status spec_verify(const spec_verify_args *a, void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
    return verify_enqueue(a, workspace, workspace_bytes, stream, nullptr, nullptr);
}

extern "C" spec_status spec_verify_round(const spec_verify_args *a, void *workspace, size_t workspace_bytes,
                                         const spec_compact_args *compact, double alpha_prev, double c,
                                         int32_t gamma_min, int32_t gamma_max, int32_t *gamma_out,
                                         double *alpha_out, cudaStream_t stream) {
    if (!a || !compact) return SPEC_ERR_INVALID_ARG;
    CompactParams C;
    GammaParams G;
    spec_status st = compact_params(compact, C);
    if (st != SPEC_OK) return st;
    if (compact->B != a->B || compact->total_rows != a->total_rows) return SPEC_ERR_INVALID_ARG;
    st = gamma_params(a->alpha_sum, a->alpha_count, alpha_prev, c, gamma_min, gamma_max, gamma_out, alpha_out, G);
    if (st != SPEC_OK) return st;
    return verify_enqueue(a, workspace, workspace_bytes, stream, &C, &G);
}

extern "C" const char *spec_version(void) { return "spec-verify-gb300 0.1 (sm_103a)"; }

// ------------------------------------------------------------------------------------------
// spec_verify_noalloc: spec_verify for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they verify a round: a serving
// engine whose memory planner has already reserved every byte of the device, a plugin that
// runs inside another runtime's allocator or scheduler callbacks, or a latency-critical loop
// where an allocation's implicit synchronisation and possible failure are not acceptable.
// For them this entry point takes its workspace from a fixed array in the library's own
// device memory instead of from the caller.
//
// The array lives in every GPU that loads the library until the process exits. Its address
// is looked up once per device, on the first call made with that device current; make that
// first call before any stream capture. All calls share the one array and it keeps the last
// call's contents (the kernels write every workspace entry before reading it, so nothing
// needs clearing); calls that overlap on the GPU, on two streams or from two threads, race
// on it and must be serialised by the caller.

namespace spec {
constexpr int32_t kNoallocMaxRows = 16384;  // target rows per call: T = sum_i (K_i + 1)
constexpr size_t kNoallocScratchBytes = 9 * 65536;  // = workspace of kNoallocMaxRows rows
static __device__ __align__(256) unsigned char noalloc_scratch[kNoallocScratchBytes];

static std::mutex noalloc_mu;
static void *noalloc_ptr[64] = {nullptr};
}  // namespace spec

extern "C" spec_status spec_verify_noalloc(const spec_verify_args *a, cudaStream_t stream) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->total_rows > kNoallocMaxRows) return SPEC_ERR_UNSUPPORTED;  // beyond the fixed scratch
    const size_t need = ws_layout(a->B, a->total_rows).total;
    if (need > kNoallocScratchBytes) return SPEC_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPEC_ERR_CUDA;
    void *ptr = nullptr;
    {
        std::lock_guard<std::mutex> lock(noalloc_mu);
        if (!noalloc_ptr[dev]) {
            // host code must not use the array's name as a device address: ask the runtime
            if (cudaGetSymbolAddress(&noalloc_ptr[dev], noalloc_scratch) != cudaSuccess) {
                noalloc_ptr[dev] = nullptr;
                return SPEC_ERR_CUDA;
            }
        }
        ptr = noalloc_ptr[dev];
    }
    return spec_verify(a, ptr, kNoallocScratchBytes, stream);
}

extern "C" const char *spec_verify_plan(int32_t B, int32_t V, int32_t total_rows, spec_dtype dtype, int32_t *cluster,
                                        int32_t *clusters) {
    if (B <= 0 || V <= 0 || total_rows < B || (dtype != SPEC_BF16 && dtype != SPEC_F32)) return nullptr;
    const int per_vec = (dtype == SPEC_BF16) ? 8 : 4;
    if (V % per_vec != 0) return nullptr;
    const int nvec_row = V / per_vec;
    const Plan plan = (dtype == SPEC_BF16) ? choose_plan<SPEC_BF16>(nvec_row, total_rows, B)
                                           : choose_plan<SPEC_F32>(nvec_row, total_rows, B);
    if (!plan.ok) return nullptr;
    if (cluster) *cluster = plan.opt.C;
    if (clusters) *clusters = std::min(plan.opt.active, total_rows);
    return plan.streaming ? "spec_stream_kernel" : "spec_rows_kernel";
}
