// Batched speculative-decoding verifier for GB300 (sm_103a): spec_verify.
//
// The rule is the one of "SOTA-227: Decode with a draft model and an accept-reject rule"
// ("What to do", steps 3-4) and SDCP Rules 1 and 2 ("Acceptance Rules"); the C ABI and its
// conventions are documented in include/spec_verify.h.
//
// Four kernels per call (five with top-k / top-p, whose cut of each target row comes first), all in
// spec_kernels.cuh: the statistics kernel reads every logit once (pass 1) on a persistent grid; the
// decision kernel decides every (request, position) and marks each request's frontier; pass 2
// reads the pairs again (mostly from L2) for alpha and the frontier's residual; the finishing
// kernel draws the tokens, selects each request's result (first rejection, emitted tokens,
// stopping), reduces alpha for the gamma controller and, for spec_verify_round, compacts the round
// and chooses gamma. Each kernel after the first is launched to start as the one before drains.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <mutex>

#include "spec_device.cuh"
#include "spec_verify.h"

#include "spec_kernels.cuh"
#include "spec_trunc.cuh"
#include "spec_tail.cuh"

namespace spec {

// ------------------------------------------------------------------------------------------
// Host side

// Workspace of one call. It needs no preparation: the statistics kernel zeroes the counters the
// later kernels use, and every record is written before it is read within the call.
struct WsLayout {
    size_t rec, xrec, desc, dec, alpha_c, zc, req_first, req_st, ctl, agg, cut, total;
    int32_t nvec_row, nchunk;
};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static WsLayout ws_layout(int32_t B, int32_t V, int32_t total_rows, spec_dtype dtype) {
    WsLayout L = {};
    const size_t T = static_cast<size_t>(total_rows > 0 ? total_rows : 0);
    const size_t nb = static_cast<size_t>(B > 0 ? B : 0);
    const size_t eb = (dtype == SPEC_BF16) ? 2 : 4;
    const size_t nvec = V > 0 ? (static_cast<size_t>(V) * eb) / 16 : 0;
    L.nvec_row = static_cast<int32_t>(nvec);
    L.nchunk = static_cast<int32_t>((nvec + vk::kChunkVecs - 1) / vk::kChunkVecs);
    const size_t chunks = T * static_cast<size_t>(L.nchunk);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    L.ctl = take(vk::kCtlWords * 4);
    L.agg = take(vk::kAggWords * 4);
    L.req_first = take(nb * 4);
    L.req_st = take(nb * 4);
    L.rec = take(chunks * 16);
    L.alpha_c = take(chunks * 4);
    L.zc = take(chunks * 4);
    L.xrec = take(T * 16);
    L.desc = take(T * sizeof(vk::ItemDesc));
    L.dec = take(T * sizeof(vk::ItemDec));
    L.cut = take(T * 8);  // top-k / top-p cut per target row
    L.total = off;
    return L;
}

// The persistent grid of the statistics kernel on the current device: every SM filled with as many
// CTAs as fit.
template <int DT>
static cudaError_t stats_grid(int &ctas, int *p2 = nullptr) {
    static std::mutex mu;
    static int ctas_of[64] = {0}, p2_of[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!ctas_of[dev]) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vk::spec_stats_kernel<DT>, vk::kStatsBlock, 0);
        if (e != cudaSuccess) return e;
        ctas_of[dev] = sms * per_sm;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vk::spec_pass2_kernel<DT>, vk::kFinBlock, 0);
        if (e != cudaSuccess) return e;
        p2_of[dev] = sms * per_sm;
    }
    ctas = ctas_of[dev];
    if (p2) *p2 = p2_of[dev];
    return cudaSuccess;
}

template <int DT>
static spec_status launch_verify(const vk::VerifyParams &P, cudaStream_t stream, cudaEvent_t stats_end) {
    int ctas = 0, p2_ctas = 0;
    if (stats_grid<DT>(ctas, &p2_ctas) != cudaSuccess) return SPEC_ERR_CUDA;
    if (ctas <= 0 || p2_ctas <= 0) return SPEC_ERR_UNSUPPORTED;
    vk::spec_stats_kernel<DT><<<ctas, vk::kStatsBlock, 0, stream>>>(P);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
    if (stats_end && cudaEventRecord(stats_end, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    if (launch_after(vk::spec_decide_kernel<DT>, dim3(static_cast<unsigned>(P.B)), dim3(vk::kDecWarps * kWarp), 0,
                     stream, P) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (launch_after(vk::spec_pass2_kernel<DT>, dim3(static_cast<unsigned>(p2_ctas)), dim3(vk::kFinBlock), 0, stream,
                     P) != cudaSuccess)
        return SPEC_ERR_CUDA;
    const unsigned fin_ctas = static_cast<unsigned>((P.total_rows + vk::kFinWarps - 1) / vk::kFinWarps);
    if (launch_after(vk::spec_finish_kernel<DT>, dim3(fin_ctas), dim3(vk::kFinBlock), 0, stream, P) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

}  // namespace spec

using namespace spec;

extern "C" size_t spec_verify_workspace_size(int32_t B, int32_t V, int32_t total_rows, spec_dtype dtype) {
    return ws_layout(B, V, total_rows, dtype).total;
}

// spec_verify's checks and launches (the truncation kernel when top-k / top-p is given, then the
// statistics, decision, pass-2 and finishing kernels); with C and G the finishing kernel also runs
// the round's compaction and gamma choice.
// Nothing is enqueued when a check fails.
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
    if (row_bytes / 16 > static_cast<size_t>(INT_MAX / 2)) return SPEC_ERR_UNSUPPORTED;
    if (!a->temperature && !(a->temperature_scalar >= 0.0f && std::isfinite(a->temperature_scalar)))
        return SPEC_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(a->B, a->V, a->total_rows, a->dtype);
    if (static_cast<int64_t>(a->total_rows) * L.nchunk > INT_MAX / 2) return SPEC_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < L.total || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return SPEC_ERR_WORKSPACE;

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    vk::VerifyParams P = {};
    P.target = a->target_logits;
    P.draft = a->draft_logits;
    P.row_off = a->row_off;
    P.draft_tokens = a->draft_tokens;
    P.uniforms = a->uniforms;
    P.temperature = a->temperature;
    P.temperature_scalar = a->temperature_scalar;
    P.top_p = a->top_p;
    P.stop_token = a->stop_token;
    P.max_new = a->max_new;
    P.B = a->B;
    P.V = a->V;
    P.K_max = a->K_max;
    P.total_rows = a->total_rows;
    P.nvec_row = L.nvec_row;
    P.nchunk = L.nchunk;
    P.rec = reinterpret_cast<int4 *>(ws + L.rec);
    P.xrec = reinterpret_cast<float4 *>(ws + L.xrec);
    P.desc = reinterpret_cast<vk::ItemDesc *>(ws + L.desc);
    P.dec = reinterpret_cast<vk::ItemDec *>(ws + L.dec);
    P.alpha_c = reinterpret_cast<float *>(ws + L.alpha_c);
    P.zc = reinterpret_cast<float *>(ws + L.zc);
    P.req_first = reinterpret_cast<int32_t *>(ws + L.req_first);
    P.req_st = reinterpret_cast<int32_t *>(ws + L.req_st);
    P.ctl = reinterpret_cast<uint32_t *>(ws + L.ctl);
    P.agg = reinterpret_cast<uint32_t *>(ws + L.agg);
    P.accept_len = a->accept_len;
    P.n_emitted = a->n_emitted;
    P.out_tokens = a->out_tokens;
    P.req_status = a->req_status;
    P.fallback = a->fallback;
    P.alpha_count = a->alpha_count;
    P.depth_reached = a->depth_reached;
    P.depth_accepted = a->depth_accepted;
    P.alpha_rows = a->alpha_rows;
    P.rho_rows = a->rho_rows;
    P.resid_rows = a->resid_rows;
    P.frontier_prob = a->frontier_prob;
    P.frontier_margin = a->frontier_margin;
    P.alpha_sum = a->alpha_sum;
    P.round = (C && G) ? 1 : 0;
    if (C) P.C = *C;
    if (G) P.G = *G;
    P.trunc = nullptr;
    if (a->top_k || a->top_p) {
        // top-k / top-p: the cut of every target row, before the statistics kernel reads it
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
    const spec_status st = (a->dtype == SPEC_BF16) ? launch_verify<SPEC_BF16>(P, stream, a->stats_event_end)
                                                   : launch_verify<SPEC_F32>(P, stream, a->stats_event_end);
    if (st != SPEC_OK) return st;
    if (a->rows_event_end && cudaEventRecord(a->rows_event_end, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
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

#ifdef SPEC_DEBUG
extern "C" const char *spec_version(void) { return "spec-verify-gb300 0.1 (sm_103a, index-checked debug build)"; }

namespace spec {
cudaError_t debug_take_compact(unsigned int out[4]);
}

extern "C" spec_status spec_debug_fetch(unsigned int *out) {
    if (!out) return SPEC_ERR_INVALID_ARG;
    unsigned int a[4] = {0u, 0u, 0u, 0u}, b[4] = {0u, 0u, 0u, 0u};
    if (cudaDeviceSynchronize() != cudaSuccess) return SPEC_ERR_CUDA;
    if (spec::spec_dbg_take(a) != cudaSuccess || spec::debug_take_compact(b) != cudaSuccess) return SPEC_ERR_CUDA;
    const unsigned int *first = a[0] ? a : b;
    out[0] = first[0];
    out[1] = first[1];
    out[2] = first[2];
    out[3] = a[3] + b[3];
    return SPEC_OK;
}
#else
extern "C" const char *spec_version(void) { return "spec-verify-gb300 0.1 (sm_103a)"; }
#endif

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
// The array lives in every GPU that loads the library until the process exits; a workspace needs
// no preparation between calls, so every call finds it ready. Its address is looked up once
// per device, on the first call made with that device current; make that first call before any
// stream capture. All calls share the one array and it keeps the last call's contents; calls
// that overlap on the GPU, on two streams or from two threads, race on it and must be
// serialised by the caller.

namespace spec {
constexpr int32_t kNoallocMaxRows = 16384;             // target rows per call: T = sum_i (K_i + 1)
constexpr size_t kNoallocScratchBytes = 16u << 20;     // 16 MiB of device memory per GPU
static __device__ __align__(256) unsigned char noalloc_scratch[kNoallocScratchBytes];

static std::mutex noalloc_mu;
static void *noalloc_ptr[64] = {nullptr};
}  // namespace spec

extern "C" spec_status spec_verify_noalloc(const spec_verify_args *a, cudaStream_t stream) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->total_rows > kNoallocMaxRows) return SPEC_ERR_UNSUPPORTED;  // beyond the fixed scratch
    const size_t need = ws_layout(a->B, a->V, a->total_rows, a->dtype).total;
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
    int ctas = 0;
    const cudaError_t e = (dtype == SPEC_BF16) ? stats_grid<SPEC_BF16>(ctas) : stats_grid<SPEC_F32>(ctas);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (ctas <= 0) return nullptr;
    if (cluster) *cluster = 1;
    if (clusters) *clusters = ctas;
    return "spec_stats_kernel";
}
