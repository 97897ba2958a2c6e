// Linear verification ("Accelerating Sonar through speculation",
// §Speculative decoding and §Target-Draft): row statistics of every target
// and draft row (this file's two-pass kernel, or the one-read kernel of
// rows_topp.cu for bf16 rows under top-p), then a finishing launch that
// takes every request's accept tests, accepted length and packed offsets
// (this file); then per request the residual or bonus draw and, for the
// compacting call, the gather of the accepted positions' hidden rows
// (draw_stream.cu, decide.cu); the C entry points.
#include <mutex>

#include "../../include/specverify.h"
#include "decisions.cuh"
#include "launch.cuh"
#include "linear_args.cuh"
#include "sample.cuh"

namespace sv {

// One CTA per row (persistent).  MODE 0 greedy, 1 sampled, 2 sampled + top-p.
// finish = 0: every row.  finish = 1: the launch after the statistics
// (every row written by an earlier launch): when some rows were left by the
// one-read top-p pass it recomputes them and its last CTA then takes every
// request's decisions; otherwise each warp takes one request's decisions at
// once.  Either way the last CTA to finish writes the packed offsets.
template <typename T, int MODE>
__global__ void __launch_bounds__(kNT, 4) k_linear_rowstats(LinearArgs a, int finish) {
    extern __shared__ uint4 dyn_smem[];
    __shared__ BlockScratch s;
    __shared__ SampleScratch ss;
    __shared__ unsigned sh_ticket;
    uint8_t* topsmem = reinterpret_cast<uint8_t*>(dyn_smem);
    const int nt = a.B * (a.k + 1);
    const int R = nt + (MODE > 0 ? a.B * a.k : 0);
    const T* tgt = static_cast<const T*>(a.tgt);
    const T* drf = static_cast<const T*>(a.drf);
    grid_dep_wait();     // the finishing launch reads what the launch before it wrote
    grid_dep_trigger();  // the next launch may be scheduled; it waits for this grid
    const bool redo = finish && __ldcg(a.done + 2) != 0u;  // the same value in every thread
    if (finish && !redo) {  // every record final: one warp per request
        const int warp = threadIdx.x >> 5;
        for (int b = blockIdx.x * kNW + warp; b < a.B; b += gridDim.x * kNW) warp_request_decisions<MODE>(a, b);
        if (last_cta_done(a, &sh_ticket, 0)) linear_offsets(a, s);
        return;
    }
    for (int r = blockIdx.x; r < R; r += gridDim.x) {
        if (redo && !(a.stats[r].flags & kRowRedo)) continue;  // the same value in every thread
        const T* row;
        int tok;
        if (r < nt) {
            const int b = r / (a.k + 1), i = r - b * (a.k + 1);
            row = tgt + (size_t)r * a.V;
            tok = (i < a.k) ? a.drafts[(size_t)b * a.k + i] : -1;
        } else {
            const int rr = r - nt;
            row = drf + (size_t)rr * a.V;
            tok = a.drafts[rr];
        }
        const RowStat st = row_stats<T, MODE>(row, a.V, a.c, a.top_p, tok, topsmem, s, ss);
        if (threadIdx.x == 0) a.stats[r] = st;
        __syncthreads();
    }
    if (finish && last_cta_done(a, &sh_ticket, 0)) {  // the recomputed rows are in: every request
        const int warp = threadIdx.x >> 5;
        for (int b = warp; b < a.B; b += kNW) warp_request_decisions<MODE>(a, b);
        __syncthreads();
        linear_offsets(a, s);
    }
}

// Zeroes the call's counters, device error word and length histogram in
// one launch (the statistics launch after it may start while it ends).
__global__ void k_zero_counters(unsigned* done, int32_t* dev_error, int32_t* len_hist, int nh) {
    grid_dep_wait();
    grid_dep_trigger();
    const int t = threadIdx.x;
    if (t < 4) done[t] = 0u;
    if (t == 0 && dev_error) *dev_error = 0;
    if (len_hist)
        for (int i = t; i < nh; i += blockDim.x) len_hist[i] = 0;
}

// Stage 1: statistics of every target and draft row into the workspace,
// then the finishing launch (decisions and offsets).  bf16 rows under top-p
// take the one-read kernel (rows_topp.cu) first; the finishing launch then
// also recomputes the rows it left.
template <typename T, int MODE>
static spec_status launch_stats(LinearArgs& a, cudaStream_t st) {
    const int nt = a.B * (a.k + 1);
    const int R = nt + (MODE > 0 ? a.B * a.k : 0);
    constexpr bool kOnePass = (MODE == 2 && sizeof(T) == 2);
    const size_t dyn = (MODE == 2 && sizeof(T) == 2) ? (size_t)kTopSmemBytes : 0;
    auto* k1 = k_linear_rowstats<T, MODE>;
    int grid = 0;
    if (!launch_grid(k1, dyn, R, &grid, kNT)) return SPEC_ERR_CUDA;
    if (kOnePass) {
        const spec_status r = launch_rows_topp_onepass(a, st);
        if (r != SPEC_OK) return r;
    } else {
        if (launch_dependent(k1, dim3(grid), dim3(kNT), dyn, st, a, 0) != cudaSuccess) return SPEC_ERR_CUDA;
    }
    if (launch_dependent(k1, dim3(grid), dim3(kNT), dyn, st, a, 1) != cudaSuccess) return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

template <typename T>
static spec_status launch_stage(LinearArgs& a, int mode, int stage, cudaStream_t st) {
    if (stage == 0) {
        if (mode == 0) return launch_stats<T, 0>(a, st);
        if (mode == 1) return launch_stats<T, 1>(a, st);
        return launch_stats<T, 2>(a, st);
    }
    return launch_decide_stage(a, sizeof(T) == 2 ? SPEC_BF16 : SPEC_F32, mode, st);
}

// Host-side checks shared by the linear entry points; fills `a` and `mode`.
static spec_status prepare_linear(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                  const int32_t* draft_tokens, int B, int k, int V, const int64_t* request_ids,
                                  const int64_t* positions, const spec_sampling_params* params, void* workspace,
                                  size_t workspace_bytes, LinearArgs& a, int& mode) {
    if (!params || !target_logits || !draft_tokens) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
    if (B < 1 || k < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
    if (k > 64) return SPEC_ERR_UNSUPPORTED;
    const float T = params->temperature, top_p = params->top_p;
    if (!(T >= 0.0f) || !(T < INFINITY) || !(top_p > 0.0f)) return SPEC_ERR_INVALID_ARG;
    const bool greedy = (T == 0.0f);
    if (!greedy && !draft_logits) return SPEC_ERR_INVALID_ARG;
    if ((int64_t)V > kMaxVocab) return SPEC_ERR_UNSUPPORTED;
    if ((int64_t)B * (2 * k + 1) > 0x7fffffffLL / 2) return SPEC_ERR_UNSUPPORTED;
    const LinearWorkspace lw = linear_workspace(B, k);
    if (!workspace || workspace_bytes < lw.total || (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return SPEC_ERR_WORKSPACE;
    if (!select_device_of(target_logits)) return SPEC_ERR_INVALID_ARG;
    a = LinearArgs{};
    a.tgt = target_logits;
    a.drf = draft_logits;
    a.drafts = draft_tokens;
    a.B = B; a.k = k; a.V = V;
    a.req = request_ids;
    a.pos = positions;
    a.T = T;
    a.top_p = top_p;
    a.c = greedy ? 0.0f : (float)(1.4426950408889634 / (double)T);
    a.seed = params->seed;
    char* w = static_cast<char*>(workspace);
    a.stats = reinterpret_cast<RowStat*>(w);
    a.dec = reinterpret_cast<int32_t*>(w + lw.dec);
    a.woff = reinterpret_cast<int32_t*>(w + lw.woff);
    a.done = reinterpret_cast<unsigned*>(w + lw.done);
    mode = greedy ? 0 : (top_p < 1.0f ? 2 : 1);
    return SPEC_OK;
}

static spec_status run_stage(LinearArgs& a, spec_dtype dtype, int mode, int stage, cudaStream_t st) {
    return dtype == SPEC_BF16 ? launch_stage<__nv_bfloat16>(a, mode, stage, st) : launch_stage<float>(a, mode, stage, st);
}

}  // namespace sv

using namespace sv;

extern "C" spec_status spec_linear_stats_decide(const void* target_logits, const void* draft_logits,
                                                spec_dtype dtype, const int32_t* draft_tokens, int B, int k, int V,
                                                const int64_t* request_ids, const int64_t* positions,
                                                const spec_sampling_params* params, int32_t* accepted_len,
                                                float* accept_prob, float* token_probs, int32_t* len_hist,
                                                int32_t* dev_error, void* workspace, size_t workspace_bytes,
                                                spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    if (!accepted_len) return SPEC_ERR_INVALID_ARG;
    LinearArgs a;
    int mode = 0;
    spec_status r = prepare_linear(target_logits, draft_logits, dtype, draft_tokens, B, k, V, request_ids, positions,
                                   params, workspace, workspace_bytes, a, mode);
    if (r != SPEC_OK) return r;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (launch_dependent(k_zero_counters, dim3(1), dim3(64), 0, st, a.done, dev_error, len_hist, k + 1) != cudaSuccess)
        return SPEC_ERR_CUDA;
    a.acc_len = accepted_len;
    a.accept_prob = accept_prob;
    a.token_probs = token_probs;
    a.len_hist = len_hist;
    a.dev_error = dev_error;
    return run_stage(a, dtype, mode, 0, st);
}

extern "C" spec_status spec_linear_draw(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                        const int32_t* draft_tokens, int B, int k, int V,
                                        const int64_t* request_ids, const int64_t* positions,
                                        const spec_sampling_params* params, const void* hidden, int H,
                                        int32_t* out_tokens, void* out_hidden, int32_t* offsets,
                                        int32_t* next_tokens, const void* workspace, size_t workspace_bytes,
                                        spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    if (!out_tokens) return SPEC_ERR_INVALID_ARG;
    if (hidden && (H < 1 || !out_hidden || !offsets || !next_tokens)) return SPEC_ERR_INVALID_ARG;
    if (hidden && (int64_t)B * (k + 1) >= 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
    LinearArgs a;
    int mode = 0;
    spec_status r = prepare_linear(target_logits, draft_logits, dtype, draft_tokens, B, k, V, request_ids, positions,
                                   params, const_cast<void*>(workspace), workspace_bytes, a, mode);
    if (r != SPEC_OK) return r;
    a.out_tokens = out_tokens;
    if (hidden) {
        a.hidden = static_cast<const uint16_t*>(hidden);
        a.H = H;
        a.out_hidden = static_cast<uint16_t*>(out_hidden);
        a.offsets = offsets;
        a.next_tokens = next_tokens;
        a.vec_ok = ((size_t)H * 2) % 16 == 0 && (reinterpret_cast<uintptr_t>(hidden) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(out_hidden) & 15u) == 0;
    }
    return run_stage(a, dtype, mode, 1, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" spec_status spec_verify_linear(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                          const int32_t* draft_tokens, int B, int k, int V,
                                          const int64_t* request_ids, const int64_t* positions,
                                          const spec_sampling_params* params, int32_t* accepted_len,
                                          int32_t* out_tokens, float* accept_prob, float* token_probs,
                                          int32_t* len_hist, int32_t* dev_error, void* workspace,
                                          size_t workspace_bytes, spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    if (!accepted_len || !out_tokens) return SPEC_ERR_INVALID_ARG;
    const spec_status r =
        spec_linear_stats_decide(target_logits, draft_logits, dtype, draft_tokens, B, k, V, request_ids, positions,
                                 params, accepted_len, accept_prob, token_probs, len_hist, dev_error, workspace,
                                 workspace_bytes, stream);
    if (r != SPEC_OK) return r;
    return spec_linear_draw(target_logits, draft_logits, dtype, draft_tokens, B, k, V, request_ids, positions,
                            params, nullptr, 0, out_tokens, nullptr, nullptr, nullptr, workspace, workspace_bytes,
                            stream);
}

extern "C" spec_status spec_verify_linear_compact(const void* target_logits, const void* draft_logits,
                                                  spec_dtype dtype, const int32_t* draft_tokens, int B, int k, int V,
                                                  const int64_t* request_ids, const int64_t* positions,
                                                  const spec_sampling_params* params, const void* hidden, int H,
                                                  int32_t* accepted_len, int32_t* out_tokens, float* accept_prob,
                                                  float* token_probs, int32_t* len_hist, void* out_hidden,
                                                  int32_t* offsets, int32_t* next_tokens, int32_t* dev_error,
                                                  void* workspace, size_t workspace_bytes, spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    if (!accepted_len || !out_tokens || !hidden || H < 1 || !out_hidden || !offsets || !next_tokens)
        return SPEC_ERR_INVALID_ARG;
    const spec_status r =
        spec_linear_stats_decide(target_logits, draft_logits, dtype, draft_tokens, B, k, V, request_ids, positions,
                                 params, accepted_len, accept_prob, token_probs, len_hist, dev_error, workspace,
                                 workspace_bytes, stream);
    if (r != SPEC_OK) return r;
    return spec_linear_draw(target_logits, draft_logits, dtype, draft_tokens, B, k, V, request_ids, positions,
                            params, hidden, H, out_tokens, out_hidden, offsets, next_tokens, workspace,
                            workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Variant of spec_verify_linear that allocates nothing and takes no
// workspace.  Some callers cannot allocate device memory when they verify:
// code running inside a custom allocator or memory pool, code that must not
// grow its memory after start-up, or code whose buffers are all handed to it
// by a host framework.  This variant keeps the per-row statistics in a
// fixed array that lives in the library's device image, so the caller only
// passes inputs and outputs.
//
// The array holds the workspace of up to kNoAllocMaxRows rows (about 2.3
// MiB: the row records, the decisions, the offsets and a counter); every GPU
// that loads the library keeps it until the process exits.  Calls with
// B * (2k + 1) rows above that limit return SPEC_ERR_UNSUPPORTED.  All calls
// share the array, so calls that overlap on the GPU (on different streams,
// or from different host threads) race on it.  Each call clears the counter
// and writes every record before reading it, so nothing in the array needs
// to start at zero.
// ---------------------------------------------------------------------------
namespace sv {

constexpr int kNoAllocMaxRows = 65536;
// every (B, k) within the row limit has B <= kNoAllocMaxRows / 3
constexpr size_t kNoAllocMaxB = kNoAllocMaxRows / 3;
constexpr size_t kNoAllocBytes = kNoAllocMaxRows * sizeof(RowStat) + 2 * (((kNoAllocMaxB + 1) * 4 + 255) / 256 * 256) + 256;
static __device__ __align__(256) uint8_t g_noalloc_stats[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
static std::mutex g_noalloc_mutex;
static void* g_noalloc_ptr[kNoAllocMaxDevices];

// Device address of the array on the current device.  The first call on a
// device resolves it (once), so make that first call before any stream
// capture begins.
static spec_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return SPEC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_stats) != cudaSuccess || !p) return SPEC_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SPEC_OK;
}

}  // namespace sv

extern "C" spec_status spec_verify_linear_noalloc(const void* target_logits, const void* draft_logits,
                                                  spec_dtype dtype, const int32_t* draft_tokens, int B, int k, int V,
                                                  const int64_t* request_ids, const int64_t* positions,
                                                  const spec_sampling_params* params, int32_t* accepted_len,
                                                  int32_t* out_tokens, float* accept_prob, float* token_probs,
                                                  int32_t* len_hist, int32_t* dev_error, spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    if (B < 1 || k < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
    if ((int64_t)B * (2 * (int64_t)k + 1) > kNoAllocMaxRows) return SPEC_ERR_UNSUPPORTED;
    if (linear_workspace(B, k).total > kNoAllocBytes) return SPEC_ERR_UNSUPPORTED;
    if (!target_logits || !select_device_of(target_logits)) return SPEC_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const spec_status r = noalloc_scratch(&scratch);
    if (r != SPEC_OK) return r;
    return spec_verify_linear(target_logits, draft_logits, dtype, draft_tokens, B, k, V, request_ids, positions,
                              params, accepted_len, out_tokens, accept_prob, token_probs, len_hist, dev_error,
                              scratch, kNoAllocBytes, stream);
}
