// Linear verification ("Accelerating Sonar through speculation",
// §Speculative decoding and §Target-Draft): row statistics of every target
// and draft row (this file), then per request the accept tests, the
// accepted length and the residual or bonus draw (decide.cu); the C entry
// points.
#include <mutex>

#include "../../include/specverify.h"
#include "launch.cuh"
#include "linear_args.cuh"
#include "sample.cuh"

namespace sv {

// One CTA per row (persistent).  MODE 0 greedy, 1 sampled, 2 sampled + top-p.
// redo_only: take only the rows the one-read top-p kernel marked kRowRedo.
template <typename T, int MODE>
__global__ void __launch_bounds__(kNT, 4) k_linear_rowstats(LinearArgs a, int redo_only) {
    extern __shared__ uint4 dyn_smem[];
    __shared__ BlockScratch s;
    __shared__ SampleScratch ss;
    uint8_t* topsmem = reinterpret_cast<uint8_t*>(dyn_smem);
    const int nt = a.B * (a.k + 1);
    const int R = nt + (MODE > 0 ? a.B * a.k : 0);
    const T* tgt = static_cast<const T*>(a.tgt);
    const T* drf = static_cast<const T*>(a.drf);
    for (int r = blockIdx.x; r < R; r += gridDim.x) {
        if (redo_only && !(a.stats[r].flags & kRowRedo)) continue;  // the same value in every thread
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
}

// Stage 1: statistics of every target and draft row into the workspace.
// bf16 rows under top-p take the one-read kernel (rows_topp.cu) first; the
// two-pass kernel then takes only the rows it left.
template <typename T, int MODE>
static spec_status launch_stats(LinearArgs& a, cudaStream_t st) {
    const int nt = a.B * (a.k + 1);
    const int R = nt + (MODE > 0 ? a.B * a.k : 0);
    constexpr bool kOnePass = (MODE == 2 && sizeof(T) == 2);
    if (kOnePass) {
        const spec_status r = launch_rows_topp_onepass(a, st);
        if (r != SPEC_OK) return r;
    }
    const size_t dyn = kOnePass ? (size_t)kTopSmemBytes : 0;
    auto* k1 = k_linear_rowstats<T, MODE>;
    int grid = 0;
    if (!launch_grid(k1, dyn, R, &grid, kNT)) return SPEC_ERR_CUDA;
    k1<<<grid, kNT, dyn, st>>>(a, kOnePass ? 1 : 0);
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
    const size_t need = spec_workspace_size(SPEC_OP_LINEAR, B, k, V, dtype);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15u))
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
    a.stats = static_cast<RowStat*>(workspace);
    mode = greedy ? 0 : (top_p < 1.0f ? 2 : 1);
    return SPEC_OK;
}

static spec_status run_stage(LinearArgs& a, spec_dtype dtype, int mode, int stage, cudaStream_t st) {
    return dtype == SPEC_BF16 ? launch_stage<__nv_bfloat16>(a, mode, stage, st) : launch_stage<float>(a, mode, stage, st);
}

}  // namespace sv

using namespace sv;

extern "C" spec_status spec_verify_linear(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                          const int32_t* draft_tokens, int B, int k, int V,
                                          const int64_t* request_ids, const int64_t* positions,
                                          const spec_sampling_params* params, int32_t* accepted_len,
                                          int32_t* out_tokens, float* accept_prob, float* token_probs,
                                          int32_t* len_hist, int32_t* dev_error, void* workspace,
                                          size_t workspace_bytes, spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    if (!accepted_len || !out_tokens) return SPEC_ERR_INVALID_ARG;
    LinearArgs a;
    int mode = 0;
    spec_status r = prepare_linear(target_logits, draft_logits, dtype, draft_tokens, B, k, V, request_ids, positions,
                                   params, workspace, workspace_bytes, a, mode);
    if (r != SPEC_OK) return r;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dev_error && cudaMemsetAsync(dev_error, 0, sizeof(int32_t), st) != cudaSuccess) return SPEC_ERR_CUDA;
    if (len_hist && cudaMemsetAsync(len_hist, 0, sizeof(int32_t) * (size_t)(k + 1), st) != cudaSuccess)
        return SPEC_ERR_CUDA;
    a.acc_len = accepted_len;
    a.out_tokens = out_tokens;
    a.accept_prob = accept_prob;
    a.token_probs = token_probs;
    a.len_hist = len_hist;
    a.dev_error = dev_error;
    r = run_stage(a, dtype, mode, 0, st);
    if (r != SPEC_OK) return r;
    return run_stage(a, dtype, mode, 1, st);
}

extern "C" spec_status spec_linear_stats(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                         const int32_t* draft_tokens, int B, int k, int V,
                                         const spec_sampling_params* params, void* workspace, size_t workspace_bytes,
                                         spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    LinearArgs a;
    int mode = 0;
    const spec_status r = prepare_linear(target_logits, draft_logits, dtype, draft_tokens, B, k, V, nullptr, nullptr,
                                         params, workspace, workspace_bytes, a, mode);
    if (r != SPEC_OK) return r;
    return run_stage(a, dtype, mode, 0, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" spec_status spec_linear_decide(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                          const int32_t* draft_tokens, int B, int k, int V,
                                          const int64_t* request_ids, const int64_t* positions,
                                          const spec_sampling_params* params, int32_t* accepted_len,
                                          int32_t* out_tokens, float* accept_prob, float* token_probs,
                                          int32_t* len_hist, int32_t* dev_error, const void* workspace,
                                          size_t workspace_bytes, spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    if (!accepted_len || !out_tokens) return SPEC_ERR_INVALID_ARG;
    LinearArgs a;
    int mode = 0;
    spec_status r = prepare_linear(target_logits, draft_logits, dtype, draft_tokens, B, k, V, request_ids, positions,
                                   params, const_cast<void*>(workspace), workspace_bytes, a, mode);
    if (r != SPEC_OK) return r;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dev_error && cudaMemsetAsync(dev_error, 0, sizeof(int32_t), st) != cudaSuccess) return SPEC_ERR_CUDA;
    if (len_hist && cudaMemsetAsync(len_hist, 0, sizeof(int32_t) * (size_t)(k + 1), st) != cudaSuccess)
        return SPEC_ERR_CUDA;
    a.acc_len = accepted_len;
    a.out_tokens = out_tokens;
    a.accept_prob = accept_prob;
    a.token_probs = token_probs;
    a.len_hist = len_hist;
    a.dev_error = dev_error;
    return run_stage(a, dtype, mode, 1, st);
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
// The array holds kNoAllocMaxRows rows (2 MiB); every GPU that loads the
// library keeps it until the process exits.  Calls with B * (2k + 1) rows
// above that limit return SPEC_ERR_UNSUPPORTED.  All calls share the array,
// so calls that overlap on the GPU (on different streams, or from different
// host threads) race on it.  Each call writes every row's statistics before
// reading them, so nothing in the array needs to start at zero.
// ---------------------------------------------------------------------------
namespace sv {

constexpr int kNoAllocMaxRows = 65536;
static __device__ __align__(256) RowStat g_noalloc_stats[kNoAllocMaxRows];

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
    if (!target_logits || !select_device_of(target_logits)) return SPEC_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const spec_status r = noalloc_scratch(&scratch);
    if (r != SPEC_OK) return r;
    return spec_verify_linear(target_logits, draft_logits, dtype, draft_tokens, B, k, V, request_ids, positions,
                              params, accepted_len, out_tokens, accept_prob, token_probs, len_hist, dev_error,
                              scratch, sizeof(RowStat) * (size_t)kNoAllocMaxRows, stream);
}
