// Linear verification ("Accelerating Sonar through speculation",
// §Speculative decoding and §Target-Draft): row statistics of every target
// and draft row, then per request the accept tests, the accepted length
// and the residual or bonus draw.
#include <mutex>

#include "../../include/specverify.h"
#include "launch.cuh"
#include "sample.cuh"

namespace sv {

struct LinearArgs {
    const void* tgt;
    const void* drf;
    const int32_t* drafts;
    int B, k, V;
    const int64_t* req;
    const int64_t* pos;
    float T, top_p, c;
    uint64_t seed;
    int32_t* acc_len;
    int32_t* out_tokens;
    float* accept_prob;
    float* token_probs;
    int32_t* len_hist;
    int32_t* dev_error;
    RowStat* stats;  // target rows [B*(k+1)], then draft rows [B*k]
};

__device__ __forceinline__ int tgt_row(const LinearArgs& a, int b, int i) { return b * (a.k + 1) + i; }
__device__ __forceinline__ int drf_row(const LinearArgs& a, int b, int i) { return a.B * (a.k + 1) + b * a.k + i; }

// One CTA per row (persistent).  MODE 0 greedy, 1 sampled, 2 sampled + top-p.
template <typename T, int MODE>
__global__ void __launch_bounds__(kNT, 4) k_linear_rowstats(LinearArgs a) {
    extern __shared__ uint4 dyn_smem[];
    __shared__ BlockScratch s;
    __shared__ SampleScratch ss;
    uint8_t* topsmem = reinterpret_cast<uint8_t*>(dyn_smem);
    const int nt = a.B * (a.k + 1);
    const int R = nt + (MODE > 0 ? a.B * a.k : 0);
    const T* tgt = static_cast<const T*>(a.tgt);
    const T* drf = static_cast<const T*>(a.drf);
    for (int r = blockIdx.x; r < R; r += gridDim.x) {
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

// One CTA per request: warp 0 takes the accept decisions, then the whole
// CTA draws the residual or bonus token.
template <typename T, int MODE>
__global__ void __launch_bounds__(kNT, 2) k_linear_finalize(LinearArgs a) {
    __shared__ BlockScratch s;
    __shared__ DrawScratch ds;
    __shared__ int sh_a, sh_inval;
    const int b = blockIdx.x, k = a.k, V = a.V;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t req = a.req ? a.req[b] : (int64_t)b;
    const int64_t pos = a.pos ? a.pos[b] : 0;
    const int32_t* d = a.drafts + (size_t)b * k;

    if (warp == 0) {
        int inval = 0;
        for (int i = lane; i <= k; i += 32)
            if (a.stats[tgt_row(a, b, i)].flags & kRowInvalid) inval |= kDevErrNonfinite;
        if (MODE > 0)
            for (int i = lane; i < k; i += 32)
                if (a.stats[drf_row(a, b, i)].flags & kRowInvalid) inval |= kDevErrNonfinite;
        for (int i = lane; i < k; i += 32)
            if (d[i] < 0 || d[i] >= V) inval |= kDevErrToken;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) inval |= __shfl_xor_sync(0xffffffffu, inval, o);
        int first_reject = k;
        for (int i0 = 0; i0 < k; i0 += 32) {
            const int i = i0 + lane;
            bool acc = true;
            float ap = 0.0f, pp = 0.0f, qq = 0.0f;
            if (i < k && !inval) {
                const RowStat sp = a.stats[tgt_row(a, b, i)];
                if (MODE == 0) {
                    acc = (d[i] == sp.argmax);
                    ap = acc ? 1.0f : 0.0f;
                    pp = ap;
                    qq = 1.0f;
                } else {
                    const RowStat sq = a.stats[drf_row(a, b, i)];
                    pp = (sp.flags & kRowTokMember) ? weight_of(sp.x_tok, a.c, scaled_max(sp.m, a.c)) * sp.inv_zn : 0.0f;
                    qq = (sq.flags & kRowTokMember) ? weight_of(sq.x_tok, a.c, scaled_max(sq.m, a.c)) * sq.inv_zn : 0.0f;
                    const float ratio = qq > 0.0f ? pp / qq : 0.0f;
                    ap = fminf(1.0f, ratio);
                    acc = uniform01(a.seed, req, pos + i + 1, kPurposeAccept, 0) < ratio;
                }
            }
            if (i < k) {
                if (a.accept_prob) a.accept_prob[(size_t)b * k + i] = inval ? 0.0f : ap;
                if (a.token_probs) {
                    a.token_probs[((size_t)b * k + i) * 2 + 0] = inval ? 0.0f : pp;
                    a.token_probs[((size_t)b * k + i) * 2 + 1] = inval ? 0.0f : qq;
                }
            }
            const unsigned rej = __ballot_sync(0xffffffffu, i < k && !acc);
            if (rej && first_reject == k) first_reject = i0 + __ffs(rej) - 1;
        }
        if (lane == 0) {
            sh_a = inval ? 0 : first_reject;
            sh_inval = inval;
        }
    }
    __syncthreads();
    const int acnt = sh_a, inval = sh_inval;
    const T* tgt = static_cast<const T*>(a.tgt) + (size_t)b * (k + 1) * V;
    int t = -1;
    if (inval) {
        t = row_argmax_finite<T>(tgt, V, s);
    } else if (MODE == 0) {
        t = a.stats[tgt_row(a, b, acnt)].argmax;
    } else {
        const RowStat sp = a.stats[tgt_row(a, b, acnt)];
        const T* prow = tgt + (size_t)acnt * V;
        const RowView<T> rv(prow, V);
        FilteredRow<T> P(prow, sp, a.c, 0x7fffffff);
        const bool resid = acnt < k;
        const float u = uniform01(a.seed, req, pos + acnt + 1, resid ? kPurposeResidual : kPurposeBonus, 0);
        if (resid) {
            const RowStat sq = a.stats[drf_row(a, b, acnt)];
            const T* qrow = static_cast<const T*>(a.drf) + ((size_t)b * k + acnt) * V;
            FilteredRow<T> Q(qrow, sq, a.c, 0x7fffffff);
            t = draw_linear<T, true, (MODE == 2)>(rv, P, Q, u, s, ds);
            if (t < 0) t = draw_linear<T, false, (MODE == 2)>(rv, P, Q, u, s, ds);  // p == q: draw from p
        } else {
            t = draw_linear<T, false, (MODE == 2)>(rv, P, P, u, s, ds);
        }
    }
    if (threadIdx.x == 0) {
        a.acc_len[b] = acnt;
        int32_t* o = a.out_tokens + (size_t)b * (k + 1);
        for (int j = 0; j <= k; ++j) o[j] = (j < acnt) ? d[j] : (j == acnt ? t : -1);
        if (a.len_hist) atomicAdd(a.len_hist + acnt, 1);
        if (inval && a.dev_error) atomicOr(a.dev_error, inval);
    }
}

// Stage 1: statistics of every target and draft row into the workspace.
template <typename T, int MODE>
static spec_status launch_stats(LinearArgs& a, cudaStream_t st) {
    const int nt = a.B * (a.k + 1);
    const int R = nt + (MODE > 0 ? a.B * a.k : 0);
    const size_t dyn = (MODE == 2 && sizeof(T) == 2) ? (size_t)kTopSmemBytes : 0;
    auto* k1 = k_linear_rowstats<T, MODE>;
    int grid = 0;
    if (!launch_grid(k1, dyn, R, &grid, kNT)) return SPEC_ERR_CUDA;
    k1<<<grid, kNT, dyn, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Stage 2: accept tests, accepted length and the residual / bonus draw.
template <typename T, int MODE>
static spec_status launch_decide(LinearArgs& a, cudaStream_t st) {
    k_linear_finalize<T, MODE><<<a.B, kNT, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

template <typename T>
static spec_status launch_stage(LinearArgs& a, int mode, int stage, cudaStream_t st) {
    if (stage == 0) {
        if (mode == 0) return launch_stats<T, 0>(a, st);
        if (mode == 1) return launch_stats<T, 1>(a, st);
        return launch_stats<T, 2>(a, st);
    }
    if (mode == 0) return launch_decide<T, 0>(a, st);
    if (mode == 1) return launch_decide<T, 1>(a, st);
    return launch_decide<T, 2>(a, st);
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
