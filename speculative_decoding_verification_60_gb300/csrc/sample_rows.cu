// Draft-side sampling ("Accelerating Sonar through speculation",
// §Target-Draft: the draft model samples its tokens; §MTP schedule for a
// single token: sampling stays on the GPU so that the next draft run needs
// no host round trip).  One token per logit row from filter(softmax(row /
// T)), by the same row statistics and inverse-CDF draw as the bonus token
// of linear verification, with the DRAFT purpose in the Philox counter.
// bf16 rows under top-p take the one-read pass first (rows_topp.cu), which
// marks the rows it cannot finish; this kernel then takes only those.
// Built with 512-thread CTAs: one row per CTA at a time.
#include "../../include/specverify.h"
#include "launch.cuh"
#include "linear_args.cuh"
#include "sample.cuh"

namespace sv {

struct SampleArgs {
    const void* logits;
    int R, V;
    const int64_t* req;
    const int64_t* pos;
    float c, top_p;
    uint64_t seed;
    int32_t* out;
    int32_t* dev_error;
    bool redo_only;  // take only the rows whose out holds kSampleRedo
};

template <typename T, int MODE>
__global__ void __launch_bounds__(kNT, 2) k_sample_rows(SampleArgs a) {
    extern __shared__ uint4 dyn_smem[];
    __shared__ BlockScratch s;
    __shared__ SampleScratch ss;
    __shared__ DrawScratch ds;
    uint8_t* topsmem = reinterpret_cast<uint8_t*>(dyn_smem);
    grid_dep_wait();  // after the one-read pass: its marks are in out
    for (int r = blockIdx.x; r < a.R; r += gridDim.x) {
        if (a.redo_only && a.out[r] != kSampleRedo) continue;  // the same for the whole CTA
        const T* row = static_cast<const T*>(a.logits) + (size_t)r * a.V;
        const RowStat st = row_stats<T, MODE>(row, a.V, a.c, a.top_p, -1, topsmem, s, ss);
        int t;
        int err = 0;
        if (st.flags & kRowInvalid) {
            t = row_argmax_finite<T>(row, a.V, s);
            err = (MODE > 0) ? kDevErrNonfinite : 0;
        } else if (MODE == 0) {
            t = st.argmax;
        } else {
            const RowView<T> rv(row, a.V);
            FilteredRow<T> P(row, st, a.c, 0x7fffffff);
            const int64_t req = a.req ? a.req[r] : (int64_t)r;
            const int64_t pos = a.pos ? a.pos[r] : 0;
            const float u = uniform01(a.seed, req, pos, kPurposeDraft, 0);
            t = draw_linear<T, false, (MODE == 2)>(rv, P, P, u, s, ds);
        }
        if (threadIdx.x == 0) {
            a.out[r] = t;
            if (err && a.dev_error) atomicOr(a.dev_error, err);
        }
        __syncthreads();
    }
}

template <typename T, int MODE>
static spec_status launch_sample(SampleArgs& a, cudaStream_t st) {
    const size_t dyn = (MODE == 2 && sizeof(T) == 2) ? (size_t)kTopSmemBytes : 0;
    auto* kern = k_sample_rows<T, MODE>;
    int grid = 0;
    if (!launch_grid(kern, dyn, a.R, &grid, kNT)) return SPEC_ERR_CUDA;
    if (launch_dependent(kern, dim3(grid), dim3(kNT), dyn, st, a) != cudaSuccess) return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

template <typename T>
static spec_status launch_sample_t(SampleArgs& a, int mode, cudaStream_t st) {
    if (mode == 0) return launch_sample<T, 0>(a, st);
    if (mode == 1) return launch_sample<T, 1>(a, st);
    return launch_sample<T, 2>(a, st);
}

}  // namespace sv

using namespace sv;

extern "C" spec_status spec_sample_rows(const void* logits, spec_dtype dtype, int R, int V,
                                        const int64_t* request_ids, const int64_t* positions,
                                        const spec_sampling_params* params, int32_t* out_tokens,
                                        int32_t* dev_error, spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    if (!logits || !params || !out_tokens) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
    if (R < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
    const float T = params->temperature, top_p = params->top_p;
    if (!(T >= 0.0f) || !(T < INFINITY) || !(top_p > 0.0f)) return SPEC_ERR_INVALID_ARG;
    if ((int64_t)V > kMaxVocab) return SPEC_ERR_UNSUPPORTED;
    if (!select_device_of(logits)) return SPEC_ERR_INVALID_ARG;
    SampleArgs a{};
    a.logits = logits;
    a.R = R;
    a.V = V;
    a.req = request_ids;
    a.pos = positions;
    const bool greedy = (T == 0.0f);
    a.c = greedy ? 0.0f : (float)(1.4426950408889634 / (double)T);
    a.top_p = top_p;
    a.seed = params->seed;
    a.out = out_tokens;
    a.dev_error = dev_error;
    const int mode = greedy ? 0 : (top_p < 1.0f ? 2 : 1);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dev_error && cudaMemsetAsync(dev_error, 0, sizeof(int32_t), st) != cudaSuccess) return SPEC_ERR_CUDA;
    if (dtype == SPEC_BF16 && mode == 2) {
        // one read per row, then the two-pass route on the rows it leaves
        LinearArgs la{};
        la.tgt = logits;
        la.B = R;
        la.k = 0;
        la.V = V;
        la.req = request_ids;
        la.pos = positions;
        la.c = a.c;
        la.top_p = top_p;
        la.seed = a.seed;
        la.dev_error = dev_error;
        la.sample_out = out_tokens;
        const spec_status s1 = launch_sample_onepass(la, st);
        if (s1 != SPEC_OK) return s1;
        a.redo_only = true;
    }
    return dtype == SPEC_BF16 ? launch_sample_t<__nv_bfloat16>(a, mode, st) : launch_sample_t<float>(a, mode, st);
}
