// Arguments of the two launches of a linear verification (row statistics,
// then decisions and the draw), shared by linear.cu and decide.cu, which are
// compiled with different CTA sizes.
#pragma once

#include "../../include/specverify.h"
#include "common.cuh"

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

// Stage 1 for bf16 rows under top-p (rows_topp.cu): one read per row; rows
// it cannot finish are marked kRowRedo for the two-pass kernel.
spec_status launch_rows_topp_onepass(LinearArgs& a, cudaStream_t st);

// Stage 2 (decide.cu): accept tests, accepted length and the residual or
// bonus draw, one CTA per request.
spec_status launch_decide_stage(LinearArgs& a, spec_dtype dtype, int mode, cudaStream_t st);

}  // namespace sv
