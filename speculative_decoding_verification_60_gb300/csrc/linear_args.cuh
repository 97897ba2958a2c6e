// Arguments of the two launch groups of a linear verification (row
// statistics with every request's accept decisions, then the draw with the
// optional compaction), shared by linear.cu, rows_topp.cu and decide.cu,
// which are compiled with different CTA sizes; and the layout of the
// caller's workspace.
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
    RowStat* stats;  // workspace: target rows [B*(k+1)], then draft rows [B*k]
    int32_t* dec;    // workspace: per request a | (invalid bits << 16)
    int32_t* woff;   // workspace: packed offsets of the accepted positions [B+1]
    // workspace counters (zeroed by the call): [0] CTAs of the finishing
    // launch that are done, [2] rows the one-read top-p pass left for the
    // two-pass kernel
    unsigned* done;
    // compaction in the draw launch (hidden NULL: none), as spec_compact_accepted
    // with T = W = k + 1 and the linear layout
    const uint16_t* hidden;  // [B, k+1, H]
    int H;
    uint16_t* out_hidden;    // [B*(k+1), H]
    int32_t* offsets;        // [B+1]
    int32_t* next_tokens;    // [B*(k+1)]
    bool vec_ok;             // H*2 % 16 == 0 and both hidden pointers 16-byte aligned
    // draft-side sampler on the one-read pass (B rows of logits in tgt, k = 0):
    // the token of each row, or kSampleRedo for the two-pass sampler
    int32_t* sample_out;
};

constexpr int32_t kSampleRedo = -2;

__device__ __forceinline__ int tgt_row(const LinearArgs& a, int b, int i) { return b * (a.k + 1) + i; }
__device__ __forceinline__ int drf_row(const LinearArgs& a, int b, int i) { return a.B * (a.k + 1) + b * a.k + i; }

// Workspace of a linear call: the row records, the decisions, the offsets
// and the completion counter, each on a 256-byte boundary.
struct LinearWorkspace {
    size_t dec, woff, done, total;
};
__host__ __device__ inline size_t ws_round(size_t x) { return (x + 255) & ~(size_t)255; }
__host__ __device__ inline LinearWorkspace linear_workspace(int B, int k) {
    const size_t rows = (size_t)B * (2 * (size_t)k + 1);
    LinearWorkspace w;
    w.dec = ws_round(rows * sizeof(RowStat));
    w.woff = w.dec + ws_round((size_t)B * 4);
    w.done = w.woff + ws_round(((size_t)B + 1) * 4);
    w.total = w.done + 256;
    return w;
}

// Stage 1 for bf16 rows under top-p (rows_topp.cu): one read per row; rows
// it cannot finish are marked kRowRedo for the two-pass kernel.
spec_status launch_rows_topp_onepass(LinearArgs& a, cudaStream_t st);
// The draft-side sampler's first launch (rows_topp.cu): tokens of bf16 rows
// under top-p in one read each; kSampleRedo where the row needs the two-pass route.
spec_status launch_sample_onepass(LinearArgs& a, cudaStream_t st);

// Stage 2 for bf16 sampled rows with 16-byte aligned units (draw_stream.cu):
// the rows streamed through shared memory by bulk copies.
bool draw_stream_applies(const LinearArgs& a, int mode);
spec_status launch_draw_stream(LinearArgs& a, int mode, cudaStream_t st);

// Stage 2 (decide.cu): the residual or bonus draw and the optional
// compaction, one CTA per request.
spec_status launch_decide_stage(LinearArgs& a, spec_dtype dtype, int mode, cudaStream_t st);

}  // namespace sv
