// Linear verification, stage 2 ("Accelerating Sonar through speculation",
// §Speculative decoding and §Target-Draft; the cited rule): per request the
// draw from norm(max(0, p - q)) at the first rejection or from the last
// target row after a full accept (the accept tests and the accepted length
// come from the statistics launch), and the optional compaction.  Built
// with 512-thread CTAs: one request per CTA, so more warps per request
// shorten its draw.
#include "launch.cuh"
#include "linear_args.cuh"
#include "draw_bf16.cuh"
#include "sample.cuh"

namespace sv {

// One CTA per request: the residual or bonus draw at the request's accept
// decisions (taken by the statistics launch), its output tokens and, for
// the compacting call, its accepted hidden rows and their next tokens at
// the packed offset (§MTP: token t_{i+1} pairs with hidden state H_i;
// §MTP schedule for a single token: the next tokens are inserted on the
// GPU, without a host round trip).
template <typename T, int MODE>
__global__ void __launch_bounds__(kNT, 2) k_linear_finalize(LinearArgs a) {
    __shared__ BlockScratch s;
    __shared__ union {
        DrawScratch d;    // fp32 rows
        BDrawScratch b;   // bf16 rows
    } ds;
    const int b = blockIdx.x, k = a.k, V = a.V;
    grid_dep_wait();  // the decisions and offsets come from the launch before
    const int64_t req = a.req ? a.req[b] : (int64_t)b;
    const int64_t pos = a.pos ? a.pos[b] : 0;
    const int32_t* d = a.drafts + (size_t)b * k;
    const int dv = a.dec[b];
    const int acnt = dv & 0xffff, inval = dv >> 16;
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
        const bool resid = acnt < k;
        const float u = uniform01(a.seed, req, pos + acnt + 1, resid ? kPurposeResidual : kPurposeBonus, 0);
        const RowStat sq = resid ? a.stats[drf_row(a, b, acnt)] : sp;
        const T* qrow = resid ? static_cast<const T*>(a.drf) + ((size_t)b * k + acnt) * V : prow;
        if constexpr (sizeof(T) == 2) {
            BRow P(reinterpret_cast<const uint16_t*>(prow), sp, a.c, MODE == 2);
            if (resid) {
                BRow Q(reinterpret_cast<const uint16_t*>(qrow), sq, a.c, MODE == 2);
                t = draw_linear_bf16<true, (MODE == 2)>(rv, P, Q, a.c, u, s, ds.b);
                if (t < 0) t = draw_linear_bf16<false, (MODE == 2)>(rv, P, P, a.c, u, s, ds.b);  // p == q: draw from p
            } else {
                t = draw_linear_bf16<false, (MODE == 2)>(rv, P, P, a.c, u, s, ds.b);
            }
        } else {
            FilteredRow<T> P(prow, sp, a.c, 0x7fffffff);
            if (resid) {
                FilteredRow<T> Q(qrow, sq, a.c, 0x7fffffff);
                t = draw_linear<T, true, (MODE == 2)>(rv, P, Q, u, s, ds.d);
                if (t < 0) t = draw_linear<T, false, (MODE == 2)>(rv, P, Q, u, s, ds.d);  // p == q: draw from p
            } else {
                t = draw_linear<T, false, (MODE == 2)>(rv, P, P, u, s, ds.d);
            }
        }
    }
    if (threadIdx.x == 0) {
        int32_t* o = a.out_tokens + (size_t)b * (k + 1);
        for (int j = 0; j <= k; ++j) o[j] = (j < acnt) ? d[j] : (j == acnt ? t : -1);
    }
    if (a.hidden) {  // rows 0 .. a of this request, packed at its offset
        const int off = a.woff[b];
        for (int r = 0; r <= acnt; ++r) {
            const uint16_t* in = a.hidden + ((size_t)b * (k + 1) + r) * a.H;
            uint16_t* out = a.out_hidden + (size_t)(off + r) * a.H;
            if (a.vec_ok) {
                const uint4* vi = reinterpret_cast<const uint4*>(in);
                uint4* vo = reinterpret_cast<uint4*>(out);
                for (int i = threadIdx.x; i < a.H / 8; i += kNT) vo[i] = __ldg(vi + i);
            } else {
                for (int i = threadIdx.x; i < a.H; i += kNT) out[i] = in[i];
            }
        }
        if (threadIdx.x == 0) {
            for (int r = 0; r <= acnt; ++r) a.next_tokens[off + r] = (r < acnt) ? d[r] : t;
            a.offsets[b + 1] = a.woff[b + 1];
            if (b == 0) a.offsets[0] = 0;
        }
    }
}

template <typename T, int MODE>
static spec_status launch_decide(LinearArgs& a, cudaStream_t st) {
    if (launch_dependent(k_linear_finalize<T, MODE>, dim3(a.B), dim3(kNT), 0, st, a) != cudaSuccess) return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

template <typename T>
static spec_status launch_decide_t(LinearArgs& a, int mode, cudaStream_t st) {
    if (mode == 0) return launch_decide<T, 0>(a, st);
    if (mode == 1) return launch_decide<T, 1>(a, st);
    return launch_decide<T, 2>(a, st);
}

spec_status launch_decide_stage(LinearArgs& a, spec_dtype dtype, int mode, cudaStream_t st) {
    if (dtype == SPEC_BF16 && draw_stream_applies(a, mode)) return launch_draw_stream(a, mode, st);
    return dtype == SPEC_BF16 ? launch_decide_t<__nv_bfloat16>(a, mode, st) : launch_decide_t<float>(a, mode, st);
}

}  // namespace sv
