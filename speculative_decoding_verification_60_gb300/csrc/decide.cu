// Linear verification, stage 2 ("Accelerating Sonar through speculation",
// §Speculative decoding and §Target-Draft; the cited rule): per request the
// accept tests u_i < p(d_i) / q(d_i) in order, the accepted length, and the
// draw from norm(max(0, p - q)) at the first rejection or from the last
// target row after a full accept.  Built with 512-thread CTAs: one request
// per CTA, so more warps per request shorten its draw.
#include "launch.cuh"
#include "linear_args.cuh"
#include "sample.cuh"

namespace sv {

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
                    const bool pm = (sp.flags & kRowTokMember) != 0, qm = (sq.flags & kRowTokMember) != 0;
                    const float lp = fmaf(sp.x_tok, a.c, -scaled_max(sp.m, a.c));  // log2 of the weights
                    const float lq = fmaf(sq.x_tok, a.c, -scaled_max(sq.m, a.c));
                    pp = pm ? ex2(lp) * sp.inv_zn : 0.0f;
                    qq = qm ? ex2(lq) * sq.inv_zn : 0.0f;
                    // q = 0 (the token outside q's nucleus) rejects; a weight
                    // that only underflowed in fp32 takes the ratio from the
                    // logits, differenced before scaling (the exponents
                    // themselves are large and would lose digits)
                    float ratio = 0.0f;
                    if (pm && qm)
                        ratio = (pp > 0.0f && qq > 0.0f)
                                    ? pp / qq
                                    : ex2(((sp.x_tok - sq.x_tok) - (sp.m - sq.m)) * a.c) * (sp.inv_zn / sq.inv_zn);
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

template <typename T, int MODE>
static spec_status launch_decide(LinearArgs& a, cudaStream_t st) {
    k_linear_finalize<T, MODE><<<a.B, kNT, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

template <typename T>
static spec_status launch_decide_t(LinearArgs& a, int mode, cudaStream_t st) {
    if (mode == 0) return launch_decide<T, 0>(a, st);
    if (mode == 1) return launch_decide<T, 1>(a, st);
    return launch_decide<T, 2>(a, st);
}

spec_status launch_decide_stage(LinearArgs& a, spec_dtype dtype, int mode, cudaStream_t st) {
    return dtype == SPEC_BF16 ? launch_decide_t<__nv_bfloat16>(a, mode, st) : launch_decide_t<float>(a, mode, st);
}

}  // namespace sv
