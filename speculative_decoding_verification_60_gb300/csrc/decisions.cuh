// Accept decisions of every request of a linear verification, and the
// packed row offsets of the accepted positions ("Accelerating Sonar through
// speculation", §Speculative decoding and §Target-Draft, with the rule of
// the cited "Fast Inference from Transformers via Speculative Decoding":
// d_i is accepted iff u_i < p(d_i) / q(d_i), the first rejection ends the
// run; §MTP: the accepted positions' hidden rows are packed for the next
// draft step).
//
// They run in the launch that follows the row statistics (every record is
// final then): one warp per request across the grid, lanes over the drafts,
// then the offsets in the last CTA to finish, which learns that it is last
// from a completion counter (each CTA adds one when its requests are
// written), so nothing waits.
#pragma once

#include "linear_args.cuh"

namespace sv {

// A row record read through L2 (other CTAs of this launch wrote it).
__device__ __forceinline__ RowStat load_stat_l2(const RowStat* p) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    const uint4 a = __ldcg(q), b = __ldcg(q + 1);
    RowStat st;
    st.m = __uint_as_float(a.x);
    st.inv_zn = __uint_as_float(a.y);
    st.x_tok = __uint_as_float(a.z);
    st.argmax = (int)a.w;
    st.tau = __uint_as_float(b.x);
    st.n_keep = (int)b.y;
    st.c_tau = (int)b.z;
    st.flags = (int)b.w;
    return st;
}

// One request's decisions on one warp, lanes over the drafts (so that the
// row records' loads overlap).  Writes accept_prob, token_probs (zeros for
// an invalid request), accepted_len, the length histogram, the device error
// bits and dec[b] = a | (invalid bits << 16).
template <int MODE>
__device__ void warp_request_decisions(const LinearArgs& a, int b) {
    const int k = a.k, lane = threadIdx.x & 31;
    const int32_t* d = a.drafts + (size_t)b * k;
    const int64_t req = a.req ? a.req[b] : (int64_t)b;
    const int64_t pos = a.pos ? a.pos[b] : 0;
    int inval = 0;
    for (int i = lane; i <= k; i += 32) {
        if (load_stat_l2(a.stats + tgt_row(a, b, i)).flags & kRowInvalid) inval |= kDevErrNonfinite;
        if (i < k) {
            if (MODE > 0 && (load_stat_l2(a.stats + drf_row(a, b, i)).flags & kRowInvalid)) inval |= kDevErrNonfinite;
            if (d[i] < 0 || d[i] >= a.V) inval |= kDevErrToken;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) inval |= __shfl_xor_sync(0xffffffffu, inval, o);
    int first_reject = k;
    for (int i0 = 0; i0 < k; i0 += 32) {
        const int i = i0 + lane;
        bool acc = true;
        float ap = 0.0f, pp = 0.0f, qq = 0.0f;
        if (i < k && !inval) {
            const RowStat sp = load_stat_l2(a.stats + tgt_row(a, b, i));
            if (MODE == 0) {
                acc = (d[i] == sp.argmax);
                ap = acc ? 1.0f : 0.0f;
                pp = ap;
                qq = 1.0f;
            } else {
                const RowStat sq = load_stat_l2(a.stats + drf_row(a, b, i));
                const bool pm = (sp.flags & kRowTokMember) != 0, qm = (sq.flags & kRowTokMember) != 0;
                pp = pm ? weight_of(sp.x_tok, a.c, scaled_max(sp.m, a.c)) * sp.inv_zn : 0.0f;
                qq = qm ? weight_of(sq.x_tok, a.c, scaled_max(sq.m, a.c)) * sq.inv_zn : 0.0f;
                // q = 0 (the token outside q's nucleus) rejects; a weight that
                // only underflowed in fp32 takes the ratio from the logits,
                // differenced before scaling (the exponents themselves are
                // large and would lose digits)
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
        const int acnt = inval ? 0 : first_reject;
        a.acc_len[b] = acnt;
        a.dec[b] = acnt | (inval << 16);
        if (a.len_hist) atomicAdd(a.len_hist + acnt, 1);
        if (inval && a.dev_error) atomicOr(a.dev_error, inval);
    }
}

// The offsets woff[b] = sum over b' < b of (a_b' + 1), woff[B] the total,
// from dec[] (written by this launch's CTAs, so read through L2).  All kNT
// threads of one CTA.
__device__ inline void linear_offsets(const LinearArgs& a, BlockScratch& s) {
    int carry = 0;
    for (int b0 = 0; b0 < a.B; b0 += kNT) {
        const int b = b0 + (int)threadIdx.x;
        const int rows = (b < a.B) ? (__ldcg(a.dec + b) & 0xffff) + 1 : 0;
        int tot;
        const int ex = block_exclusive_scan_i(rows, s, &tot);
        if (b < a.B) a.woff[b] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) a.woff[a.B] = carry;
}

// The last CTA of a launch to get here (counted in done[which]) returns true.
__device__ inline bool last_cta_done(const LinearArgs& a, unsigned* sh_ticket, int which) {
    row_sync();  // this CTA's writes are issued
    if (threadIdx.x == 0) {
        __threadfence();
        *sh_ticket = atomicAdd(a.done + which, 1u);
    }
    row_sync();
    if (*sh_ticket != gridDim.x - 1) return false;
    __threadfence();  // the other CTAs' writes are visible
    return true;
}

}  // namespace sv
