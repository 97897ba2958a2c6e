// The residual or bonus draw of a linear verification over bf16 rows
// ("Accelerating Sonar through speculation", §Target-Draft; the cited rule:
// at the first rejection the token is drawn from norm(max(0, p - q)), after
// a full accept from p).  The draw is the smallest v with C(v) > u * C(last),
// C the running sum of the weights in index order.
//
// Same result as draw_linear, with less work per element, because only the
// selected rows are read and each element is touched once:
//  - weights are taken relative to p's normaliser: max(0, p - q) / (1/Z_p) =
//    max(0, e_p - (Z_p/Z_q) e_q) with e = 2^((x - m) c), so an element costs
//    one fused multiply-add, not a scale of each row and a difference;
//  - nucleus membership is one packed bf16x2 compare per element pair, and
//    a non-member is replaced by -inf before the exponent (its weight is 0);
//  - a lane sums 16 units (128 elements) of a step in fp32 before the
//    float-float warp sum, so a step (512 units) costs one warp reduction;
//  - tokens valued exactly at a row's nucleus boundary tau (kept only up to
//    the row's cut, not known before the row is read) are only flagged per
//    unit in the pass; each lane then revisits its flagged units (a few in a
//    step, from L1) for the per-step counts and corrections.
#pragma once

#include "sample.cuh"

namespace sv {

constexpr int kBSub = kNW;                  // 32-unit sub-steps of a step: one per warp
constexpr int kBDrawUnits = kBSub;          // units per lane in a step
constexpr int kBDrawStep = 32 * kBDrawUnits;
constexpr int kBDrawMaxSteps = (int)((kMaxVocab / 8 + 2 + kBDrawStep - 1) / kBDrawStep);

struct BDrawScratch {
    float base_h[kBDrawMaxSteps], base_l[kBDrawMaxSteps];  // step sums, every tau-valued token kept
    float dp[kBDrawMaxSteps];   // change when the step's tau_p-valued tokens are dropped
    float dq[kBDrawMaxSteps];   // ... its tau_q-valued tokens
    float dpq[kBDrawMaxSteps];  // the extra change when both are dropped
    int cpq[kBDrawMaxSteps];    // tau_p-valued count | tau_q-valued count << 16
    float sub_h[kBSub], sub_l[kBSub];
    int sub_i[kBSub], sub_j[kBSub];
};

// Packed bf16x2 compares: each half 0xffff where true, else 0.
__device__ __forceinline__ uint32_t bf2_ge(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf2_eq(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("set.eq.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// Bits of the smallest bf16 above the finite value with bits t.
__device__ __forceinline__ uint32_t bf16_above(uint32_t t) {
    if ((t & 0x7fffu) == 0u) return 1u;  // +-0: the smallest positive subnormal
    return (t & 0x8000u) ? t - 1u : t + 1u;
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int j) {
    return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// One filtered bf16 row as the draw reads it.
struct BRow {
    const uint16_t* row;
    float nmc;        // -m c
    float inv;        // 1 / kept mass: p = e inv
    float tau;        // nucleus boundary value (-inf: every token kept)
    uint32_t tau1;    // its bits; tau2 = both halves
    uint32_t tau2, above2;  // x >= tau; x > tau as x >= the next bf16 up
    uint32_t flag2;   // tau2 when the row drops tau-valued tokens, else a NaN (matches nothing)
    int cut;          // tau-valued tokens with index <= cut are kept
    int n_keep_minus1;  // the cut is the (n_keep)-th tau-valued token
    bool need;        // some tau-valued tokens are dropped: the cut must be found
    __device__ BRow(const uint16_t* r, const RowStat& st, float c, bool topp) : row(r) {
        nmc = -scaled_max(st.m, c);
        inv = st.inv_zn;
        tau = topp ? st.tau : -INFINITY;
        need = topp && st.tau > -INFINITY && st.n_keep < st.c_tau;
        tau1 = (__float_as_uint(st.tau) >> 16) & 0xffffu;
        tau2 = tau1 | (tau1 << 16);
        const uint32_t a1 = bf16_above(tau1);
        above2 = a1 | (a1 << 16);
        flag2 = need ? tau2 : 0x7fc07fc0u;
        cut = 0x7fffffff;
        n_keep_minus1 = st.n_keep - 1;
    }
};

// e = 2^((x - m) c) of the element pair in word x at indices i, i + 1, with
// non-members of the nucleus at 0.  EXACT: membership at the row's cut;
// otherwise every tau-valued token counts as kept.
template <bool TOPP, bool EXACT>
__device__ __forceinline__ float2 pair_exp(const BRow& R, float c, uint32_t x, int i) {
    if (TOPP) {
        uint32_t thr = R.tau2;
        if (EXACT) {
            const uint32_t a1 = R.above2 & 0xffffu;
            thr = ((i <= R.cut) ? R.tau1 : a1) | (((i + 1 <= R.cut) ? R.tau1 : a1) << 16);
        }
        const uint32_t m = bf2_ge(x, thr);
        x = (x & m) | (0xff80ff80u & ~m);  // non-members become -inf
    }
    const float2 t = __ffma2_rn(make_float2(bf16_lo(x), bf16_hi(x)), make_float2(c, c), make_float2(R.nmc, R.nmc));
    return make_float2(ex2(t.x), ex2(t.y));
}

// Weights of one unit (8 elements from index i0; padding slots hold -inf):
// w = max(0, e_p - r e_q) (RESID) or e_p, and pw = e_p; returns their sum
// added pairwise into acc.
template <bool RESID, bool TOPP, bool EXACT>
__device__ __forceinline__ void unit_weights(const BRow& P, const BRow& Q, float c, float r, const uint4& vp,
                                             const uint4& vq, int i0, float2& acc, float* w, float* pw) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 ep = pair_exp<TOPP, EXACT>(P, c, word_of(vp, j), i0 + 2 * j);
        float2 ww = ep;
        if (RESID) {
            const float2 eq = pair_exp<TOPP, EXACT>(Q, c, word_of(vq, j), i0 + 2 * j);
            const float2 d = __ffma2_rn(eq, make_float2(-r, -r), ep);
            ww = make_float2(fmaxf(d.x, 0.0f), fmaxf(d.y, 0.0f));
        }
        acc = __fadd2_rn(acc, ww);
        w[2 * j] = ww.x;
        w[2 * j + 1] = ww.y;
        pw[2 * j] = ep.x;
        pw[2 * j + 1] = ep.y;
    }
}

// The 16 bytes of elements [i0, i0 + cnt) of a bf16 row, -inf padded.
__device__ __forceinline__ uint4 bf16_unit(const uint16_t* row, int i0, int cnt) {
    const uint16_t* q = row + i0;
    if (cnt == 8 && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) return __ldg(reinterpret_cast<const uint4*>(q));
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t lo = (2 * j < cnt) ? q[2 * j] : 0xff80u;
        const uint32_t hi = (2 * j + 1 < cnt) ? q[2 * j + 1] : 0xff80u;
        w[j] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Step pass of one warp over its steps: base sums with every tau-valued
// token kept; with TRACK, the counts and corrections of the tau-valued
// tokens.  fastq: Q's units are aligned as P's.
template <bool RESID, bool TOPP, bool TRACK>
__device__ void bdraw_steps(const RowView<__nv_bfloat16>& rv, const BRow& P, const BRow& Q, float c, float r,
                            bool fastq, BDrawScratch& ds) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int units = rv.units();
    const int nsteps = (units + kBDrawStep - 1) / kBDrawStep;
    const uint16_t* pbody = P.row + rv.head;
    const uint16_t* qbody = Q.row + rv.head;
    const uint4 ninf = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
    auto load = [&](const uint16_t* row, int u, bool fast, int& i0) -> uint4 {
        if (fast) {
            i0 = rv.head + (u - 1) * 8;
            return __ldg(reinterpret_cast<const uint4*>(row + i0));
        }
        int cnt = 0;
        i0 = 0;
        if (u < units) rv.unit_range(u, i0, cnt);
        return cnt ? bf16_unit(row, i0, cnt) : ninf;
    };
    for (int st = warp; st < nsteps; st += kNW) {
        const int ub = st * kBDrawStep + lane;  // this lane's first unit of the step
        const bool fast = st * kBDrawStep >= 1 && (st + 1) * kBDrawStep - 1 <= rv.nvec;
        float2 acc = make_float2(0.0f, 0.0f);
        uint32_t flags = 0u;
        float w[8], pw[8];
        if (fast && (fastq || !RESID)) {
            const uint4* pv = reinterpret_cast<const uint4*>(pbody) + (ub - 1);
            const uint4* qv = reinterpret_cast<const uint4*>(qbody) + (ub - 1);
#pragma unroll 1
            for (int g0 = 0; g0 < kBDrawUnits; g0 += 4) {
                uint4 vp[4], vq[4];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    vp[g] = __ldg(pv + (g0 + g) * 32);
                    vq[g] = RESID ? __ldg(qv + (g0 + g) * 32) : ninf;
                }
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int i0 = rv.head + (ub - 1 + (g0 + g) * 32) * 8;
                    unit_weights<RESID, TOPP, false>(P, Q, c, r, vp[g], vq[g], i0, acc, w, pw);
                    if (TRACK) {
                        uint32_t e = bf2_eq(vp[g].x, P.flag2) | bf2_eq(vp[g].y, P.flag2) | bf2_eq(vp[g].z, P.flag2) |
                                     bf2_eq(vp[g].w, P.flag2);
                        if (RESID)
                            e |= bf2_eq(vq[g].x, Q.flag2) | bf2_eq(vq[g].y, Q.flag2) | bf2_eq(vq[g].z, Q.flag2) |
                                 bf2_eq(vq[g].w, Q.flag2);
                        if (e) flags |= 1u << (g0 + g);
                    }
                }
            }
        } else {
#pragma unroll 1
            for (int g = 0; g < kBDrawUnits; ++g) {
                const int u = ub + g * 32;
                int i0;
                const uint4 vp = load(P.row, u, false, i0);
                const uint4 vq = RESID ? load(Q.row, u, false, i0) : ninf;
                unit_weights<RESID, TOPP, false>(P, Q, c, r, vp, vq, i0, acc, w, pw);
                if (TRACK) {
                    uint32_t e = bf2_eq(vp.x, P.flag2) | bf2_eq(vp.y, P.flag2) | bf2_eq(vp.z, P.flag2) |
                                 bf2_eq(vp.w, P.flag2);
                    if (RESID)
                        e |= bf2_eq(vq.x, Q.flag2) | bf2_eq(vq.y, Q.flag2) | bf2_eq(vq.z, Q.flag2) |
                             bf2_eq(vq.w, Q.flag2);
                    if (e) flags |= 1u << g;
                }
            }
        }
        const ff t = warp_sum_ff(ff_from(acc.x + acc.y));
        float dp = 0.0f, dq = 0.0f, dpq = 0.0f;
        int npq = 0;
        if (TRACK) {
            // the flagged units again (from L1): per-element counts and corrections
            uint32_t f = flags;
            while (f) {
                const int g = __ffs(f) - 1;
                f &= f - 1u;
                const int u = ub + g * 32;
                int i0;
                const bool vf = fast && (fastq || !RESID);
                const uint4 vp = load(P.row, u, vf, i0);
                const uint4 vq = RESID ? load(Q.row, u, vf, i0) : ninf;
                float2 dummy = make_float2(0.0f, 0.0f);
                unit_weights<RESID, TOPP, false>(P, Q, c, r, vp, vq, i0, dummy, w, pw);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t wp = word_of(vp, j >> 1), wq = word_of(vq, j >> 1);
                    const float xp = (j & 1) ? bf16_hi(wp) : bf16_lo(wp);
                    const float xq = (j & 1) ? bf16_hi(wq) : bf16_lo(wq);
                    const bool ip = P.need && xp == P.tau;
                    const bool iq = RESID && Q.need && xq == Q.tau;
                    if (ip) dp -= w[j];               // p dropped: max(0, 0 - q) = 0
                    if (iq) dq += pw[j] - w[j];       // q dropped: max(0, p - 0) = p
                    if (ip && iq) dpq += w[j] - pw[j];  // both dropped: 0
                    npq += (ip ? 1 : 0) + (iq ? 0x10000 : 0);
                }
            }
            if (__any_sync(0xffffffffu, flags != 0u)) {
                dp = warp_sum_f(dp);
                dq = warp_sum_f(dq);
                dpq = warp_sum_f(dpq);
                npq = warp_sum_i(npq);
            }
        }
        if (lane == 0) {
            ds.base_h[st] = t.hi;
            ds.base_l[st] = t.lo;
            ds.dp[st] = dp;
            ds.dq[st] = dq;
            ds.dpq[st] = dpq;
            ds.cpq[st] = npq;
        }
    }
}

// Inverse-CDF draw over the bf16 row pair with weights max(0, p - q) (RESID)
// or p: the smallest v with C(v) > u * C(last).  On return P.cut and Q.cut
// are set.  Returns -1 when every weight is zero.
template <bool RESID, bool TOPP>
__device__ int draw_linear_bf16(const RowView<__nv_bfloat16>& rv, BRow& P, BRow& Q, float c, float u, BlockScratch& s,
                                BDrawScratch& ds) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int units = rv.units();
    const int nsteps = (units + kBDrawStep - 1) / kBDrawStep;
    const uint4 ninf = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
    // max(0, p - q) = (1 / Z_p) max(0, e_p - r e_q) with r = Z_p / Z_q
    const float r = RESID ? Q.inv / P.inv : 0.0f;
    const bool needP = TOPP && P.need, needQ = TOPP && RESID && Q.need;
    const bool fastq = !RESID || ((reinterpret_cast<uintptr_t>(Q.row) - reinterpret_cast<uintptr_t>(P.row)) & 15u) == 0;
    P.cut = 0x7fffffff;
    Q.cut = 0x7fffffff;
    // A: step sums (every tau-valued token kept), counts and corrections
    if (needP || needQ)
        bdraw_steps<RESID, TOPP, true>(rv, P, Q, c, r, fastq, ds);
    else
        bdraw_steps<RESID, TOPP, false>(rv, P, Q, c, r, fastq, ds);
    row_sync();
    // unit u of the row pair, -inf padded (units past the end: all -inf)
    auto load2 = [&](int uu, uint4& vp, uint4& vq) -> int {
        int i0 = 0, cnt = 0;
        if (uu < units) rv.unit_range(uu, i0, cnt);
        vp = cnt ? bf16_unit(P.row, i0, cnt) : ninf;
        vq = (RESID && cnt) ? bf16_unit(Q.row, i0, cnt) : ninf;
        return i0;
    };
    // B1: the steps holding the cuts (warp 0): the n_keep-th tau-valued token of each row
    if (warp == 0) {
        auto cut_step = [&](int shift, int n, int& js, int& pre) {
            js = -1;
            pre = 0;
            const int per = (nsteps + 31) / 32;
            int ls = 0;
            for (int i = 0; i < per; ++i) {
                const int st = lane * per + i;
                if (st < nsteps) ls += (ds.cpq[st] >> shift) & 0xffff;
            }
            const int incl = warp_inclusive_scan_i(ls);
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            if (n < 0 || n >= total) return;  // every tau-valued token kept
            const unsigned bal = __ballot_sync(0xffffffffu, incl > n);
            const int L = __ffs(bal) - 1;
            if (lane == L) {
                int run = incl - ls;
                for (int i = 0; i < per; ++i) {
                    const int st = lane * per + i;
                    const int cn = (ds.cpq[st] >> shift) & 0xffff;
                    if (run + cn > n) { js = st; pre = run; break; }
                    run += cn;
                }
            }
            js = __shfl_sync(0xffffffffu, js, L);
            pre = __shfl_sync(0xffffffffu, pre, L);
        };
        int jsp = -1, prep = 0, jsq = -1, preq = 0;
        if (needP) cut_step(0, P.n_keep_minus1, jsp, prep);
        if (needQ) cut_step(16, Q.n_keep_minus1, jsq, preq);
        if (lane == 0) {
            s.bcast_i[0] = jsp;
            s.bcast_i[1] = prep;
            s.bcast_i[2] = jsq;
            s.bcast_i[3] = preq;
        }
    }
    row_sync();
    const int jsp = s.bcast_i[0], prep = s.bcast_i[1], jsq = s.bcast_i[2], preq = s.bcast_i[3];
    row_sync();
    // B2: the cut index inside its step; warp w takes the step's sub-step w
    auto locate = [&](int js, int pre, int n, bool isq) -> int {
        const BRow& R = isq ? Q : P;
        uint4 vp, vq;
        const int i0 = load2(js * kBDrawStep + warp * 32 + lane, vp, vq);
        const uint4 v = isq ? vq : vp;
        unsigned msk = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t wd = word_of(v, j >> 1);
            if (((j & 1) ? bf16_hi(wd) : bf16_lo(wd)) == R.tau) msk |= 1u << j;
        }
        const int cw = warp_sum_i(__popc(msk));
        if (lane == 0) ds.sub_i[warp] = cw;
        if (threadIdx.x == 0) s.bcast_i[4] = 0x7fffffff;
        row_sync();
        int base = pre, gsel = -1, gpre = 0;
        for (int g = 0; g < kBSub; ++g) {
            if (gsel < 0 && base + ds.sub_i[g] > n) { gsel = g; gpre = base; }
            base += ds.sub_i[g];
        }
        if (warp == gsel) {
            const int cl = __popc(msk);
            const int ic = warp_inclusive_scan_i(cl);
            if (gpre + ic > n && gpre + ic - cl <= n) {
                int kk = n - (gpre + ic - cl);
                for (int j = 0; j < 8; ++j)
                    if (msk & (1u << j)) {
                        if (kk == 0) { s.bcast_i[4] = i0 + j; break; }
                        --kk;
                    }
            }
        }
        row_sync();
        const int res = s.bcast_i[4];
        row_sync();
        return res;
    };
    if (jsp >= 0) P.cut = locate(jsp, prep, P.n_keep_minus1, false);
    if (jsq >= 0) Q.cut = locate(jsq, preq, Q.n_keep_minus1, true);
    // B3: exact sums of the cut steps (with the cuts now known)
    auto exact_step = [&](int js) -> ff {
        uint4 vp, vq;
        const int i0 = load2(js * kBDrawStep + warp * 32 + lane, vp, vq);
        float2 acc = make_float2(0.0f, 0.0f);
        float w[8], pw[8];
        unit_weights<RESID, TOPP, true>(P, Q, c, r, vp, vq, i0, acc, w, pw);
        const ff t = warp_sum_ff(ff_from(acc.x + acc.y));
        if (lane == 0) {
            ds.sub_h[warp] = t.hi;
            ds.sub_l[warp] = t.lo;
        }
        row_sync();
        ff res = ff{0.0f, 0.0f};
        for (int g = 0; g < kBSub; ++g) res = ff_add(res, ff{ds.sub_h[g], ds.sub_l[g]});
        row_sync();
        return res;
    };
    const ff exact_p = (jsp >= 0) ? exact_step(jsp) : ff{0.0f, 0.0f};
    const ff exact_q = (jsq >= 0 && jsq != jsp) ? exact_step(jsq) : exact_p;
    auto step_sum = [&](int st) -> ff {
        if (st == jsp) return exact_p;
        if (st == jsq) return exact_q;
        ff v = ff{ds.base_h[st], ds.base_l[st]};
        const bool past_p = jsp >= 0 && st > jsp, past_q = jsq >= 0 && st > jsq;
        float d = 0.0f;
        if (past_p) d += ds.dp[st];
        if (past_q) d += ds.dq[st];
        if (past_p && past_q) d += ds.dpq[st];
        return d != 0.0f ? ff_add_f(v, d) : v;
    };
    // B4: the crossing step (warp 0)
    if (warp == 0) {
        const int per = (nsteps + 31) / 32;
        ff ls = ff{0.0f, 0.0f};
        int lastpos = -1;
        for (int i = 0; i < per; ++i) {
            const int st = lane * per + i;
            if (st < nsteps) {
                const ff sv = step_sum(st);
                ls = ff_add(ls, sv);
                if (sv.hi > 0.0f) lastpos = st;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
        const ff incl = warp_inclusive_scan_ff(ls);
        const ff tot = ff_shfl(incl, 31);
        int js = -1;
        ff pre = ff{0.0f, 0.0f}, tgt = ff{0.0f, 0.0f};
        if (tot.hi > 0.0f) {
            tgt = ff_mul_f(tot, u);
            const ff up = ff_shfl_up(incl, 1);
            const ff before = lane == 0 ? ff{0.0f, 0.0f} : up;
            const unsigned bal = __ballot_sync(0xffffffffu, ls.hi > 0.0f && ff_lt(tgt, incl));
            if (bal) {
                const int L = __ffs(bal) - 1;
                if (lane == L) {
                    ff run = before;
                    for (int i = 0; i < per; ++i) {
                        const int st = lane * per + i;
                        if (st >= nsteps) break;
                        const ff sv = step_sum(st);
                        const ff nx = ff_add(run, sv);
                        if (sv.hi > 0.0f && ff_lt(tgt, nx)) { js = st; pre = run; break; }
                        run = nx;
                    }
                }
                js = __shfl_sync(0xffffffffu, js, L);
                pre = ff_shfl(pre, L);
            }
            if (js < 0) {  // rounding: the draw falls in the last step with weight
                js = lastpos;
                pre = ff{0.0f, 0.0f};
                tgt = ff{INFINITY, 0.0f};
            }
        }
        if (lane == 0) {
            s.bcast_i[5] = js;
            s.bcast_f[0] = pre.hi;
            s.bcast_f[1] = pre.lo;
            s.bcast_f[2] = tgt.hi;
            s.bcast_f[3] = tgt.lo;
        }
    }
    row_sync();
    const int js = s.bcast_i[5];
    const ff tgt = ff{s.bcast_f[2], s.bcast_f[3]};
    ff run = ff{s.bcast_f[0], s.bcast_f[1]};
    row_sync();
    if (js < 0) return -1;  // every weight is zero
    // C: the crossing step, warp w on its sub-step w
    uint4 vp, vq;
    const int i0 = load2(js * kBDrawStep + warp * 32 + lane, vp, vq);
    float2 acc = make_float2(0.0f, 0.0f);
    float w[8], pw[8];
    unit_weights<RESID, TOPP, true>(P, Q, c, r, vp, vq, i0, acc, w, pw);
    const float a_own = acc.x + acc.y;
    {
        const ff t = warp_sum_ff(ff_from(a_own));
        int mylast = -1;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (w[j] > 0.0f) mylast = i0 + j;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mylast = max(mylast, __shfl_xor_sync(0xffffffffu, mylast, o));
        if (lane == 0) {
            ds.sub_h[warp] = t.hi;
            ds.sub_l[warp] = t.lo;
            ds.sub_j[warp] = mylast;
        }
    }
    row_sync();
    int g_cross = -1, lastw = -1;
    ff pre_cross = run;
    for (int g = 0; g < kBSub; ++g) {  // the same order in every warp
        const ff sv = ff{ds.sub_h[g], ds.sub_l[g]};
        const ff nx = ff_add(run, sv);
        if (ds.sub_j[g] >= 0) lastw = ds.sub_j[g];
        if (g_cross < 0 && sv.hi > 0.0f && ff_lt(tgt, nx)) { g_cross = g; pre_cross = run; }
        run = nx;
    }
    if (threadIdx.x == 0 && g_cross < 0) s.bcast_i[6] = lastw;  // otherwise the crossing warp writes it
    if (warp == g_cross) {
        const ff ia = warp_inclusive_scan_ff(ff_from(a_own));
        const ff ua = ff_shfl_up(ia, 1);
        const ff ex = ff_add(pre_cross, lane == 0 ? ff{0.0f, 0.0f} : ua);
        const unsigned cb = __ballot_sync(0xffffffffu, a_own > 0.0f && ff_lt(tgt, ff_add(ex, ff_from(a_own))));
        int p = ds.sub_j[g_cross];  // rounding: the last weighted element of this sub-step
        if (cb) {
            const int L = __ffs(cb) - 1;
            int q = -1;
            if (lane == L) {
                ff rr = ex;
                int mylast = -1;
                for (int j = 0; j < 8 && q < 0; ++j) {
                    if (w[j] > 0.0f) mylast = i0 + j;
                    rr = ff_add_f(rr, w[j]);
                    if (w[j] > 0.0f && ff_lt(tgt, rr)) q = i0 + j;
                }
                if (q < 0) q = mylast;
            }
            p = __shfl_sync(0xffffffffu, q, L);
        }
        if (lane == 0) s.bcast_i[6] = p;
    }
    row_sync();
    const int res = s.bcast_i[6];
    row_sync();
    return res;
}

}  // namespace sv
