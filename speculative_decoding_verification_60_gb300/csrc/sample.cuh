// Block-wide inverse-CDF draw over one vocabulary row (or row pair).
//
// "Accelerating Sonar through speculation", §Target-Draft: at the
// mismatch, or after the last draft, the target logits are sampled for one
// more token; the cited rule draws that token from norm(max(0, p - q)) at a
// rejection and from p after a full accept.  The draw is the smallest v with
// C(v) > u * C(V-1), C the running sum of the weights in index order.
//
// The row is walked in the step layout of the block-wide searches (per-step
// sums, one barrier); warp 0 then finds the crossing step and walks it.  Only the selected row(s) are
// read, once plus one step.
#pragma once

#include "rowstats.cuh"

namespace sv {

// WeightFn: void operator()(int unit, float* w /*[VEC]*/, int& idx0, int& cnt) const
// Returns the drawn index, or -1 when every weight is zero.
template <int VEC, typename WeightFn>
__device__ int block_inverse_cdf(int units, float u, const WeightFn& wf, BlockScratch& s, SampleScratch& ss) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nsteps = (units + kStepUnits - 1) / kStepUnits;
    const int spw = steps_per_warp(units);
    auto unit_sum = [&](int unit, float* w, int& i0, int& cnt) -> float {
        float a = 0.0f;
        i0 = 0;
        cnt = 0;
        if (unit < units) {
            wf(unit, w, i0, cnt);
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (j < cnt) a += w[j];
        }
        return a;
    };
    // A: step sums
    for (int st = warp * spw; st < (warp + 1) * spw && st < nsteps; ++st) {
        float a = 0.0f;
#pragma unroll
        for (int g = 0; g < kStepUnits / 32; ++g) {
            float w[VEC];
            int i0, cnt;
            a += unit_sum(st * kStepUnits + g * 32 + lane, w, i0, cnt);
        }
        const ff t = warp_sum_ff(ff_from(a));
        if (lane == 0) {
            ss.sh[st] = t.hi;
            ss.sl[st] = t.lo;
        }
    }
    row_sync();
    // B + C: warp 0 finds the crossing step and walks it
    if (warp == 0) {
        const int per = (nsteps + 31) / 32;
        ff ls = ff{0.0f, 0.0f};
        for (int i = 0; i < per; ++i) {
            const int st = lane * per + i;
            if (st < nsteps) ls = ff_add(ls, ff{ss.sh[st], ss.sl[st]});
        }
        const ff incl = warp_inclusive_scan_ff(ls);
        const ff tot = ff_shfl(incl, 31);
        int pick = -1;
        if (tot.hi > 0.0f) {
            const ff target = ff_mul_f(tot, u);
            const ff up = ff_shfl_up(incl, 1);
            const ff before = lane == 0 ? ff{0.0f, 0.0f} : up;
            // crossing lane: the first whose running sum exceeds the target
            const unsigned bal = __ballot_sync(0xffffffffu, ls.hi > 0.0f && ff_lt(target, incl));
            // last step with weight (for a crossing lost to rounding)
            int lastpos = -1;
            for (int i = 0; i < per; ++i) {
                const int st = lane * per + i;
                if (st < nsteps && ss.sh[st] > 0.0f) lastpos = st;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
            int js = -1;
            ff pre = ff{0.0f, 0.0f};
            if (bal) {
                const int L = __ffs(bal) - 1;
                if (lane == L) {
                    ff run = before;
                    for (int i = 0; i < per; ++i) {
                        const int st = lane * per + i;
                        if (st >= nsteps) break;
                        const ff sv = ff{ss.sh[st], ss.sl[st]};
                        const ff nx = ff_add(run, sv);
                        if (sv.hi > 0.0f && ff_lt(target, nx)) { js = st; pre = run; break; }
                        run = nx;
                    }
                }
                js = __shfl_sync(0xffffffffu, js, L);
                pre = ff_shfl(pre, L);
            }
            ff tgt = target;
            if (js < 0) {  // rounding: the draw falls in the last step with weight
                js = lastpos;
                pre = ff{0.0f, 0.0f};
                tgt = ff{INFINITY, 0.0f};
            }
            // C: walk step js, 32 units at a time
            int lastw = -1;
            for (int g = 0; g < kStepUnits / 32 && pick < 0; ++g) {
                float w[VEC];
                int i0, cnt;
                const float a = unit_sum(js * kStepUnits + g * 32 + lane, w, i0, cnt);
                const ff ia = warp_inclusive_scan_ff(ff_from(a));
                const ff ua = ff_shfl_up(ia, 1);
                const ff ex = ff_add(pre, lane == 0 ? ff{0.0f, 0.0f} : ua);
                int mylast = -1;
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (j < cnt && w[j] > 0.0f) mylast = i0 + j;
                const unsigned cb = __ballot_sync(0xffffffffu, a > 0.0f && ff_lt(tgt, ff_add(ex, ff_from(a))));
                int p = -1;
                if (cb) {
                    const int L = __ffs(cb) - 1;
                    if (lane == L) {
                        ff run = ex;
                        for (int j = 0; j < VEC && p < 0; ++j) {
                            if (j >= cnt) break;
                            run = ff_add_f(run, w[j]);
                            if (w[j] > 0.0f && ff_lt(tgt, run)) p = i0 + j;
                        }
                        if (p < 0) p = mylast;
                    }
                    p = __shfl_sync(0xffffffffu, p, L);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mylast = max(mylast, __shfl_xor_sync(0xffffffffu, mylast, o));
                if (mylast >= 0) lastw = mylast;
                pick = p;
                pre = ff_add(pre, ff_shfl(ia, 31));
            }
            if (pick < 0) pick = lastw;  // the step's sums fell short by rounding
        }
        if (lane == 0) s.bcast_i[7] = pick;
    }
    row_sync();
    const int r = s.bcast_i[7];
    row_sync();
    return r;
}

// Sum over a row of a per-unit weight function (float-float, fixed order).
template <int VEC, typename WeightFn>
__device__ ff block_weight_total(int units, const WeightFn& wf, BlockScratch& s) {
    ff acc = ff{0.0f, 0.0f};
    for (int unit = threadIdx.x; unit < units; unit += kNT) {
        float w[VEC];
        int i0, cnt;
        wf(unit, w, i0, cnt);
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (j < cnt) a += w[j];
        acc = ff_add_f(acc, a);
    }
    return block_sum_ff(acc, s);
}

// Filtered probabilities of a filtered row over an index range of at most
// VEC elements (vector load when the range is one aligned 16-byte vector).
template <typename T>
struct FilteredRow {
    const T* row;
    RowStat st;
    float c, mc;
    int cut;  // boundary-valued tokens with index <= cut are kept
    __device__ FilteredRow(const T* row_, const RowStat& s_, float c_, int cut_)
        : row(row_), st(s_), c(c_), mc(scaled_max(s_.m, c_)), cut(cut_) {}
    __device__ __forceinline__ void probs(int i0, int cnt, float* p) const {
        constexpr int VEC = ElemT<T>::VEC;
        float x[VEC];
        const T* q = row + i0;
        if (cnt == VEC && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) {
            ElemT<T>::unpack(__ldg(reinterpret_cast<const uint4*>(q)), x);
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) x[j] = (j < cnt) ? ElemT<T>::load(q + j) : -INFINITY;
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const bool member = (x[j] > st.tau) || (x[j] == st.tau && i0 + j <= cut);
            p[j] = (j < cnt && member) ? weight_of(x[j], c, mc) * st.inv_zn : 0.0f;
        }
    }
    // The 16 bytes holding elements [i0, i0 + cnt) (cnt <= VEC): one vector
    // load when aligned, else element loads padded with -inf.
    __device__ __forceinline__ uint4 raw(int i0, int cnt) const {
        constexpr int VEC = ElemT<T>::VEC;
        const T* q = row + i0;
        if (cnt == VEC && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) return __ldg(reinterpret_cast<const uint4*>(q));
        uint32_t w[4];
        if (sizeof(T) == 2) {
            const unsigned short* h = reinterpret_cast<const unsigned short*>(q);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t lo = (2 * j < cnt) ? h[2 * j] : 0xff80u;
                const uint32_t hi = (2 * j + 1 < cnt) ? h[2 * j + 1] : 0xff80u;
                w[j] = lo | (hi << 16);
            }
        } else {
            const uint32_t* f = reinterpret_cast<const uint32_t*>(q);
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = (j < cnt) ? f[j] : 0xff800000u;
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ __forceinline__ void probs_raw(const uint4& v, int i0, int cnt, float* p) const {
        constexpr int VEC = ElemT<T>::VEC;
        float x[VEC];
        ElemT<T>::unpack(v, x);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const bool member = (x[j] > st.tau) || (x[j] == st.tau && i0 + j <= cut);
            p[j] = (j < cnt && member) ? weight_of(x[j], c, mc) * st.inv_zn : 0.0f;
        }
    }
    // probs_raw with one membership threshold per unit: x >= tau before the
    // cut, x > tau after it (as x >= the next float above tau); the unit that
    // holds the cut takes the exact per-element test.  TOPP = false: every
    // token is kept.  Padding slots hold -inf and get 0.
    template <bool TOPP>
    __device__ __forceinline__ void probs_fast(const uint4& v, int i0, int cnt, float* p) const {
        constexpr int VEC = ElemT<T>::VEC;
        if (TOPP && i0 <= cut && i0 + VEC - 1 > cut) {
            probs_raw(v, i0, cnt, p);
            return;
        }
        float x[VEC];
        ElemT<T>::unpack(v, x);
        float thr = -INFINITY;
        if (TOPP) {
            thr = st.tau;
            if (i0 > cut) {  // strictly above tau: the next float up
                const uint32_t b = __float_as_uint(thr);
                thr = (thr == 0.0f) ? __uint_as_float(1u) : __uint_as_float((b & 0x80000000u) ? b - 1u : b + 1u);
            }
        }
        const float2 cc = make_float2(c, c), nmc = make_float2(-mc, -mc), inv = make_float2(st.inv_zn, st.inv_zn);
#pragma unroll
        for (int j = 0; j < VEC; j += 2) {
            float2 t = __ffma2_rn(make_float2(x[j], x[j + 1]), cc, nmc);
            if (TOPP) {
                t.x = (x[j] >= thr) ? t.x : -INFINITY;
                t.y = (x[j + 1] >= thr) ? t.y : -INFINITY;
            }
            const float2 w = __fmul2_rn(make_float2(ex2(t.x), ex2(t.y)), inv);
            p[j] = w.x;
            p[j + 1] = w.y;
        }
    }
    __device__ __forceinline__ float prob_at(int v) const {
        const float x = ElemT<T>::load(row + v);
        const bool member = (x > st.tau) || (x == st.tau && v <= cut);
        return member ? weight_of(x, c, mc) * st.inv_zn : 0.0f;
    }
};

// Index of the last kept boundary-valued token of a filtered row.
template <typename T>
__device__ int nucleus_cut(const T* row, int V, const RowStat& st, BlockScratch& s, SampleScratch& ss) {
    if (!(st.tau > -INFINITY) || st.n_keep >= st.c_tau) return 0x7fffffff;
    return row_find_nth_equal<T>(row, V, st.tau, st.n_keep - 1, 0x7fffffff, nullptr, s, ss);
}

// ------------------------------------------------ linear residual / bonus --
// The draw of the linear step reads the selected rows once from HBM.  A step
// is kDrawStep consecutive units; warp w takes steps w, w + kNW, ... and lane
// l units l, l + 32, ... of each, with all of a step's loads (both rows)
// issued before any is used.
//
// With top-p, a token whose logit equals the row's boundary value tau is
// kept only up to the n_keep-th such token in index order (the cut), which
// is not known before the row is read.  So the first pass sums every step
// as if all tau-valued tokens were kept, and records per step how much the
// sum changes when its tau_p-valued tokens, its tau_q-valued tokens, or
// both, are dropped, and how many there are.  From the counts the cut steps
// follow; the cut indices and the two cut steps' exact sums come from one
// re-read of those steps, and every other step's sum is its recorded sum
// plus the corrections of the cuts it lies past.
constexpr int kDrawUnitsPerLane = kNT <= 256 ? 8 : 4;  // fewer registers for larger CTAs
constexpr int kDrawStep = 32 * kDrawUnitsPerLane;
constexpr int kSub = kDrawUnitsPerLane;  // 32-unit sub-steps of a step
constexpr int kDrawMaxSteps = 1024;
static_assert((long long)kDrawMaxSteps * kDrawStep >= kMaxRowUnits, "draw steps do not cover the largest row");

struct DrawScratch {
    float base_h[kDrawMaxSteps], base_l[kDrawMaxSteps];  // step sums, every tau-valued token kept
    float dp[kDrawMaxSteps];   // change when the step's tau_p-valued tokens are dropped
    float dq[kDrawMaxSteps];   // ... its tau_q-valued tokens
    float dpq[kDrawMaxSteps];  // the extra change when both are dropped (tokens tau-valued in both rows)
    int cp[kDrawMaxSteps], cq[kDrawMaxSteps];
    float sub_h[kSub], sub_l[kSub];  // per sub-step results of a re-read step
    int sub_i[kSub], sub_j[kSub];
};

// Inverse-CDF draw over the units of rv with weights max(0, p - q) (RESID)
// or p: the smallest v with C(v) > u * C(last), C the running sum in index
// order.  P and Q carry their rows' statistics; on return their cuts are
// set.  Returns -1 when every weight is zero.
template <typename T, bool RESID, bool TOPP>
__device__ int draw_linear(const RowView<T>& rv, FilteredRow<T>& P, FilteredRow<T>& Q, float u, BlockScratch& s,
                           DrawScratch& ds) {
    constexpr int VEC = ElemT<T>::VEC;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int units = rv.units();
    const int nsteps = (units + kDrawStep - 1) / kDrawStep;
    const bool needP = TOPP && P.st.tau > -INFINITY && P.st.n_keep < P.st.c_tau;
    const bool needQ = TOPP && RESID && Q.st.tau > -INFINITY && Q.st.n_keep < Q.st.c_tau;
    const float tp = P.st.tau, tq = Q.st.tau;
    P.cut = 0x7fffffff;
    Q.cut = 0x7fffffff;
    // weights with the current cuts; also the tau masks of the unit (bit j: element j is tau-valued)
    auto weights = [&](const uint4& rp, const uint4& rq, int i0, int cnt, float* w, float* pw, unsigned& mp,
                       unsigned& mq) -> float {
        P.template probs_fast<TOPP>(rp, i0, cnt, pw);
        float q[VEC];
        if (RESID) Q.template probs_fast<TOPP>(rq, i0, cnt, q);
        mp = 0u;
        mq = 0u;
        if (needP || needQ) {
            float xp[VEC], xq[VEC];
            ElemT<T>::unpack(rp, xp);
            if (RESID) ElemT<T>::unpack(rq, xq);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                if (needP && xp[j] == tp) mp |= 1u << j;
                if (needQ && xq[j] == tq) mq |= 1u << j;
            }
        }
#pragma unroll
        for (int j = 0; j < VEC; j += 2) {
            if (RESID) {
                const float2 d = __fadd2_rn(make_float2(pw[j], pw[j + 1]), make_float2(-q[j], -q[j + 1]));
                w[j] = fmaxf(0.0f, d.x);
                w[j + 1] = fmaxf(0.0f, d.y);
            } else {
                w[j] = pw[j];
                w[j + 1] = pw[j + 1];
            }
        }
        float2 a2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < VEC; j += 2) a2 = __fadd2_rn(a2, make_float2(w[j], w[j + 1]));
        return a2.x + a2.y;
    };
    auto unit_of = [&](int st, int g, int& i0, int& cnt) {
        const int uu = st * kDrawStep + g * 32 + lane;
        i0 = 0;
        cnt = 0;
        if (uu < units) rv.unit_range(uu, i0, cnt);
    };
    // A: per-step sums with every tau-valued token kept, corrections and counts
    for (int st = warp; st < nsteps; st += kNW) {
        uint4 vp[kDrawUnitsPerLane], vq[kDrawUnitsPerLane];
#pragma unroll
        for (int g = 0; g < kDrawUnitsPerLane; ++g) {
            int i0, cnt;
            unit_of(st, g, i0, cnt);
            vp[g] = cnt ? P.raw(i0, cnt) : make_uint4(0u, 0u, 0u, 0u);
            vq[g] = (RESID && cnt) ? Q.raw(i0, cnt) : make_uint4(0u, 0u, 0u, 0u);
        }
        float a = 0.0f, dp = 0.0f, dq = 0.0f, dpq = 0.0f;
        int np = 0, nq = 0;
#pragma unroll
        for (int g = 0; g < kDrawUnitsPerLane; ++g) {
            int i0, cnt;
            unit_of(st, g, i0, cnt);
            if (!cnt) continue;
            float w[VEC], pw[VEC];
            unsigned mp, mq;
            a += weights(vp[g], vq[g], i0, cnt, w, pw, mp, mq);
            if (mp | mq) {  // rare: tau-valued tokens in this unit
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const bool ip = (mp >> j) & 1u, iq = (mq >> j) & 1u;
                    if (ip) dp -= w[j];            // p dropped: max(0, 0 - q) = 0
                    if (iq) dq += pw[j] - w[j];    // q dropped: max(0, p - 0) = p
                    if (ip && iq) dpq += w[j] - pw[j];  // both dropped: 0
                }
                np += __popc(mp);
                nq += __popc(mq);
            }
        }
        const ff t = warp_sum_ff(ff_from(a));
        dp = warp_sum_f(dp);
        dq = warp_sum_f(dq);
        dpq = warp_sum_f(dpq);
        np = warp_sum_i(np);
        nq = warp_sum_i(nq);
        if (lane == 0) {
            ds.base_h[st] = t.hi;
            ds.base_l[st] = t.lo;
            ds.dp[st] = dp;
            ds.dq[st] = dq;
            ds.dpq[st] = dpq;
            ds.cp[st] = np;
            ds.cq[st] = nq;
        }
    }
    row_sync();
    // B1: the steps holding the cuts (warp 0): the n_keep-th tau-valued token of each row
    if (warp == 0) {
        auto cut_step = [&](const int* cnts, int n, int& js, int& pre) {
            js = -1;
            pre = 0;
            const int per = (nsteps + 31) / 32;
            int ls = 0;
            for (int i = 0; i < per; ++i) {
                const int st = lane * per + i;
                if (st < nsteps) ls += cnts[st];
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
                    if (run + cnts[st] > n) { js = st; pre = run; break; }
                    run += cnts[st];
                }
            }
            js = __shfl_sync(0xffffffffu, js, L);
            pre = __shfl_sync(0xffffffffu, pre, L);
        };
        int jsp = -1, prep = 0, jsq = -1, preq = 0;
        if (needP) cut_step(ds.cp, P.st.n_keep - 1, jsp, prep);
        if (needQ) cut_step(ds.cq, Q.st.n_keep - 1, jsq, preq);
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
    // B2: the cut index inside its step, one 32-unit sub-step per warp
    auto locate = [&](int js, int pre, int n, const FilteredRow<T>& R, float tau) -> int {
        unsigned msk = 0u;
        int i0 = 0, cnt = 0;
        if (warp < kSub) {
            unit_of(js, warp, i0, cnt);
            if (cnt) {
                float x[VEC];
                ElemT<T>::unpack(R.raw(i0, cnt), x);
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (j < cnt && x[j] == tau) msk |= 1u << j;
            }
            const int c = warp_sum_i(__popc(msk));
            if (lane == 0) ds.sub_i[warp] = c;
        }
        if (threadIdx.x == 0) s.bcast_i[4] = 0x7fffffff;
        row_sync();
        int base = pre, gsel = -1, gpre = 0;
        for (int g = 0; g < kSub; ++g) {
            if (gsel < 0 && base + ds.sub_i[g] > n) { gsel = g; gpre = base; }
            base += ds.sub_i[g];
        }
        if (warp == gsel) {
            const int c = __popc(msk);
            const int ic = warp_inclusive_scan_i(c);
            if (gpre + ic > n && gpre + ic - c <= n) {
                int kk = n - (gpre + ic - c);
                for (int j = 0; j < VEC; ++j)
                    if (msk & (1u << j)) {
                        if (kk == 0) { s.bcast_i[4] = i0 + j; break; }
                        --kk;
                    }
            }
        }
        row_sync();
        const int r = s.bcast_i[4];
        row_sync();
        return r;
    };
    if (jsp >= 0) P.cut = locate(jsp, prep, P.st.n_keep - 1, P, tp);
    if (jsq >= 0) Q.cut = locate(jsq, preq, Q.st.n_keep - 1, Q, tq);
    // B3: exact sums of the cut steps (with the cuts now known), one sub-step per warp
    auto exact_step = [&](int js) -> ff {
        if (warp < kSub) {
            int i0, cnt;
            unit_of(js, warp, i0, cnt);
            float a = 0.0f;
            if (cnt) {
                float w[VEC], pw[VEC];
                unsigned mp, mq;
                a = weights(P.raw(i0, cnt), RESID ? Q.raw(i0, cnt) : make_uint4(0u, 0u, 0u, 0u), i0, cnt, w, pw, mp,
                            mq);
            }
            const ff t = warp_sum_ff(ff_from(a));
            if (lane == 0) {
                ds.sub_h[warp] = t.hi;
                ds.sub_l[warp] = t.lo;
            }
        }
        row_sync();
        ff r = ff{0.0f, 0.0f};
        for (int g = 0; g < kSub; ++g) r = ff_add(r, ff{ds.sub_h[g], ds.sub_l[g]});
        row_sync();
        return r;
    };
    const ff exact_p = (jsp >= 0) ? exact_step(jsp) : ff{0.0f, 0.0f};
    const ff exact_q = (jsq >= 0 && jsq != jsp) ? exact_step(jsq) : exact_p;
    // the true sum of step st
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
    // C: the crossing step, one sub-step per warp
    float w[VEC];
    float a_own = 0.0f;
    int i0 = 0, cnt = 0;
#pragma unroll
    for (int j = 0; j < VEC; ++j) w[j] = 0.0f;
    if (warp < kSub) {
        unit_of(js, warp, i0, cnt);
        if (cnt) {
            float pw[VEC];
            unsigned mp, mq;
            a_own = weights(P.raw(i0, cnt), RESID ? Q.raw(i0, cnt) : make_uint4(0u, 0u, 0u, 0u), i0, cnt, w, pw, mp, mq);
        }
        const ff t = warp_sum_ff(ff_from(a_own));
        int mylast = -1;
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (j < cnt && w[j] > 0.0f) mylast = i0 + j;
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
    for (int g = 0; g < kSub; ++g) {  // the same order in every warp
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
                for (int j = 0; j < VEC && q < 0; ++j) {
                    if (j >= cnt) break;
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
    const int r = s.bcast_i[6];
    row_sync();
    return r;
}

}  // namespace sv
