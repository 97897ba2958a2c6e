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

#include <cooperative_groups.h>

#include "rowstats.cuh"

namespace sv {

namespace cg = cooperative_groups;

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
    __syncthreads();
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
    __syncthreads();
    const int r = s.bcast_i[7];
    __syncthreads();
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
// The draw of the linear step reads the selected rows from HBM, so it is
// spread over a cluster of kDecCluster CTAs (one request per cluster) and
// organised for memory parallelism: a step is kDrawStep consecutive units,
// lane l takes units l, l + 32, ... of it, and all of a step's loads (for
// both rows) are issued before any is used.  CTA r of the cluster owns a
// contiguous quarter of the steps; per-step results meet through
// distributed shared memory.  Every cluster barrier below is reached by
// all CTAs of the cluster (the control flow around them is uniform).
constexpr int kDecCluster = 1;
constexpr int kDrawUnitsPerLane = 8;
constexpr int kDrawStep = 32 * kDrawUnitsPerLane;
constexpr int kSub = kDrawUnitsPerLane;  // 32-unit sub-steps of a step
static_assert((long long)(kMaxSteps - 2 * kSub) * kDrawStep >= kMaxRowUnits, "step sums do not cover the largest row");
static_assert(kSub % kNW == 0 || kNW % kSub == 0, "sub-steps per warp");

struct ClusterSteps {
    int units, nsteps, lo, hi;  // this CTA's steps [lo, hi)
    __device__ ClusterSteps(int units_, int rank) : units(units_) {
        nsteps = (units + kDrawStep - 1) / kDrawStep;
        const int per = (nsteps + kDecCluster - 1) / kDecCluster;
        lo = rank * per;
        hi = min(nsteps, lo + per);
    }
};

// Owner CTA of step st.
__device__ __forceinline__ int step_owner(const ClusterSteps& cs, int st) {
    const int per = (cs.nsteps + kDecCluster - 1) / kDecCluster;
    return st / per;
}

// Last kept boundary-valued index of P and, when Q is given, of Q (INT_MAX
// when every boundary-valued token is kept), known to every CTA of the
// cluster on return.  One pass over both rows counts the boundary-valued
// elements per step; each CTA then locates the n_keep-th one of each row.
template <typename T>
__device__ void nucleus_cuts(cg::cluster_group& cl, const RowView<T>& rv, FilteredRow<T>& P, FilteredRow<T>* Q,
                             BlockScratch& s, SampleScratch& ss) {
    constexpr int VEC = ElemT<T>::VEC;
    const bool needP = P.st.tau > -INFINITY && P.st.n_keep < P.st.c_tau;
    const bool needQ = Q && Q->st.tau > -INFINITY && Q->st.n_keep < Q->st.c_tau;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const ClusterSteps cs(rv.units(), (int)cl.block_rank());
    int* cp = reinterpret_cast<int*>(ss.sh);
    int* cq = reinterpret_cast<int*>(ss.sl);
    const float tp = P.st.tau, tq = Q ? Q->st.tau : 0.0f;
    auto eq_mask = [&](const uint4& v, float tau, int cnt) -> unsigned {
        float x[VEC];
        ElemT<T>::unpack(v, x);
        unsigned m = 0u;
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (j < cnt && x[j] == tau) m |= 1u << j;
        return m;
    };
    // elements equal to tau among the unit's 16 bytes (padding is -inf and tau is finite)
    auto eq_count = [&](const uint4& v, float tau, int cnt) -> int {
        if constexpr (sizeof(T) == 2) {
            if (tau != 0.0f) {  // bit equality is value equality away from +-0 (rows hold no NaN)
                const uint32_t tb = __float_as_uint(tau) >> 16;
                const uint32_t t2 = tb | (tb << 16);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                int n = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t d = w4[j] ^ t2;
                    n += ((d & 0xffffu) == 0u) + ((d >> 16) == 0u);
                }
                return n;
            }
        }
        return __popc(eq_mask(v, tau, cnt));
    };
    if (needP || needQ) {
        for (int st = cs.lo + warp; st < cs.hi; st += kNW) {
            uint4 vp[kDrawUnitsPerLane], vq[kDrawUnitsPerLane];
#pragma unroll
            for (int g = 0; g < kDrawUnitsPerLane; ++g) {
                const int u = st * kDrawStep + g * 32 + lane;
                int i0 = 0, cnt = 0;
                if (u < cs.units) rv.unit_range(u, i0, cnt);
                vp[g] = (needP && cnt) ? P.raw(i0, cnt) : make_uint4(0u, 0u, 0u, 0u);
                vq[g] = (needQ && cnt) ? Q->raw(i0, cnt) : make_uint4(0u, 0u, 0u, 0u);
            }
            int np = 0, nq = 0;
#pragma unroll
            for (int g = 0; g < kDrawUnitsPerLane; ++g) {
                const int u = st * kDrawStep + g * 32 + lane;
                int i0 = 0, cnt = 0;
                if (u < cs.units) rv.unit_range(u, i0, cnt);
                if (needP) np += eq_count(vp[g], tp, cnt);
                if (needQ) nq += eq_count(vq[g], tq, cnt);
            }
            np = warp_sum_i(np);
            nq = warp_sum_i(nq);
            if (lane == 0) {
                cp[st] = np;
                cq[st] = nq;
            }
        }
    }
    cl.sync();
    // every CTA: the step holding the n-th element (warp 0 over all steps), then
    // its sub-steps, one warp each
    auto locate = [&](int which, const FilteredRow<T>& R, int n) -> int {
        if (warp == 0) {
            const int per = (cs.nsteps + 31) / 32;
            int ls = 0;
            for (int i = 0; i < per; ++i) {
                const int st = lane * per + i;
                if (st < cs.nsteps) {
                    const int* src = cl.map_shared_rank(which ? cq : cp, step_owner(cs, st));
                    ls += src[st];
                }
            }
            const int incl = warp_inclusive_scan_i(ls);
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            int js = -1, pre = 0;
            if (n >= 0 && n < total) {
                const unsigned bal = __ballot_sync(0xffffffffu, incl > n);
                const int L = __ffs(bal) - 1;
                if (lane == L) {
                    int run = incl - ls;
                    for (int i = 0; i < per; ++i) {
                        const int st = lane * per + i;
                        const int* src = cl.map_shared_rank(which ? cq : cp, step_owner(cs, st));
                        if (run + src[st] > n) { js = st; pre = run; break; }
                        run += src[st];
                    }
                }
                js = __shfl_sync(0xffffffffu, js, L);
                pre = __shfl_sync(0xffffffffu, pre, L);
            }
            if (lane == 0) { s.bcast_i[0] = js; s.bcast_i[1] = pre; }
        }
        __syncthreads();
        const int js = s.bcast_i[0];
        int pre = s.bcast_i[1];
        __syncthreads();
        if (js < 0) return 0x7fffffff;
        int* subc = reinterpret_cast<int*>(s.pf3);  // kSub counts (kSub <= kNW)
        unsigned msk = 0u;
        int i0 = 0;
        const int g = warp;
        if (g < kSub) {
            const int u = js * kDrawStep + g * 32 + lane;
            int cnt = 0;
            if (u < cs.units) rv.unit_range(u, i0, cnt);
            msk = cnt ? eq_mask(R.raw(i0, cnt), R.st.tau, cnt) : 0u;
            const int c = warp_sum_i(__popc(msk));
            if (lane == 0) subc[g] = c;
        }
        __syncthreads();
        int base = pre, gsel = -1, gpre = 0;
        for (int gg = 0; gg < kSub; ++gg) {
            if (gsel < 0 && base + subc[gg] > n) { gsel = gg; gpre = base; }
            base += subc[gg];
        }
        if (threadIdx.x == 0) s.bcast_i[2] = 0x7fffffff;
        __syncthreads();
        if (g == gsel) {
            const int c = __popc(msk);
            const int ic = warp_inclusive_scan_i(c);
            if (gpre + ic > n && gpre + ic - c <= n) {
                int kk = n - (gpre + ic - c);
                for (int j = 0; j < VEC; ++j)
                    if (msk & (1u << j)) {
                        if (kk == 0) { s.bcast_i[2] = i0 + j; break; }
                        --kk;
                    }
            }
        }
        __syncthreads();
        const int r = s.bcast_i[2];
        __syncthreads();
        return r;
    };
    static_assert(kSub <= kNW, "one sub-step per warp in the locate");
    P.cut = needP ? locate(0, P, P.st.n_keep - 1) : 0x7fffffff;
    if (Q) Q->cut = needQ ? locate(1, *Q, Q->st.n_keep - 1) : 0x7fffffff;
    cl.sync();  // the counts may be overwritten from here on
}

// Inverse-CDF draw over the units of rv with weights max(0, p - q) (RESID)
// or p: the smallest v with C(v) > u * C(last), C the running sum in index
// order.  Returns, in every CTA of the cluster, the drawn index or -1 when
// every weight is zero.
template <typename T, bool RESID, bool TOPP>
__device__ int draw_filtered(cg::cluster_group& cl, const RowView<T>& rv, const FilteredRow<T>& P,
                             const FilteredRow<T>& Q, float u, BlockScratch& s, SampleScratch& ss) {
    constexpr int VEC = ElemT<T>::VEC;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rank = (int)cl.block_rank();
    const ClusterSteps cs(rv.units(), rank);
    auto weights = [&](const uint4& rp, const uint4& rq, int i0, int cnt, float* w) -> float {
        P.template probs_fast<TOPP>(rp, i0, cnt, w);
        if (RESID) {
            float q[VEC];
            Q.template probs_fast<TOPP>(rq, i0, cnt, q);
#pragma unroll
            for (int j = 0; j < VEC; j += 2) {
                const float2 d = __fadd2_rn(make_float2(w[j], w[j + 1]), make_float2(-q[j], -q[j + 1]));
                w[j] = fmaxf(0.0f, d.x);
                w[j + 1] = fmaxf(0.0f, d.y);
            }
        }
        float2 a2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < VEC; j += 2) a2 = __fadd2_rn(a2, make_float2(w[j], w[j + 1]));
        return a2.x + a2.y;
    };
    // A: this CTA's step sums
    for (int st = cs.lo + warp; st < cs.hi; st += kNW) {
        uint4 vp[kDrawUnitsPerLane], vq[kDrawUnitsPerLane];
#pragma unroll
        for (int g = 0; g < kDrawUnitsPerLane; ++g) {
            const int uu = st * kDrawStep + g * 32 + lane;
            int i0 = 0, cnt = 0;
            if (uu < cs.units) rv.unit_range(uu, i0, cnt);
            vp[g] = cnt ? P.raw(i0, cnt) : make_uint4(0u, 0u, 0u, 0u);
            vq[g] = (RESID && cnt) ? Q.raw(i0, cnt) : make_uint4(0u, 0u, 0u, 0u);
        }
        float a = 0.0f;
#pragma unroll
        for (int g = 0; g < kDrawUnitsPerLane; ++g) {
            const int uu = st * kDrawStep + g * 32 + lane;
            int i0 = 0, cnt = 0;
            if (uu < cs.units) rv.unit_range(uu, i0, cnt);
            float w[VEC];
            if (cnt) a += weights(vp[g], vq[g], i0, cnt, w);
        }
        const ff t = warp_sum_ff(ff_from(a));
        if (lane == 0) {
            ss.sh[st] = t.hi;
            ss.sl[st] = t.lo;
        }
    }
    cl.sync();
    // B: every CTA finds the crossing step from all step sums (warp 0)
    if (warp == 0) {
        const int per = (cs.nsteps + 31) / 32;
        ff ls = ff{0.0f, 0.0f};
        int lastpos = -1;
        for (int i = 0; i < per; ++i) {
            const int st = lane * per + i;
            if (st < cs.nsteps) {
                const int o = step_owner(cs, st);
                const ff sv = ff{cl.map_shared_rank(ss.sh, o)[st], cl.map_shared_rank(ss.sl, o)[st]};
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
                        if (st >= cs.nsteps) break;
                        const int o = step_owner(cs, st);
                        const ff sv = ff{cl.map_shared_rank(ss.sh, o)[st], cl.map_shared_rank(ss.sl, o)[st]};
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
            s.bcast_i[4] = js;
            s.bcast_f[0] = pre.hi;
            s.bcast_f[1] = pre.lo;
            s.bcast_f[2] = tgt.hi;
            s.bcast_f[3] = tgt.lo;
        }
    }
    cl.sync();  // every CTA has read the step sums
    const int js = s.bcast_i[4];
    if (js < 0) return -1;  // uniform across the cluster
    // C: warp g takes sub-steps g, g + kNW, ... (32 units each) of step js
    constexpr int KW = (kSub + kNW - 1) / kNW;
    float* sub_h = ss.sh;  // free again after the cluster barrier
    float* sub_l = ss.sl;
    int* sub_last = reinterpret_cast<int*>(ss.sh + kSub);
    float w[KW][VEC];
    float a_own[KW];
    int i0s[KW], cnts[KW];
#pragma unroll
    for (int k2 = 0; k2 < KW; ++k2) {
        const int g = warp + k2 * kNW;
        a_own[k2] = 0.0f;
        i0s[k2] = 0;
        cnts[k2] = 0;
#pragma unroll
        for (int j = 0; j < VEC; ++j) w[k2][j] = 0.0f;
        if (g >= kSub) continue;
        const int uu = js * kDrawStep + g * 32 + lane;
        int i0 = 0, cnt = 0;
        if (uu < cs.units) rv.unit_range(uu, i0, cnt);
        if (cnt) a_own[k2] = weights(P.raw(i0, cnt), RESID ? Q.raw(i0, cnt) : make_uint4(0u, 0u, 0u, 0u), i0, cnt, w[k2]);
        i0s[k2] = i0;
        cnts[k2] = cnt;
        const ff t = warp_sum_ff(ff_from(a_own[k2]));
        int mylast = -1;
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (j < cnt && w[k2][j] > 0.0f) mylast = i0 + j;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mylast = max(mylast, __shfl_xor_sync(0xffffffffu, mylast, o));
        if (lane == 0) {
            sub_h[g] = t.hi;
            sub_l[g] = t.lo;
            sub_last[g] = mylast;
        }
    }
    __syncthreads();
    const ff tgt = ff{s.bcast_f[2], s.bcast_f[3]};
    ff run = ff{s.bcast_f[0], s.bcast_f[1]};
    int g_cross = -1, lastw = -1;
    ff pre_cross = run;
    for (int g = 0; g < kSub; ++g) {  // the same order in every warp
        const ff sv = ff{sub_h[g], sub_l[g]};
        const ff nx = ff_add(run, sv);
        if (sub_last[g] >= 0) lastw = sub_last[g];
        if (g_cross < 0 && sv.hi > 0.0f && ff_lt(tgt, nx)) { g_cross = g; pre_cross = run; }
        run = nx;
    }
    if (threadIdx.x == 0 && g_cross < 0) s.bcast_i[7] = lastw;  // otherwise the crossing warp writes it
#pragma unroll
    for (int k2 = 0; k2 < KW; ++k2) {
        const int g = warp + k2 * kNW;
        if (g != g_cross) continue;  // warp-uniform
        const ff ia = warp_inclusive_scan_ff(ff_from(a_own[k2]));
        const ff ua = ff_shfl_up(ia, 1);
        const ff ex = ff_add(pre_cross, lane == 0 ? ff{0.0f, 0.0f} : ua);
        const unsigned cb = __ballot_sync(0xffffffffu, a_own[k2] > 0.0f && ff_lt(tgt, ff_add(ex, ff_from(a_own[k2]))));
        int p = sub_last[g];  // rounding: the last weighted element of this sub-step
        if (cb) {
            const int L = __ffs(cb) - 1;
            int q = -1;
            if (lane == L) {
                ff rr = ex;
                int mylast = -1;
                for (int j = 0; j < VEC && q < 0; ++j) {
                    if (j >= cnts[k2]) break;
                    if (w[k2][j] > 0.0f) mylast = i0s[k2] + j;
                    rr = ff_add_f(rr, w[k2][j]);
                    if (w[k2][j] > 0.0f && ff_lt(tgt, rr)) q = i0s[k2] + j;
                }
                if (q < 0) q = mylast;
            }
            p = __shfl_sync(0xffffffffu, q, L);
        }
        if (lane == 0) s.bcast_i[7] = p;
    }
    __syncthreads();
    const int r = s.bcast_i[7];
    __syncthreads();
    return r;
}

}  // namespace sv
