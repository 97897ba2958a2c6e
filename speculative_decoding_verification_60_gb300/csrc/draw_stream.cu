// Linear verification, stage 2 for bf16 rows with 16-byte aligned units
// ("Accelerating Sonar through speculation", §Speculative decoding and
// §Target-Draft; the cited rule: at the first rejection the token is drawn
// from norm(max(0, p - q)), after a full accept from p; §MTP and §MTP
// schedule for a single token: the accepted positions' hidden rows and the
// next tokens are packed on the GPU).  The draw is the smallest v with
// C(v) > u * C(last), C the running sum of the weights in index order.
//
// One CTA per request: kNT compute threads, a copy warp and a compaction
// warp.  The copy warp streams the selected rows through a ring of
// shared-memory slots with bulk copies (16 KiB of each row per slot), so
// many copies are in flight without holding registers; the compute warps
// take each slot's weights once.  A slot is cut into regions of 128 units
// (1024 elements), one per warp, in index order; within a region, sub-row j
// is units 32j .. 32j+31, lane l taking unit 32j + l (conflict-free shared
// reads).  The compaction warp packs the accepted hidden rows meanwhile.
//
// Under top-p, a token valued exactly at a row's nucleus boundary tau is
// kept only up to the row's cut, the n_keep-th such token in index order.
// Until the cut is passed, each slot's regions first count their
// tau-valued tokens; the counts (shared after a barrier) tell each region
// whether its tau-valued tokens are kept, dropped, or split by the cut,
// which the region's warp then locates.  So every region sum is exact, and
// warp 0 needs only the crossing region again (2 KiB of each row, from L2).
#include "bulk.cuh"
#include "draw_bf16.cuh"
#include "launch.cuh"
#include "linear_args.cuh"

namespace sv {

namespace {

constexpr int kDSlots = 3;
constexpr int kDChunkUnits = 1024;                  // units of each row per slot (16 KiB)
constexpr int kDLaneUnits = 4;                      // units per lane in a slot: sub-rows of a region
constexpr int kDRegionUnits = 32 * kDLaneUnits;     // units per warp region
static_assert(kDRegionUnits * kNW == kDChunkUnits, "a slot is one region per compute warp");
constexpr int kDMaxChunks = (int)((kMaxVocab / 8 + kDChunkUnits - 1) / kDChunkUnits);
constexpr int kDMaxRegions = kDMaxChunks * kNW;
constexpr int kDThreads = kNT + 64;                 // compute threads, the copy warp, the compaction warp
constexpr int kDCopyWarp = kNW, kDPackWarp = kNW + 1;
constexpr uint64_t kDWaitLimitNs = 2000000000ull;   // 2 s: a bulk copy that long has failed

struct DrawSmem {
    union {
        uint4 ring[kDSlots][2][kDChunkUnits];       // [slot][P, Q][unit]
        BDrawScratch fallback;                      // the p == q redraw, after the stream
    };
    float wsum[kDMaxRegions];    // exact region sums (lane partials in fp32, then a warp sum)
    int cnt[2][kNW];             // tau_p | tau_q << 16 counts of a slot's regions (by slot parity)
    int cut[2];                  // the cuts of P and Q (0x7fffffff: none)
    uint64_t full[kDSlots];      // slot holds its copies (1 arrival + bytes)
    uint64_t empty[kDSlots];     // slot read by every compute warp (kNW arrivals)
    BlockScratch s;
    int aborted;
    int tok;
};

__device__ __forceinline__ int count_eq(const uint4& v, uint32_t t2) {
    return (__popc(bf2_eq(v.x, t2)) + __popc(bf2_eq(v.y, t2)) + __popc(bf2_eq(v.z, t2)) + __popc(bf2_eq(v.w, t2))) >> 4;
}

// e = 2^((x - m) c) of the pair in word x with members x >= thr (per half).
template <bool TOPP>
__device__ __forceinline__ float2 pair_exp_thr(float nmc, float c, uint32_t x, uint32_t thr) {
    if (TOPP) {
        const uint32_t m = bf2_ge(x, thr);
        x = (x & m) | (0xff80ff80u & ~m);
    }
    const float2 t = __ffma2_rn(make_float2(bf16_lo(x), bf16_hi(x)), make_float2(c, c), make_float2(nmc, nmc));
    return make_float2(ex2(t.x), ex2(t.y));
}

// Membership threshold pair of a row for elements i, i + 1 at its cut.
__device__ __forceinline__ uint32_t thr_at(const BRow& R, int i) {
    const uint32_t a1 = R.above2 & 0xffffu;
    return ((i <= R.cut) ? R.tau1 : a1) | (((i + 1 <= R.cut) ? R.tau1 : a1) << 16);
}

// Sum of one unit's weights, max(0, e_p - r e_q) (RESID) or e_p, with
// membership thresholds given per pair (EXACT: from the rows' cuts at
// element i0) or for the whole unit (tp, tq).  w: the 8 weights.
template <bool RESID, bool TOPP, bool EXACT>
__device__ __forceinline__ float unit_sum(const BRow& P, const BRow& Q, float c, float r, const uint4& vp,
                                          const uint4& vq, uint32_t tp, uint32_t tq, int i0, float* w) {
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 ep = pair_exp_thr<TOPP>(P.nmc, c, word_of(vp, j), EXACT ? thr_at(P, i0 + 2 * j) : tp);
        float2 ww = ep;
        if (RESID) {
            const float2 eq = pair_exp_thr<TOPP>(Q.nmc, c, word_of(vq, j), EXACT ? thr_at(Q, i0 + 2 * j) : tq);
            const float2 d = __ffma2_rn(eq, make_float2(-r, -r), ep);
            ww = make_float2(fmaxf(d.x, 0.0f), fmaxf(d.y, 0.0f));
        }
        acc = __fadd2_rn(acc, ww);
        w[2 * j] = ww.x;
        w[2 * j + 1] = ww.y;
    }
    return acc.x + acc.y;
}

// Index of the (n+1)-th tau-valued token (0-based n) of a warp's region
// whose first unit is u0, given the count before the region; lane l holds
// unit u0 + 32j + l in v[j].
__device__ __forceinline__ int locate_cut(const uint4* v, float tau, int u0, int before, int n) {
    const int lane = threadIdx.x & 31;
    int idx = 0x7fffffff;
    int run = before;
#pragma unroll
    for (int j = 0; j < kDLaneUnits; ++j) {
        uint32_t msk = 0u;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t wd = word_of(v[j], e >> 1);
            if (((e & 1) ? bf16_hi(wd) : bf16_lo(wd)) == tau) msk |= 1u << e;
        }
        const int cl = __popc(msk);
        const int ic = warp_inclusive_scan_i(cl);
        int kk = n - (run + ic - cl);
        if (kk >= 0 && kk < cl) {
            for (int e = 0; e < 8; ++e)
                if (msk & (1u << e)) {
                    if (kk == 0) { idx = (u0 + 32 * j + lane) * 8 + e; break; }
                    --kk;
                }
        }
        run += __shfl_sync(0xffffffffu, ic, 31);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
    return idx;
}

template <int MODE>
__global__ void __launch_bounds__(kDThreads, 2) k_draw_stream(LinearArgs a) {
    constexpr bool TOPP = (MODE == 2);
    extern __shared__ __align__(128) uint8_t draw_raw[];
    DrawSmem& sm = *reinterpret_cast<DrawSmem*>(draw_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x, k = a.k, V = a.V;
    const int nvec = V / 8;
    grid_dep_wait();  // the decisions and offsets come from the launch before
    const int dv = a.dec[b];
    const int acnt = dv & 0xffff, inval = dv >> 16;
    const bool resid = acnt < k;
    const uint16_t* prow = static_cast<const uint16_t*>(a.tgt) + ((size_t)b * (k + 1) + acnt) * V;
    const uint16_t* qrow = resid ? static_cast<const uint16_t*>(a.drf) + ((size_t)b * k + acnt) * V : prow;
    const int nch = (nvec + kDChunkUnits - 1) / kDChunkUnits;
    const int32_t* d = a.drafts + (size_t)b * k;
    volatile int* aborted = &sm.aborted;
    if (tid == 0) {
        for (int i = 0; i < kDSlots; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kNW);
        }
        sm.aborted = 0;
        sm.cut[0] = sm.cut[1] = 0x7fffffff;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == kDCopyWarp) {  // ---------------------------------- copy warp
        if (lane != 0 || inval) return;
        int issued = 0;
        bool ok = true;
        for (int ch = 0; ch < nch && ok; ++ch) {
            const int slot = ch % kDSlots;
            if (ch >= kDSlots && !mbar_wait(&sm.empty[slot], ((ch / kDSlots) - 1) & 1, kDWaitLimitNs)) {
                ok = false;
                break;
            }
            if (*aborted) break;
            const uint32_t nb = (uint32_t)min(kDChunkUnits, nvec - ch * kDChunkUnits) * 16u;
            mbar_arrive_expect_tx(&sm.full[slot], resid ? 2u * nb : nb);
            bulk_load(sm.ring[slot][0], reinterpret_cast<const uint4*>(prow) + (size_t)ch * kDChunkUnits, nb,
                      &sm.full[slot]);
            if (resid)
                bulk_load(sm.ring[slot][1], reinterpret_cast<const uint4*>(qrow) + (size_t)ch * kDChunkUnits, nb,
                          &sm.full[slot]);
            ++issued;
        }
        if (!ok) *aborted = 1;
        // every copy issued has landed before the CTA may end
        for (int i = max(0, issued - kDSlots); i < issued; ++i)
            mbar_wait(&sm.full[i % kDSlots], (i / kDSlots) & 1, kDWaitLimitNs);
        return;
    }
    if (warp == kDPackWarp) {  // ---------------------- compaction warp
        // rows 0 .. a of the request are contiguous in hidden, and so are
        // their places at the packed offset: one flat copy
        if (!a.hidden) return;
        const size_t n = (size_t)(acnt + 1) * a.H;
        const uint16_t* in = a.hidden + (size_t)b * (k + 1) * a.H;
        uint16_t* out = a.out_hidden + (size_t)a.woff[b] * a.H;
        if (a.vec_ok) {
            const uint4* vi = reinterpret_cast<const uint4*>(in);
            uint4* vo = reinterpret_cast<uint4*>(out);
            const size_t nv = n / 8;
            for (size_t i0 = 0; i0 < nv; i0 += 32 * 8) {
                uint4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const size_t i = i0 + (size_t)j * 32 + lane;
                    if (i < nv) v[j] = __ldg(vi + i);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const size_t i = i0 + (size_t)j * 32 + lane;
                    if (i < nv) vo[i] = v[j];
                }
            }
        } else {
            for (size_t i = lane; i < n; i += 32) out[i] = in[i];
        }
        return;
    }

    // ------------------------------------------------------- compute threads
    const int64_t req = a.req ? a.req[b] : (int64_t)b;
    const int64_t pos = a.pos ? a.pos[b] : 0;
    const float c = a.c;
    int t = -1;
    if (inval) {
        t = row_argmax_finite<__nv_bfloat16>(reinterpret_cast<const __nv_bfloat16*>(prow), V, sm.s);
    } else {
        const RowStat sp = a.stats[tgt_row(a, b, acnt)];
        const RowStat sq = resid ? a.stats[drf_row(a, b, acnt)] : sp;
        BRow P(prow, sp, c, TOPP), Q(qrow, sq, c, TOPP);
        const float r = resid ? Q.inv / P.inv : 0.0f;
        const bool needP = TOPP && P.need, needQ = TOPP && resid && Q.need;
        const int nP = P.n_keep_minus1 + 1, nQ = Q.n_keep_minus1 + 1;  // tau-valued tokens kept
        const float u = uniform01(a.seed, req, pos + acnt + 1, resid ? kPurposeResidual : kPurposeBonus, 0);
        const uint4 ninf = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);

        // 1. stream: exact region sums
        bool ab = false;
        int cumP = 0, cumQ = 0;  // tau-valued tokens of the slots before
        for (int ch = 0; ch < nch; ++ch) {
            const int slot = ch % kDSlots;
            if (!ab && !mbar_test(&sm.full[slot], (ch / kDSlots) & 1)) {
                if (*aborted || !mbar_wait(&sm.full[slot], (ch / kDSlots) & 1, kDWaitLimitNs)) {
                    ab = true;
                    *aborted = 1;
                }
            }
            const int nu = ab ? 0 : min(kDChunkUnits, nvec - ch * kDChunkUnits);
            const int ru0 = warp * kDRegionUnits;          // the region's first unit in the slot
            const int u0 = ch * kDChunkUnits + ru0;        // ... in the row
            uint4 vp[kDLaneUnits], vq[kDLaneUnits];
#pragma unroll
            for (int j = 0; j < kDLaneUnits; ++j) {
                const bool ok = ru0 + 32 * j + lane < nu;
                vp[j] = ok ? sm.ring[slot][0][ru0 + 32 * j + lane] : ninf;
                vq[j] = (resid && ok) ? sm.ring[slot][1][ru0 + 32 * j + lane] : ninf;
            }
            // thresholds of this region: every tau-valued token kept before
            // the cut, dropped after it (counted while the cut lies ahead)
            uint32_t tp = (needP && cumP >= nP) ? P.above2 : P.tau2;
            uint32_t tq = (needQ && cumQ >= nQ) ? Q.above2 : Q.tau2;
            bool exact = false;
            const bool cntP = needP && cumP < nP, cntQ = needQ && cumQ < nQ;  // the same in every warp
            if (cntP || cntQ) {
                int lp = 0, lq = 0;
#pragma unroll
                for (int j = 0; j < kDLaneUnits; ++j) {
                    if (cntP) lp += count_eq(vp[j], P.tau2);
                    if (cntQ) lq += count_eq(vq[j], Q.tau2);
                }
                const int rcp = warp_sum_i(lp), rcq = warp_sum_i(lq);
                if (lane == 0) sm.cnt[ch & 1][warp] = rcp | (rcq << 16);
                row_sync();
                int bp = cumP, bq = cumQ;
                for (int w = 0; w < kNW; ++w) {
                    const int cw = sm.cnt[ch & 1][w];
                    if (w < warp) {
                        bp += cw & 0xffff;
                        bq += cw >> 16;
                    }
                    cumP += cw & 0xffff;
                    cumQ += cw >> 16;
                }
                // the region holding the nP-th tau-valued token (the last one
                // kept) locates it, also when it is the region's last: the
                // re-read of the crossing region takes its thresholds from it
                if (cntP) {
                    if (bp >= nP) tp = P.above2;
                    else if (bp + rcp >= nP) {  // the cut lies in this region
                        P.cut = locate_cut(vp, P.tau, u0, bp, nP - 1);
                        if (lane == 0) sm.cut[0] = P.cut;
                        exact = true;
                    }
                }
                if (cntQ) {
                    if (bq >= nQ) tq = Q.above2;
                    else if (bq + rcq >= nQ) {
                        Q.cut = locate_cut(vq, Q.tau, u0, bq, nQ - 1);
                        if (lane == 0) sm.cut[1] = Q.cut;
                        exact = true;
                    }
                }
            }
            float us[kDLaneUnits], w[8];
            if (exact) {  // once per row: per-element thresholds at the cuts
                if (!(P.cut < 0x7fffffff)) P.cut = (tp == P.tau2) ? 0x7fffffff : -1;
                if (!(Q.cut < 0x7fffffff)) Q.cut = (tq == Q.tau2) ? 0x7fffffff : -1;
                float s4 = 0.0f;
#pragma unroll 1
                for (int j = 0; j < kDLaneUnits; ++j) {  // units from the slot (kept out of registers)
                    const int uu = ru0 + 32 * j + lane;
                    const bool ok = uu < nu;
                    const uint4 xp = ok ? sm.ring[slot][0][uu] : ninf;
                    const uint4 xq = (resid && ok) ? sm.ring[slot][1][uu] : ninf;
                    const int ie = (u0 + 32 * j + lane) * 8;
                    const float su = resid ? unit_sum<true, TOPP, true>(P, Q, c, r, xp, xq, 0, 0, ie, w)
                                           : unit_sum<false, TOPP, true>(P, P, c, 0.0f, xp, xp, 0, 0, ie, w);
                    s4 = (j == 0) ? su : s4 + su;
                }
                us[0] = s4;
                us[1] = us[2] = us[3] = 0.0f;
                P.cut = Q.cut = 0x7fffffff;
            } else {
#pragma unroll
                for (int j = 0; j < kDLaneUnits; ++j)
                    us[j] = resid ? unit_sum<true, TOPP, false>(P, Q, c, r, vp[j], vq[j], tp, tq, 0, w)
                                  : unit_sum<false, TOPP, false>(P, P, c, 0.0f, vp[j], vp[j], tp, tp, 0, w);
            }
            const float ws = warp_sum_f(((us[0] + us[1]) + us[2]) + us[3]);
            __syncwarp();
            if (lane == 0) {
                sm.wsum[ch * kNW + warp] = ws;
                if (!ab) mbar_arrive(&sm.empty[slot]);
            }
        }
        row_sync();
        if (*aborted) {
            // a bulk copy did not land in time: the request keeps its
            // decisions and takes the argmax of its row
            if (tid == 0 && a.dev_error) atomicOr(a.dev_error, kDevErrTimeout);
            t = sp.argmax;
        } else {
            // 2. warp 0: the crossing region, then its lane and element
            const int nreg = nch * kNW;
            if (warp == 0) {
                P.cut = sm.cut[0];
                Q.cut = sm.cut[1];
                const int per = (nreg + 31) / 32;
                ff ls = ff{0.0f, 0.0f};
                int lastpos = -1;
                for (int i = 0; i < per; ++i) {
                    const int rg = lane * per + i;
                    if (rg < nreg) {
                        const float sv = sm.wsum[rg];
                        ls = ff_add_f(ls, sv);
                        if (sv > 0.0f) lastpos = rg;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
                const ff incl = warp_inclusive_scan_ff(ls);
                const ff tot = ff_shfl(incl, 31);
                int rx = -1;
                ff pre = ff{0.0f, 0.0f}, tgt = ff{0.0f, 0.0f};
                if (tot.hi > 0.0f) {
                    tgt = ff_mul_f(tot, u);
                    const ff up = ff_shfl_up(incl, 1);
                    const unsigned bal = __ballot_sync(0xffffffffu, ls.hi > 0.0f && ff_lt(tgt, incl));
                    if (bal) {
                        const int L = __ffs(bal) - 1;
                        if (lane == L) {
                            ff run = lane == 0 ? ff{0.0f, 0.0f} : up;
                            for (int i = 0; i < per; ++i) {
                                const int rg = lane * per + i;
                                if (rg >= nreg) break;
                                const float sv = sm.wsum[rg];
                                const ff nx = ff_add_f(run, sv);
                                if (sv > 0.0f && ff_lt(tgt, nx)) { rx = rg; pre = run; break; }
                                run = nx;
                            }
                        }
                        rx = __shfl_sync(0xffffffffu, rx, L);
                        pre = ff_shfl(pre, L);
                    }
                    if (rx < 0) {  // rounding: the draw falls in the last region with weight
                        rx = lastpos;
                        pre = ff{0.0f, 0.0f};
                        tgt = ff{INFINITY, 0.0f};
                    }
                }
                int tok = -1;
                if (rx >= 0) {
                    // the region again (from L2), at the cuts; its units in
                    // index order are (sub-row j, lane l)
                    const int u0 = (rx / kNW) * kDChunkUnits + (rx % kNW) * kDRegionUnits;
                    int lastw = -1;
                    tok = -2;
                    ff run = pre;
                    for (int j = 0; j < kDLaneUnits && tok == -2; ++j) {
                        const int uu = u0 + 32 * j + lane;
                        const bool ok = uu < nvec;
                        const uint4 xp = ok ? __ldg(reinterpret_cast<const uint4*>(prow) + uu) : ninf;
                        const uint4 xq = (ok && resid) ? __ldg(reinterpret_cast<const uint4*>(qrow) + uu) : ninf;
                        float w[8];
                        const float su = resid ? unit_sum<true, TOPP, true>(P, Q, c, r, xp, xq, 0, 0, uu * 8, w)
                                               : unit_sum<false, TOPP, true>(P, P, c, 0.0f, xp, xp, 0, 0, uu * 8, w);
                        int mylast = -1;
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (w[e] > 0.0f) mylast = uu * 8 + e;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) mylast = max(mylast, __shfl_xor_sync(0xffffffffu, mylast, o));
                        if (mylast >= 0) lastw = mylast;
                        const ff ia = warp_inclusive_scan_ff(ff_from(su));
                        const ff ua = ff_shfl_up(ia, 1);  // every lane takes part in the shuffle
                        const ff ex = ff_add(run, lane == 0 ? ff{0.0f, 0.0f} : ua);
                        const unsigned cb = __ballot_sync(0xffffffffu, su > 0.0f && ff_lt(tgt, ff_add(ex, ff_from(su))));
                        if (cb) {
                            const int L = __ffs(cb) - 1;
                            int q = -1;
                            if (lane == L) {
                                ff rr = ex;
                                int last = -1;
                                for (int e = 0; e < 8 && q < 0; ++e) {
                                    if (w[e] > 0.0f) last = uu * 8 + e;
                                    rr = ff_add_f(rr, w[e]);
                                    if (w[e] > 0.0f && ff_lt(tgt, rr)) q = uu * 8 + e;
                                }
                                if (q < 0) q = last;  // rounding: the unit's last weighted element
                            }
                            tok = __shfl_sync(0xffffffffu, q, L);
                        }
                        run = ff_add(run, ff_shfl(ia, 31));
                    }
                    if (tok == -2) tok = lastw;  // rounding: the last weighted element of the region
                }
                if (lane == 0) sm.tok = tok;
            }
            row_sync();
            t = sm.tok;
            row_sync();
            if (t < 0 && resid) {
                // every residual weight is zero (p == q): draw from p
                const RowView<__nv_bfloat16> rv(reinterpret_cast<const __nv_bfloat16*>(prow), V);
                BRow P0(prow, sp, c, TOPP);
                t = draw_linear_bf16<false, TOPP>(rv, P0, P0, c, u, sm.s, sm.fallback);
            }
        }
    }
    if (tid == 0) {
        int32_t* o = a.out_tokens + (size_t)b * (k + 1);
        for (int j = 0; j <= k; ++j) o[j] = (j < acnt) ? d[j] : (j == acnt ? t : -1);
        if (a.hidden) {
            const int off = a.woff[b];
            for (int rr = 0; rr <= acnt; ++rr) a.next_tokens[off + rr] = (rr < acnt) ? d[rr] : t;
            a.offsets[b + 1] = a.woff[b + 1];
            if (b == 0) a.offsets[0] = 0;
        }
    }
}

template <int MODE>
spec_status launch_mode(LinearArgs& a, cudaStream_t st) {
    const size_t smem = sizeof(DrawSmem);
    if (!set_dyn_smem(k_draw_stream<MODE>, smem, kDThreads)) return SPEC_ERR_CUDA;
    if (launch_dependent(k_draw_stream<MODE>, dim3(a.B), dim3(kDThreads), smem, st, a) != cudaSuccess) return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

bool draw_stream_applies(const LinearArgs& a, int mode) {
    return mode >= 1 && a.V % 8 == 0 && (reinterpret_cast<uintptr_t>(a.tgt) & 15u) == 0 &&
           (reinterpret_cast<uintptr_t>(a.drf) & 15u) == 0 && a.drf != nullptr;
}

spec_status launch_draw_stream(LinearArgs& a, int mode, cudaStream_t st) {
    return mode == 2 ? launch_mode<2>(a, st) : launch_mode<1>(a, st);
}

}  // namespace sv
