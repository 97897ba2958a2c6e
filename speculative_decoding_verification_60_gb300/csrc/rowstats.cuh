// Row statistics of one logit row, computed by one CTA of kNT threads.
//
// "Accelerating Sonar through speculation", §Target-Draft: acceptance
// compares the full probability distributions of draft and target, so every
// row needs its normaliser; with top-p filtering also the exact nucleus.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int kUnroll = 8;             // 16-byte vectors in flight per thread
// Shared memory of a top-p row (bf16): one region of kTopSmemBytes, carved as
//   sample  [0, 16 KiB)      bf16 bit patterns of the systematic sample
//   scount  [16, 24 KiB)     sample counts per value bin of the estimate
//   tcount  [24, 32 KiB)     thread-maximum counts per value bin
//   wtot    [32, 32.5 KiB)   per-warp prefix totals of the estimate
//   tmax    [32.5, 33.5 KiB) each thread's maximum from pass 1
// After the estimate, [0, 32 KiB) holds the key histogram of the exact
// count (up to kFullBins consecutive bf16 keys).
constexpr int kSampleCap = 8192;       // sample slots (2 per batch of kUnroll vectors)
constexpr int kEstBins = 2048;         // value-linear bins of the estimate
constexpr int kBinsPerThread = kEstBins / kNT;
constexpr int kSCountOffset = 16384;
constexpr int kTCountOffset = kSCountOffset + kEstBins * 4;
constexpr int kWTotOffset = kTCountOffset + kEstBins * 4;
constexpr int kTmaxOffset = kWTotOffset + 512;
constexpr int kTopSmemBytes = kTmaxOffset + kNT * 4;
constexpr int kFullBins = 8192;        // widest key window counted in one pass
static_assert(kSampleCap * 2 <= kSCountOffset, "sample overlaps the estimate bins");
static_assert(kNW * 16 <= 512, "estimate warp totals overlap the thread maxima");
static_assert(kFullBins * 4 <= kWTotOffset, "histogram overlaps what the estimate still reads");
static_assert(kEstBins % (4 * kNT) == 0, "whole uint4 groups of bins per thread");

struct Pass1 {
    float m;     // max (NaN-free); -inf if the row has no non-NaN value
    ff z;        // sum of 2^(x*c - m*c) over the row (when requested)
    int argmax;  // lowest index holding m
    bool bad;    // a NaN was seen
};

template <typename T>
__device__ __forceinline__ void batch_max(const uint4* v, float& mx, bool& nan);

template <>
__device__ __forceinline__ void batch_max<__nv_bfloat16>(const uint4* v, float& mx, bool& nan) {
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v[0].x);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) a = __hmax2_nan(a, *reinterpret_cast<const __nv_bfloat162*>(&w[j]));
    }
    const float lo = __low2float(a), hi = __high2float(a);
    nan = (lo != lo) || (hi != hi);
    mx = fmaxf(lo, hi);
}

template <>
__device__ __forceinline__ void batch_max<float>(const uint4* v, float& mx, bool& nan) {
    float a = -INFINITY;
    bool n = false;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const float f[4] = {__uint_as_float(v[u].x), __uint_as_float(v[u].y), __uint_as_float(v[u].z),
                            __uint_as_float(v[u].w)};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            n |= (f[j] != f[j]);
            a = fmaxf(a, f[j]);
        }
    }
    nan = n;
    mx = a;
}

template <typename T> __device__ __forceinline__ uint4 neg_inf_vec();
template <> __device__ __forceinline__ uint4 neg_inf_vec<__nv_bfloat16>() {
    return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
}
template <> __device__ __forceinline__ uint4 neg_inf_vec<float>() {
    return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
}

// Sum of weights of a batch relative to mc.
template <typename T>
__device__ __forceinline__ float batch_weight_sum(const uint4* v, float c, float mc);

template <>
__device__ __forceinline__ float batch_weight_sum<__nv_bfloat16>(const uint4* v, float c, float mc) {
    float2 acc = make_float2(0.0f, 0.0f);
    const float2 cc = make_float2(c, c), nm = make_float2(-mc, -mc);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 x = make_float2(bf16_lo(w[j]), bf16_hi(w[j]));
            const float2 t = __ffma2_rn(x, cc, nm);
            acc = __fadd2_rn(acc, make_float2(ex2(t.x), ex2(t.y)));
        }
    }
    return acc.x + acc.y;
}

template <>
__device__ __forceinline__ float batch_weight_sum<float>(const uint4* v, float c, float mc) {
    float acc = 0.0f;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const float f[4] = {__uint_as_float(v[u].x), __uint_as_float(v[u].y), __uint_as_float(v[u].z),
                            __uint_as_float(v[u].w)};
#pragma unroll
        for (int j = 0; j < 4; ++j) acc += weight_of(f[j], c, mc);
    }
    return acc;
}

// The block result of pass 1 from each thread's (max, sum rescaled to it,
// lowest index holding the max or INT_MAX, NaN seen).  Each warp takes its
// max, rescales every lane's sum to it once and adds them in a fixed
// float-float tree; warp 0 does the same over the warps.  Two barriers.
template <bool kSum>
__device__ __forceinline__ Pass1 reduce_pass1(float m, ff z, int idx, bool bad, float c, BlockScratch& s) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const float mw = warp_max(m);
    idx = warp_min_i(m == mw ? idx : 0x7fffffff);
    const int bw = __any_sync(0xffffffffu, bad) ? 1 : 0;
    ff zw = ff{0.0f, 0.0f};
    if (kSum) zw = warp_sum_ff((m > -INFINITY) ? ff_scale(z, ex2((m - mw) * c)) : ff{0.0f, 0.0f});
    if (lane == 0) {
        s.pf[w] = mw;
        s.pf2[w] = zw.hi;
        s.pf3[w] = zw.lo;
        s.pi[w] = idx;
        s.pi2[w] = bw;
    }
    row_sync();
    if (w == 0) {
        const float mi = (lane < kNW) ? s.pf[lane] : -INFINITY;
        const float M = warp_max(mi);
        const int I = warp_min_i((lane < kNW && mi == M) ? s.pi[lane] : 0x7fffffff);
        const int Bd = __any_sync(0xffffffffu, lane < kNW && s.pi2[lane] != 0) ? 1 : 0;
        ff Z = ff{0.0f, 0.0f};
        if (kSum) {
            const ff zi = (lane < kNW && mi > -INFINITY) ? ff_scale(ff{s.pf2[lane], s.pf3[lane]}, ex2((mi - M) * c))
                                                          : ff{0.0f, 0.0f};
            Z = warp_sum_ff(zi);
        }
        if (lane == 0) {
            s.rf[kNW] = M;
            s.rf[kNW + 1] = Z.hi;
            s.rf2[kNW] = Z.lo;
            s.ri[kNW] = I;
            s.ri[kNW + 1] = Bd;
        }
    }
    row_sync();
    Pass1 r;
    r.m = s.rf[kNW];
    r.z = ff{s.rf[kNW + 1], s.rf2[kNW]};
    r.argmax = (s.ri[kNW] == 0x7fffffff) ? 0 : s.ri[kNW];
    r.bad = s.ri[kNW + 1] != 0;
    return r;
}

// Pass 1: one streaming read of the row.  kSum adds the sum of weights
// (online: the running sum is rescaled whenever the running max grows).
// When `sample` is given (bf16 rows), two elements of the first vector of
// every batch are stored in slot order, a systematic sample of 1/32 of the
// row; unused slots keep the NaN pattern they were set to.
template <typename T, bool kSum>
__device__ Pass1 row_pass1(const T* __restrict__ row, int V, float c, BlockScratch& s,
                           uint16_t* sample = nullptr, float* tmax = nullptr) {
    constexpr int VEC = ElemT<T>::VEC;
    const RowView<T> rv(row, V);
    const int tid = threadIdx.x;
    float m_t = -INFINITY, z_t = 0.0f, z_c = 0.0f, best_bm = -INFINITY;  // z_c: Kahan compensation
    int best_batch = -1;
    bool bad = false;
    float x_head = -INFINITY, x_tail = -INFINITY;

    if (sample) {
        const int nslots = min(kSampleCap, 2 * kNT * ((rv.nvec + kUnroll * kNT - 1) / (kUnroll * kNT)));
        for (int i = tid; i < (nslots + 7) / 8; i += kNT)
            reinterpret_cast<uint4*>(sample)[i] = make_uint4(0x7fff7fffu, 0x7fff7fffu, 0x7fff7fffu, 0x7fff7fffu);
        row_sync();
    }
    auto take_scalar = [&](float x) {
        bad |= (x != x);
        if (x > m_t) {
            if (kSum) z_t *= ex2((m_t - x) * c);
            m_t = x;
        }
        if (kSum && m_t > -INFINITY) z_t += weight_of(x, c, scaled_max(m_t, c));
    };
    if (tid < rv.head) {
        x_head = ElemT<T>::load(row + tid);
        take_scalar(x_head);
    }
    const uint4* vp = rv.vec();
    int batch = 0;
    for (int base = tid; base < rv.nvec; base += kUnroll * kNT, ++batch) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int vi = base + u * kNT;
            v[u] = (vi < rv.nvec) ? __ldg(vp + vi) : neg_inf_vec<T>();
        }
        if (sample) {
            const int slot = (batch * kNT + tid) * 2;
            if (slot + 1 < kSampleCap) {
                sample[slot] = (uint16_t)(v[0].x & 0xffffu);
                sample[slot + 1] = (uint16_t)(v[0].z & 0xffffu);
            }
        }
        float bm;
        bool nan;
        batch_max<T>(v, bm, nan);
        bad |= nan;
        if (bm > m_t) {
            if (kSum) {
                const float sc = ex2((m_t - bm) * c);
                z_t *= sc;
                z_c *= sc;
            }
            m_t = bm;
            best_batch = base;
            best_bm = bm;
        }
        if (kSum && m_t > -INFINITY) {
            const float y = batch_weight_sum<T>(v, c, scaled_max(m_t, c)) - z_c;
            const float t = z_t + y;
            z_c = (t - z_t) - y;
            z_t = t;
        }
    }
    if (tid < rv.tail) {
        x_tail = ElemT<T>::load(row + rv.head + rv.nvec * VEC + tid);
        take_scalar(x_tail);
    }

    // Lowest index of this thread holding m_t (head < body < tail), searched
    // only by the lanes that hold their warp's max.
    int idx = 0x7fffffff;
    const bool holds = (m_t == warp_max(m_t));
    if (!holds) {
    } else if (tid < rv.head && x_head == m_t) {
        idx = tid;
    } else if (best_batch >= 0 && best_bm == m_t) {
        for (int u = 0; u < kUnroll && idx == 0x7fffffff; ++u) {
            const int vi = best_batch + u * kNT;
            if (vi >= rv.nvec) break;
            float f[VEC];
            ElemT<T>::unpack(__ldg(vp + vi), f);
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (f[j] == m_t && idx == 0x7fffffff) idx = rv.head + vi * VEC + j;
        }
    } else if (tid < rv.tail && x_tail == m_t) {
        idx = rv.head + rv.nvec * VEC + tid;
    }

    if (tmax) tmax[tid] = m_t;
    return reduce_pass1<kSum>(m_t, ff_add(ff{z_t, 0.0f}, ff{-z_c, 0.0f}), idx, bad, c, s);
}

// Lowest-index argmax over entries that are neither NaN nor +inf (the
// fallback token of an invalid request); 0 when no such entry exists.
template <typename T>
__device__ int row_argmax_finite(const T* __restrict__ row, int V, BlockScratch& s) {
    constexpr int VEC = ElemT<T>::VEC;
    const RowView<T> rv(row, V);
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    for (int u = threadIdx.x; u < rv.units(); u += kNT) {
        float f[VEC];
        int i0, cnt;
        rv.load_unit(u, f, i0, cnt);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            if (j >= cnt) break;
            const float x = f[j];
            if (x != x || x == INFINITY) continue;
            if (bidx == 0x7fffffff || x > best) { best = x; bidx = i0 + j; }
        }
    }
    const float m = block_max(bidx == 0x7fffffff ? -INFINITY : best, s);
    const int any = block_min_i(bidx, s);
    const int r = block_min_i((bidx != 0x7fffffff && best == m) ? bidx : 0x7fffffff, s);
    return any == 0x7fffffff ? 0 : r;
}

// Step layout of the block-wide searches: the row's units (RowView: head,
// 16-byte vectors, tail) are cut into steps of kStepUnits consecutive units;
// warp w owns a contiguous range of steps and lane l takes units l, l + 32,
// ... of each step, so loads are coalesced and one barrier publishes the
// per-step results.
constexpr int kStepUnits = 128;        // 4 units per lane
constexpr int kMaxSteps = 1024;        // rows of up to kMaxSteps * kStepUnits units
constexpr long long kMaxRowUnits = (long long)kMaxSteps * kStepUnits;
// Largest vocabulary the row kernels accept (fp32 rows of 4 elements per unit).
constexpr long long kMaxVocab = 4 * (kMaxRowUnits - 2);

struct SampleScratch {
    float sh[kMaxSteps];  // per-step results (float-float sums, or counts)
    float sl[kMaxSteps];
};

__device__ __forceinline__ int steps_per_warp(int units) {
    const int nsteps = (units + kStepUnits - 1) / kStepUnits;
    return (nsteps + kNW - 1) / kNW;
}

// Index of the n-th (0-based) element, in index order, among those with
// index < limit that equal `val`; INT_MAX when there are fewer.  *count
// receives how many such elements there are.
template <typename T>
__device__ int row_find_nth_equal(const T* __restrict__ row, int V, float val, int n, int limit, int* count,
                                  BlockScratch& s, SampleScratch& ss) {
    constexpr int VEC = ElemT<T>::VEC;
    const RowView<T> rv(row, V);
    const int units = rv.units();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nsteps = (units + kStepUnits - 1) / kStepUnits;
    const int spw = steps_per_warp(units);
    int* sc = reinterpret_cast<int*>(ss.sh);
    auto matches = [&](int unit, int& i0) -> unsigned {  // bit j: element j of the unit matches
        unsigned msk = 0u;
        i0 = 0;
        if (unit < units) {
            float f[VEC];
            int cnt;
            rv.load_unit(unit, f, i0, cnt);
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (j < cnt && i0 + j < limit && f[j] == val) msk |= 1u << j;
        }
        return msk;
    };
    for (int st = warp * spw; st < (warp + 1) * spw && st < nsteps; ++st) {
        int c = 0;
#pragma unroll
        for (int g = 0; g < kStepUnits / 32; ++g) {
            int i0;
            c += __popc(matches(st * kStepUnits + g * 32 + lane, i0));
        }
        c = warp_sum_i(c);
        if (lane == 0) sc[st] = c;
    }
    row_sync();
    if (warp == 0) {
        const int per = (nsteps + 31) / 32;
        int ls = 0;
        for (int i = 0; i < per; ++i) {
            const int st = lane * per + i;
            if (st < nsteps) ls += sc[st];
        }
        const int incl = warp_inclusive_scan_i(ls);
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        int found = 0x7fffffff;
        if (n >= 0 && n < total) {
            const unsigned bal = __ballot_sync(0xffffffffu, incl > n);
            const int L = __ffs(bal) - 1;
            int js = -1, pre = 0;
            if (lane == L) {
                int run = incl - ls;
                for (int i = 0; i < per; ++i) {
                    const int st = lane * per + i;
                    if (run + sc[st] > n) { js = st; pre = run; break; }
                    run += sc[st];
                }
            }
            js = __shfl_sync(0xffffffffu, js, L);
            pre = __shfl_sync(0xffffffffu, pre, L);
            for (int g = 0; g < kStepUnits / 32 && found == 0x7fffffff; ++g) {
                int i0;
                const unsigned msk = matches(js * kStepUnits + g * 32 + lane, i0);
                const int c = __popc(msk);
                const int ic = warp_inclusive_scan_i(c);
                int hit = 0x7fffffff;
                if (pre + ic > n && pre + ic - c <= n) {
                    int k = n - (pre + ic - c);
                    for (int j = 0; j < VEC; ++j) {
                        if (msk & (1u << j)) {
                            if (k == 0) { hit = i0 + j; break; }
                            --k;
                        }
                    }
                }
                found = warp_min_i(hit);
                pre += __shfl_sync(0xffffffffu, ic, 31);
            }
        }
        if (lane == 0) {
            s.bcast_i[5] = total;
            s.bcast_i[6] = found;
        }
    }
    row_sync();
    const int r = s.bcast_i[6];
    if (count) *count = s.bcast_i[5];
    row_sync();
    return r;
}

// ------------------------------------------------------------------ top-p --
// Nucleus of a row (the pages' filter, with ties broken by lower index):
// walking tokens in decreasing logit order, a token is kept while the mass
// of the tokens before it is below top_p * Z.  All tokens of one logit value
// share one weight, so the nucleus is a key tau (the boundary value), the
// number n_keep of tau-valued tokens kept (the lowest-index ones), and the
// kept mass.
struct Topp {
    float tau;     // boundary logit (-inf: every token kept)
    int n_keep;    // boundary-valued tokens kept
    int c_tau;     // boundary-valued tokens in the row
    ff mass;       // nucleus mass (weights relative to the max)
};

// Key of a bf16 value with -0 folded onto +0.
__device__ __forceinline__ uint32_t value_key(float x) {
    return x == 0.0f ? 0x8000u : okey16(__float_as_uint(x) >> 16);
}
__device__ __forceinline__ float key_value(int key) { return bf16_bits_to_float(okey16_to_bits((uint32_t)key)); }

// Smallest n in [1, cnt] with F + n * w >= pZ, for F < pZ <= F + cnt * w
// (products formed exactly, differences in float-float).
__device__ __forceinline__ int keep_count(ff F, ff pZ, float w, int cnt) {
    const ff d = ff_sub(pZ, F);
    int n = (int)ceilf(ff_to_float(d) / w);
    n = n < 1 ? 1 : (n > cnt ? cnt : n);
    if (n > 1 && ff_ge(ff_two_prod((float)(n - 1), w), d)) --n;
    else if (n < cnt && ff_lt(ff_two_prod((float)n, w), d)) ++n;
    return n;
}

// Number of 16-byte vectors of a bf16 row (as RowView counts them).
__device__ __forceinline__ int rv_nvec(const __nv_bfloat16* row, int V) { return RowView<__nv_bfloat16>(row, V).nvec; }

// Lower bound on the nucleus boundary: a token of weight w <= (1 - top_p) *
// Z / V cannot be kept (the tail from that token on holds at most V tokens,
// none heavier, so it weighs at most (1 - top_p) * Z and everything before
// it already reaches top_p * Z).  Returned as a value a little below that.
__device__ __forceinline__ float nucleus_lower_bound(float m, ff Z, float top_p, int V, float c) {
    const float wb = 0.5f * (1.0f - top_p) * ff_to_float(Z) / (float)V;
    if (!(wb > 0.0f)) return -INFINITY;
    return m + log2f(wb) / c;
}

// Walk of consecutive keys from the top (position 0 holds key key_top,
// position p key key_top - p) from mass F0 above key_top, looking for the
// key where the running mass reaches pZ.  ASC = false: hist[p] is the
// count at position p; ASC = true: hist[nbins - 1 - p].  A map may put a
// "lump" at one position: the values too close to zero to count key by key,
// given by their exact total mass; positions after it continue from
// key_below.  Position masses are formed exactly per key (count * weight as
// a pair) and summed in float-float; the crossing chunk is the lowest-index
// one whose end reaches pZ, and its owner walks it.  WARP = true: warp 0
// walks (the other warps only meet the barriers).
// found: 0 the window ends first (*F_end: mass above its bottom); 1 found;
// 2 the crossing lies inside the lump (F_lump: the mass above the lump).
struct WalkMap {
    int key_top;
    int lump;       // position of the lump, or -1
    int key_below;  // key at position lump + 1
    ff lump_mass;
};
__device__ __forceinline__ WalkMap plain_map(int key_top) { return WalkMap{key_top, -1, 0, ff{0.0f, 0.0f}}; }
struct WalkOut {
    int found;
    Topp r;
    ff F_lump;
};
template <bool WARP, bool ASC = false>
__device__ WalkOut walk_keys(const uint32_t* hist, int nbins, const WalkMap& map, float c, float mc, ff F0, ff pZ,
                             ff* F_end, BlockScratch& s) {
    auto count_at = [&](int p) -> uint32_t { return hist[ASC ? nbins - 1 - p : p]; };
    auto key_at = [&](int p) -> int {
        return (map.lump < 0 || p < map.lump) ? map.key_top - p : map.key_below - (p - map.lump - 1);
    };
    const int tid = threadIdx.x, lane = tid & 31;
    const int nparts = WARP ? 32 : kNT;
    const int part = WARP ? lane : tid;
    const bool active = !WARP || tid < 32;
    const int per = (nbins + nparts - 1) / nparts;
    const int b0 = part * per;
    ff M = ff{0.0f, 0.0f};
    if (active) {
        for (int i = 0; i < per; ++i) {
            const int b = b0 + i;
            if (b >= nbins) break;
            if (b == map.lump) {
                M = ff_add(M, map.lump_mass);
                continue;
            }
            const uint32_t cnt = count_at(b);
            if (cnt == 0) continue;
            M = ff_add(M, ff_two_prod((float)cnt, weight_of(key_value(key_at(b)), c, mc)));
        }
    }
    ff before = ff{0.0f, 0.0f}, tot = ff{0.0f, 0.0f};
    if (WARP) {
        if (active) {
            const ff incl = warp_inclusive_scan_ff(M);
            const ff up = ff_shfl_up(incl, 1);
            before = lane == 0 ? ff{0.0f, 0.0f} : up;
            tot = ff_shfl(incl, 31);
        }
    } else {
        before = block_exclusive_scan_ff(M, s, &tot);
    }
    // lowest part whose end reaches pZ
    int cand = 0x7fffffff;
    if (active && M.hi > 0.0f && ff_ge(ff_add(ff_add(F0, before), M), pZ)) cand = part;
    int first = 0x7fffffff;
    if (WARP) {
        if (active) {
            const unsigned bal = __ballot_sync(0xffffffffu, cand != 0x7fffffff);
            first = bal ? __ffs(bal) - 1 : 0x7fffffff;
        }
    } else {
        first = block_min_i(cand, s);
    }
    if (first == 0x7fffffff && tid == 0) s.bcast_i[0] = 0;  // otherwise the crossing part writes it
    if (active && part == first) {
        ff F = ff_add(F0, before);
        int last = -1;
        ff F_last = F;  // mass above the last nonzero position
        int res = 0;
        for (int i = 0; i < per; ++i) {
            const int b = b0 + i;
            if (b >= nbins) break;
            if (b == map.lump) {
                if (!(map.lump_mass.hi > 0.0f)) continue;
                const ff nxt = ff_add(F, map.lump_mass);
                if (ff_ge(nxt, pZ)) {
                    s.bcast_f[1] = F.hi;
                    s.bcast_f[2] = F.lo;
                    res = 2;
                    break;
                }
                F_last = F;
                F = nxt;
                last = b;
                continue;
            }
            const uint32_t cnt = count_at(b);
            if (cnt == 0) continue;
            const float w = weight_of(key_value(key_at(b)), c, mc);
            const ff nxt = ff_add(F, ff_two_prod((float)cnt, w));
            if (ff_ge(nxt, pZ)) {
                const int nk = keep_count(F, pZ, w, (int)cnt);
                const ff mass = ff_add(F, ff_two_prod((float)nk, w));
                s.bcast_f[0] = key_value(key_at(b));
                s.bcast_f[1] = mass.hi;
                s.bcast_f[2] = mass.lo;
                s.bcast_i[1] = nk;
                s.bcast_i[2] = (int)cnt;
                res = 1;
                break;
            }
            F_last = F;
            F = nxt;
            last = b;
        }
        if (res == 0 && last >= 0) {  // the sequential sum fell short by rounding: take the last bucket
            if (last == map.lump) {
                s.bcast_f[1] = F_last.hi;
                s.bcast_f[2] = F_last.lo;
                res = 2;
            } else {
                s.bcast_f[0] = key_value(key_at(last));
                s.bcast_f[1] = F.hi;
                s.bcast_f[2] = F.lo;
                s.bcast_i[1] = (int)count_at(last);
                s.bcast_i[2] = (int)count_at(last);
                res = 1;
            }
        }
        s.bcast_i[0] = res;
    }
    if (WARP && tid < 32) {  // the total for F_end, from lane 0
        if (lane == 0) { s.bcast_f[3] = tot.hi; s.bcast_f[4] = tot.lo; }
    } else if (!WARP && tid == 0) {
        s.bcast_f[3] = tot.hi;
        s.bcast_f[4] = tot.lo;
    }
    row_sync();
    WalkOut o;
    o.found = s.bcast_i[0];
    o.r.tau = s.bcast_f[0];
    o.r.mass = ff{s.bcast_f[1], s.bcast_f[2]};
    o.r.n_keep = s.bcast_i[1];
    o.r.c_tau = s.bcast_i[2];
    o.F_lump = o.r.mass;
    if (F_end) *F_end = ff_add(F0, ff{s.bcast_f[3], s.bcast_f[4]});
    row_sync();
    return o;
}

// Counts of the keys in [klo, khi] into hist[khi - key]; -0 is counted as
// +0 when both are in the window.
__device__ inline void count_key_window(const __nv_bfloat16* __restrict__ row, int V, int klo, int khi,
                                        uint32_t* hist) {
    const RowView<__nv_bfloat16> rv(row, V);
    const int tid = threadIdx.x;
    const int nb = khi - klo + 1;
    auto take = [&](uint32_t b) {
        const uint32_t idx = (uint32_t)(khi - (int)okey16(b));
        if (idx < (uint32_t)nb) atomicAdd(&hist[idx], 1u);
    };
    if (tid < rv.head) take(*reinterpret_cast<const unsigned short*>(row + tid));
    const uint4* vp = rv.vec();
    constexpr int kU2 = 4;
    for (int base = tid; base < rv.nvec; base += kU2 * kNT) {
        uint4 v[kU2];
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
            const int vi = base + u * kNT;
            v[u] = (vi < rv.nvec) ? __ldg(vp + vi) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
        }
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
            const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                take(w4[j] & 0xffffu);
                take(w4[j] >> 16);
            }
        }
    }
    if (tid < rv.tail) take(*reinterpret_cast<const unsigned short*>(row + rv.head + rv.nvec * 8 + tid));
    row_sync();
    if (tid == 0 && khi >= 0x8000 && klo <= 0x7fff) {
        hist[khi - 0x8000] += hist[khi - 0x7fff];
        hist[khi - 0x7fff] = 0u;
    }
}

// Counts of the keys of a window on one side of zero: one predicated shared
// reduction per element, at an address formed from the element's bits.
// NEG = false (klo > +0): position key - klo, since a positive element's key
// is its bits + 0x8000; NEG = true (khi < -0): position khi - key, since a
// negative element's key is 0xffff - its bits.  TOP: khi is the row's
// largest key, so no element lies above the window.  COPIES interleaved
// copies of the histogram (hist[pos * COPIES + copy], the copy chosen by
// lane / (32 / COPIES)) put lanes of different groups in different banks;
// the caller sums them.
template <bool NEG, bool TOP, int COPIES>
__device__ inline void count_window_signed(const __nv_bfloat16* __restrict__ row, int V, int klo, int khi,
                                           uint32_t* hist) {
    static_assert(COPIES == 1 || COPIES == 2 || COPIES == 4 || COPIES == 8, "copies: a power of two up to 8");
    constexpr int kLgC = COPIES == 8 ? 3 : (COPIES == 4 ? 2 : (COPIES == 2 ? 1 : 0));
    const RowView<__nv_bfloat16> rv(row, V);
    const int tid = threadIdx.x;
    const float t_lo = key_value(klo), t_hi = key_value(khi);
    const uint32_t copy = (uint32_t)(tid & 31) >> (5 - kLgC);
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(hist) + 4u * copy;
    const uint32_t kb = NEG ? base - 4u * COPIES * (uint32_t)(0xffff - khi) : base - 4u * COPIES * (uint32_t)(klo - 0x8000);
    auto take = [&](uint32_t xb) {  // xb: the element's float bit pattern (bf16 bits << 16)
        const uint32_t addr = kb + (xb >> (14 - kLgC));
        if (TOP) {
            asm volatile("{\n\t.reg .pred p;\n\tsetp.ge.f32 p, %0, %1;\n\t@p red.shared.add.u32 [%2], 1;\n\t}"
                         ::"f"(__uint_as_float(xb)), "f"(t_lo), "r"(addr)
                         : "memory");
        } else {
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ge.f32 p, %0, %1;\n\tsetp.le.and.f32 p, %0, %3, p;\n\t"
                "@p red.shared.add.u32 [%2], 1;\n\t}"
                ::"f"(__uint_as_float(xb)), "f"(t_lo), "r"(addr), "f"(t_hi)
                : "memory");
        }
    };
    if (tid < rv.head) take((uint32_t)(*reinterpret_cast<const unsigned short*>(row + tid)) << 16);
    const uint4* vp = rv.vec();
    const uint64_t last_use = l2_evict_first_policy();
    constexpr int kU2 = 8;  // L2 (partly DRAM) re-read: 8 vectors in flight per thread
    for (int base_v = tid; base_v < rv.nvec; base_v += kU2 * kNT) {
        uint4 v[kU2];
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
            const int vi = base_v + u * kNT;
            v[u] = (vi < rv.nvec) ? ldg_last_use(vp + vi, last_use) : neg_inf_vec<__nv_bfloat16>();
        }
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
            const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                take(w4[j] << 16);
                take(w4[j] & 0xffff0000u);
            }
        }
    }
    if (tid < rv.tail)
        take((uint32_t)(*reinterpret_cast<const unsigned short*>(row + rv.head + rv.nvec * 8 + tid)) << 16);
}

// Sums the 8 interleaved copies of an nb-position histogram (nb <= 4 * kNT)
// into hist[0, nb).
__device__ inline void merge_copies8(uint32_t* hist, int nb) {
    uint32_t sum[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int i = threadIdx.x + j * kNT;
        sum[j] = 0u;
        if (i < nb) {
            const uint4 a = reinterpret_cast<const uint4*>(hist)[2 * i];
            const uint4 b = reinterpret_cast<const uint4*>(hist)[2 * i + 1];
            sum[j] = (a.x + a.y) + (a.z + a.w) + (b.x + b.y) + (b.z + b.w);
        }
    }
    row_sync();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int i = threadIdx.x + j * kNT;
        if (i < nb) hist[i] = sum[j];
    }
}

// One-signed window count, interleaved 8 ways when the window is narrow.
template <bool NEG>
__device__ inline void count_window_one_sign(const __nv_bfloat16* __restrict__ row, int V, int klo, int khi,
                                             bool top, uint32_t* hist) {
    const int nb = khi - klo + 1;
    if (nb <= 4 * kNT && 8 * nb <= kFullBins) {
        for (int i = threadIdx.x; i < 8 * nb; i += kNT) hist[i] = 0u;
        row_sync();
        if (top) count_window_signed<NEG, true, 8>(row, V, klo, khi, hist);
        else count_window_signed<NEG, false, 8>(row, V, klo, khi, hist);
        row_sync();
        merge_copies8(hist, nb);
    } else {
        for (int i = threadIdx.x; i < nb; i += kNT) hist[i] = 0u;
        row_sync();
        if (top) count_window_signed<NEG, true, 1>(row, V, klo, khi, hist);
        else count_window_signed<NEG, false, 1>(row, V, klo, khi, hist);
    }
}

// Exact nucleus by counting key windows from key_top down to key_floor,
// starting at mass F0 above key_top.  Each window is one pass over the row
// (from L2) and one walk.  The first window stops at first_lo when that is
// higher; top: key_top is the row's largest key.
__device__ inline Topp topp_windows(const __nv_bfloat16* __restrict__ row, int V, float c, float mc, ff Z, ff pZ,
                                    int key_top, int key_floor, ff F0, uint32_t* hist, BlockScratch& s,
                                    int first_lo = 0, bool top = false) {
    if (key_floor == 0x8000) key_floor = 0x7fff;  // -0 belongs with +0
    for (int hi = key_top; hi >= key_floor;) {
        int lo = hi - kFullBins + 1;
        if (lo < key_floor) lo = key_floor;
        if (hi == key_top && lo < first_lo) lo = first_lo;
        if (lo == 0x8000 && hi > 0x8000) lo = 0x8001;  // keep +0 and -0 in one window
        const int nb = hi - lo + 1;
        const bool pos = lo > 0x8000, neg = hi < 0x7fff, at_top = top && hi == key_top;
        if (pos) {
            count_window_one_sign<false>(row, V, lo, hi, at_top, hist);
        } else if (neg) {
            count_window_one_sign<true>(row, V, lo, hi, at_top, hist);
        } else {
            for (int i = threadIdx.x; i < nb; i += kNT) hist[i] = 0u;
            row_sync();
            count_key_window(row, V, lo, hi, hist);
        }
        row_sync();
        ff F_end;
        WalkOut o;
        if (pos) {  // warp 0 alone walks short windows; the block walks longer ones
            o = (nb <= 256) ? walk_keys<true, true>(hist, nb, plain_map(hi), c, mc, F0, pZ, &F_end, s)
                             : walk_keys<false, true>(hist, nb, plain_map(hi), c, mc, F0, pZ, &F_end, s);
        } else {
            o = (nb <= 2048) ? walk_keys<true, false>(hist, nb, plain_map(hi), c, mc, F0, pZ, &F_end, s)
                             : walk_keys<false, false>(hist, nb, plain_map(hi), c, mc, F0, pZ, &F_end, s);
        }
        if (o.found == 1) return o.r;
        F0 = F_end;
        hi = lo - 1;
    }
    Topp r;  // reached only by rounding: keep every token
    r.tau = -INFINITY;
    r.n_keep = 0;
    r.c_tau = 0;
    r.mass = Z;
    return r;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Second pass of a bracket below -0, one read of the row (from L2): the
// exact mass of the elements above t_b (returned as this thread's part) and
// the exact counts of the keys in [t_a, t_b], in hist[key_b - key].  A count
// is addressed by one add to the element's float bit pattern shifted right
// by 14 (4 * its bf16 bits), since a negative element's key is 0xffff - its
// bits.
__device__ inline ff band_pass_neg(const __nv_bfloat16* __restrict__ row, int V, float c, float mc, int key_a, int key_b,
                            uint32_t* hist) {
    const RowView<__nv_bfloat16> rv(row, V);
    const int tid = threadIdx.x;
    const float t_a = key_value(key_a), t_b = key_value(key_b);
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(hist);
    const uint32_t kb = base - 4u * (uint32_t)(0xffff - key_b);
    // One element, branch-free: returns x's exponent argument when x is above
    // t_b (-inf otherwise) and counts x when it lies inside [t_a, t_b]; xb is
    // x's float bit pattern (bf16 bits << 16).
    auto element = [&](float x, uint32_t xb, float t) -> float {
        float r;
        asm volatile(
            "{\n\t.reg .pred pa, pb;\n\t"
            "setp.gt.f32 pa, %1, %3;\n\t"
            "selp.f32 %0, %2, 0fFF800000, pa;\n\t"
            "setp.ge.and.f32 pb, %1, %4, !pa;\n\t"
            "@pb red.shared.add.u32 [%5], 1;\n\t}"
            : "=f"(r)
            : "f"(x), "f"(t), "f"(t_b), "f"(t_a), "r"(kb + (xb >> 14))
            : "memory");
        return r;
    };
    const float2 cc = make_float2(c, c), nmc = make_float2(-mc, -mc);
    float fsum = 0.0f, fcomp = 0.0f;  // Kahan pair across batches
    auto vec_mass = [&](const uint4& v) -> float {
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t xl = w4[j] << 16, xh = w4[j] & 0xffff0000u;
            const float2 x = make_float2(__uint_as_float(xl), __uint_as_float(xh));
            float2 t = __ffma2_rn(x, cc, nmc);
            t.x = element(x.x, xl, t.x);
            t.y = element(x.y, xh, t.y);
            acc = __fadd2_rn(acc, make_float2(ex2(t.x), ex2(t.y)));
        }
        return acc.x + acc.y;
    };
    auto take_scalar = [&](uint32_t b) {
        const uint32_t xb = b << 16;
        const float x = __uint_as_float(xb);
        fsum += ex2(element(x, xb, fmaf(x, c, -mc)));
    };
    if (tid < rv.head) take_scalar(*reinterpret_cast<const unsigned short*>(row + tid));
    const uint4* vp = rv.vec();
    constexpr int kU2 = 4;  // the re-read comes from L2: fewer vectors in flight suffice
    const uint64_t last_use = l2_evict_first_policy();  // the row's last read
    for (int base_v = tid; base_v < rv.nvec; base_v += kU2 * kNT) {
        uint4 v[kU2];
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
            const int vi = base_v + u * kNT;
            v[u] = (vi < rv.nvec) ? ldg_last_use(vp + vi, last_use) : neg_inf_vec<__nv_bfloat16>();
        }
        float bsum = 0.0f;
#pragma unroll
        for (int u = 0; u < kU2; ++u) bsum += vec_mass(v[u]);
        const float y = bsum - fcomp;
        const float t = fsum + y;
        fcomp = (t - fsum) - y;
        fsum = t;
    }
    if (tid < rv.tail) take_scalar(*reinterpret_cast<const unsigned short*>(row + rv.head + rv.nvec * 8 + tid));
    return ff_add(ff{fsum, 0.0f}, ff{-fcomp, 0.0f});
}

// Key layout of a bracket that spans zero.  bf16 keys crowd near zero (every
// binade down to the denormals), so values with |x| < 2^-10 form one lump,
// measured by its exact mass; the keys above and below it are counted key by
// key: positions [0, Wp) hold keys key_b, key_b - 1, ..., position Wp the
// lump, positions after it keys kn_top, kn_top - 1, ... down to key_a.
constexpr int kLumpPosKey = 0xBA80;  // key of +2^-10: smallest positive key counted one by one
constexpr int kLumpNegKey = 0x457F;  // key of -2^-10: largest negative key counted one by one
struct MixedLayout {
    int key_a, key_b, Wp, Wn, kn_top;
    __device__ MixedLayout(int ka, int kb) : key_a(ka), key_b(kb) {
        Wp = (kb >= kLumpPosKey) ? kb - (ka > kLumpPosKey ? ka : kLumpPosKey) + 1 : 0;
        kn_top = kb < kLumpNegKey ? kb : kLumpNegKey;
        Wn = (ka <= kLumpNegKey) ? kn_top - ka + 1 : 0;
    }
    __device__ int bins() const { return Wp + 1 + Wn; }
};

// Second pass for a bracket spanning zero (layout above): exact mass above
// t_b, exact mass of the lump, exact counts of the other keys inside.
// Branch-free per element: the count goes through one predicated shared
// reduction at a position computed for every element.
__device__ inline void band_pass_mixed(const __nv_bfloat16* __restrict__ row, int V, float c, float mc,
                                       const MixedLayout& L, uint32_t* hist, ff& above, ff& lump) {
    const RowView<__nv_bfloat16> rv(row, V);
    const int tid = threadIdx.x;
    const float t_a = key_value(L.key_a), t_b = key_value(L.key_b);
    const float s0 = 0.0009765625f;  // 2^-10
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(hist);
    const int pos_top = L.key_b, lump_pos = L.Wp, neg_top = L.Wp + 1 + L.kn_top;
    // one element: its exponent argument, its lump weight share, and its count
    auto take = [&](uint32_t b, float& fa, float& fl) {
        const float x = bf16_bits_to_float(b);
        const int k = (int)okey16(b);
        const bool in_band = (x >= t_a) && (x <= t_b);
        const bool in_lump = fabsf(x) < s0;
        const bool abv = x > t_b;
        const int idx = (k >= kLumpPosKey) ? pos_top - k : (in_lump ? lump_pos : neg_top - k);
        const float w = ex2((abv || (in_band && in_lump)) ? fmaf(x, c, -mc) : -INFINITY);
        fa += abv ? w : 0.0f;
        fl += (in_band && in_lump) ? w : 0.0f;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t@p red.shared.add.u32 [%0], 1;\n\t}"
            ::"r"(base + 4u * (uint32_t)idx), "r"((uint32_t)in_band)
            : "memory");
    };
    float fa = 0.0f, fl = 0.0f, ca = 0.0f;
    if (tid < rv.head) take(*reinterpret_cast<const unsigned short*>(row + tid), fa, fl);
    const uint4* vp = rv.vec();
    const uint64_t last_use = l2_evict_first_policy();
    constexpr int kU2 = 4;
    for (int base_v = tid; base_v < rv.nvec; base_v += kU2 * kNT) {
        uint4 v[kU2];
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
            const int vi = base_v + u * kNT;
            v[u] = (vi < rv.nvec) ? ldg_last_use(vp + vi, last_use) : neg_inf_vec<__nv_bfloat16>();
        }
        float ba = 0.0f;
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
            const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                take(w4[j] & 0xffffu, ba, fl);
                take(w4[j] >> 16, ba, fl);
            }
        }
        const float y = ba - ca;  // Kahan across batches
        const float t = fa + y;
        ca = (t - fa) - y;
        fa = t;
    }
    if (tid < rv.tail) take(*reinterpret_cast<const unsigned short*>(row + rv.head + rv.nvec * 8 + tid), fa, fl);
    above = ff_add(ff{fa, 0.0f}, ff{-ca, 0.0f});
    lump = ff{fl, 0.0f};
}

// Exact nucleus of a bf16 row, guided by the pass-1 sample.
//  1. Estimate (warp 0, from value-binned counts of the 1/32 sample and of
//     the threads' maxima):
//     - peaked rows: the thread maxima are distinct elements, so when those
//       at or above some t already weigh top_p * Z (counted at lower-bound
//       weights), the boundary provably lies at or above t; if few elements
//       are estimated above t, they are all counted exactly (one pass, no
//       weights needed);
//     - otherwise the tail below the boundary is made of many light tokens
//       and the sample estimates its mass with a computable standard error:
//       the bracket [t_a, t_b] is where the estimated tail mass crosses
//       (1 - top_p) * Z widened by four standard errors and one bin.
//  2. One pass from L2.  A bracket above zero: exact counts of every key
//     from t_a up to the max (the walk then starts at the max).  Otherwise:
//     exact mass above t_b and exact key counts inside the bracket.
//  3. Walk the key counts.  When the boundary is outside the bracket, the
//     exact counted windows take over from the side it lies on.
// smem: kTopSmemBytes holding the pass-1 sample and thread maxima.
__device__ inline Topp row_topp_bf16(const __nv_bfloat16* __restrict__ row, int V, float c, float m, ff Z,
                                     float top_p, uint8_t* smem, BlockScratch& s) {
    const uint16_t* sample = reinterpret_cast<const uint16_t*>(smem);
    uint32_t* scount = reinterpret_cast<uint32_t*>(smem + kSCountOffset);
    uint32_t* tcount = reinterpret_cast<uint32_t*>(smem + kTCountOffset);
    const float* tmax = reinterpret_cast<const float*>(smem + kTmaxOffset);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float mc = scaled_max(m, c);
    const ff pZ = ff_mul_f(Z, top_p);
    const float tlo = nucleus_lower_bound(m, Z, top_p, V, c);
    const int kmax = (int)value_key(m);
    int key_lo = (tlo > -INFINITY) ? (int)value_key(bf16_bits_to_float(bf16_bits_round_down(tlo))) - 2 : 0x80;
    if (key_lo < 0x80) key_lo = 0x80;  // keys below are -inf and negative NaNs: zero weight
    if (key_lo > kmax) key_lo = kmax;
    const float span = m - tlo;
    int route = 0, key_a = key_lo, key_b = kmax;  // route 0: counted windows from the top
    if (span > 0.0f && span < INFINITY) {
        const float inv_w = (float)kEstBins / span;
        const float cdl = span / (float)kEstBins * c;  // log2 weight step of one bin
        for (int i = tid; i < kEstBins / 4; i += kNT) {
            reinterpret_cast<uint4*>(scount)[i] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4*>(tcount)[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        row_sync();
        auto bin_of = [&](float x) {
            const int j = (int)((m - x) * inv_w);
            return j < 0 ? 0 : (j > kEstBins - 1 ? kEstBins - 1 : j);
        };
        {
            const float x = tmax[tid];
            if (x >= tlo) atomicAdd(&tcount[bin_of(x)], 1u);
        }
        int nv = 0;
        float gb = 0.0f, vb = 0.0f;  // sampled mass (and squares) below tlo
        const int nslots = min(kSampleCap, 2 * kNT * ((rv_nvec(row, V) + kUnroll * kNT - 1) / (kUnroll * kNT)));
        for (int i = tid; i < nslots; i += kNT) {
            const uint32_t b = sample[i];
            if ((b & 0x7fffu) > 0x7f80u) continue;  // empty slot
            const float x = bf16_bits_to_float(b);
            ++nv;
            if (x >= tlo) {
                atomicAdd(&scount[bin_of(x)], 1u);
            } else {
                const float w = weight_of(x, c, mc);
                gb += w;
                vb += w * w;
            }
        }
        nv = warp_sum_i(nv);
        gb = warp_sum_f(gb);
        vb = warp_sum_f(vb);
        if (lane == 0) {
            s.pi[warp] = nv;
            s.pf[warp] = gb;
            s.pf2[warp] = vb;
        }
        row_sync();  // also publishes the bins
        int S = 0;
        float Gb = 0.0f, Vb = 0.0f;
        for (int w = 0; w < kNW; ++w) {  // same order in every thread: identical values
            S += s.pi[w];
            Gb += s.pf[w];
            Vb += s.pf2[w];
        }
        // this thread's bins j = kBinsPerThread * tid + i, j ascending from the max:
        // thread maxima at lower-bound weights (tm), sample mass (sm), its squares (sv), counts (sn)
        const int jt = kBinsPerThread * tid;
        float tmv[kBinsPerThread], smv[kBinsPerThread], svv[kBinsPerThread], snv[kBinsPerThread];
        float4 own = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int i4 = 0; i4 < kBinsPerThread; i4 += 4) {
            const uint4 tc4 = *reinterpret_cast<const uint4*>(tcount + jt + i4);
            const uint4 sc4 = *reinterpret_cast<const uint4*>(scount + jt + i4);
            const uint32_t tca[4] = {tc4.x, tc4.y, tc4.z, tc4.w}, sca[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = i4 + q;
                const float jf = (float)(jt + i);
                const float wc = ex2(-(jf + 0.5f) * cdl);
                tmv[i] = tca[q] ? (float)tca[q] * ex2(-(jf + 2.0f) * cdl) : 0.0f;
                smv[i] = (float)sca[q] * wc;
                svv[i] = smv[i] * wc;
                snv[i] = (float)sca[q];
                own.x += tmv[i]; own.y += smv[i]; own.z += svv[i]; own.w += snv[i];
            }
        }
        // prefixes over bins in j order (four quantities), warp by warp
        float4 inc = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float a = __shfl_up_sync(0xffffffffu, inc.x, o), b = __shfl_up_sync(0xffffffffu, inc.y, o);
            const float d = __shfl_up_sync(0xffffffffu, inc.z, o), e = __shfl_up_sync(0xffffffffu, inc.w, o);
            if (lane >= o) { inc.x += a; inc.y += b; inc.z += d; inc.w += e; }
        }
        float4* wtot = reinterpret_cast<float4*>(smem + kWTotOffset);
        if (lane == 31) wtot[warp] = inc;
        row_sync();
        float4 base = make_float4(0.0f, 0.0f, 0.0f, 0.0f), all = base;
        for (int w = 0; w < kNW; ++w) {
            const float4 t = wtot[w];
            if (w < warp) { base.x += t.x; base.y += t.y; base.z += t.z; base.w += t.w; }
            all.x += t.x; all.y += t.y; all.z += t.z; all.w += t.w;
        }
        // exclusive prefixes at this thread's first bin
        const float pt0 = base.x + inc.x - own.x, pm0 = base.y + inc.y - own.y;
        const float pv0 = base.z + inc.z - own.z, pn0 = base.w + inc.w - own.w;
        // tail of the sample at bin j (values up to bin j's upper edge): G(j) = Gb + all.y - prefix_m(j)
        const float thr_pk = pZ.hi * (1.0f + 1.0f / 4096.0f);
        const float lower = 1.0f - 1.0f / 4096.0f;  // covers the rounding of the weights and sums
        const float T0 = (1.0f - top_p) * ff_to_float(Z) * (float)S / (float)V;
        int jp = 0x7fffffff, j0 = -1;
        {
            float rt = pt0, rm = pm0;
#pragma unroll
            for (int i = 0; i < kBinsPerThread; ++i) {
                const int j = jt + i;
                rt += tmv[i];
                if (jp == 0x7fffffff && rt * lower >= thr_pk) jp = j;
                if (Gb + (all.y - rm) >= T0) j0 = j;
                rm += smv[i];
            }
            if (tid == 0 && Gb >= T0) j0 = max(j0, kEstBins);  // the position below tlo
        }
        int r1 = warp_min_i(jp), r2 = -warp_min_i(-j0);
        if (lane == 0) { s.pi[warp] = r1; s.pi2[warp] = r2; }
        row_sync();
        int Jp = 0x7fffffff, J0 = -1;
        for (int w = 0; w < kNW; ++w) { Jp = min(Jp, s.pi[w]); J0 = max(J0, s.pi2[w]); }
        // the owners of bins Jp + 2 and J0 publish the sample count and the squares there
        {
            float rn = pn0, rv = pv0;
#pragma unroll
            for (int i = 0; i < kBinsPerThread; ++i) {
                const int j = jt + i;
                rn += snv[i];
                if (Jp != 0x7fffffff && j == min(Jp + 2, kEstBins - 1)) s.bcast_f[5] = rn;
                if (j == J0) s.bcast_f[6] = Vb + (all.z - rv);
                rv += svv[i];
            }
            if (tid == 0 && J0 == kEstBins) s.bcast_f[6] = Vb;
        }
        row_sync();
        const float ns = s.bcast_f[5], v0 = s.bcast_f[6];
        if (Jp != 0x7fffffff && (S < 256 || 16.0f * ns <= (float)S)) {
            route = 1;
            const float t_f = m - (float)(Jp + 2) / inv_w;
            key_a = (int)value_key(bf16_bits_to_float(bf16_bits_round_down(t_f < tlo ? tlo : t_f)));
            if (key_a < key_lo) key_a = key_lo;
        } else if (S >= 256 && J0 >= 0 && T0 > 0.0f) {
            float eps = 4.0f * sqrtf(v0) / T0 + 2.0f * cdl + 0.002f;
            eps = eps > 0.9f ? 0.9f : eps;
            const float Ta = T0 * (1.0f - eps), Tb = T0 * (1.0f + eps);
            int ja = -1, jb = -1;
            float rm = pm0;
#pragma unroll
            for (int i = 0; i < kBinsPerThread; ++i) {
                const int j = jt + i;
                const float G = Gb + (all.y - rm);
                if (G >= Ta) ja = j;
                if (G >= Tb) jb = j;
                rm += smv[i];
            }
            if (tid == 0 && Gb >= Ta) ja = max(ja, kEstBins);
            if (tid == 0 && Gb >= Tb) jb = max(jb, kEstBins);
            r1 = -warp_min_i(-ja);
            r2 = -warp_min_i(-jb);
            row_sync();  // everyone has read the previous partials
            if (lane == 0) { s.pi[warp] = r1; s.pi2[warp] = r2; }
            row_sync();
            int JA = -1, JB = -1;
            for (int w = 0; w < kNW; ++w) { JA = max(JA, s.pi[w]); JB = max(JB, s.pi2[w]); }
            // one bin of slack on each side
            float ta = (JA >= kEstBins - 1) ? tlo : m - (float)(JA + 2) / inv_w;
            float tb = m - (float)(JB - 1) / inv_w;
            ta = ta < tlo ? tlo : ta;
            tb = tb > m ? m : tb;
            int ka = (int)value_key(bf16_bits_to_float(bf16_bits_round_down(ta)));
            int kb = (int)value_key(bf16_bits_to_float(bf16_bits_round_down(tb)));
            if (ka < key_lo) ka = key_lo;
            if (kb > kmax) kb = kmax;
            const bool spans = ka <= 0x8000 && kb >= 0x8000;
            const int nb = spans ? MixedLayout(ka, kb).bins() : kb - ka + 1;
            if (kb >= ka && nb <= kFullBins) {
                route = 2;
                key_a = ka;
                key_b = kb;
            }
        }
        row_sync();  // the estimate's shared memory becomes the histogram
    }
    if (route == 1) return topp_windows(row, V, c, mc, Z, pZ, kmax, key_a, ff{0.0f, 0.0f}, hist, s, 0, true);
    if (route == 0) return topp_windows(row, V, c, mc, Z, pZ, kmax, key_lo, ff{0.0f, 0.0f}, hist, s, 0, true);
    // A bracket above zero: counting every key from t_a up to the max costs
    // less per element than weighing the elements above t_b.
    if (key_a > 0x8000) return topp_windows(row, V, c, mc, Z, pZ, kmax, key_lo, ff{0.0f, 0.0f}, hist, s, key_a, true);

    const bool spans = key_a <= 0x8000 && key_b >= 0x8000;
    const MixedLayout L(key_a, key_b);
    const int W = spans ? L.bins() : key_b - key_a + 1;
    for (int i = tid; i < W; i += kNT) hist[i] = 0u;
    row_sync();
    ff part, lpart = ff{0.0f, 0.0f};
    if (!spans) part = band_pass_neg(row, V, c, mc, key_a, key_b, hist);
    else band_pass_mixed(row, V, c, mc, L, hist, part, lpart);
    const ff F_above = block_sum_ff(part, s);  // its barriers also publish the counts
    const ff lump = spans ? block_sum_ff(lpart, s) : ff{0.0f, 0.0f};
    if (ff_ge(F_above, pZ))  // the boundary lies above the bracket
        return topp_windows(row, V, c, mc, Z, pZ, kmax, key_b + 1, ff{0.0f, 0.0f}, hist, s);
    ff F_end;
    const WalkMap map = spans ? WalkMap{key_b, L.Wp, L.kn_top, lump} : plain_map(key_b);
    const WalkOut o = (W <= 2048) ? walk_keys<true, false>(hist, W, map, c, mc, F_above, pZ, &F_end, s)
                                  : walk_keys<false, false>(hist, W, map, c, mc, F_above, pZ, &F_end, s);
    if (o.found == 1) return o.r;
    if (o.found == 2) {  // inside the lump: count its keys exactly, from the mass above it
        const int top = key_b < kLumpPosKey - 1 ? key_b : kLumpPosKey - 1;
        return topp_windows(row, V, c, mc, Z, pZ, top, key_lo, o.F_lump, hist, s);
    }
    // below the bracket: continue downwards from the exact mass above it
    return topp_windows(row, V, c, mc, Z, pZ, key_a - 1, key_lo, F_end, hist, s);
}

// Exact nucleus by bisection over 32-bit ordered keys (any element type):
// the largest key K with mass(key >= K) >= top_p * Z.  One pass per step,
// float-float sums in a fixed order.
template <typename T>
__device__ Topp row_topp_bisect(const T* __restrict__ row, int V, float c, float m, ff Z, float top_p,
                                BlockScratch& s) {
    constexpr int VEC = ElemT<T>::VEC;
    const RowView<T> rv(row, V);
    const float mc = scaled_max(m, c);
    const ff pZ = ff_mul_f(Z, top_p);
    auto mass_ge = [&](uint32_t K, int* cnt_out) -> ff {
        ff acc = ff{0.0f, 0.0f};
        int cnt = 0;
        for (int u = threadIdx.x; u < rv.units(); u += kNT) {
            float f[VEC];
            int i0, n;
            rv.load_unit(u, f, i0, n);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                if (j < n && okey32(f[j]) >= K) {
                    acc = ff_add_f(acc, weight_of(f[j], c, mc));
                    ++cnt;
                }
            }
        }
        if (cnt_out) *cnt_out = block_sum_i(cnt, s);
        return block_sum_ff(acc, s);
    };
    // invariant: mass(>= lo) >= pZ, mass(>= hi) < pZ (hi = one above the max key)
    uint32_t lo = 0x00800000u, hi = okey32(m) + 1u;  // keys below 0x00800000 are -inf and NaNs
    ff F_hi = ff{0.0f, 0.0f};
    while (hi - lo > 1u) {
        const uint32_t mid = lo + (hi - lo) / 2u;
        int cm;
        const ff Fm = mass_ge(mid, &cm);
        if (ff_ge(Fm, pZ)) lo = mid;
        else { hi = mid; F_hi = Fm; }
    }
    Topp r;
    r.tau = okey32_to_float(lo);
    int c_lo;
    mass_ge(lo, &c_lo);
    int c_hi;
    mass_ge(hi, &c_hi);
    r.c_tau = c_lo - c_hi;
    const float w = weight_of(r.tau, c, mc);
    r.n_keep = (r.c_tau > 0) ? keep_count(F_hi, pZ, w, r.c_tau) : 0;
    r.mass = ff_add(F_hi, ff_two_prod((float)r.n_keep, w));
    return r;
}

// Full statistics of one row.  MODE 0: greedy (max/argmax only); 1:
// sampled; 2: sampled with top-p.  tok: the row's token of interest or -1.
// smem: kTopSmemBytes of shared memory (MODE 2 with bf16 only).
template <typename T, int MODE>
__device__ RowStat row_stats(const T* __restrict__ row, int V, float c, float top_p, int tok, uint8_t* smem,
                             BlockScratch& s, SampleScratch& ss) {
    constexpr bool kBand = (MODE == 2 && sizeof(T) == 2);
    const Pass1 p1 = row_pass1<T, (MODE > 0)>(row, V, c, s, kBand ? reinterpret_cast<uint16_t*>(smem) : nullptr,
                                              kBand ? reinterpret_cast<float*>(smem + kTmaxOffset) : nullptr);
    RowStat st;
    st.m = p1.m;
    st.argmax = p1.argmax;
    st.tau = -INFINITY;
    st.n_keep = 0;
    st.c_tau = 0;
    st.flags = 0;
    st.inv_zn = 0.0f;
    st.x_tok = (tok >= 0 && tok < V) ? ElemT<T>::load(row + tok) : __int_as_float(0x7fffffff);
    bool valid = !p1.bad && p1.m > -INFINITY && p1.m < INFINITY;
    if (MODE > 0) valid = valid && (p1.z.hi > 0.0f) && (p1.z.hi < INFINITY);
    if (!valid) {
        st.flags = kRowInvalid;
        return st;
    }
    if (MODE == 0) {
        st.flags = kRowTokMember;
        return st;
    }
    ff mass = p1.z;
    bool member = true;
    if (MODE == 2) {
        Topp tp;
        if constexpr (sizeof(T) == 2) tp = row_topp_bf16(row, V, c, p1.m, p1.z, top_p, smem, s);
        else tp = row_topp_bisect<T>(row, V, c, p1.m, p1.z, top_p, s);
        st.tau = tp.tau;
        st.n_keep = tp.n_keep;
        st.c_tau = tp.c_tau;
        mass = tp.mass;
        const float xt = st.x_tok;
        if (xt == st.tau && tp.n_keep < tp.c_tau) {
            int before = 0;
            row_find_nth_equal<T>(row, V, st.tau, -1, tok, &before, s, ss);
            member = before < tp.n_keep;
        } else {
            member = xt >= st.tau;
        }
    }
    st.inv_zn = 1.0f / ff_to_float(mass);
    st.flags = member ? kRowTokMember : 0;
    return st;
}

}  // namespace sv
