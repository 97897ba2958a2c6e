// Row statistics of one logit row, computed by one CTA of kNT threads.
//
// "Accelerating Sonar through speculation", §Target-Draft: acceptance
// compares the full probability distributions of draft and target, so every
// row needs its normaliser; with top-p filtering also the exact nucleus.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int kUnroll = 8;             // 16-byte vectors in flight per thread
// Shared memory of a top-p row (bf16): one 64 KiB region, carved as
//   sample  [0, 16 KiB)      bf16 bit patterns of the systematic sample
//   band    [16, 44 KiB)     counts of the keys inside the bracket: one
//                            histogram per warp (brackets up to
//                            kBandBinsWarp keys) or one shared histogram
//   coarse  [44, 52.25 KiB)  per-warp sample counts of the estimate (u16 pairs)
//   tmcount [52.25, 53.3 KiB) counts of the thread maxima per coarse bin
//   tmax    [60, 62 KiB)     each thread's maximum from pass 1
// and reused whole by the exact full-window fallback.  Per-warp histograms
// keep same-address shared atomics inside one warp instruction.
constexpr int kTopSmemBytes = 64 * 1024;
constexpr int kSampleCap = 8192;       // sample slots (2 per batch of kUnroll vectors)
constexpr int kBandBins = 4096;        // widest bracket, in bf16 keys (shared histogram)
constexpr int kBandBinsWarp = 448;     // widest bracket counted with per-warp histograms
constexpr int kBandOffset = 16384;
constexpr int kCoarseOffset = 45056;
constexpr int kCoarseWords = (257 + 1) / 2;  // 257 u16 counters per warp
constexpr int kTmCountOffset = kCoarseOffset + kNW * kCoarseWords * 4;
constexpr int kCoarseBins = 256;       // value-linear bins of the estimate
constexpr int kFullBins = kTopSmemBytes / 4;  // key window of the fallback histogram
constexpr int kTmaxOffset = 61440;
static_assert(kSampleCap * 2 <= kBandOffset, "sample overlaps the bracket histograms");
static_assert(kBandOffset + kNW * kBandBinsWarp * 4 <= kCoarseOffset, "bracket histograms overlap the estimate");
static_assert(kBandOffset + kBandBins * 4 <= kCoarseOffset, "shared bracket histogram overlaps the estimate");
static_assert(kTmCountOffset + (kCoarseBins + 1) * 4 <= kTmaxOffset, "estimate overlaps the thread maxima");
static_assert(kTmaxOffset + kNT * 4 <= kTopSmemBytes, "thread maxima outside the region");
// The estimate counts samples per bin (integer atomics, order-free) and
// weighs each bin in fixed point (w * 2^40, truncated, which only lowers a
// sum), so every choice made from it is deterministic.
constexpr double kFix = 1099511627776.0;
constexpr float kFixF = 1099511627776.0f;

struct Pass1 {
    float m;     // max (NaN-free); -inf if the row has no non-NaN value
    double z;    // sum of 2^(x*c - m*c) over the row (when requested)
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

// One block reduction of pass 1's per-thread results: the max, the sum of
// weights rescaled to it (fp64), the lowest index holding it, and the NaN
// flag.  Warps merge with shuffles; one barrier publishes the warp results,
// which every thread then merges in the same order.
template <bool kSum>
__device__ __forceinline__ Pass1 reduce_pass1(float m, ff z, int idx, bool bad, float c, BlockScratch& s) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int nb = bad ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
        nb |= __shfl_xor_sync(0xffffffffu, nb, o);
        if (kSum) {
            const ff z2 = ff_shfl_xor(z, o);
            const float mn = fmaxf(m, m2);
            const ff a = (m > -INFINITY) ? ff_scale(z, ex2((m - mn) * c)) : ff{0.0f, 0.0f};
            const ff b = (m2 > -INFINITY) ? ff_scale(z2, ex2((m2 - mn) * c)) : ff{0.0f, 0.0f};
            z = ff_add(a, b);
        }
        idx = (m == m2) ? min(idx, i2) : (m > m2 ? idx : i2);
        m = fmaxf(m, m2);
    }
    if (lane == 0) {
        s.red_m[w] = m;
        s.red_zh[w] = z.hi;
        s.red_zl[w] = z.lo;
        s.red_i[w] = idx;
        s.red_b[w] = nb;
    }
    __syncthreads();
    Pass1 r;
    float M = s.red_m[0];
#pragma unroll 4
    for (int i = 1; i < kNW; ++i) M = fmaxf(M, s.red_m[i]);
    ff Z = ff{0.0f, 0.0f};
    int I = 0x7fffffff, B = 0;
    for (int i = 0; i < kNW; ++i) {
        const float mi = s.red_m[i];
        if (kSum && mi > -INFINITY) Z = ff_add(Z, ff_scale(ff{s.red_zh[i], s.red_zl[i]}, ex2((mi - M) * c)));
        if (mi == M) I = min(I, s.red_i[i]);
        B |= s.red_b[i];
    }
    r.m = M;
    r.z = kSum ? ff_to_double(Z) : 0.0;
    r.argmax = (I == 0x7fffffff) ? 0 : I;
    r.bad = B != 0;
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
        for (int i = tid; i < kSampleCap / 8; i += kNT)
            reinterpret_cast<uint4*>(sample)[i] = make_uint4(0x7fff7fffu, 0x7fff7fffu, 0x7fff7fffu, 0x7fff7fffu);
        __syncthreads();
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

    // Lowest index of this thread holding m_t: head < body < tail.
    int idx = 0x7fffffff;
    if (tid < rv.head && x_head == m_t) {
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

// Index of the n-th (0-based) element, in index order, among those with
// index < limit that equal `val`; INT_MAX when there are fewer.  *count
// receives how many such elements were seen (all of them when n is out of
// reach, which makes this a counter of equals below `limit`).
template <typename T>
__device__ int row_find_nth_equal(const T* __restrict__ row, int V, float val, int n, int limit, int* count,
                                  BlockScratch& s) {
    constexpr int VEC = ElemT<T>::VEC;
    const RowView<T> rv(row, V);
    int seen = 0, found = 0x7fffffff;
    for (int t0 = 0; t0 < rv.units(); t0 += kNT) {
        const int u = t0 + threadIdx.x;
        float f[VEC];
        int i0 = 0, cnt = 0;
        if (u < rv.units()) rv.load_unit(u, f, i0, cnt);
        int mine = 0;
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (j < cnt && i0 + j < limit && f[j] == val) ++mine;
        int tot;
        const int before = block_exclusive_scan_i(mine, s, &tot);
        if (n >= seen + before && n < seen + before + mine) {
            int k = n - seen - before;
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                if (j < cnt && i0 + j < limit && f[j] == val) {
                    if (k == 0) s.bcast_i[0] = i0 + j;
                    --k;
                }
            }
        }
        seen += tot;
        __syncthreads();
        const bool hit = n < seen;  // uniform across the CTA
        if (hit) found = s.bcast_i[0];
        __syncthreads();
        if (hit) break;
    }
    if (count) *count = seen;
    return found;
}


struct Topp {
    float tau;     // boundary logit
    int n_keep;    // boundary-valued tokens kept
    int c_tau;     // boundary-valued tokens in the row
    double mass;   // nucleus mass (weights relative to the max)
    bool ok;
};

// Key of a bf16 value with -0 folded onto +0.
__device__ __forceinline__ uint32_t value_key(float x) {
    return x == 0.0f ? 0x8000u : okey16(__float_as_uint(x) >> 16);
}

// Walk bins holding counts of consecutive keys from `key_top` downwards
// (bin i = key key_top - i), starting at mass F0 above the window, and find
// where the mass reaches pZ.  Bins are split into contiguous per-thread
// chunks; chunk masses are scanned in fp64.  Returns ok = false when the
// window ends first (then *F_end holds the mass above the window's bottom).
__device__ inline Topp scan_key_bins(const uint32_t* hist, int nbins, int key_top, float c, float mc, double F0,
                                     double pZ, double* F_end, BlockScratch& s) {
    const int per = (nbins + kNT - 1) / kNT;
    const int b0 = threadIdx.x * per;
    ff Mf = ff{0.0f, 0.0f};
    for (int i = 0; i < per; ++i) {
        const int b = b0 + i;
        if (b >= nbins) break;
        const uint32_t cnt = hist[b];
        if (cnt == 0) continue;
        const float x = bf16_bits_to_float(okey16_to_bits((uint32_t)(key_top - b)));
        const float w = weight_of(x, c, mc);
        const float p = (float)cnt * w;
        Mf = ff_add(Mf, ff{p, fmaf((float)cnt, w, -p)});  // exact product as a pair
    }
    ff totf;
    const ff Sf = block_exclusive_scan_ff(Mf, s, &totf);
    const double Mt = ff_to_double(Mf), St = ff_to_double(Sf), tot = ff_to_double(totf);
    if (threadIdx.x == 0) s.bcast_i[1] = 0;
    __syncthreads();
    if (Mt > 0.0 && F0 + St < pZ && F0 + St + Mt >= pZ) {
        double F = F0 + St;
        int last = -1;
        for (int i = 0; i < per; ++i) {
            const int b = b0 + i;
            if (b >= nbins) break;
            const uint32_t cnt = hist[b];
            if (cnt == 0) continue;
            last = b;
            const float x = bf16_bits_to_float(okey16_to_bits((uint32_t)(key_top - b)));
            const double w = (double)weight_of(x, c, mc);
            if (F + (double)cnt * w >= pZ) {
                int nk = (int)ceil((pZ - F) / w);
                nk = nk < 1 ? 1 : (nk > (int)cnt ? (int)cnt : nk);
                s.bcast_f[0] = x;
                s.bcast_i[2] = nk;
                s.bcast_i[3] = (int)cnt;
                s.bcast_d[0] = F + (double)nk * w;
                s.bcast_i[1] = 1;
                last = -2;
                break;
            }
            F += (double)cnt * w;
        }
        if (last >= 0) {  // pZ at the chunk's very end after rounding: keep the last bucket whole
            s.bcast_f[0] = bf16_bits_to_float(okey16_to_bits((uint32_t)(key_top - last)));
            s.bcast_i[2] = (int)hist[last];
            s.bcast_i[3] = (int)hist[last];
            s.bcast_d[0] = F;
            s.bcast_i[1] = 1;
        }
    }
    __syncthreads();
    Topp r;
    r.ok = s.bcast_i[1] != 0;
    r.tau = s.bcast_f[0];
    r.n_keep = s.bcast_i[2];
    r.c_tau = s.bcast_i[3];
    r.mass = s.bcast_d[0];
    if (F_end) *F_end = F0 + tot;
    __syncthreads();
    return r;
}

// Lower bound on the nucleus boundary: a token of weight w <= (1 - top_p) *
// Z / V cannot be kept (the tail from the crossing token on holds more than
// (1 - top_p) * Z in at most V tokens, none heavier than it).  Returned as a
// value a little below that bound.
__device__ __forceinline__ float nucleus_lower_bound(float m, double Z, float top_p, int V, float c) {
    const float wb = 0.5f * (1.0f - top_p) * (float)Z / (float)V;
    return m + log2f(wb) / c;
}

// Exact nucleus by count histograms of the 16-bit keys over successive
// windows of kFullBins keys below the max, walked from the top.  Keys below
// the weight bound are never counted.  Shared memory: kFullBins words.
__device__ inline Topp row_topp_bf16_full(const __nv_bfloat16* __restrict__ row, int V, float c, float m, double Z,
                                          float top_p, uint32_t* hist, BlockScratch& s, int key_floor = -1) {
    const RowView<__nv_bfloat16> rv(row, V);
    const int tid = threadIdx.x;
    const float mc = scaled_max(m, c);
    const int kmax = (int)value_key(m);
    const double pZ = (double)top_p * Z;
    // keys <= 0x7f are -inf and negative NaNs: zero weight, never the boundary
    int oklo = (int)okey16(bf16_bits_round_down(nucleus_lower_bound(m, Z, top_p, V, c))) - 2;
    if (oklo < 0x80) oklo = 0x80;
    if (key_floor > oklo) oklo = key_floor;
    double F0 = 0.0;
    for (int hi_ok = kmax; hi_ok >= oklo;) {
        int lo_ok = hi_ok - kFullBins + 1;
        if (lo_ok < oklo) lo_ok = oklo;
        if (lo_ok == 0x8000 && hi_ok > 0x8000) lo_ok = 0x8001;  // keep +0 and -0 in one window
        const int nb = hi_ok - lo_ok + 1;
        for (int i = tid; i < kFullBins / 4; i += kNT) reinterpret_cast<uint4*>(hist)[i] = make_uint4(0, 0, 0, 0);
        __syncthreads();
        const uint4* vp = rv.vec();
        for (int u = tid; u < rv.units(); u += kNT) {
            int i0, cnt;
            rv.unit_range(u, i0, cnt);
            uint32_t w[4];
            if (u >= 1 && u <= rv.nvec) {
                const uint4 v = __ldg(vp + (u - 1));
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            } else {
                const unsigned short* p16 = reinterpret_cast<const unsigned short*>(row) + i0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t lo = (2 * j < cnt) ? p16[2 * j] : 0xff80u;
                    const uint32_t hi = (2 * j + 1 < cnt) ? p16[2 * j + 1] : 0xff80u;
                    w[j] = lo | (hi << 16);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t b = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu);
                const int ok = (int)okey16(b);
                if (ok >= lo_ok && ok <= hi_ok) atomicAdd(&hist[hi_ok - ok], 1u);
            }
        }
        __syncthreads();
        // -0 and +0 are one value: fold the -0 count onto +0
        if (tid == 0 && hi_ok >= 0x8000 && lo_ok <= 0x7fff) {
            hist[hi_ok - 0x8000] += hist[hi_ok - 0x7fff];
            hist[hi_ok - 0x7fff] = 0;
        }
        __syncthreads();
        double F_end;
        const Topp r = scan_key_bins(hist, nb, hi_ok, c, mc, F0, pZ, &F_end, s);
        if (r.ok) return r;
        F0 = F_end;
        hi_ok = lo_ok - 1;
    }
    Topp r;  // not reached above key_floor (or, without a floor, only by rounding)
    r.ok = false;
    r.tau = -INFINITY;
    r.n_keep = 0;
    r.c_tau = 0;
    r.mass = F0 > 0.0 ? F0 : Z;
    return r;
}

// Exact nucleus guided by the pass-1 sample (bf16 rows).
//  1. From the sample and the exact Z, estimate where the mass strictly
//     below t reaches (1 - top_p) * Z: the tail is made of many light
//     tokens, so a 1/32 sample estimates it well, and the few heavy tokens
//     (which the sample may miss) sit far above it.  Widen by a
//     sampling-error margin into a bracket [t_a, t_b] of bf16 values.
//  2. Re-read the row (from L2): exact mass strictly above t_b, and exact
//     counts of the keys inside the bracket.
//  3. Walk the bracket from the top.  ok = false when the crossing is not
//     inside it; the caller then runs the full method.
// Before that, a peaked row takes a cheaper exact route: each thread's
// maximum is a distinct element, so when the maxima at or above t already
// weigh top_p * Z, the boundary lies above t; if few tokens are estimated
// above that t, all of them are counted exactly (no mass pass needed).
// smem: kTopSmemBytes holding the pass-1 sample and thread maxima.
__device__ inline Topp row_topp_bf16_guided(const __nv_bfloat16* __restrict__ row, int V, float c, float m, double Z,
                                            float top_p, uint8_t* smem, BlockScratch& s) {
    const uint16_t* sample = reinterpret_cast<const uint16_t*>(smem);
    uint32_t* band = reinterpret_cast<uint32_t*>(smem + kBandOffset);
    uint32_t* wcount = reinterpret_cast<uint32_t*>(smem + kCoarseOffset);  // per-warp u16 pairs
    int* tmcount = reinterpret_cast<int*>(smem + kTmCountOffset);         // thread-maximum counts
    int* ccount = reinterpret_cast<int*>(smem + kBandOffset);             // merged sample counts
    const float* tmax = reinterpret_cast<const float*>(smem + kTmaxOffset);
    const int tid = threadIdx.x;
    const float mc = scaled_max(m, c);
    const double pZ = (double)top_p * Z;
    const float tlo = nucleus_lower_bound(m, Z, top_p, V, c);
    const float span = m - tlo;
    Topp fail;
    fail.ok = false;
    if (!(span > 0.0f) || !(span < INFINITY)) return fail;

    // 1. estimate from the sample (bin kCoarseBins collects values below tlo)
    for (int i = tid; i < kNW * kCoarseWords; i += kNT) wcount[i] = 0u;
    for (int i = tid; i <= kCoarseBins; i += kNT) tmcount[i] = 0;
    __syncthreads();
    const float inv_w = (float)kCoarseBins / span;
    {
        const float x = tmax[tid];
        if (x >= tlo) {
            int bin = (int)((m - x) * inv_w);
            bin = bin < 0 ? 0 : (bin > kCoarseBins - 1 ? kCoarseBins - 1 : bin);
            atomicAdd(&tmcount[bin], 1);
        }
    }
    int nvalid = 0;
    for (int i = tid; i < kSampleCap; i += kNT) {
        const uint32_t b = sample[i];
        if ((b & 0x7fffu) > 0x7f80u) continue;  // empty slot (NaN pattern)
        const float x = bf16_bits_to_float(b);
        ++nvalid;
        int bin = kCoarseBins;
        if (x >= tlo) {
            bin = (int)((m - x) * inv_w);
            bin = bin < 0 ? 0 : (bin > kCoarseBins - 1 ? kCoarseBins - 1 : bin);
        }
        atomicAdd(&wcount[(tid >> 5) * kCoarseWords + (bin >> 1)], 1u << ((bin & 1) * 16));
    }
    const int S = block_sum_i(nvalid, s);
    // merge the per-warp counters (block_sum_i above ended with a barrier)
    for (int i = tid; i <= kCoarseBins; i += kNT) {
        int t = 0;
        for (int w = 0; w < kNW; ++w) t += (int)((wcount[w * kCoarseWords + (i >> 1)] >> ((i & 1) * 16)) & 0xffffu);
        ccount[i] = t;
    }
    __syncthreads();
    // Warp 0 turns the bins into the decision: prefix sums in fixed point,
    // crossings found by ballot.  Bottom-up positions q: q = 0 is the bin
    // below tlo, q >= 1 is coarse bin j = kCoarseBins - q (rising values).
    if (tid < 32) {
        const int lane = tid;
        // peaked route (top-down over bins j): thread maxima against top_p * Z
        int floor_key = -1;
        {
            // each thread maximum in bin j weighs at least the weight of the
            // bin's lower edge, so these masses never exceed the true ones
            unsigned long long tm[8], cum = 0ull;
            int cn[8], ccum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = 8 * lane + i;
                const float w_lo = weight_of(m - (float)(j + 1) / inv_w, c, mc);
                tm[i] = (unsigned long long)tmcount[j] * (unsigned long long)(w_lo * kFixF);
                cn[i] = ccount[j];
                cum += tm[i];
                ccum += cn[i];
            }
            unsigned long long pre = cum;
            int cpre = ccum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, pre, o);
                const int yc = __shfl_up_sync(0xffffffffu, cpre, o);
                if (lane >= o) { pre += y; cpre += yc; }
            }
            pre -= cum;
            cpre -= ccum;
            const unsigned long long pZf = (unsigned long long)(pZ * kFix);
            int hit = -1, nab = 0;
            for (int i = 0; i < 8 && hit < 0; ++i) {
                pre += tm[i];
                cpre += cn[i];
                if (pre >= pZf) { hit = 8 * lane + i; nab = cpre; }
            }
            const unsigned bal = __ballot_sync(0xffffffffu, hit >= 0);
            if (bal) {
                const int src = __ffs(bal) - 1;
                const int jp = __shfl_sync(0xffffffffu, hit, src);
                const int nabove_s = __shfl_sync(0xffffffffu, nab, src);
                const double nabove = S > 0 ? (double)nabove_s * (double)V / (double)S : (double)V;
                if (nabove <= (double)V / 64.0 || S < 512) {
                    const float edge = m - (float)(jp + 1) / inv_w;
                    floor_key = (int)value_key(bf16_bits_to_float(bf16_bits_round_down(edge < tlo ? tlo : edge))) - 1;
                }
            }
        }
        // sampled bracket (bottom-up over positions q)
        int key_a = -1, key_b = -1;
        if (floor_key < 0 && S >= 512) {
            unsigned long long mm[9], cum = 0ull;
            int cc[9], ccum = 0;
#pragma unroll
            for (int i = 0; i < 9; ++i) {
                const int q = 9 * lane + i;
                const int idx = (q == 0) ? kCoarseBins : kCoarseBins - q;
                const float xc = (q == 0) ? tlo : m - ((float)idx + 0.5f) / inv_w;  // bin centre
                cc[i] = (q <= kCoarseBins) ? ccount[idx] : 0;
                mm[i] = (unsigned long long)cc[i] * (unsigned long long)(weight_of(xc, c, mc) * kFixF);
                cum += mm[i];
                ccum += cc[i];
            }
            unsigned long long pre = cum;
            int cpre = ccum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, pre, o);
                const int yc = __shfl_up_sync(0xffffffffu, cpre, o);
                if (lane >= o) { pre += y; cpre += yc; }
            }
            pre -= cum;
            cpre -= ccum;
            const double T0 = (1.0 - (double)top_p) * Z * (double)S / (double)V;
            // first position whose running mass reaches a threshold (9*32 if none)
            auto first_ge = [&](unsigned long long thr, int* count_at) -> int {
                unsigned long long r = pre;
                int rc = cpre, hit = -1, hc = 0;
                for (int i = 0; i < 9; ++i) {
                    r += mm[i];
                    rc += cc[i];
                    if (hit < 0 && r >= thr && 9 * lane + i <= kCoarseBins) { hit = 9 * lane + i; hc = rc; }
                }
                const unsigned bal = __ballot_sync(0xffffffffu, hit >= 0);
                if (!bal) return 9 * 32;
                const int src = __ffs(bal) - 1;
                if (count_at) *count_at = __shfl_sync(0xffffffffu, hc, src);
                return __shfl_sync(0xffffffffu, hit, src);
            };
            int ncross = 0;
            const int qx = first_ge((unsigned long long)(T0 * kFix), &ncross);
            if (qx <= kCoarseBins && ncross > 0) {
                const double eps = 4.0 / sqrt((double)ncross) + 0.03;
                const int qa_next = first_ge((unsigned long long)fmax(0.0, T0 * (1.0 - eps) * kFix) + 1ull, nullptr);
                const int qb = first_ge((unsigned long long)(T0 * (1.0 + eps) * kFix), nullptr);
                if (qb <= kCoarseBins) {
                    const int qa = qa_next - 1;  // last position still at or below T0 * (1 - eps)
                    const int ja = (qa >= 1) ? kCoarseBins - qa : kCoarseBins;
                    const int jb = kCoarseBins - (qb > 1 ? qb : 1);
                    // widen by one bin on each side
                    const float ta = (ja >= kCoarseBins) ? tlo : m - (float)(ja + 2) / inv_w;
                    const float tb = m - (float)(jb - 1) / inv_w;
                    const float ta_c = ta < tlo ? tlo : ta;
                    const float tb_c = tb > m ? m : tb;
                    key_a = (int)value_key(bf16_bits_to_float(bf16_bits_round_down(ta_c)));
                    key_b = (int)value_key(bf16_bits_to_float(bf16_bits_round_down(tb_c)));
                    if (key_a <= 0x8000 && key_b >= 0x8000) key_a = key_a < 0x7fff ? key_a : 0x7fff;  // include -0
                    if (key_a < 0x80) key_a = 0x80;
                    if (key_b - key_a + 1 > kBandBins || key_b < key_a) key_a = -1;
                }
            }
        }
        if (lane == 0) {
            s.bcast_i[0] = key_a;
            s.bcast_i[1] = key_b;
            s.bcast_i[2] = floor_key;
        }
    }
    __syncthreads();
    const int floor_key = s.bcast_i[2];
    if (floor_key >= 0) {
        __syncthreads();
        return row_topp_bf16_full(row, V, c, m, Z, top_p, reinterpret_cast<uint32_t*>(smem), s, floor_key);
    }
    const int key_a = s.bcast_i[0], key_b = s.bcast_i[1];
    __syncthreads();
    if (key_a < 0) return fail;
    const int W = key_b - key_a + 1;
    const float t_b = bf16_bits_to_float(okey16_to_bits((uint32_t)key_b));
    const float t_a = bf16_bits_to_float(okey16_to_bits((uint32_t)key_a));

    // 2. exact mass above t_b and exact counts inside [t_a, t_b]
    const bool per_warp = W <= kBandBinsWarp;
    const int nwords = per_warp ? kNW * W : W;
    for (int i = tid; i < nwords; i += kNT) band[i] = 0u;
    __syncthreads();
    uint32_t* myband = per_warp ? band + (tid >> 5) * W : band;
    const RowView<__nv_bfloat16> rv(row, V);
    // Per 16-byte vector: the weights of elements above t_b (others get
    // 2^-inf = 0) summed with packed FP32 pairs, and an 8-bit mask of the
    // elements inside the bracket, whose keys are counted in one branch.
    const float2 cc = make_float2(c, c), nmc = make_float2(-mc, -mc);
    float fsum = 0.0f, fcomp = 0.0f;  // Kahan pair across batches
    // Histogram index key_b - key(b): one add when the bracket lies on one
    // side of zero (keys of one sign are affine in the bit pattern).
    const int sgn = (key_a >= 0x8000) ? 0 : (key_b <= 0x7fff ? 1 : 2);
    const uint32_t kpos = (uint32_t)(key_b - 0x8000), kneg = (uint32_t)(key_b - 0xffff);
    auto count_key = [&](uint32_t b) {
        if (sgn == 0) atomicAdd(&myband[kpos - b], 1u);
        else if (sgn == 1) atomicAdd(&myband[kneg + b], 1u);
        else {
            const uint32_t idx = (uint32_t)(key_b - (int)okey16(b));
            if (idx < (uint32_t)W) atomicAdd(&myband[idx], 1u);
        }
    };
    auto vec_mass = [&](const uint4& v) -> float {
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 x = make_float2(bf16_lo(w4[j]), bf16_hi(w4[j]));
            float2 t = __ffma2_rn(x, cc, nmc);
            const bool ax = x.x > t_b, ay = x.y > t_b;
            t.x = ax ? t.x : -INFINITY;
            t.y = ay ? t.y : -INFINITY;
            acc = __fadd2_rn(acc, make_float2(ex2(t.x), ex2(t.y)));
            if (!ax && x.x >= t_a) count_key(w4[j] & 0xffffu);
            if (!ay && x.y >= t_a) count_key(w4[j] >> 16);
        }
        return acc.x + acc.y;
    };
    auto take_scalar = [&](uint32_t b) {
        const float x = bf16_bits_to_float(b);
        fsum += (x > t_b) ? weight_of(x, c, mc) : 0.0f;
        if (x >= t_a && x <= t_b) count_key(b);
    };
    if (tid < rv.head) take_scalar(*reinterpret_cast<const unsigned short*>(row + tid));
    const uint4* vp = rv.vec();
    constexpr int kU2 = 4;  // the re-read comes from L2: fewer vectors in flight suffice
    for (int base = tid; base < rv.nvec; base += kU2 * kNT) {
        uint4 v[kU2];
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
            const int vi = base + u * kNT;
            v[u] = (vi < rv.nvec) ? __ldg(vp + vi) : neg_inf_vec<__nv_bfloat16>();
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
    const double F_above = ff_to_double(block_sum_ff(ff_add(ff{fsum, 0.0f}, ff{-fcomp, 0.0f}), s));
    if (per_warp) {  // fold the warps' histograms into the first one
        for (int i = tid; i < W; i += kNT) {
            uint32_t t = 0u;
            for (int w = 0; w < kNW; ++w) t += band[w * W + i];
            band[i] = t;
        }
        __syncthreads();
    }
    if (tid == 0 && key_b >= 0x8000 && key_a <= 0x7fff) {
        band[key_b - 0x8000] += band[key_b - 0x7fff];
        band[key_b - 0x7fff] = 0;
    }
    __syncthreads();
    if (F_above >= pZ) return fail;  // the boundary lies above the bracket

    // 3. walk the bracket
    return scan_key_bins(band, W, key_b, c, mc, F_above, pZ, nullptr, s);
}

// Exact top-p nucleus by bisection over 32-bit ordered keys (any element
// type): the largest key K with mass(key >= K) >= top_p * Z.  One pass per
// step, deterministic sums.
template <typename T>
__device__ Topp row_topp_bisect(const T* __restrict__ row, int V, float c, float m, double Z, float top_p,
                                BlockScratch& s) {
    constexpr int VEC = ElemT<T>::VEC;
    const RowView<T> rv(row, V);
    const float mc = scaled_max(m, c);
    const double pZ = (double)top_p * Z;
    auto mass_ge = [&](uint32_t K, int* cnt_out) -> double {
        double acc = 0.0;
        int cnt = 0;
        for (int u = threadIdx.x; u < rv.units(); u += kNT) {
            float f[VEC];
            int i0, n;
            rv.load_unit(u, f, i0, n);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                if (j < n && f[j] == f[j] && okey32(f[j]) >= K) {
                    acc += (double)weight_of(f[j], c, mc);
                    ++cnt;
                }
            }
        }
        *cnt_out = block_sum_i(cnt, s);
        return block_sum_d(acc, s);
    };
    const uint32_t kmax = okey32(m);
    uint64_t lo = 0, hi = (uint64_t)kmax + 1;  // mass(>= lo) >= pZ > mass(>= hi)
    double F_hi = 0.0;
    int c_hi = 0;
    while (hi - lo > 1) {
        const uint64_t mid = lo + (hi - lo) / 2;
        int cm;
        const double Fm = mass_ge((uint32_t)mid, &cm);
        if (Fm >= pZ) lo = mid;
        else { hi = mid; F_hi = Fm; c_hi = cm; }
    }
    int c_lo;
    mass_ge((uint32_t)lo, &c_lo);
    Topp r;
    r.ok = true;
    r.tau = okey32_to_float((uint32_t)lo);
    r.c_tau = c_lo - c_hi;
    const double w = (double)weight_of(r.tau, c, mc);
    int nk = (int)ceil((pZ - F_hi) / w);
    nk = nk < 1 ? 1 : (nk > r.c_tau ? r.c_tau : nk);
    r.n_keep = nk;
    r.mass = F_hi + (double)nk * w;
    return r;
}

// Full statistics of one row.  MODE 0: greedy (max/argmax only); 1:
// sampled; 2: sampled with top-p.  tok: the row's token of interest or -1.
// smem: kTopSmemBytes of shared memory (MODE 2 with bf16 only).
template <typename T, int MODE>
__device__ RowStat row_stats(const T* __restrict__ row, int V, float c, float top_p, int tok, uint8_t* smem,
                             BlockScratch& s) {
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
    if (threadIdx.x == 0) s.bcast_f[1] = (tok >= 0 && tok < V) ? ElemT<T>::load(row + tok) : __int_as_float(0x7fffffff);
    __syncthreads();
    st.x_tok = s.bcast_f[1];
    __syncthreads();
    bool valid = !p1.bad && p1.m > -INFINITY && p1.m < INFINITY;
    if (MODE > 0) valid = valid && (p1.z > 0.0) && (p1.z < 1e300);
    if (!valid) {
        st.flags = kRowInvalid;
        return st;
    }
    if (MODE == 0) {
        st.flags = kRowTokMember;
        return st;
    }
    double mass = p1.z;
    bool member = true;
    if (MODE == 2) {
        Topp tp;
        if constexpr (sizeof(T) == 2) {
            tp = row_topp_bf16_guided(row, V, c, p1.m, p1.z, top_p, smem, s);
            if (!tp.ok) tp = row_topp_bf16_full(row, V, c, p1.m, p1.z, top_p, reinterpret_cast<uint32_t*>(smem), s);
        } else {
            tp = row_topp_bisect<T>(row, V, c, p1.m, p1.z, top_p, s);
        }
        st.tau = tp.tau;
        st.n_keep = tp.n_keep;
        st.c_tau = tp.c_tau;
        mass = tp.mass;
        const float xt = st.x_tok;
        if (xt == st.tau && tp.n_keep < tp.c_tau) {
            int before = 0;
            row_find_nth_equal<T>(row, V, st.tau, 0x7fffffff, tok, &before, s);
            member = before < tp.n_keep;
        } else {
            member = xt >= st.tau;
        }
    }
    st.inv_zn = 1.0f / (float)mass;
    st.flags = member ? kRowTokMember : 0;
    return st;
}

}  // namespace sv
