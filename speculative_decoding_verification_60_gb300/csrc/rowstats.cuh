// Row statistics of one logit row, computed by one CTA of kNT threads.
//
// "Accelerating Sonar through speculation", §Target-Draft: acceptance
// compares the full probability distributions of draft and target, so every
// row needs its normaliser; with top-p filtering also the exact nucleus.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int kUnroll = 8;           // 16-byte vectors in flight per thread
constexpr int kHistBins = 32768;     // bf16 key window of the top-p histogram
constexpr int kBinsPerThread = kHistBins / kNT;

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

// Pass 1: one streaming read of the row.  kSum adds the sum of weights
// (online: the running sum is rescaled whenever the running max grows).
template <typename T, bool kSum>
__device__ Pass1 row_pass1(const T* __restrict__ row, int V, float c, BlockScratch& s) {
    constexpr int VEC = ElemT<T>::VEC;
    const RowView<T> rv(row, V);
    const int tid = threadIdx.x;
    float m_t = -INFINITY, z_t = 0.0f, best_bm = -INFINITY;
    int best_batch = -1;
    bool bad = false;
    float x_head = -INFINITY, x_tail = -INFINITY;

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
    for (int base = tid; base < rv.nvec; base += kUnroll * kNT) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int vi = base + u * kNT;
            v[u] = (vi < rv.nvec) ? __ldg(vp + vi) : neg_inf_vec<T>();
        }
        float bm;
        bool nan;
        batch_max<T>(v, bm, nan);
        bad |= nan;
        if (bm > m_t) {
            if (kSum) z_t *= ex2((m_t - bm) * c);
            m_t = bm;
            best_batch = base;
            best_bm = bm;
        }
        if (kSum && m_t > -INFINITY) z_t += batch_weight_sum<T>(v, c, scaled_max(m_t, c));
    }
    if (tid < rv.tail) {
        x_tail = ElemT<T>::load(row + rv.head + rv.nvec * VEC + tid);
        take_scalar(x_tail);
    }

    // Lowest index of this thread holding m_t: head < body < tail.
    int idx = 0x7fffffff;
    {
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
    }

    Pass1 r;
    r.m = block_max(m_t, s);
    double zs = 0.0;
    if (kSum && m_t > -INFINITY) zs = (double)(z_t * ex2((m_t - r.m) * c));
    r.z = kSum ? block_sum_d(zs, s) : 0.0;
    r.argmax = block_min_i(m_t == r.m ? idx : 0x7fffffff, s);
    r.bad = block_any(bad, s);
    if (r.argmax == 0x7fffffff) r.argmax = 0;
    return r;
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
};

// Exact top-p nucleus of a bf16 row by a count histogram of its 16-bit
// keys.  A token of weight w <= (1 - top_p) * Z / V cannot be in the
// nucleus (the tail from the crossing token on holds more than
// (1 - top_p) * Z in at most V tokens, each no heavier than it), so only
// keys above half that bound are counted; the window of kHistBins keys
// below the max is scanned from the top, and a second window follows when
// the crossing lies further down.  hist: kHistBins words of shared memory.
__device__ inline Topp row_topp_bf16(const __nv_bfloat16* __restrict__ row, int V, float c, float m, double Z, float top_p,
                              uint32_t* hist, BlockScratch& s) {
    const RowView<__nv_bfloat16> rv(row, V);
    const int tid = threadIdx.x;
    const float mc = scaled_max(m, c);
    const uint32_t kmax = (m == 0.0f) ? 0x8000u : okey16(__float_as_uint(m) >> 16);
    const double pZ = (double)top_p * Z;
    const double wb = 0.5 * (1.0 - (double)top_p) * Z / (double)V;
    const float vb = m + (float)(log2(wb) / (double)c);
    // keys <= 0x7f are -inf and negative NaNs: zero weight, never the boundary
    int oklo = (int)okey16(bf16_bits_round_down(vb)) - 2;
    if (oklo < 0x80) oklo = 0x80;

    Topp res;
    res.tau = m;
    res.n_keep = 1;
    res.c_tau = 1;
    res.mass = 1.0;
    double F0 = 0.0;
    bool done = false;
    for (int win = 0; win < 2 && !done; ++win) {
        const int hi_ok = (int)kmax - win * kHistBins;
        int lo_ok = hi_ok - kHistBins + 1;
        if (lo_ok < oklo) lo_ok = oklo;
        if (hi_ok < oklo) break;
        for (int i = tid; i < kHistBins / 4; i += kNT) reinterpret_cast<uint4*>(hist)[i] = make_uint4(0, 0, 0, 0);
        __syncthreads();
        auto count_bits = [&](uint32_t b) {
            const int ok = (int)okey16(b);
            if (ok >= lo_ok && ok <= hi_ok) atomicAdd(&hist[hi_ok - ok], 1u);
        };
        if (tid < rv.head) count_bits(*reinterpret_cast<const unsigned short*>(row + tid));
        const uint4* vp = rv.vec();
        for (int base = tid; base < rv.nvec; base += kUnroll * kNT) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int vi = base + u * kNT;
                v[u] = (vi < rv.nvec) ? __ldg(vp + vi) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    count_bits(w[j] & 0xffffu);
                    count_bits(w[j] >> 16);
                }
            }
        }
        if (tid < rv.tail)
            count_bits(*reinterpret_cast<const unsigned short*>(row + rv.head + rv.nvec * 8 + tid));
        __syncthreads();
        // -0 and +0 are one value: fold the -0 count into +0.
        if (win == 0 && tid == 0 && kmax >= 0x8000u) {
            const int ip = (int)kmax - 0x8000;
            if (ip + 1 < kHistBins) {
                hist[ip] += hist[ip + 1];
                hist[ip + 1] = 0;
            }
        }
        __syncthreads();
        // Chunk masses in value-descending order, then the crossing chunk.
        double Mt = 0.0;
        const int b0 = tid * kBinsPerThread;
        for (int i = 0; i < kBinsPerThread; ++i) {
            const uint32_t cnt = hist[b0 + i];
            if (cnt == 0) continue;
            const float x = bf16_bits_to_float(okey16_to_bits((uint32_t)(hi_ok - (b0 + i))));
            Mt += (double)cnt * (double)weight_of(x, c, mc);
        }
        double tot;
        const double St = block_exclusive_scan_d(Mt, s, &tot);
        if (tid == 0) s.bcast_i[1] = 0;
        __syncthreads();
        if (Mt > 0.0 && F0 + St < pZ && F0 + St + Mt >= pZ) {
            double F = F0 + St;
            int last = -1;
            for (int i = 0; i < kBinsPerThread; ++i) {
                const uint32_t cnt = hist[b0 + i];
                if (cnt == 0) continue;
                last = b0 + i;
                const float x = bf16_bits_to_float(okey16_to_bits((uint32_t)(hi_ok - (b0 + i))));
                const double w = (double)weight_of(x, c, mc);
                if (F + (double)cnt * w >= pZ) {
                    int nk = (int)ceil((pZ - F) / w);
                    if (nk < 1) nk = 1;
                    if (nk > (int)cnt) nk = (int)cnt;
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
            if (last >= 0) {  // rounding put pZ at the chunk's very end: keep the whole last bucket
                const uint32_t cnt = hist[last];
                s.bcast_f[0] = bf16_bits_to_float(okey16_to_bits((uint32_t)(hi_ok - last)));
                s.bcast_i[2] = (int)cnt;
                s.bcast_i[3] = (int)cnt;
                s.bcast_d[0] = F;
                s.bcast_i[1] = 1;
            }
        }
        __syncthreads();
        if (s.bcast_i[1]) {
            res.tau = s.bcast_f[0];
            res.n_keep = s.bcast_i[2];
            res.c_tau = s.bcast_i[3];
            res.mass = s.bcast_d[0];
            done = true;
        } else {
            F0 += tot;
        }
        __syncthreads();
    }
    if (!done) {  // unreachable for a valid row: keep everything counted
        res.tau = -INFINITY;
        res.n_keep = 0;
        res.c_tau = 0;
        res.mass = F0 > 0.0 ? F0 : Z;
    }
    return res;
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
    r.tau = okey32_to_float((uint32_t)lo);
    r.c_tau = c_lo - c_hi;
    const double w = (double)weight_of(r.tau, c, mc);
    int nk = (int)ceil((pZ - F_hi) / w);
    if (nk < 1) nk = 1;
    if (nk > r.c_tau) nk = r.c_tau;
    r.n_keep = nk;
    r.mass = F_hi + (double)nk * w;
    return r;
}

// Full statistics of one row.  MODE 0: greedy (max/argmax only); 1:
// sampled; 2: sampled with top-p.  tok: the row's token of interest or -1.
// hist: kHistBins words of shared memory (MODE 2 with bf16 only).
template <typename T, int MODE>
__device__ RowStat row_stats(const T* __restrict__ row, int V, float c, float top_p, int tok, uint32_t* hist,
                             BlockScratch& s) {
    const Pass1 p1 = row_pass1<T, (MODE > 0)>(row, V, c, s);
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
        if constexpr (sizeof(T) == 2) tp = row_topp_bf16(row, V, c, p1.m, p1.z, top_p, hist, s);
        else tp = row_topp_bisect<T>(row, V, c, p1.m, p1.z, top_p, s);
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
    st.inv_zn = (float)(1.0 / mass);
    st.flags = member ? kRowTokMember : 0;
    return st;
}

}  // namespace sv
