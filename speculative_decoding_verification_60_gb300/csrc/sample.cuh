// Block-wide inverse-CDF draw over one vocabulary row (or row pair).
//
// "Accelerating Sonar through speculation", §Target-Draft: at the
// mismatch, or after the last draft, the target logits are sampled for one
// more token; the cited rule draws that token from norm(max(0, p - q)) at a
// rejection and from p after a full accept.  The draw is the smallest v with
// C(v) > u * C(V-1), C the running sum of the weights in index order.
//
// The row is walked in tiles of kNT "units" (RowView: head, 16-byte vectors,
// tail).  Pass A keeps one fp64 sum per tile; the crossing tile is walked
// again and scanned.  Only the selected row(s) are read, twice.
#pragma once

#include "rowstats.cuh"

namespace sv {

constexpr int kMaxTiles = 1024;

struct SampleScratch {
    double tile[kMaxTiles];
};

// WeightFn: void operator()(int unit, float* w /*[VEC]*/, int& idx0, int& cnt) const
// Returns the drawn index, or -1 when every weight is zero.
template <int VEC, typename WeightFn>
__device__ int block_inverse_cdf(int units, float u, const WeightFn& wf, BlockScratch& s, SampleScratch& ss) {
    const int ntiles = (units + kNT - 1) / kNT;
    for (int t = 0; t < ntiles; ++t) {
        const int unit = t * kNT + threadIdx.x;
        float w[VEC];
        int i0 = 0, cnt = 0;
        float acc = 0.0f;
        if (unit < units) {
            wf(unit, w, i0, cnt);
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (j < cnt) acc += w[j];
        }
        const ff ts = block_sum_ff(ff_from(acc), s);
        if (threadIdx.x == 0) ss.tile[t] = ff_to_double(ts);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int t = 0; t < ntiles; ++t) tot += ss.tile[t];
        int jt = -1;
        double pre = 0.0, target = (double)u * tot;
        if (tot > 0.0) {
            double c = 0.0;
            int lastpos = -1;
            for (int t = 0; t < ntiles; ++t) {
                if (ss.tile[t] > 0.0) lastpos = t;
                if (c + ss.tile[t] > target) { jt = t; pre = c; break; }
                c += ss.tile[t];
            }
            if (jt < 0) {  // rounding: take the last tile with weight
                jt = lastpos;
                pre = 0.0;
                for (int t = 0; t < jt; ++t) pre += ss.tile[t];
                target = pre + ss.tile[jt] * 0.999999999;
            }
        }
        s.bcast_i[4] = jt;
        s.bcast_d[1] = pre;
        s.bcast_d[2] = target;
    }
    __syncthreads();
    const int jt = s.bcast_i[4];
    const double pre = s.bcast_d[1], target = s.bcast_d[2];
    __syncthreads();
    if (jt < 0) return -1;

    const int unit = jt * kNT + threadIdx.x;
    float w[VEC];
    int i0 = 0, cnt = 0;
    float acc = 0.0f;
    if (unit < units) {
        wf(unit, w, i0, cnt);
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (j < cnt) acc += w[j];
    }
    const double before = pre + ff_to_double(block_exclusive_scan_ff(ff_from(acc), s, nullptr));
    if (threadIdx.x == 0) { s.bcast_i[5] = 0x7fffffff; s.bcast_i[6] = -1; }
    __syncthreads();
    int last_pos = -1;
#pragma unroll
    for (int j = 0; j < VEC; ++j)
        if (j < cnt && w[j] > 0.0f) last_pos = i0 + j;
    if (last_pos >= 0) atomicMax(&s.bcast_i[6], last_pos);
    if (acc > 0.0f && before <= target && before + (double)acc > target) {
        double run = before;
        int pick = -1;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            if (j < cnt && pick < 0) {
                run += (double)w[j];
                if (w[j] > 0.0f && run > target) pick = i0 + j;
            }
        }
        if (pick < 0) pick = last_pos;
        atomicMin(&s.bcast_i[5], pick);
    }
    __syncthreads();
    int r = s.bcast_i[5];
    if (r == 0x7fffffff) r = s.bcast_i[6];  // rounding at the tile's end
    __syncthreads();
    return r;
}

// Sum over a row of a per-unit weight function (fp64, deterministic).
template <int VEC, typename WeightFn>
__device__ double block_weight_total(int units, const WeightFn& wf, BlockScratch& s) {
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
    return ff_to_double(block_sum_ff(acc, s));
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
    __device__ __forceinline__ float prob_at(int v) const {
        const float x = ElemT<T>::load(row + v);
        const bool member = (x > st.tau) || (x == st.tau && v <= cut);
        return member ? weight_of(x, c, mc) * st.inv_zn : 0.0f;
    }
};

// Index of the last kept boundary-valued token of a filtered row.
template <typename T>
__device__ int nucleus_cut(const T* row, int V, const RowStat& st, BlockScratch& s) {
    if (!(st.tau > -INFINITY) || st.n_keep >= st.c_tau) return 0x7fffffff;
    return row_find_nth_equal<T>(row, V, st.tau, st.n_keep - 1, 0x7fffffff, nullptr, s);
}

}  // namespace sv
