// Device building blocks of libspecverify (sm_103a).
//
// Method: "Accelerating Sonar through speculation", sections "Speculative
// decoding", "Target-Draft", "EAGLE", "MTP"; rule of the cited "Fast
// Inference from Transformers via Speculative Decoding".
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

// Threads of a row-level CTA.  Each translation unit may set its own (the
// build passes -DSV_NT); device code is compiled per unit, so the sizes do
// not meet.
#ifndef SV_NT
#define SV_NT 256
#endif
constexpr int kNT = SV_NT;
constexpr int kNW = kNT / 32;        // warps of such a CTA
constexpr int kPurposeAccept = 1;
constexpr int kPurposeResidual = 2;
constexpr int kPurposeBonus = 3;
constexpr int kPurposeDraft = 4;

constexpr int kDevErrToken = 1;
constexpr int kDevErrNonfinite = 2;
constexpr int kDevErrParent = 4;
constexpr int kDevErrLength = 8;
constexpr int kDevErrTimeout = 16;

// ---------------------------------------------------------------- Philox --
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with a
// Weyl key schedule.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

// u in [0, 1) on the 2^-24 grid (exact in fp32):
// key = (seed lo, seed hi), counter = (req lo, pos lo, purpose | round << 8, req hi).
__device__ __forceinline__ float uniform01(uint64_t seed, int64_t req, int64_t pos, int purpose, int round) {
    const uint64_t r = (uint64_t)req;
    const uint4 c = make_uint4((uint32_t)r, (uint32_t)(uint64_t)pos, (uint32_t)purpose | ((uint32_t)round << 8),
                               (uint32_t)(r >> 32));
    const uint4 o = philox4x32_10(c, make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
    return (float)(o.x >> 8) * (1.0f / 16777216.0f);
}

// ------------------------------------------------------- cached loads --
// 16-byte read-only load marked evict-first in L2: for a second read of data
// that is not read again, so that the lines still awaiting their second read
// stay.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint4 ldg_last_use(const uint4* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

// ------------------------------------------------------------- numerics --
// 2^x on the MUFU unit (flushes results below 2^-126 to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Weight of logit x in a row with max m at c = log2(e) / T: 2^(x*c - m*c).
// Every kernel forms m*c the same way so that weights agree bit for bit.
__device__ __forceinline__ float scaled_max(float m, float c) { return m * c; }
__device__ __forceinline__ float weight_of(float x, float c, float mc) { return ex2(fmaf(x, c, -mc)); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// Order-preserving 16-bit key of a bf16 bit pattern (larger key = larger
// value; NaNs sit outside [-inf, +inf]).  -0 maps one below +0.
__device__ __forceinline__ uint32_t okey16(uint32_t b) {
    return (b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u);
}
__device__ __forceinline__ uint32_t okey16_to_bits(uint32_t k) {
    return (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
}
__device__ __forceinline__ uint32_t okey32(float f) {
    const uint32_t b = __float_as_uint(f == 0.0f ? 0.0f : f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float okey32_to_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Round a float down to a bf16 value (towards -inf), as its bit pattern.
__device__ __forceinline__ uint32_t bf16_bits_round_down(float f) {
    uint32_t b = __float_as_uint(f);
    const uint32_t t = b >> 16;
    if ((b & 0xffffu) == 0u) return t;
    return (b & 0x80000000u) ? t + 1u : t;  // negative: more negative is larger magnitude
}

// ------------------------------------------------------------- barriers --
// Barrier over the kNT threads that work on a row.  A unit whose CTAs hold
// other warps beside them (a warp issuing bulk copies) defines
// SV_ROW_BARRIER_NAMED, so that these barriers count the kNT row threads
// only (named barrier 1); elsewhere they are the CTA barrier.
// Programmatic dependent launch: a kernel lets the next kernel on its
// stream be scheduled (grid_dep_trigger, called by every CTA), and a kernel
// so launched waits for the one before it to complete and its writes to be
// visible (grid_dep_wait; a no-op after an ordinary launch).
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void row_sync() {
#ifdef SV_ROW_BARRIER_NAMED
    asm volatile("bar.sync 1, %0;" ::"n"(kNT) : "memory");
#else
    __syncthreads();
#endif
}
// row_sync that also returns whether v was true in any row thread.
__device__ __forceinline__ bool row_sync_or(bool v) {
#ifdef SV_ROW_BARRIER_NAMED
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v), "n"(kNT)
                 : "memory");
    return r != 0;
#else
    return __syncthreads_or(v ? 1 : 0) != 0;
#endif
}

// ------------------------------------------------------- block reductions --
// Every block-wide operation below follows one pattern: per-warp partials
// are published, one barrier, warp 0 merges them in a fixed order and
// publishes the result, a second barrier, every thread reads the result.
// Partials and results live in different slots, so no trailing barrier is
// needed: the next operation's warp 0 writes a result only after that
// operation's first barrier, which every reader of the previous result has
// passed.
struct BlockScratch {
    float pf[kNW];        // per-warp float partials
    float pf2[kNW];       // second float partial (float-float low parts)
    float pf3[kNW];
    int pi[kNW];          // per-warp int partials
    int pi2[kNW];
    float rf[kNW + 2];    // results: floats (scans: per-warp prefixes + total)
    float rf2[kNW + 2];
    int ri[kNW + 2];      // results: ints
    float bcast_f[8];     // free-form broadcast slots (callers own the barriers)
    int bcast_i[8];
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------- float-float arithmetic --
// FP64 runs at a small fraction of the FP32 rate on this GPU, so sums that
// must carry more than 24 bits are kept as unevaluated pairs hi + lo of
// floats, combined with error-free transformations (Knuth's two-sum,
// Dekker's product through fma).
struct ff {
    float hi, lo;
};
__device__ __forceinline__ ff ff_from(float x) { return ff{x, 0.0f}; }
__device__ __forceinline__ ff ff_add(ff a, ff b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    const float e = (a.hi - (s - bb)) + (b.hi - bb);
    const float t = e + a.lo + b.lo;
    const float h = s + t;
    return ff{h, t - (h - s)};
}
__device__ __forceinline__ ff ff_add_f(ff a, float b) { return ff_add(a, ff{b, 0.0f}); }
__device__ __forceinline__ ff ff_neg(ff a) { return ff{-a.hi, -a.lo}; }
__device__ __forceinline__ ff ff_sub(ff a, ff b) { return ff_add(a, ff_neg(b)); }
__device__ __forceinline__ ff ff_scale(ff a, float f) { return ff{a.hi * f, a.lo * f}; }
// a * b exactly, as a pair
__device__ __forceinline__ ff ff_two_prod(float a, float b) {
    const float p = a * b;
    return ff{p, fmaf(a, b, -p)};
}
__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
    const ff p = ff_two_prod(a.hi, b);
    const float lo = fmaf(a.lo, b, p.lo);
    const float h = p.hi + lo;
    return ff{h, lo - (h - p.hi)};
}
__device__ __forceinline__ float ff_to_float(ff a) { return a.hi + a.lo; }
// a >= b, decided on the pair difference (its sign is the sign of hi, or of
// lo when hi is zero)
__device__ __forceinline__ bool ff_ge(ff a, ff b) {
    const ff d = ff_sub(a, b);
    return d.hi > 0.0f || (d.hi == 0.0f && d.lo >= 0.0f);
}
__device__ __forceinline__ bool ff_lt(ff a, ff b) { return !ff_ge(a, b); }
__device__ __forceinline__ ff ff_shfl_xor(ff v, int o) {
    return ff{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ ff ff_shfl_up(ff v, int o) {
    return ff{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ ff ff_shfl(ff v, int src) {
    return ff{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}
__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
    return v;
}
// Inclusive prefix over the lanes of a warp.
__device__ __forceinline__ ff warp_inclusive_scan_ff(ff x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const ff y = ff_shfl_up(x, o);
        if (lane >= o) x = ff_add(x, y);
    }
    return x;
}
__device__ __forceinline__ int warp_inclusive_scan_i(int x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// All kNT row threads must call these.
__device__ __forceinline__ float block_max(float v, BlockScratch& s) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_max(v);
    if (lane == 0) s.pf[w] = v;
    row_sync();
    if (w == 0) {
        float r = warp_max(lane < kNW ? s.pf[lane] : -INFINITY);
        if (lane == 0) s.rf[0] = r;
    }
    row_sync();
    return s.rf[0];
}
__device__ __forceinline__ int block_min_i(int v, BlockScratch& s) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_min_i(v);
    if (lane == 0) s.pi[w] = v;
    row_sync();
    if (w == 0) {
        const int r = warp_min_i(lane < kNW ? s.pi[lane] : 0x7fffffff);
        if (lane == 0) s.ri[0] = r;
    }
    row_sync();
    return s.ri[0];
}
__device__ __forceinline__ int block_sum_i(int v, BlockScratch& s) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum_i(v);
    if (lane == 0) s.pi[w] = v;
    row_sync();
    if (w == 0) {
        const int r = warp_sum_i(lane < kNW ? s.pi[lane] : 0);
        if (lane == 0) s.ri[0] = r;
    }
    row_sync();
    return s.ri[0];
}
__device__ __forceinline__ bool block_any(bool v, BlockScratch& s) {
    return row_sync_or(v);
}
// Deterministic block sum in float-float: fixed shuffle trees.
__device__ __forceinline__ ff block_sum_ff(ff v, BlockScratch& s) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum_ff(v);
    if (lane == 0) { s.pf[w] = v.hi; s.pf2[w] = v.lo; }
    row_sync();
    if (w == 0) {
        const ff r = warp_sum_ff(lane < kNW ? ff{s.pf[lane], s.pf2[lane]} : ff{0.0f, 0.0f});
        if (lane == 0) { s.rf[0] = r.hi; s.rf2[0] = r.lo; }
    }
    row_sync();
    return ff{s.rf[0], s.rf2[0]};
}
// Exclusive prefix in thread order (float-float); *total receives the sum.
__device__ __forceinline__ ff block_exclusive_scan_ff(ff v, BlockScratch& s, ff* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const ff x = warp_inclusive_scan_ff(v);
    if (lane == 31) { s.pf[w] = x.hi; s.pf2[w] = x.lo; }
    row_sync();
    if (w == 0) {
        const ff t = (lane < kNW) ? ff{s.pf[lane], s.pf2[lane]} : ff{0.0f, 0.0f};
        const ff incl = warp_inclusive_scan_ff(t);
        if (lane < kNW) {
            const ff ex = ff_sub(incl, t);
            s.rf[lane] = ex.hi;
            s.rf2[lane] = ex.lo;
        }
        if (lane == kNW - 1) { s.rf[kNW] = incl.hi; s.rf2[kNW] = incl.lo; }
    }
    row_sync();
    if (total) *total = ff{s.rf[kNW], s.rf2[kNW]};
    return ff_add(ff{s.rf[w], s.rf2[w]}, ff_sub(x, v));
}
__device__ __forceinline__ int block_exclusive_scan_i(int v, BlockScratch& s, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int x = warp_inclusive_scan_i(v);
    if (lane == 31) s.pi[w] = x;
    row_sync();
    if (w == 0) {
        const int t = (lane < kNW) ? s.pi[lane] : 0;
        const int incl = warp_inclusive_scan_i(t);
        if (lane < kNW) s.ri[lane] = incl - t;
        if (lane == kNW - 1) s.ri[kNW] = incl;
    }
    row_sync();
    if (total) *total = s.ri[kNW];
    return s.ri[w] + x - v;
}

// ------------------------------------------------------------ row access --
// Element type traits: VEC elements per 16-byte vector.
template <typename T> struct ElemT;
template <> struct ElemT<__nv_bfloat16> {
    static constexpr int VEC = 8;
    __device__ static __forceinline__ float load(const __nv_bfloat16* p) {
        return bf16_bits_to_float(*reinterpret_cast<const unsigned short*>(p));
    }
    __device__ static __forceinline__ void unpack(const uint4& v, float* o) {
        o[0] = bf16_lo(v.x); o[1] = bf16_hi(v.x); o[2] = bf16_lo(v.y); o[3] = bf16_hi(v.y);
        o[4] = bf16_lo(v.z); o[5] = bf16_hi(v.z); o[6] = bf16_lo(v.w); o[7] = bf16_hi(v.w);
    }
};
template <> struct ElemT<float> {
    static constexpr int VEC = 4;
    __device__ static __forceinline__ float load(const float* p) { return *p; }
    __device__ static __forceinline__ void unpack(const uint4& v, float* o) {
        o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y);
        o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
    }
};

// A row split into a scalar head (until the first 16-byte boundary), a body
// of 16-byte vectors and a scalar tail.  "Units" walk it in index order:
// unit 0 is the head (possibly empty), units 1..nvec the vectors, unit
// nvec+1 the tail (possibly empty).
template <typename T>
struct RowView {
    const T* row;
    int V, head, nvec, tail;
    __device__ __forceinline__ RowView(const T* r, int v) : row(r), V(v) {
        constexpr int VEC = ElemT<T>::VEC;
        const uintptr_t a = reinterpret_cast<uintptr_t>(r);
        int h = (int)(((16u - (unsigned)(a & 15u)) & 15u) / sizeof(T));
        if (h > V) h = V;
        head = h;
        nvec = (V - h) / VEC;
        tail = V - h - nvec * VEC;
    }
    __device__ __forceinline__ int units() const { return nvec + 2; }
    // Index range of unit u without loading it.
    __device__ __forceinline__ void unit_range(int u, int& idx0, int& cnt) const {
        constexpr int VEC = ElemT<T>::VEC;
        if (u >= 1 && u <= nvec) { idx0 = head + (u - 1) * VEC; cnt = VEC; return; }
        idx0 = (u == 0) ? 0 : head + nvec * VEC;
        cnt = (u == 0) ? head : tail;
    }
    __device__ __forceinline__ const uint4* vec() const {
        return reinterpret_cast<const uint4*>(row + head);
    }
    // Loads unit u into vals (missing slots get -inf); first element index
    // and number of valid slots are returned through idx0 and cnt.
    __device__ __forceinline__ void load_unit(int u, float* vals, int& idx0, int& cnt) const {
        constexpr int VEC = ElemT<T>::VEC;
        if (u >= 1 && u <= nvec) {
            const uint4 v = __ldg(vec() + (u - 1));
            ElemT<T>::unpack(v, vals);
            idx0 = head + (u - 1) * VEC;
            cnt = VEC;
            return;
        }
        const int start = (u == 0) ? 0 : head + nvec * VEC;
        const int n = (u == 0) ? head : tail;
        idx0 = start;
        cnt = n;
#pragma unroll
        for (int j = 0; j < VEC; ++j) vals[j] = (j < n) ? ElemT<T>::load(row + start + j) : -INFINITY;
    }
};

// Per-row statistics shared between kernels (32 bytes).
struct RowStat {
    float m;       // max logit of the row
    float inv_zn;  // 1 / sum of weights kept (nucleus mass when top-p is on)
    float x_tok;   // logit at the row's token of interest (NaN if none)
    int argmax;    // lowest index holding m
    float tau;     // top-p boundary logit; -inf when top-p is off
    int n_keep;    // boundary-valued tokens kept (the lowest-index ones)
    int c_tau;     // boundary-valued tokens in the row
    int flags;     // kRowInvalid | kRowTokMember | kRowRedo
};
constexpr int kRowInvalid = 1;
constexpr int kRowTokMember = 2;
// Set by the one-read top-p pass on a row it leaves to the two-pass route
// (the record's other fields are then undefined).
constexpr int kRowRedo = 4;

// Filtered probability of a logit x given the row's statistics; `rank_ok`
// tells whether a boundary-valued token is among the kept ones.
__device__ __forceinline__ float filtered_prob(float x, const RowStat& st, float c, bool rank_ok) {
    const bool member = (x > st.tau) || (x == st.tau && rank_ok);
    return member ? weight_of(x, c, scaled_max(st.m, c)) * st.inv_zn : 0.0f;
}

}  // namespace sv
