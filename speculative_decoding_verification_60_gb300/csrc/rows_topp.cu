// Row statistics of bf16 rows under top-p with one read of each row.
//
// "Accelerating Sonar through speculation", §Target-Draft: acceptance
// compares the full probability distributions of draft and target, so each
// row needs its normaliser and, with top-p filtering (applied to p and q
// alike), its exact nucleus.
//
// Each CTA runs its rows on kNT row threads plus one copy warp.  The copy
// warp streams every row through a ring of shared-memory slots with bulk
// copies (cp.async.bulk, completion counted on one mbarrier per slot); the
// row threads read the slots, hand them back through a second mbarrier per
// slot, and never wait for DRAM directly.  Per row:
//   1. Window.  The row's first kSampleChunks copies are spread over it
//      (chunk order (i * nch) / ns first); their maximum m^ fixes the weight
//      reference and a window of kWinKeys = 2048 consecutive keys, the 16
//      binades [2^(e-11), 2^(e+5)) around m^ in [2^e, 2^(e+1)).
//   2. One pass over every slot: the sum of 2^((x - m^) c) (NaN or +inf
//      anywhere shows in it), the row maximum, and an exact count of every
//      key in the window (one predicated shared-memory reduction per
//      element, kCopies interleaved copies of the histogram).  Every key
//      weighs the same for all of its elements, so the counts give the mass
//      above any key in the window exactly.  The argmax is not taken: only
//      greedy rows read it.
//   3. The nucleus: the key counts walked down from the row maximum in
//      float-float (as the two-pass route does).
// A row this route cannot finish exactly (m^ not above zero, a maximum
// above the window, a boundary below it, a sum that is not finite, a wait
// that ran out) is marked kRowRedo and the two-pass kernel recomputes it.
//
// The same pass serves the draft-side sampler (SAMPLE): the rows are plain
// logit rows, and once a row's nucleus is known its token is drawn right
// away from the row (just streamed, so read from L2) while the copy warp
// already streams the next row; a row this route cannot finish gets the
// mark kSampleRedo in place of its token for the two-pass sampler.
#include "../../include/specverify.h"
#include "bulk.cuh"
#include "draw_bf16.cuh"
#include "launch.cuh"
#include "linear_args.cuh"
#include "rowstats.cuh"

namespace sv {

#ifndef SV_ONEPASS_CHUNK
#define SV_ONEPASS_CHUNK 12288
#endif
#ifndef SV_ONEPASS_SLOTS
#define SV_ONEPASS_SLOTS 3
#endif
#ifndef SV_ONEPASS_CTAS
#define SV_ONEPASS_CTAS 4
#endif
constexpr int kChunkBytes = SV_ONEPASS_CHUNK;        // bytes per bulk copy
constexpr int kChunkVecs = kChunkBytes / 16;         // 16-byte vectors per copy
constexpr int kVecsPerThread = kChunkVecs / kNT;
constexpr int kSlots = SV_ONEPASS_SLOTS;             // ring slots
constexpr int kSampleChunks = 2;                     // copies that give m^
constexpr int kWinKeys = 2048;                       // keys counted in the pass: 16 binades
constexpr int kWinBelow = 11;                        // binades of the window below m^'s
#ifndef SV_ONEPASS_COPIES
#define SV_ONEPASS_COPIES 1
#endif
constexpr int kCopies = SV_ONEPASS_COPIES;           // interleaved histogram copies
constexpr int kCopyShift = (kCopies == 4) ? 12 : (kCopies == 2 ? 13 : 14);  // bits >> kCopyShift = key bytes
constexpr int kOnePassThreads = kNT + 32;            // row threads + the copy warp
constexpr int kOnePassCtasPerSm = SV_ONEPASS_CTAS;
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // a wait longer than 2 s is an error
static_assert(kChunkVecs % kNT == 0, "whole vectors per row thread and copy");
static_assert((kWinKeys * kCopies) % (4 * kNT) == 0, "histogram cleared in whole uint4 per thread");
static_assert(kCopies == 1 || kCopies == 2 || kCopies == 4, "1, 2 or 4 copies (4 * kCopies bytes per key)");

struct OnePassSmem {
    uint4 ring[kSlots][kChunkVecs];
    uint32_t hist[kWinKeys * kCopies];  // count of key key_a + p in copy c at [p * kCopies + c]
    uint64_t full[kSlots];              // slot holds its copy (1 arrival + bytes)
    uint64_t empty[kSlots];             // slot read by every row warp (kNW arrivals)
    BlockScratch s;
    float xtok;
    int aborted;
};

__device__ __forceinline__ const __nv_bfloat16* onepass_row(const LinearArgs& a, int r, int& tok) {
    const int nt = a.B * (a.k + 1);
    if (r < nt) {
        const int b = r / (a.k + 1), i = r - b * (a.k + 1);
        tok = (i < a.k) ? a.drafts[(size_t)b * a.k + i] : -1;
        return static_cast<const __nv_bfloat16*>(a.tgt) + (size_t)r * a.V;
    }
    const int rr = r - nt;
    tok = a.drafts[rr];
    return static_cast<const __nv_bfloat16*>(a.drf) + (size_t)rr * a.V;
}

// A row's copy order: the ns sample chunks (i * nch) / ns first, then the
// others in increasing order.  f(s, ch) is called for positions s = 0, 1, ...
// (one division per sample chunk, none per chunk).
template <typename F>
__device__ __forceinline__ void for_each_chunk(int nch, int ns, F&& f) {
    for (int i = 0; i < ns; ++i) f(i, (i * nch) / ns);
    int s = ns;
    for (int i = 0; i < ns; ++i) {
        const int a = (i * nch) / ns + 1, b = (i + 1 < ns) ? ((i + 1) * nch) / ns : nch;
        for (int ch = a; ch < b; ++ch) f(s++, ch);
    }
}

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t w) { return *reinterpret_cast<__nv_bfloat162*>(&w); }
__device__ __forceinline__ __nv_bfloat162 vec_max(const uint4& q) {
    return __hmax2(__hmax2(as_bf162(q.x), as_bf162(q.y)), __hmax2(as_bf162(q.z), as_bf162(q.w)));
}

// Counts element xb (float bit pattern, bf16 bits << 16) at its key's
// position in the window, clamped: position 0 takes every element at or
// below the bottom key (negative ones too: as signed integers they sort
// below every positive pattern), position kWinKeys - 1 every element at or
// above the top key.  Positions 1 .. kWinKeys - 2 are exact key counts.  No
// predicate and no branch; hbk is the lane's copy base minus xb_a >> 12, so
// that the position's 16-byte slot is hbk + (clamped bits >> 12).
__device__ __forceinline__ void count_key(uint32_t xb, int lo, int hi, uint32_t hbk) {
    const uint32_t cb = (uint32_t)min(max((int)xb, lo), hi);
    asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(hbk + (cb >> kCopyShift)) : "memory");
}

static_assert(sizeof(BDrawScratch) <= sizeof(uint32_t) * kWinKeys * kCopies, "the draw's scratch fits in the histogram");

template <bool SAMPLE>
__global__ void __launch_bounds__(kOnePassThreads, kOnePassCtasPerSm) k_rows_topp_onepass(LinearArgs a) {
    extern __shared__ __align__(128) uint8_t onepass_raw[];
    OnePassSmem& sm = *reinterpret_cast<OnePassSmem*>(onepass_raw);
    grid_dep_wait();     // launched to overlap the launch before: wait for it before reading anything
    grid_dep_trigger();  // the finishing launch may be scheduled; it waits for this grid
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = a.B * (2 * a.k + 1);
    const int V = a.V;
    volatile int* aborted = &sm.aborted;
    if (tid == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kNW);
        }
        sm.aborted = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == kNW) {  // ---------------------------------------- copy warp
        if (lane != 0) return;
        uint32_t g = 0;  // copies issued by this CTA so far
        bool ok = true;
        for (int r = blockIdx.x; r < R && ok; r += gridDim.x) {
            int tok;
            const RowView<__nv_bfloat16> rv(onepass_row(a, r, tok), V);
            const int bytes = rv.nvec * 16;
            const int nch = (bytes + kChunkBytes - 1) / kChunkBytes;
            const char* base = reinterpret_cast<const char*>(rv.vec());
            for_each_chunk(nch, min(kSampleChunks, nch), [&](int, int ch) {
                if (!ok) return;
                const int slot = (int)(g % kSlots);
                if (g >= kSlots && !mbar_test(&sm.empty[slot], ((g / kSlots) - 1u) & 1u) &&
                    !mbar_wait(&sm.empty[slot], ((g / kSlots) - 1u) & 1u, kWaitLimitNs)) {
                    ok = false;
                    return;
                }
                if (*aborted) {
                    ok = false;
                    return;
                }
                const int nb = min(kChunkBytes, bytes - ch * kChunkBytes);
                mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)nb);
                bulk_load(sm.ring[slot], base + (size_t)ch * kChunkBytes, (uint32_t)nb, &sm.full[slot]);
                ++g;
            });
        }
        if (!ok) *aborted = 1;
        // every copy issued has landed before the CTA may end
        for (uint32_t i = g > (uint32_t)kSlots ? g - kSlots : 0u; i < g; ++i)
            mbar_wait(&sm.full[i % kSlots], (i / kSlots) & 1u, kWaitLimitNs);
        return;
    }

    // ------------------------------------------------------------ row threads
    const float c = a.c;
    const float top_p = a.top_p;
    const uint32_t hb = smem_addr(sm.hist) + 4u * (uint32_t)(lane & (kCopies - 1));
    uint32_t g0 = 0;  // copies of this CTA's earlier rows
    bool ab = false;  // this thread saw a wait run out
    auto wait_full = [&](uint64_t* bar, uint32_t par) {
        if (mbar_test(bar, par)) return;
        if (ab || *aborted) {
            ab = true;
            return;
        }
        if (!mbar_wait(bar, par, kWaitLimitNs)) {
            ab = true;
            *aborted = 1;
        }
    };

    for (int r = blockIdx.x; r < R; r += gridDim.x) {
        int tok;
        const __nv_bfloat16* row = onepass_row(a, r, tok);
        const RowView<__nv_bfloat16> rv(row, V);
        const int nch = (rv.nvec * 16 + kChunkBytes - 1) / kChunkBytes;
        const int ns = min(kSampleChunks, nch);
        if (tid == 0) sm.xtok = (tok >= 0 && tok < V) ? ElemT<__nv_bfloat16>::load(row + tok) : __int_as_float(0x7fffffff);
        const float xh = (tid < rv.head) ? ElemT<__nv_bfloat16>::load(row + tid) : -INFINITY;
        const float xt = (tid < rv.tail) ? ElemT<__nv_bfloat16>::load(row + rv.head + rv.nvec * 8 + tid) : -INFINITY;

        // 1. m^ over the sample chunks (copy positions 0 .. ns-1), the window
        __nv_bfloat162 smax = as_bf162(0xff80ff80u);
        for (int i = 0; i < ns; ++i) {
            const uint32_t g = g0 + i;
            wait_full(&sm.full[g % kSlots], (g / kSlots) & 1u);
            const int ch = (i * nch) / ns;
            const int nvc = min(kChunkVecs, rv.nvec - ch * kChunkVecs);
#pragma unroll
            for (int h = 0; h < kVecsPerThread; ++h) {
                const int v = tid + h * kNT;
                if (v < nvc) smax = __hmax2(smax, vec_max(sm.ring[g % kSlots][v]));
            }
        }
        for (int i = tid; i < kWinKeys * kCopies / 4; i += kNT)
            reinterpret_cast<uint4*>(sm.hist)[i] = make_uint4(0u, 0u, 0u, 0u);
        const float mh = block_max(fmaxf(__low2float(smax), __high2float(smax)), sm.s);  // also publishes the clear
        // window [2^(e-11), 2^(e+5)) for m^ in [2^e, 2^(e+1)): bf16 bits of 2^(e-11) are (e - 11 + 127) << 7
        const int be = (int)((__float_as_uint(mh) >> 23) & 0xffu) - kWinBelow;  // biased exponent of the bottom
        const bool est = mh > 0.0f && mh < INFINITY && be >= 1;
        const int key_a = 0x8000 + (be << 7);
        const uint32_t xba = (uint32_t)max(be, 1) << 23;                    // bits of the bottom key's value
        const int clo = (int)xba, chi = (int)(xba + ((uint32_t)(kWinKeys - 1) << 16));  // bottom and top keys' bits
        const uint32_t hbk = hb - (xba >> kCopyShift);

        // 2. the pass: copy positions 0 .. nch-1 (the sample chunks again first).
        // Each thread keeps one pair of partial sums per vector slot of a
        // chunk over the whole row (about V / (2 kNT kVecsPerThread) terms
        // each), merged in float-float at the end.
        const float rc = est ? mh * c : 0.0f;
        const float2 cc = make_float2(c, c), nrc = make_float2(-rc, -rc);
        float2 za[kVecsPerThread];
#pragma unroll
        for (int h = 0; h < kVecsPerThread; ++h) za[h] = make_float2(0.0f, 0.0f);
        auto take_vec = [&](const uint4& q, float2& acc) {
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t xl = w4[j] << 16, xu = w4[j] & 0xffff0000u;
                const float2 t = __ffma2_rn(make_float2(__uint_as_float(xl), __uint_as_float(xu)), cc, nrc);
                acc = __fadd2_rn(acc, make_float2(ex2(t.x), ex2(t.y)));
                count_key(xl, clo, chi, hbk);
                count_key(xu, clo, chi, hbk);
            }
        };
        const int nvc_last = rv.nvec - (nch - 1) * kChunkVecs;  // vectors of the last chunk (only it can be short)
        uint32_t slot = g0 % kSlots, par = (g0 / kSlots) & 1u;
        for_each_chunk(nch, ns, [&](int, int ch) {
            wait_full(&sm.full[slot], par);
            const uint4* sp = sm.ring[slot];
            if (ch != nch - 1 || nvc_last == kChunkVecs) {
                uint4 q[kVecsPerThread];
#pragma unroll
                for (int h = 0; h < kVecsPerThread; ++h) q[h] = sp[tid + h * kNT];
#pragma unroll
                for (int h = 0; h < kVecsPerThread; ++h) take_vec(q[h], za[h]);
            } else {
#pragma unroll
                for (int h = 0; h < kVecsPerThread; ++h)
                    if (tid + h * kNT < nvc_last) take_vec(sp[tid + h * kNT], za[h]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[slot]);
            if (++slot == kSlots) {
                slot = 0;
                par ^= 1u;
            }
        });
        g0 += (uint32_t)nch;
        ff zsum = ff{0.0f, 0.0f};
#pragma unroll
        for (int h = 0; h < kVecsPerThread; ++h) zsum = ff_add(zsum, ff_add(ff{za[h].x, 0.0f}, ff{za[h].y, 0.0f}));
        auto take_scalar = [&](float x) {
            zsum = ff_add_f(zsum, ex2(fmaf(x, c, -rc)));
            count_key(__float_as_uint(x), clo, chi, hbk);
        };
        if (tid < rv.head) take_scalar(xh);
        if (tid < rv.tail) take_scalar(xt);

        // 3. block results; NaN or +inf anywhere makes the sum NaN or +inf
        const bool abort_row = row_sync_or(ab || *aborted);
        const ff zr = block_sum_ff(zsum, sm.s);  // its barriers publish the counts
        if constexpr (kCopies > 1) {  // merge the copies into positions 0 .. kWinKeys-1
            uint32_t sum[kWinKeys / kNT];
#pragma unroll
            for (int i = 0; i < kWinKeys / kNT; ++i) {
                const int p = tid + i * kNT;
                uint32_t t = 0u;
#pragma unroll
                for (int cpy = 0; cpy < kCopies; ++cpy) t += sm.hist[p * kCopies + cpy];
                sum[i] = t;
            }
            row_sync();
#pragma unroll
            for (int i = 0; i < kWinKeys / kNT; ++i) sm.hist[tid + i * kNT] = sum[i];
            row_sync();
        }
        const float xtk = sm.xtok;

        RowStat st;
        st.m = mh;      // the weight reference: weights are 2^((x - m^) c)
        st.argmax = 0;  // read for greedy rows only
        st.tau = -INFINITY;
        st.n_keep = 0;
        st.c_tau = 0;
        st.inv_zn = 0.0f;
        st.x_tok = xtk;
        st.flags = 0;
        // leave to the two-pass route: no window, an element at or above the
        // window's top key, a sum that is not finite and positive (NaN, +inf,
        // or weights too large for fp32 relative to m^); a finite sum also
        // bounds every key's mass below
        bool redo = abort_row || !est || sm.hist[kWinKeys - 1] != 0u || !(zr.hi > 0.0f && zr.hi < INFINITY);
        if (redo) {
            // every thread has read the sentinel and xtok before the next row
            // clears the histogram and writes xtok (the walk's barriers do
            // this on the other branch), so all take the same branch
            row_sync();
        } else {
            const float mc = scaled_max(mh, c);
            const ff pZ = ff_mul_f(zr, top_p);
            // positions 1 .. kWinKeys-2 walked down from the top by the block
            // (empty positions cost a load)
            const int ktop = key_a + kWinKeys - 2;
            ff F_end;
            const WalkOut o = walk_keys<false, true>(sm.hist + 1, kWinKeys - 2, plain_map(ktop), c, mc, ff{0.0f, 0.0f},
                                                     pZ, &F_end, sm.s);
            if (o.found != 1) {
                redo = true;  // the boundary lies at or below the bottom key
            } else {
                st.tau = o.r.tau;
                st.n_keep = o.r.n_keep;
                st.c_tau = o.r.c_tau;
                bool member;
                if (xtk == st.tau && o.r.n_keep < o.r.c_tau) {
                    int before = 0;
                    row_find_nth_equal<__nv_bfloat16>(row, V, st.tau, -1, tok, &before, sm.s,
                                                      *reinterpret_cast<SampleScratch*>(sm.hist));
                    member = before < o.r.n_keep;
                } else {
                    member = xtk >= st.tau;
                }
                st.inv_zn = 1.0f / ff_to_float(o.r.mass);
                st.flags = member ? kRowTokMember : 0;
            }
        }
        if (redo) st.flags = kRowRedo;
        if constexpr (SAMPLE) {
            // the token at the DRAFT-purpose uniform, drawn from the row (in
            // L2 now); the histogram's space holds the draw's scratch
            int t = kSampleRedo;
            if (!redo) {
                const int64_t req = a.req ? a.req[r] : (int64_t)r;
                const int64_t pos = a.pos ? a.pos[r] : 0;
                const float u = uniform01(a.seed, req, pos, kPurposeDraft, 0);
                BRow P(reinterpret_cast<const uint16_t*>(row), st, c, true);
                t = draw_linear_bf16<false, true>(rv, P, P, c, u, sm.s, *reinterpret_cast<BDrawScratch*>(sm.hist));
                if (t < 0) t = kSampleRedo;
            }
            if (tid == 0) a.sample_out[r] = t;
        } else {
            if (tid == 0) {
                a.stats[r] = st;
                if (redo && a.dec) atomicAdd(a.done + 2, 1u);
            }
        }
        if (abort_row) {  // leave every remaining row to the two-pass kernel
            if (tid == 0) {
                if (a.dev_error) atomicOr(a.dev_error, kDevErrTimeout);
                for (int r2 = r + gridDim.x; r2 < R; r2 += gridDim.x) {
                    if constexpr (SAMPLE)
                        a.sample_out[r2] = kSampleRedo;
                    else
                        a.stats[r2].flags = kRowRedo;
                }
                if (a.dec) atomicAdd(a.done + 2, 1u);
            }
            break;
        }
        // the walk and the boundary search end on a barrier, so the next row
        // may clear the histogram and overwrite xtok right away
    }
}

spec_status launch_rows_topp_onepass(LinearArgs& a, cudaStream_t st) {
    const long long R = (long long)a.B * (2 * a.k + 1);
    const size_t smem = sizeof(OnePassSmem);
    int grid = 0;
    if (!launch_grid(k_rows_topp_onepass<false>, smem, R, &grid, kOnePassThreads)) return SPEC_ERR_CUDA;
    if (launch_dependent(k_rows_topp_onepass<false>, dim3(grid), dim3(kOnePassThreads), smem, st, a) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status launch_sample_onepass(LinearArgs& a, cudaStream_t st) {
    const size_t smem = sizeof(OnePassSmem);
    int grid = 0;
    if (!launch_grid(k_rows_topp_onepass<true>, smem, a.B, &grid, kOnePassThreads)) return SPEC_ERR_CUDA;
    k_rows_topp_onepass<true><<<grid, kOnePassThreads, smem, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace sv
