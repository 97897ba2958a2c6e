// Tree verification ("Accelerating Sonar through speculation", §EAGLE: a
// static draft tree explored with the Top-K candidates of each node; the
// longest accepted root-to-leaf path is kept plus one target token).
// One CTA walks one request's tree: at each node it takes the statistics of
// the node's target (and draft) row, tests the children in index order with
// the residual updates of recursive rejection sampling, and descends into
// the first accepted child.  The tree is the same for every request (a
// fixed tree, EAGLE) or each request's own (a dynamically shaped tree,
// EAGLE-2 in the page's citation): parent [B, N] and a node count per
// request, the walk itself unchanged.
#include "../../include/specverify.h"
#include "launch.cuh"
#include "sample.cuh"

namespace sv {

constexpr int kMaxChildren = 64;
constexpr int kMaxNodes = 1024;

struct TreeArgs {
    const void* tgt;
    const void* drf;
    const int32_t* tok;
    const int32_t* parent;    // [N], or [B, N] with parent_stride = N
    int parent_stride;        // 0: one tree for every request
    const int32_t* n_nodes;   // [B] nodes of each request's tree, or NULL: N
    int B, N, V, W;  // N: nodes (rows) per request in the inputs; W = max_depth + 1
    const int64_t* req;
    const int64_t* pos;
    float top_p, c;
    uint64_t seed;
    int mode;  // spec_child_mode
    int32_t* acc_len;
    int32_t* path;
    int32_t* out_tokens;
    int32_t* dev_error;
};

// State of the rejected rounds at the current node.
struct Rounds {
    int n;                        // rounds rejected so far
    int tok[kMaxChildren];        // rejected token of each round
    float inv_norm[kMaxChildren]; // 1 / (IID/WOR: residual mass N_i;  DET: 1 - P_i(x_i)); 0 => P unchanged
    float qscale[kMaxChildren];   // WOR: 1 / (1 - Q_i(x_i)), 0 when that mass is 1
};

// P_j(v), Q_j(v) after the recorded rejected rounds, from the filtered
// probabilities p, q of token v.
__device__ __forceinline__ void chain(float& P, float& Q, int v, const Rounds& R, int mode) {
    for (int i = 0; i < R.n; ++i) {
        const float in = R.inv_norm[i];
        if (mode == SPEC_CHILD_DETERMINISTIC) {
            P = (v == R.tok[i]) ? 0.0f : (in > 0.0f ? P * in : P);
        } else {
            P = in > 0.0f ? fmaxf(0.0f, P - Q) * in : P;
            if (mode == SPEC_CHILD_WOR) Q = (v == R.tok[i]) ? 0.0f : Q * R.qscale[i];
        }
    }
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kNT, 1) k_tree(TreeArgs a) {
    extern __shared__ uint4 dyn_smem[];
    uint8_t* topsmem = reinterpret_cast<uint8_t*>(dyn_smem);
    __shared__ BlockScratch s;
    __shared__ SampleScratch ss;
    __shared__ Rounds R;
    __shared__ int ch[kMaxChildren];
    __shared__ int sh_m, sh_inval, sh_next;
    __shared__ int depth[kMaxNodes];
    constexpr int VEC = ElemT<T>::VEC;
    const int b = blockIdx.x, N = a.N, V = a.V, W = a.W, tid = threadIdx.x;
    const int64_t req = a.req ? a.req[b] : (int64_t)b;
    const int64_t pos = a.pos ? a.pos[b] : 0;
    const T* tgt = static_cast<const T*>(a.tgt) + (size_t)b * N * V;
    const T* drf = a.drf ? static_cast<const T*>(a.drf) + (size_t)b * N * V : nullptr;
    const int32_t* tok = a.tok + (size_t)b * N;
    const bool use_q = (MODE > 0) && a.mode != SPEC_CHILD_DETERMINISTIC;
    const int32_t* par = a.parent + (size_t)b * a.parent_stride;
    int Nt = N;  // nodes of this request's tree
    bool bad_count = false;
    if (a.n_nodes) {
        Nt = a.n_nodes[b];
        if (Nt < 1 || Nt > N) {
            bad_count = true;
            Nt = 1;
        }
    }

    // Validate the parent array (depth <= max_depth) and the node tokens.
    if (tid == 0) {
        int inval = bad_count ? kDevErrParent : 0;
        if (par[0] != -1) inval |= kDevErrParent;
        sh_inval = inval;
    }
    __syncthreads();
    {
        int inval = 0;
        for (int i = 1 + tid; i < Nt; i += kNT) {
            const int p = par[i];
            if (p < 0 || p >= i) inval |= kDevErrParent;
            if (tok[i] < 0 || tok[i] >= V) inval |= kDevErrToken;
        }
        if (inval) atomicOr(&sh_inval, inval);
    }
    __syncthreads();
    if (tid == 0 && !(sh_inval & kDevErrParent)) {
        // depth[i] = depth[parent[i]] + 1 (parent[i] < i was checked above)
        int dmax = 0;
        depth[0] = 0;
        for (int i = 1; i < Nt; ++i) {
            depth[i] = depth[par[i]] + 1;
            if (depth[i] > dmax) dmax = depth[i];
        }
        if (dmax > W - 1) sh_inval |= kDevErrParent;
    }
    __syncthreads();

    int n = 0, dep = 0, t = -1;
    for (int i = tid; i < W; i += kNT) {
        a.path[(size_t)b * W + i] = (i == 0) ? 0 : -1;
        a.out_tokens[(size_t)b * W + i] = -1;
    }
    bool inval = sh_inval != 0;
    while (!inval) {
        // children of n, in index order
        {
            int found = 0;
            for (int c0 = n + 1; c0 < Nt; c0 += kNT) {  // children have larger indices than their parent
                const int i = c0 + tid;
                const bool is_child = (i < Nt && par[i] == n);
                int tot;
                const int at = found + block_exclusive_scan_i(is_child ? 1 : 0, s, &tot);
                if (is_child && at < kMaxChildren) ch[at] = i;
                found += tot;
            }
            if (tid == 0) sh_m = found;
            __syncthreads();
        }
        const int m = sh_m;
        if (m > kMaxChildren) {  // every mode: a node with more children than the kernel tests
            if (tid == 0) atomicOr(&sh_inval, kDevErrParent);
            inval = true;
            break;
        }
        const T* prow = tgt + (size_t)n * V;
        const RowStat sp = row_stats<T, MODE>(prow, V, a.c, a.top_p, -1, topsmem, s, ss);
        if (sp.flags & kRowInvalid) {
            if (tid == 0) atomicOr(&sh_inval, kDevErrNonfinite);
            inval = true;
            break;
        }
        if (MODE == 0) {
            if (tid == 0) {
                int next = -1;
                for (int j = 0; j < m && j < kMaxChildren; ++j)
                    if (tok[ch[j]] == sp.argmax) { next = ch[j]; break; }
                sh_next = next;
            }
            __syncthreads();
            const int next = sh_next;
            __syncthreads();
            if (next < 0) { t = sp.argmax; break; }
            ++dep;
            if (tid == 0) {
                a.path[(size_t)b * W + dep] = next;
                a.out_tokens[(size_t)b * W + dep - 1] = tok[next];
            }
            n = next;
            continue;
        }
        const RowView<T> rv(prow, V);
        const FilteredRow<T> P(prow, sp, a.c, nucleus_cut<T>(prow, V, sp, s, ss));
        const float up = uniform01(a.seed, req, pos + dep + 1, m == 0 ? kPurposeBonus : kPurposeResidual, 0);
        if (m == 0) {
            auto wp = [&](int unit, float* w, int& i0, int& cnt) {
                rv.unit_range(unit, i0, cnt);
                P.probs(i0, cnt, w);
            };
            t = block_inverse_cdf<VEC>(rv.units(), up, wp, s, ss);
            break;
        }
        RowStat sq = sp;
        const T* qrow = drf ? drf + (size_t)n * V : prow;
        if (use_q) {
            sq = row_stats<T, MODE>(qrow, V, a.c, a.top_p, -1, topsmem, s, ss);
            if (sq.flags & kRowInvalid) {
                if (tid == 0) atomicOr(&sh_inval, kDevErrNonfinite);
                inval = true;
                break;
            }
        }
        const FilteredRow<T> Q(qrow, sq, a.c, use_q ? nucleus_cut<T>(qrow, V, sq, s, ss) : 0x7fffffff);
        if (tid == 0) R.n = 0;
        __syncthreads();
        int next = -1;
        for (int j = 0; j < m; ++j) {
            const int x = tok[ch[j]];
            if (tid == 0) {
                float Px = P.prob_at(x), Qx = use_q ? Q.prob_at(x) : 0.0f;
                chain(Px, Qx, x, R, a.mode);
                float ratio;
                if (a.mode == SPEC_CHILD_DETERMINISTIC) ratio = Px;
                else ratio = Qx > 0.0f ? Px / Qx : 0.0f;
                const float u = uniform01(a.seed, req, pos + dep + 1, kPurposeAccept, j);
                sh_next = (u < ratio) ? ch[j] : -1;
                R.tok[j] = x;
                if (a.mode == SPEC_CHILD_DETERMINISTIC) R.inv_norm[j] = (Px < 1.0f) ? 1.0f / (1.0f - Px) : 0.0f;
                R.qscale[j] = (Qx < 1.0f) ? 1.0f / (1.0f - Qx) : 0.0f;
            }
            __syncthreads();
            next = sh_next;
            __syncthreads();
            if (next >= 0) break;
            if (a.mode != SPEC_CHILD_DETERMINISTIC) {
                auto wres = [&](int unit, float* w, int& i0, int& cnt) {
                    rv.unit_range(unit, i0, cnt);
                    float p[VEC], q[VEC];
                    P.probs(i0, cnt, p);
                    Q.probs(i0, cnt, q);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        float Pv = p[e], Qv = q[e];
                        chain(Pv, Qv, i0 + e, R, a.mode);
                        w[e] = fmaxf(0.0f, Pv - Qv);
                    }
                };
                const ff Nj = block_weight_total<VEC>(rv.units(), wres, s);
                if (tid == 0) R.inv_norm[j] = Nj.hi > 0.0f ? 1.0f / ff_to_float(Nj) : 0.0f;
            }
            if (tid == 0) R.n = j + 1;
            __syncthreads();
        }
        if (next >= 0) {
            ++dep;
            if (tid == 0) {
                a.path[(size_t)b * W + dep] = next;
                a.out_tokens[(size_t)b * W + dep - 1] = tok[next];
            }
            n = next;
            continue;
        }
        auto wfin = [&](int unit, float* w, int& i0, int& cnt) {
            rv.unit_range(unit, i0, cnt);
            float q[VEC];
            P.probs(i0, cnt, w);
            if (use_q) Q.probs(i0, cnt, q);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float Qv = use_q ? q[e] : 0.0f;
                chain(w[e], Qv, i0 + e, R, a.mode);
            }
        };
        t = block_inverse_cdf<VEC>(rv.units(), up, wfin, s, ss);
        break;
    }
    __syncthreads();
    const int bad = sh_inval;
    if (bad) {
        t = row_argmax_finite<T>(tgt, V, s);
        dep = 0;
        for (int i = tid; i < W; i += kNT) {
            a.path[(size_t)b * W + i] = (i == 0) ? 0 : -1;
            a.out_tokens[(size_t)b * W + i] = (i == 0) ? t : -1;
        }
    }
    if (tid == 0) {
        a.acc_len[b] = dep;
        if (!bad) a.out_tokens[(size_t)b * W + dep] = t;
        if (bad && a.dev_error) atomicOr(a.dev_error, bad);
    }
}

template <typename T, int MODE>
static spec_status launch_tree(TreeArgs& a, cudaStream_t st) {
    const size_t dyn = (MODE == 2 && sizeof(T) == 2) ? (size_t)kTopSmemBytes : 0;
    auto* k = k_tree<T, MODE>;
    if (!set_dyn_smem(k, dyn, kNT)) return SPEC_ERR_CUDA;
    k<<<a.B, kNT, dyn, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace sv

using namespace sv;

static spec_status tree_entry(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                              const int32_t* node_tokens, const int32_t* parent, int parent_stride,
                              const int32_t* n_nodes, int B, int N, int V, int max_depth, const int64_t* request_ids,
                              const int64_t* positions, const spec_sampling_params* params, int32_t* accepted_len,
                              int32_t* path_nodes, int32_t* out_tokens, int32_t* dev_error, spec_stream_t stream) {
    if (!params || !target_logits || !node_tokens || !parent || !accepted_len || !path_nodes || !out_tokens)
        return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
    if (B < 1 || N < 1 || V < 1 || max_depth < 0 || max_depth >= N) return SPEC_ERR_INVALID_ARG;
    if (N > kMaxNodes) return SPEC_ERR_UNSUPPORTED;
    const float T = params->temperature, top_p = params->top_p;
    if (!(T >= 0.0f) || !(T < INFINITY) || !(top_p > 0.0f)) return SPEC_ERR_INVALID_ARG;
    const int cm = params->child_mode;
    if (cm != SPEC_CHILD_WOR && cm != SPEC_CHILD_IID && cm != SPEC_CHILD_DETERMINISTIC) return SPEC_ERR_INVALID_ARG;
    const bool greedy = (T == 0.0f);
    if (!greedy && cm != SPEC_CHILD_DETERMINISTIC && !draft_logits) return SPEC_ERR_INVALID_ARG;
    if ((int64_t)V > kMaxVocab) return SPEC_ERR_UNSUPPORTED;
    if (!select_device_of(target_logits)) return SPEC_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dev_error && cudaMemsetAsync(dev_error, 0, sizeof(int32_t), st) != cudaSuccess) return SPEC_ERR_CUDA;
    TreeArgs a;
    a.tgt = target_logits;
    a.drf = draft_logits;
    a.tok = node_tokens;
    a.parent = parent;
    a.parent_stride = parent_stride;
    a.n_nodes = n_nodes;
    a.B = B; a.N = N; a.V = V; a.W = max_depth + 1;
    a.req = request_ids;
    a.pos = positions;
    a.top_p = top_p;
    a.c = greedy ? 0.0f : (float)(1.4426950408889634 / (double)T);
    a.seed = params->seed;
    a.mode = cm;
    a.acc_len = accepted_len;
    a.path = path_nodes;
    a.out_tokens = out_tokens;
    a.dev_error = dev_error;
    const int mode = greedy ? 0 : (top_p < 1.0f ? 2 : 1);
    if (dtype == SPEC_BF16) {
        if (mode == 0) return launch_tree<__nv_bfloat16, 0>(a, st);
        if (mode == 1) return launch_tree<__nv_bfloat16, 1>(a, st);
        return launch_tree<__nv_bfloat16, 2>(a, st);
    }
    if (mode == 0) return launch_tree<float, 0>(a, st);
    if (mode == 1) return launch_tree<float, 1>(a, st);
    return launch_tree<float, 2>(a, st);
}

extern "C" spec_status spec_verify_tree(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                        const int32_t* node_tokens, const int32_t* parent, int B, int N, int V,
                                        int max_depth, const int64_t* request_ids, const int64_t* positions,
                                        const spec_sampling_params* params, int32_t* accepted_len,
                                        int32_t* path_nodes, int32_t* out_tokens, int32_t* dev_error,
                                        void* workspace, size_t workspace_bytes, spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    (void)workspace;
    (void)workspace_bytes;
    return tree_entry(target_logits, draft_logits, dtype, node_tokens, parent, 0, nullptr, B, N, V, max_depth,
                      request_ids, positions, params, accepted_len, path_nodes, out_tokens, dev_error, stream);
}

extern "C" spec_status spec_verify_tree_dynamic(const void* target_logits, const void* draft_logits,
                                                spec_dtype dtype, const int32_t* node_tokens, const int32_t* parent,
                                                const int32_t* n_nodes, int B, int N, int V, int max_depth,
                                                const int64_t* request_ids, const int64_t* positions,
                                                const spec_sampling_params* params, int32_t* accepted_len,
                                                int32_t* path_nodes, int32_t* out_tokens, int32_t* dev_error,
                                                void* workspace, size_t workspace_bytes, spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    (void)workspace;
    (void)workspace_bytes;
    if (!n_nodes) return SPEC_ERR_INVALID_ARG;
    return tree_entry(target_logits, draft_logits, dtype, node_tokens, parent, N, n_nodes, B, N, V, max_depth,
                      request_ids, positions, params, accepted_len, path_nodes, out_tokens, dev_error, stream);
}
