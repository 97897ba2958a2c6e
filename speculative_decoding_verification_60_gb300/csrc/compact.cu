// Compaction for the next draft step ("Accelerating Sonar through
// speculation", §MTP: token t_{i+1} is drawn from logits computed from
// hidden state H_i, so the token buffer sits one step left of the hidden
// states; §MTP schedule for a single token: a kernel inserts the next
// target tokens into their slots, with no host synchronisation).
// One CTA per request: its output offset is the sum of (a_b' + 1) over the
// requests before it; it then copies its a_b + 1 hidden rows with 16-byte
// vectors and writes the paired next tokens.
#include "../../include/specverify.h"
#include "common.cuh"
#include "launch.cuh"

namespace sv {

constexpr int kCompactNT = 256;

struct CompactArgs {
    const uint16_t* hidden;
    int B, T, H, W;
    const int32_t* acc;
    const int32_t* path;
    const int32_t* out_tokens;
    uint16_t* out_hidden;
    int32_t* offsets;
    int32_t* next_tokens;
    int32_t* dev_error;
    bool vec_ok;  // H*2 % 16 == 0 and both base pointers 16-byte aligned
};

__device__ __forceinline__ int rows_of(const CompactArgs& a, int b) {
    const int acc = a.acc[b];
    if (acc < 0 || acc >= a.W) return 0;
    for (int r = 0; r <= acc; ++r) {
        const int src = a.path ? a.path[(size_t)b * a.W + r] : r;
        if (src < 0 || src >= a.T) return 0;
    }
    return acc + 1;
}

__global__ void __launch_bounds__(kCompactNT) k_compact(CompactArgs a) {
    __shared__ int part[kCompactNT / 32];
    __shared__ int sh_off, sh_rows;
    const int b = blockIdx.x, tid = threadIdx.x;
    int mine = 0;
    for (int j = tid; j < b; j += kCompactNT) mine += rows_of(a, j);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
    if ((tid & 31) == 0) part[tid >> 5] = mine;
    __syncthreads();
    if (tid == 0) {
        int off = 0;
        for (int w = 0; w < kCompactNT / 32; ++w) off += part[w];
        const int rows = rows_of(a, b);
        sh_off = off;
        sh_rows = rows;
        a.offsets[b + 1] = off + rows;
        if (b == 0) a.offsets[0] = 0;
        if (rows == 0 && a.dev_error) atomicOr(a.dev_error, kDevErrLength);
    }
    __syncthreads();
    const int off = sh_off, rows = sh_rows;
    for (int r = 0; r < rows; ++r) {
        const int src = a.path ? a.path[(size_t)b * a.W + r] : r;
        const uint16_t* in = a.hidden + ((size_t)b * a.T + src) * a.H;
        uint16_t* out = a.out_hidden + (size_t)(off + r) * a.H;
        if (a.vec_ok) {
            const uint4* vi = reinterpret_cast<const uint4*>(in);
            uint4* vo = reinterpret_cast<uint4*>(out);
            for (int i = tid; i < a.H / 8; i += kCompactNT) vo[i] = __ldg(vi + i);
        } else {
            for (int i = tid; i < a.H; i += kCompactNT) out[i] = in[i];
        }
        if (tid == 0) a.next_tokens[off + r] = a.out_tokens[(size_t)b * a.W + r];
    }
}

}  // namespace sv

using namespace sv;

extern "C" spec_status spec_compact_accepted(const void* hidden, int B, int T, int H, const int32_t* accepted_len,
                                             const int32_t* path_nodes, const int32_t* out_tokens, int W,
                                             void* out_hidden, int32_t* offsets, int32_t* next_tokens,
                                             int32_t* dev_error, spec_stream_t stream) {
    DeviceGuard device_guard;  // the caller's current device is put back on return
    if (!hidden || !accepted_len || !out_tokens || !out_hidden || !offsets || !next_tokens)
        return SPEC_ERR_INVALID_ARG;
    if (B < 1 || T < 1 || H < 1 || W < 1) return SPEC_ERR_INVALID_ARG;
    if ((int64_t)B * W >= 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
    if (!select_device_of(hidden)) return SPEC_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dev_error && cudaMemsetAsync(dev_error, 0, sizeof(int32_t), st) != cudaSuccess) return SPEC_ERR_CUDA;
    CompactArgs a;
    a.hidden = static_cast<const uint16_t*>(hidden);
    a.B = B; a.T = T; a.H = H; a.W = W;
    a.acc = accepted_len;
    a.path = path_nodes;
    a.out_tokens = out_tokens;
    a.out_hidden = static_cast<uint16_t*>(out_hidden);
    a.offsets = offsets;
    a.next_tokens = next_tokens;
    a.dev_error = dev_error;
    a.vec_ok = ((size_t)H * 2) % 16 == 0 && (reinterpret_cast<uintptr_t>(hidden) & 15u) == 0 &&
               (reinterpret_cast<uintptr_t>(out_hidden) & 15u) == 0;
    k_compact<<<B, kCompactNT, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
