// Entry points of libspecverify that launch nothing: status names and
// workspace sizes.
#include "../../include/specverify.h"
#include "linear_args.cuh"

extern "C" const char* spec_status_string(spec_status status) {
    switch (status) {
        case SPEC_OK: return "SPEC_OK";
        case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
        case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
        case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
        case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    }
    return "SPEC_ERR_UNKNOWN";
}

// Linear: one 32-byte RowStat per target and draft row, the requests'
// decisions and packed offsets, a counter.  Tree: no scratch.
extern "C" size_t spec_workspace_size(spec_op op, int B, int k_or_N, int V, spec_dtype dtype) {
    (void)dtype;
    if (B < 1 || k_or_N < 1 || V < 1) return 0;
    if (op == SPEC_OP_LINEAR) {
        return sv::linear_workspace(B, k_or_N).total;
    }
    if (op == SPEC_OP_TREE) return 256;
    return 0;
}
