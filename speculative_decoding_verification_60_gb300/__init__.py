"""libspecverify: batched speculative-decoding verification on GB300.

Python face of the C ABI in include/specverify.h (see that header for the
exact semantics).  The work runs in hand-written CUDA kernels for sm_103a;
this package marshals torch tensors into the C calls.
"""

from ._binding import (  # noqa: F401
    CHILD_DETERMINISTIC,
    CHILD_IID,
    CHILD_WOR,
    DEVERR_LENGTH,
    DEVERR_NONFINITE,
    DEVERR_PARENT,
    DEVERR_TOKEN,
    EXPORTS,
    LIB_PATH,
    SPEC_OP_LINEAR,
    SPEC_OP_TREE,
    SamplingParams,
    SpecError,
    compact_accepted,
    load,
    sample_rows,
    status_string,
    verify_linear,
    verify_linear_compact,
    verify_tree,
    verify_tree_dynamic,
    workspace_size,
)
