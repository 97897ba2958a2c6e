"""ctypes binding of libspecverify (argument marshalling only).

Every step of verification runs in the library's CUDA kernels; this module
only checks tensor shapes and dtypes, allocates output tensors with PyTorch
and passes raw device pointers and the current CUDA stream.  It fails loudly
when the library has not been built: there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspecverify.so")

SPEC_OK = 0
SPEC_BF16, SPEC_F32 = 0, 1
SPEC_OP_LINEAR, SPEC_OP_TREE = 0, 1
CHILD_WOR, CHILD_IID, CHILD_DETERMINISTIC = 0, 1, 2
DEVERR_TOKEN, DEVERR_NONFINITE, DEVERR_PARENT, DEVERR_LENGTH = 1, 2, 4, 8

# Every symbol declared in include/specverify.h.
EXPORTS = ("spec_workspace_size", "spec_verify_linear", "spec_verify_linear_compact", "spec_linear_stats_decide",
           "spec_linear_draw", "spec_verify_linear_noalloc", "spec_verify_tree", "spec_verify_tree_dynamic",
           "spec_compact_accepted",
           "spec_sample_rows", "spec_status_string")


class SamplingParams(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_p", ctypes.c_float), ("seed", ctypes.c_uint64),
                ("child_mode", ctypes.c_int32)]


class SpecError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} returned {status_string(status)} ({status})")
        self.status = status


_lib = None


def load() -> ctypes.CDLL:
    """Load libspecverify.so; raises when it is missing (build it with
    ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libspecverify.so not found at {LIB_PATH}: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.spec_workspace_size.argtypes = [I, I, I, I, I]
    lib.spec_workspace_size.restype = Z
    lib.spec_verify_linear.argtypes = [P, P, I, P, I, I, I, P, P, ctypes.POINTER(SamplingParams),
                                       P, P, P, P, P, P, P, Z, P]
    lib.spec_verify_linear.restype = I
    lib.spec_verify_linear_compact.argtypes = [P, P, I, P, I, I, I, P, P, ctypes.POINTER(SamplingParams), P, I,
                                               P, P, P, P, P, P, P, P, P, P, Z, P]
    lib.spec_verify_linear_compact.restype = I
    lib.spec_linear_stats_decide.argtypes = [P, P, I, P, I, I, I, P, P, ctypes.POINTER(SamplingParams),
                                             P, P, P, P, P, P, Z, P]
    lib.spec_linear_stats_decide.restype = I
    lib.spec_linear_draw.argtypes = [P, P, I, P, I, I, I, P, P, ctypes.POINTER(SamplingParams), P, I,
                                     P, P, P, P, P, Z, P]
    lib.spec_linear_draw.restype = I
    lib.spec_verify_linear_noalloc.argtypes = [P, P, I, P, I, I, I, P, P, ctypes.POINTER(SamplingParams),
                                               P, P, P, P, P, P, P]
    lib.spec_verify_linear_noalloc.restype = I
    lib.spec_verify_tree.argtypes = [P, P, I, P, P, I, I, I, I, P, P, ctypes.POINTER(SamplingParams),
                                     P, P, P, P, P, Z, P]
    lib.spec_verify_tree.restype = I
    lib.spec_verify_tree_dynamic.argtypes = [P, P, I, P, P, P, I, I, I, I, P, P, ctypes.POINTER(SamplingParams),
                                             P, P, P, P, P, Z, P]
    lib.spec_verify_tree_dynamic.restype = I
    lib.spec_compact_accepted.argtypes = [P, I, I, I, P, P, P, I, P, P, P, P, P]
    lib.spec_compact_accepted.restype = I
    lib.spec_sample_rows.argtypes = [P, I, I, I, P, P, ctypes.POINTER(SamplingParams), P, P, P]
    lib.spec_sample_rows.restype = I
    lib.spec_status_string.argtypes = [I]
    lib.spec_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().spec_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _check(t, name, dtype=None, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def workspace_size(op: int, B: int, k_or_N: int, V: int, dtype_code: int = SPEC_BF16) -> int:
    return int(load().spec_workspace_size(op, B, k_or_N, V, dtype_code))


def verify_linear(target, draft, draft_tokens, temperature: float, top_p: float = 1.0, seed: int = 0,
                  request_ids=None, positions=None, workspace=None, out=None, stream=None) -> dict:
    """``spec_verify_linear`` on torch tensors.

    target [B, k+1, V] and draft [B, k, V] (bf16 or fp32; draft may be None
    when temperature == 0), draft_tokens [B, k] int32, request_ids and
    positions [B] int64 or None.  Returns a dict of device tensors:
    accepted_len [B], out_tokens [B, k+1], accept_prob [B, k],
    token_probs [B, k, 2], len_hist [k+1], dev_error [1]."""
    lib = load()
    B, k1, V = target.shape
    k = k1 - 1
    dt = _dtype_code(target)
    _check(target, "target")
    _check(draft, "draft", target.dtype, (B, k, V))
    _check(draft_tokens, "draft_tokens", torch.int32, (B, k))
    _check(request_ids, "request_ids", torch.int64, (B,))
    _check(positions, "positions", torch.int64, (B,))
    dev = target.device
    if out is None:
        out = dict(
            accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
            out_tokens=torch.empty(B, k + 1, dtype=torch.int32, device=dev),
            accept_prob=torch.empty(B, k, dtype=torch.float32, device=dev),
            token_probs=torch.empty(B, k, 2, dtype=torch.float32, device=dev),
            len_hist=torch.empty(k + 1, dtype=torch.int32, device=dev),
            dev_error=torch.empty(1, dtype=torch.int32, device=dev),
        )
    need = workspace_size(SPEC_OP_LINEAR, B, k, V, dt)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    sp = SamplingParams(float(temperature), float(top_p), int(seed) & (2**64 - 1), 0)
    st = lib.spec_verify_linear(_ptr(target), _ptr(draft), dt, _ptr(draft_tokens), B, k, V, _ptr(request_ids),
                                _ptr(positions), ctypes.byref(sp), _ptr(out["accepted_len"]),
                                _ptr(out["out_tokens"]), _ptr(out.get("accept_prob")),
                                _ptr(out.get("token_probs")), _ptr(out.get("len_hist")),
                                _ptr(out.get("dev_error")), _ptr(workspace), workspace.numel(), _stream(stream))
    if st != SPEC_OK:
        raise SpecError("spec_verify_linear", st)
    return out


def verify_linear_compact(target, draft, draft_tokens, hidden, temperature: float, top_p: float = 1.0,
                          seed: int = 0, request_ids=None, positions=None, stream=None) -> dict:
    """``spec_verify_linear_compact`` on torch tensors: verify_linear plus
    hidden [B, k+1, H] bf16; the dict adds out_hidden [B*(k+1), H],
    offsets [B+1] and next_tokens [B*(k+1)] (rows past offsets[B] are not
    written)."""
    lib = load()
    B, k1, V = target.shape
    k = k1 - 1
    H = hidden.shape[-1]
    dt = _dtype_code(target)
    _check(target, "target")
    _check(draft, "draft", target.dtype, (B, k, V))
    _check(draft_tokens, "draft_tokens", torch.int32, (B, k))
    _check(hidden, "hidden", torch.bfloat16, (B, k + 1, H))
    _check(request_ids, "request_ids", torch.int64, (B,))
    _check(positions, "positions", torch.int64, (B,))
    dev = target.device
    out = dict(
        accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
        out_tokens=torch.empty(B, k + 1, dtype=torch.int32, device=dev),
        accept_prob=torch.empty(B, k, dtype=torch.float32, device=dev),
        token_probs=torch.empty(B, k, 2, dtype=torch.float32, device=dev),
        len_hist=torch.empty(k + 1, dtype=torch.int32, device=dev),
        out_hidden=torch.zeros(B * (k + 1), H, dtype=torch.bfloat16, device=dev),
        offsets=torch.empty(B + 1, dtype=torch.int32, device=dev),
        next_tokens=torch.full((B * (k + 1),), -1, dtype=torch.int32, device=dev),
        dev_error=torch.empty(1, dtype=torch.int32, device=dev),
    )
    need = workspace_size(SPEC_OP_LINEAR, B, k, V, dt)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    sp = SamplingParams(float(temperature), float(top_p), int(seed) & (2**64 - 1), 0)
    st = lib.spec_verify_linear_compact(_ptr(target), _ptr(draft), dt, _ptr(draft_tokens), B, k, V,
                                        _ptr(request_ids), _ptr(positions), ctypes.byref(sp), _ptr(hidden), H,
                                        _ptr(out["accepted_len"]), _ptr(out["out_tokens"]), _ptr(out["accept_prob"]),
                                        _ptr(out["token_probs"]), _ptr(out["len_hist"]), _ptr(out["out_hidden"]),
                                        _ptr(out["offsets"]), _ptr(out["next_tokens"]), _ptr(out["dev_error"]),
                                        _ptr(ws), ws.numel(), _stream(stream))
    if st != SPEC_OK:
        raise SpecError("spec_verify_linear_compact", st)
    return out


def verify_tree(target, draft, node_tokens, parent, max_depth: int, temperature: float, top_p: float = 1.0,
                seed: int = 0, child_mode: int = CHILD_WOR, request_ids=None, positions=None, stream=None) -> dict:
    """``spec_verify_tree`` on torch tensors: target/draft [B, N, V],
    node_tokens [B, N] int32, parent [N] int32 (device).  Returns
    accepted_len [B], path_nodes [B, W], out_tokens [B, W], dev_error [1]
    with W = max_depth + 1."""
    lib = load()
    B, N, V = target.shape
    dt = _dtype_code(target)
    _check(target, "target")
    _check(draft, "draft", target.dtype, (B, N, V))
    _check(node_tokens, "node_tokens", torch.int32, (B, N))
    _check(parent, "parent", torch.int32, (N,))
    _check(request_ids, "request_ids", torch.int64, (B,))
    _check(positions, "positions", torch.int64, (B,))
    dev = target.device
    W = int(max_depth) + 1
    out = dict(
        accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
        path_nodes=torch.empty(B, W, dtype=torch.int32, device=dev),
        out_tokens=torch.empty(B, W, dtype=torch.int32, device=dev),
        dev_error=torch.empty(1, dtype=torch.int32, device=dev),
    )
    need = workspace_size(SPEC_OP_TREE, B, N, V, dt)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    sp = SamplingParams(float(temperature), float(top_p), int(seed) & (2**64 - 1), int(child_mode))
    st = lib.spec_verify_tree(_ptr(target), _ptr(draft), dt, _ptr(node_tokens), _ptr(parent), B, N, V,
                              int(max_depth), _ptr(request_ids), _ptr(positions), ctypes.byref(sp),
                              _ptr(out["accepted_len"]), _ptr(out["path_nodes"]), _ptr(out["out_tokens"]),
                              _ptr(out["dev_error"]), _ptr(ws), ws.numel(), _stream(stream))
    if st != SPEC_OK:
        raise SpecError("spec_verify_tree", st)
    return out


def verify_tree_dynamic(target, draft, node_tokens, parent, n_nodes, max_depth: int, temperature: float,
                        top_p: float = 1.0, seed: int = 0, child_mode: int = CHILD_WOR, request_ids=None,
                        positions=None, stream=None) -> dict:
    """``spec_verify_tree_dynamic``: as verify_tree with a tree per request,
    parent [B, N] int32 and n_nodes [B] int32 (device)."""
    lib = load()
    B, N, V = target.shape
    dt = _dtype_code(target)
    _check(target, "target")
    _check(draft, "draft", target.dtype, (B, N, V))
    _check(node_tokens, "node_tokens", torch.int32, (B, N))
    _check(parent, "parent", torch.int32, (B, N))
    _check(n_nodes, "n_nodes", torch.int32, (B,))
    _check(request_ids, "request_ids", torch.int64, (B,))
    _check(positions, "positions", torch.int64, (B,))
    if n_nodes is None:
        raise ValueError("n_nodes is required")
    dev = target.device
    W = int(max_depth) + 1
    out = dict(
        accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
        path_nodes=torch.empty(B, W, dtype=torch.int32, device=dev),
        out_tokens=torch.empty(B, W, dtype=torch.int32, device=dev),
        dev_error=torch.empty(1, dtype=torch.int32, device=dev),
    )
    need = workspace_size(SPEC_OP_TREE, B, N, V, dt)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    sp = SamplingParams(float(temperature), float(top_p), int(seed) & (2**64 - 1), int(child_mode))
    st = lib.spec_verify_tree_dynamic(_ptr(target), _ptr(draft), dt, _ptr(node_tokens), _ptr(parent), _ptr(n_nodes),
                                      B, N, V, int(max_depth), _ptr(request_ids), _ptr(positions), ctypes.byref(sp),
                                      _ptr(out["accepted_len"]), _ptr(out["path_nodes"]), _ptr(out["out_tokens"]),
                                      _ptr(out["dev_error"]), _ptr(ws), ws.numel(), _stream(stream))
    if st != SPEC_OK:
        raise SpecError("spec_verify_tree_dynamic", st)
    return out


def compact_accepted(hidden, accepted_len, out_tokens, path_nodes=None, stream=None) -> dict:
    """``spec_compact_accepted``: hidden [B, T, H] (2-byte elements),
    accepted_len [B], out_tokens [B, W], path_nodes [B, W] or None.
    Returns out_hidden [B*W, H] (rows past offsets[B] untouched),
    offsets [B+1], next_tokens [B*W], dev_error [1]."""
    lib = load()
    B, T, H = hidden.shape
    W = out_tokens.shape[1]
    if hidden.element_size() != 2:
        raise TypeError("hidden must have 2-byte elements (bf16)")
    _check(hidden, "hidden")
    _check(accepted_len, "accepted_len", torch.int32, (B,))
    _check(out_tokens, "out_tokens", torch.int32, (B, W))
    _check(path_nodes, "path_nodes", torch.int32, (B, W))
    dev = hidden.device
    out = dict(
        out_hidden=torch.empty(B * W, H, dtype=hidden.dtype, device=dev),
        offsets=torch.empty(B + 1, dtype=torch.int32, device=dev),
        next_tokens=torch.empty(B * W, dtype=torch.int32, device=dev),
        dev_error=torch.empty(1, dtype=torch.int32, device=dev),
    )
    st = lib.spec_compact_accepted(_ptr(hidden), B, T, H, _ptr(accepted_len), _ptr(path_nodes), _ptr(out_tokens), W,
                                   _ptr(out["out_hidden"]), _ptr(out["offsets"]), _ptr(out["next_tokens"]),
                                   _ptr(out["dev_error"]), _stream(stream))
    if st != SPEC_OK:
        raise SpecError("spec_compact_accepted", st)
    return out


def sample_rows(logits, temperature: float, top_p: float = 1.0, seed: int = 0, request_ids=None, positions=None,
                out=None, stream=None) -> dict:
    """``spec_sample_rows`` on torch tensors: one token per row of logits
    [R, V] (bf16 or fp32) from filter(softmax(row / temperature)).
    request_ids and positions [R] int64 or None.  Returns a dict of device
    tensors: out_tokens [R] int32, dev_error [1] int32."""
    lib = load()
    R, V = logits.shape
    dt = _dtype_code(logits)
    _check(logits, "logits")
    _check(request_ids, "request_ids", torch.int64, (R,))
    _check(positions, "positions", torch.int64, (R,))
    dev = logits.device
    if out is None:
        out = dict(out_tokens=torch.empty(R, dtype=torch.int32, device=dev),
                   dev_error=torch.empty(1, dtype=torch.int32, device=dev))
    sp = SamplingParams(float(temperature), float(top_p), int(seed) & (2**64 - 1), 0)
    st = lib.spec_sample_rows(_ptr(logits), dt, R, V, _ptr(request_ids), _ptr(positions), ctypes.byref(sp),
                              _ptr(out["out_tokens"]), _ptr(out.get("dev_error")), _stream(stream))
    if st != SPEC_OK:
        raise SpecError("spec_sample_rows", st)
    return out
