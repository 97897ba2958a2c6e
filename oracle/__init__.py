"""Plain fp64 CPU oracle for batched speculative-decoding verification.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and bench.py's
``cpu_baseline`` leg are the only users.  The product library never imports,
links or runs anything here, and nothing here imports the product package.

The arithmetic lives in ``oracle.c`` (C, fp64, its own Philox4x32-10); this
module compiles it with gcc on first use and converts inputs to fp64.  Each
function cites the passage of "Accelerating Sonar through speculation" it
follows (see ``oracle.c`` for the full statement of the method and of the
readings taken where the page is silent).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERR_ARG = 1
ERR_NONFINITE = 2
ERR_TOKEN = 4
ERR_PARENT = 8
ERR_LENGTH = 16

PURPOSE_ACCEPT = 1
PURPOSE_RESIDUAL = 2
PURPOSE_BONUS = 3
PURPOSE_DRAFT = 4

CHILD_WOR = 0
CHILD_IID = 1
CHILD_DET = 2


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, IEEE fp64)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".{os.getpid()}.tmp"
            subprocess.check_call(
                ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
            )
            os.replace(tmp, _LIB)
    return _LIB


class _Trace(ctypes.Structure):
    _fields_ = [
        ("n_dec", ctypes.c_int),
        ("ratio", ctypes.c_double * 256),
        ("accepted", ctypes.c_int * 256),
        ("final_kind", ctypes.c_int),
        ("final_w", ctypes.POINTER(ctypes.c_double)),
    ]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, u64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        lib.orc_philox4x32_10.argtypes = [P, P, P]
        lib.orc_uniform.argtypes = [u64, i64, i64, ctypes.c_int, ctypes.c_int]
        lib.orc_uniform.restype = dbl
        lib.orc_argmax.argtypes = [P, ctypes.c_int]
        lib.orc_row_probs.argtypes = [P, ctypes.c_int, dbl, dbl, P, P]
        lib.orc_sample_inverse_cdf.argtypes = [P, ctypes.c_int, dbl, P]
        lib.orc_linear_request.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, dbl, dbl, P, P, dbl,
                                           P, P, P, P, P, ctypes.POINTER(_Trace)]
        lib.orc_verify_linear.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, dbl, dbl,
                                          u64, P, P, P, P, P, P, P]
        lib.orc_tree_depths.argtypes = [P, ctypes.c_int, P]
        lib.orc_tree_request.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int, dbl, dbl, ctypes.c_int,
                                         P, ctypes.c_int, P, P, P, P, P, P, ctypes.POINTER(_Trace)]
        lib.orc_verify_tree.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, dbl, dbl,
                                        u64, ctypes.c_int, P, P, P, P, P]
        lib.orc_compact.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_int,
                                    P, P, P, P]
        lib.orc_sample_rows.argtypes = [P, ctypes.c_int, ctypes.c_int, dbl, dbl, u64, P, P, P]
        lib.orc_draw_children.argtypes = [P, ctypes.c_int, dbl, dbl, ctypes.c_int, ctypes.c_int, u64,
                                          i64, i64, P]
        for name in ("orc_argmax", "orc_row_probs", "orc_sample_inverse_cdf", "orc_linear_request",
                     "orc_verify_linear", "orc_tree_depths", "orc_tree_request", "orc_verify_tree",
                     "orc_compact", "orc_sample_rows", "orc_draw_children"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def to_f64(x) -> np.ndarray:
    """Exact widening of bf16 / fp16 / fp32 / fp64 logits to fp64.

    bf16 arrives as a torch tensor or as raw uint16 bit patterns; each bf16
    value is the top half of an fp32, so the widening is exact."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype == torch.bfloat16:
                bits = x.contiguous().view(torch.int16).numpy().view(np.uint16)
                return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            return x.to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


# ---------------------------------------------------------------- RNG ----

def philox4x32_10(ctr, key) -> np.ndarray:
    """One Philox4x32-10 block (Salmon et al., SC'11)."""
    lib = _load()
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib.orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def uniform(seed: int, req: int, pos: int, purpose: int, rnd: int = 0) -> float:
    """u = (word0 >> 8) * 2^-24 of Philox(key = seed, counter = (req lo,
    pos lo, purpose | round << 8, req hi))."""
    return _load().orc_uniform(seed & (2**64 - 1), req, pos, purpose, rnd)


# ------------------------------------------------------- distributions ----

def argmax(x) -> int:
    x = np.ascontiguousarray(to_f64(x))
    return _load().orc_argmax(_p(x), x.shape[-1])


def row_probs(x, T: float, top_p: float = 1.0):
    """Filtered probabilities of one row (§Target-Draft: "full probability
    distributions"); returns (p, status, topp_margin)."""
    x = np.ascontiguousarray(to_f64(x))
    V = x.shape[-1]
    p = np.zeros(V, dtype=np.float64)
    m = np.zeros(1, dtype=np.float64)
    st = _load().orc_row_probs(_p(x), V, float(T), float(top_p), _p(p), _p(m))
    return p, st, float(m[0])


def sample_inverse_cdf(w, u: float):
    """Smallest v with C(v) > u * C(V-1); returns (token or -1, margin)."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    m = np.zeros(1, dtype=np.float64)
    t = _load().orc_sample_inverse_cdf(_p(w), w.shape[-1], float(u), _p(m))
    return t, float(m[0])


# ----------------------------------------------------------- linear ------

def linear_request(tgt, drf, d, T, top_p, u_acc, u_res, u_bon, want_trace=False):
    """One request of linear verification with explicit uniforms
    (§Speculative decoding, §Target-Draft).  Returns a dict."""
    tgt = np.ascontiguousarray(to_f64(tgt))
    k = tgt.shape[0] - 1
    V = tgt.shape[1]
    drf = None if drf is None else np.ascontiguousarray(to_f64(drf))
    d = np.ascontiguousarray(d, dtype=np.int32)
    u_acc = np.ascontiguousarray(u_acc, dtype=np.float64)
    u_res = np.ascontiguousarray(u_res, dtype=np.float64)
    a = np.zeros(1, dtype=np.int32)
    toks = np.zeros(k + 1, dtype=np.int32)
    accp = np.zeros(max(k, 1), dtype=np.float64)
    tokp = np.zeros(max(2 * k, 1), dtype=np.float64)
    mg = np.zeros(1, dtype=np.float64)
    tr = None
    fw = None
    if want_trace:
        tr = _Trace()
        fw = np.zeros(V, dtype=np.float64)
        tr.final_w = fw.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    st = _load().orc_linear_request(_p(tgt), _p(drf), _p(d), k, V, float(T), float(top_p), _p(u_acc),
                                    _p(u_res), float(u_bon), _p(a), _p(toks), _p(accp), _p(tokp), _p(mg),
                                    ctypes.byref(tr) if tr is not None else None)
    out = dict(status=st, a=int(a[0]), tokens=toks, accept_prob=accp[:k], tok_p=tokp[:2 * k].reshape(k, 2),
               margin=float(mg[0]))
    if tr is not None:
        out["trace"] = dict(ratio=[tr.ratio[i] for i in range(tr.n_dec)],
                            accepted=[tr.accepted[i] for i in range(tr.n_dec)],
                            final_kind=tr.final_kind, final_w=fw)
    return out


def verify_linear(target, draft, drafts, T, top_p, seed, req_ids=None, positions=None):
    """Batched linear verification with Philox uniforms; mirrors
    ``spec_verify_linear``.  target [B,k+1,V], draft [B,k,V] (or None when
    T == 0), drafts [B,k] int."""
    tgt = np.ascontiguousarray(to_f64(target))
    B, k1, V = tgt.shape
    k = k1 - 1
    drf = None if draft is None else np.ascontiguousarray(to_f64(draft))
    d = np.ascontiguousarray(np.asarray(drafts), dtype=np.int32).reshape(B, k)
    req = None if req_ids is None else np.ascontiguousarray(req_ids, dtype=np.int64)
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int64)
    acc = np.zeros(B, dtype=np.int32)
    toks = np.zeros((B, k + 1), dtype=np.int32)
    accp = np.zeros((B, max(k, 1)), dtype=np.float64)
    tokp = np.zeros((B, max(k, 1), 2), dtype=np.float64)
    hist = np.zeros(k + 1, dtype=np.int32)
    mg = np.zeros(B, dtype=np.float64)
    err = np.zeros(1, dtype=np.int32)
    _load().orc_verify_linear(_p(tgt), _p(drf), _p(d), B, k, V, _p(req), _p(pos), float(T), float(top_p),
                              seed & (2**64 - 1), _p(acc), _p(toks), _p(accp), _p(tokp), _p(hist), _p(mg),
                              _p(err))
    return dict(accepted_len=acc, out_tokens=toks, accept_prob=accp[:, :k], tok_p=tokp[:, :k],
                len_hist=hist, margin=mg, dev_error=int(err[0]))


# ------------------------------------------------------------- tree ------

def tree_depths(parent) -> tuple[int, np.ndarray]:
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    depth = np.zeros(len(parent), dtype=np.int32)
    dmax = _load().orc_tree_depths(_p(parent), len(parent), _p(depth))
    return dmax, depth


def tree_request(tgt, drf, tok, parent, T, top_p, mode, u_acc, u_res, u_bon, want_trace=False):
    """One request of tree verification with explicit uniforms (§EAGLE).
    u_acc is [Dmax+1, Kmax]; u_res, u_bon are [Dmax+1]."""
    tgt = np.ascontiguousarray(to_f64(tgt))
    N, V = tgt.shape
    drf = None if drf is None else np.ascontiguousarray(to_f64(drf))
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    u_acc = np.ascontiguousarray(u_acc, dtype=np.float64)
    Kmax = u_acc.shape[1]
    u_res = np.ascontiguousarray(u_res, dtype=np.float64)
    u_bon = np.ascontiguousarray(u_bon, dtype=np.float64)
    dmax, _ = tree_depths(parent)
    W = max(dmax, 0) + 1
    a = np.zeros(1, dtype=np.int32)
    path = np.zeros(W, dtype=np.int32)
    toks = np.zeros(W, dtype=np.int32)
    mg = np.zeros(1, dtype=np.float64)
    tr = None
    fw = None
    if want_trace:
        tr = _Trace()
        fw = np.zeros(V, dtype=np.float64)
        tr.final_w = fw.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    st = _load().orc_tree_request(_p(tgt), _p(drf), _p(tok), _p(parent), N, V, float(T), float(top_p), int(mode),
                                  _p(u_acc), Kmax, _p(u_res), _p(u_bon), _p(a), _p(path), _p(toks), _p(mg),
                                  ctypes.byref(tr) if tr is not None else None)
    out = dict(status=st, a=int(a[0]), path=path, tokens=toks, margin=float(mg[0]))
    if tr is not None:
        out["trace"] = dict(ratio=[tr.ratio[i] for i in range(tr.n_dec)],
                            accepted=[tr.accepted[i] for i in range(tr.n_dec)],
                            final_kind=tr.final_kind, final_w=fw)
    return out


def verify_tree(target, draft, node_tokens, parent, T, top_p, seed, mode=CHILD_WOR, req_ids=None, positions=None):
    """Batched tree verification with Philox uniforms; mirrors
    ``spec_verify_tree``."""
    tgt = np.ascontiguousarray(to_f64(target))
    B, N, V = tgt.shape
    drf = None if draft is None else np.ascontiguousarray(to_f64(draft))
    tok = np.ascontiguousarray(np.asarray(node_tokens), dtype=np.int32).reshape(B, N)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    dmax, _ = tree_depths(parent)
    W = max(dmax, 0) + 1
    req = None if req_ids is None else np.ascontiguousarray(req_ids, dtype=np.int64)
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int64)
    acc = np.zeros(B, dtype=np.int32)
    path = np.zeros((B, W), dtype=np.int32)
    toks = np.zeros((B, W), dtype=np.int32)
    mg = np.zeros(B, dtype=np.float64)
    err = np.zeros(1, dtype=np.int32)
    _load().orc_verify_tree(_p(tgt), _p(drf), _p(tok), _p(parent), B, N, V, _p(req), _p(pos), float(T),
                            float(top_p), seed & (2**64 - 1), int(mode), _p(acc), _p(path), _p(toks), _p(mg),
                            _p(err))
    return dict(accepted_len=acc, path_nodes=path, out_tokens=toks, margin=mg, dev_error=int(err[0]))


# ------------------------------------------------------- compaction ------

def compact(hidden_u16, accepted_len, out_tokens, path_nodes=None):
    """Gather of accepted hidden rows and shifted next tokens (§MTP,
    §MTP schedule for a single token).  hidden_u16 [B,T,H] uint16 bits."""
    h = np.ascontiguousarray(hidden_u16, dtype=np.uint16)
    B, T, H = h.shape
    acc = np.ascontiguousarray(accepted_len, dtype=np.int32)
    ot = np.ascontiguousarray(out_tokens, dtype=np.int32)
    W = ot.shape[1]
    pn = None if path_nodes is None else np.ascontiguousarray(path_nodes, dtype=np.int32)
    out_h = np.zeros((B * W, H), dtype=np.uint16)
    offs = np.zeros(B + 1, dtype=np.int32)
    nt = np.full(B * W, -1, dtype=np.int32)
    err = np.zeros(1, dtype=np.int32)
    _load().orc_compact(_p(h), B, T, H, _p(acc), _p(pn), _p(ot), W, _p(out_h), _p(offs), _p(nt), _p(err))
    n = int(offs[B])
    return dict(out_hidden=out_h[:n], offsets=offs, next_tokens=nt[:n], dev_error=int(err[0]))


# ------------------------------------------------------ draft draws ------

def sample_rows(x, T, top_p, seed, req, pos) -> np.ndarray:
    """One token per row from filter(softmax(x/T)) (draft-side draws for the
    harness: §Target-Draft, the draft model samples its tokens)."""
    x = np.ascontiguousarray(to_f64(x))
    R, V = x.shape
    req = np.ascontiguousarray(np.broadcast_to(np.asarray(req, dtype=np.int64), (R,)))
    pos = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.int64), (R,)))
    out = np.zeros(R, dtype=np.int32)
    _load().orc_sample_rows(_p(x), R, V, float(T), float(top_p), seed & (2**64 - 1), _p(req), _p(pos), _p(out))
    return out


def draw_children(x, T, top_p, K, mode, seed, req, pos) -> np.ndarray:
    """K child tokens of one tree node from filter(softmax(x/T)) per child
    mode (§EAGLE: Top-K candidates per node)."""
    x = np.ascontiguousarray(to_f64(x))
    out = np.zeros(K, dtype=np.int32)
    _load().orc_draw_children(_p(x), x.shape[-1], float(T), float(top_p), int(K), int(mode),
                              seed & (2**64 - 1), int(req), int(pos), _p(out))
    return out
