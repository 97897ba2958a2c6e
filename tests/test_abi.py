"""The C-ABI library builds, loads, and exports every function declared in
include/specverify.h; host-side argument checks reject bad calls before any
CUDA work (these run without a GPU)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_60_gb300 import build

    build.build()
    import speculative_decoding_verification_60_gb300 as svp

    return svp.load()


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(spec_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert set(declared) >= {"spec_verify_linear", "spec_verify_tree", "spec_compact_accepted",
                             "spec_workspace_size", "spec_status_string"}
    for name in declared:
        assert hasattr(lib, name), name
    import speculative_decoding_verification_60_gb300 as svp

    assert set(svp.EXPORTS) == set(declared)


def test_status_strings(lib):
    import speculative_decoding_verification_60_gb300 as svp

    assert svp.status_string(0) == "SPEC_OK"
    assert svp.status_string(3) == "SPEC_ERR_WORKSPACE"
    assert svp.status_string(99) == "SPEC_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    import speculative_decoding_verification_60_gb300 as svp

    assert svp.workspace_size(svp.SPEC_OP_LINEAR, 256, 8, 128256) >= 256 * 17 * 32
    assert svp.workspace_size(svp.SPEC_OP_LINEAR, 0, 8, 128256) == 0
    assert svp.workspace_size(svp.SPEC_OP_TREE, 32, 60, 128256) > 0


def test_host_argument_checks_return_status(lib):
    from speculative_decoding_verification_60_gb300 import SamplingParams

    sp = SamplingParams(1.0, 1.0, 0, 0)
    dummy = ctypes.c_void_p(16)
    # no params / null logits / bad sizes / bad temperature: rejected before any CUDA call
    assert lib.spec_verify_linear(dummy, dummy, 0, dummy, 1, 1, 8, None, None, None, dummy, dummy,
                                  None, None, None, None, dummy, 1 << 20, None) == 1
    assert lib.spec_verify_linear(None, dummy, 0, dummy, 1, 1, 8, None, None, ctypes.byref(sp), dummy, dummy,
                                  None, None, None, None, dummy, 1 << 20, None) == 1
    assert lib.spec_verify_linear(dummy, dummy, 0, dummy, 0, 1, 8, None, None, ctypes.byref(sp), dummy, dummy,
                                  None, None, None, None, dummy, 1 << 20, None) == 1
    bad = SamplingParams(-1.0, 1.0, 0, 0)
    assert lib.spec_verify_linear(dummy, dummy, 0, dummy, 1, 1, 8, None, None, ctypes.byref(bad), dummy, dummy,
                                  None, None, None, None, dummy, 1 << 20, None) == 1
    assert lib.spec_verify_linear(dummy, dummy, 0, dummy, 1, 65, 8, None, None, ctypes.byref(sp), dummy, dummy,
                                  None, None, None, None, dummy, 1 << 20, None) == 2
    assert lib.spec_verify_linear(dummy, dummy, 0, dummy, 1, 1, 8, None, None, ctypes.byref(sp), dummy, dummy,
                                  None, None, None, None, dummy, 8, None) == 3
    assert lib.spec_verify_tree(dummy, dummy, 0, dummy, dummy, 1, 3, 8, 3, None, None, ctypes.byref(sp),
                                dummy, dummy, dummy, None, dummy, 256, None) == 1
    # the per-request tree call: n_nodes required; the limits of the static call
    assert lib.spec_verify_tree_dynamic(dummy, dummy, 0, dummy, dummy, None, 1, 3, 8, 2, None, None,
                                        ctypes.byref(sp), dummy, dummy, dummy, None, dummy, 256, None) == 1
    assert lib.spec_verify_tree_dynamic(dummy, dummy, 0, dummy, dummy, dummy, 1, 3, 8, 3, None, None,
                                        ctypes.byref(sp), dummy, dummy, dummy, None, dummy, 256, None) == 1
    assert lib.spec_verify_tree_dynamic(dummy, dummy, 0, dummy, dummy, dummy, 1, 2000, 8, 2, None, None,
                                        ctypes.byref(sp), dummy, dummy, dummy, None, dummy, 256, None) == 2
    assert lib.spec_compact_accepted(None, 1, 1, 8, dummy, None, dummy, 1, dummy, dummy, dummy, None, None) == 1
    # the compacting call needs its hidden buffers; the split calls check like the one-call form
    assert lib.spec_verify_linear_compact(dummy, dummy, 0, dummy, 1, 1, 8, None, None, ctypes.byref(sp), None, 16,
                                          dummy, dummy, None, None, None, dummy, dummy, dummy, None, dummy, 1 << 20,
                                          None) == 1
    assert lib.spec_linear_stats_decide(dummy, dummy, 0, dummy, 1, 1, 8, None, None, ctypes.byref(sp), None,
                                        None, None, None, None, dummy, 1 << 20, None) == 1
    assert lib.spec_linear_draw(dummy, dummy, 0, dummy, 1, 1, 8, None, None, ctypes.byref(sp), None, 0, None,
                                None, None, None, dummy, 1 << 20, None) == 1
    assert lib.spec_linear_stats_decide(dummy, dummy, 0, dummy, 1, 65, 8, None, None, ctypes.byref(sp), dummy,
                                        None, None, None, None, dummy, 1 << 20, None) == 2


def test_sample_rows_host_checks(lib):
    """spec_sample_rows rejects bad calls before any CUDA call."""
    from speculative_decoding_verification_60_gb300 import SamplingParams

    sp = SamplingParams(0.7, 0.9, 0, 0)
    dummy = ctypes.c_void_p(16)
    call = lambda logits, dt, R, V, p, out: lib.spec_sample_rows(logits, dt, R, V, None, None, p, out, None, None)
    assert call(None, 0, 1, 8, ctypes.byref(sp), dummy) == 1  # no logits
    assert call(dummy, 0, 1, 8, None, dummy) == 1  # no params
    assert call(dummy, 0, 1, 8, ctypes.byref(sp), None) == 1  # no output
    assert call(dummy, 7, 1, 8, ctypes.byref(sp), dummy) == 1  # unknown dtype
    assert call(dummy, 0, 0, 8, ctypes.byref(sp), dummy) == 1  # R < 1
    assert call(dummy, 0, 1, 0, ctypes.byref(sp), dummy) == 1  # V < 1
    for T, p in ((-1.0, 0.9), (float("inf"), 0.9), (float("nan"), 0.9), (0.7, 0.0), (0.7, float("nan"))):
        bad = SamplingParams(T, p, 0, 0)
        assert call(dummy, 0, 1, 8, ctypes.byref(bad), dummy) == 1, (T, p)
    assert call(dummy, 0, 1, 524281, ctypes.byref(sp), dummy) == 2  # V above the limit


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import speculative_decoding_verification_60_gb300._binding as b

    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not found"):
        b.load()


def test_sample_rows_binding_checks(lib):
    """The Python binding refuses what the C call cannot take before calling it."""
    import torch

    import speculative_decoding_verification_60_gb300 as svp

    with pytest.raises(ValueError, match="CUDA"):
        svp.sample_rows(torch.zeros(2, 8, dtype=torch.bfloat16), 0.7, 0.9)  # host tensor
    with pytest.raises(TypeError, match="bfloat16 or float32"):
        svp.sample_rows(torch.zeros(2, 8, dtype=torch.float16), 0.7, 0.9)
    with pytest.raises(ValueError):
        svp.sample_rows(torch.zeros(2, 3, 8, dtype=torch.bfloat16), 0.7, 0.9)  # not [R, V]
