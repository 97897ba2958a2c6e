"""The pins must be able to fail: plant plausible mistakes in a scratch copy
of the oracle (on the CPU) and check that the exact enumeration rejects each
one."""

import importlib
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTATIONS = {
    "residual-sign": ("double r = Pa[v] - Qa[v]; w[v]", "double r = Qa[v] - Pa[v]; w[v]", "linear", 1.0),
    "ratio-inverted": ("ratio[i] = q > 0.0 ? p / q : 0.0;", "ratio[i] = p > 0.0 ? q / p : 0.0;", "linear", 1.0),
    "accept-le": ("int acc = u_acc[a] < ratio[a];", "int acc = u_acc[a] < 0.5 * (1.0 + ratio[a]);", "linear", 1.0),
    "bonus-from-draft": ("memcpy(w, Pa, sizeof(double) * (size_t)V);\n                t = orc_sample_inverse_cdf(w, V, u_bon, &sm);",
                         "memcpy(w, Q, sizeof(double) * (size_t)V);\n                t = orc_sample_inverse_cdf(w, V, u_bon, &sm);",
                         "linear", 1.0),
    "top-p-boundary": ("if (before < top_p) {", "if (before <= top_p + 0.05) {", "linear", 0.8),
    "wor-no-q-update": ("if (mode == ORC_CHILD_WOR) {", "if (0) {", "tree", 1.0),
    "det-no-removal": ("P[x] = 0.0;\n                for (int v = 0; v < V; ++v) s += P[v];",
                       "for (int v = 0; v < V; ++v) s += P[v];", "tree-det", 1.0),
}

SCRIPT = """
import sys
sys.path.insert(0, {scratch!r}); sys.path.insert(1, {tests!r})
import exact_enum as E, oracle
kind, top_p = {kind!r}, {top_p!r}
try:
    if kind == "linear":
        w = E.ToyWorld(4, 2, seed=42, T=1.0, top_p=top_p)
        print(E.max_abs_diff(E.linear_emitted_distribution(w, 2), w.target_joint(3)))
    else:
        mode = oracle.CHILD_DET if kind == "tree-det" else oracle.CHILD_WOR
        w = E.ToyWorld(3, 2, seed=7, T=1.0, top_p=1.0)
        print(E.max_abs_diff(E.tree_emitted_distribution(w, [-1, 0, 0, 1, 1, 2, 2], mode), w.target_joint(3)))
except E.ThresholdMismatch:
    print(1.0)
"""


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    before, after, kind, top_p = MUTATIONS[name]
    scratch = tmp_path / "scratch"
    (scratch / "oracle").mkdir(parents=True)
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert before in src, name
    (scratch / "oracle" / "oracle.c").write_text(src.replace(before, after, 1))
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), scratch / "oracle" / "__init__.py")
    code = SCRIPT.format(scratch=str(scratch), tests=HERE, kind=kind, top_p=top_p)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    assert float(res.stdout.strip().splitlines()[-1]) > 1e-6, name
