"""The oracle's pins catch plausible mistakes in the oracle itself.

Each case plants one mistake in a scratch copy of the oracle's C source (a
swapped nibble order, a wrong exponent bias, a dropped normalisation, the
gate and up operands exchanged, a shifted rank weight, a reversed LRU rule,
...), builds that copy, and runs the pins (tests/test_oracle_pins.py) against
it in a subprocess with the copy first on the import path.  Every planted
mistake must fail at least one pin; the unmodified copy must pass them all.
CPU only: nothing here touches the library or a GPU.
"""
import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")

# name: (text in oracle.c, replacement, replace every occurrence)
MUTANTS = {
    "nibble_order": ("unsigned code = (i & 1) ? (byte >> 4) : (byte & 15u);",
                     "unsigned code = (i & 1) ? (byte & 15u) : (byte >> 4);", False),
    "e2m1_bias": ("mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);",
                  "mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 2);", False),
    "e4m3_bias": ("mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);",
                  "mag = ldexp(1.0 + (double)m / 8.0, (int)e - 8);", False),
    "scale_block_32": ("orc_e4m3(srow[i / 16])", "orc_e4m3(srow[i / 32])", False),
    "bf16_shift": ("(uint32_t)(bits & 0xFFFFu) << 16", "(uint32_t)(bits & 0xFFFFu) << 15", False),
    "scale_bytes": ("*Bs = weights / 16;", "*Bs = weights / 8;", False),
    "tie_higher_id": ("  if (l[a] < l[b]) return 0;\n  return a < b;",
                      "  if (l[a] < l[b]) return 0;\n  return a > b;", False),
    "no_renormalise": ("for (int j = 0; j < k; ++j) w[j] /= sum;", "(void)sum;", False),
    "swiglu_swapped": ("h[r] = g[r] / (1.0 + exp(-g[r])) * u[r];",
                       "h[r] = u[r] / (1.0 + exp(-u[r])) * g[r];", False),
    "sigmoid_not_silu": ("h[r] = g[r] / (1.0 + exp(-g[r])) * u[r];",
                         "h[r] = 1.0 / (1.0 + exp(-g[r])) * u[r];", False),
    "gate_reads_up_rows": ("orc_nvfp4_matvec(w_e, s_e, (double)gs3[0], I, H, x, g);",
                           "orc_nvfp4_matvec(w_e + I * (H / 2), s_e + I * (H / 16), "
                           "(double)gs3[0], I, H, x, g);", False),
    "down_of_u_not_h": ("(double)gs3[2], H, I, h, y);", "(double)gs3[2], H, I, u, y);", False),
    "down_gscale_of_up": ("(double)gs3[2], H, I, h, y);", "(double)gs3[1], H, I, h, y);", False),
    "rank_weight_shift": ("o[i] += wts[m * k + j] * y[i];",
                          "o[i] += wts[m * k + (j + 1) % k] * y[i];", False),
    "lru_largest_stamp": ("if (best < 0 || stamp[v] < stamp[best]) best = v;",
                          "if (best < 0 || stamp[v] > stamp[best]) best = v;", False),
    "lru_tie_high_slot": ("if (best < 0 || stamp[v] < stamp[best]) best = v;",
                          "if (best < 0 || stamp[v] <= stamp[best]) best = v;", False),
    "misses_descending": ("  for (int e = 0; e < E; ++e) {\n    if (!inU[e] || map[e] >= 0) continue;\n"
                          "    int best = -1;",
                          "  for (int e = E - 1; e >= 0; --e) {\n    if (!inU[e] || map[e] >= 0) continue;\n"
                          "    int best = -1;", False),
    "bypass_at_S": ("if (nU > S) {", "if (nU >= S) {", True),
    "gate_gscale_of_up": ("orc_nvfp4_matvec(w_e, s_e, (double)gs3[0], I, H, x, g);",
                          "orc_nvfp4_matvec(w_e, s_e, (double)gs3[1], I, H, x, g);", False),
    "softmax_over_all_E": ("for (int j = 0; j < k; ++j) w[j] /= sum;",
                           "{ double se = 0.0; for (int e2 = 0; e2 < E; ++e2) se += "
                           "isnan(logits[e2]) ? 0.0 : exp((double)logits[e2] - lmax); "
                           "for (int j = 0; j < k; ++j) w[j] /= se; (void)sum; }", False),
    "max_not_subtracted": ("w[j] = (l == lmax) ? 1.0 : exp(l - lmax);", "w[j] = exp(l);", False),
    "hits_not_restamped":("      used[v] = 1;\n      stamp[v] = t;", "      used[v] = 1;", False),
    "nan_ranks_first": ("    if (na && nb) return a < b;\n    return nb;",
                        "    if (na && nb) return a < b;\n    return na;", False),
    "list_victim_recent_end": ("    for (int pos = 0; pos < S; ++pos) {\n      if (!used[order[pos]]) {",
                               "    for (int pos = S - 1; pos >= 0; --pos) {\n"
                               "      if (!used[order[pos]]) {", False),
    "list_used_descending": ("  for (int v = 0; v < S; ++v)\n    if (used[v]) next[n++] = v;",
                             "  for (int v = S - 1; v >= 0; --v)\n    if (used[v]) next[n++] = v;",
                             False),
}


def _run_pins(tmp_root: str, name: str, mutant) -> tuple[int, str]:
    """Copy the oracle into tmp_root/name/oracle, plant `mutant` (None: none),
    run the pins against the copy; returns (exit code, pytest's output)."""
    base = os.path.join(tmp_root, name)
    dst = os.path.join(base, "oracle")
    os.makedirs(dst)
    for f in ("__init__.py", "oracle.c", "oracle.h"):
        shutil.copy(os.path.join(ORACLE, f), dst)
    if mutant is not None:
        old, new, every = mutant
        p = os.path.join(dst, "oracle.c")
        src = open(p).read()
        n = src.count(old)
        assert n >= 1 and (every or n == 1), f"{name}: {n} matches"
        open(p, "w").write(src.replace(old, new))
    # run from the copy's directory: `python -m` puts the working directory
    # first on the import path, ahead of the repository's own oracle
    env = dict(os.environ, PYTHONPATH=base + os.pathsep + ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests",
                        "test_oracle_pins.py"), "-x", "-q", "-rf", "-p", "no:cacheprovider"],
                       cwd=base, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout + r.stderr


def test_pins_catch_planted_oracle_mistakes(tmp_path):
    cases = [("control", None)] + sorted(MUTANTS.items())
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        results = dict(zip([c[0] for c in cases],
                           ex.map(lambda c: _run_pins(str(tmp_path), c[0], c[1]), cases)))
    rc, out = results.pop("control")
    assert rc == 0, "the unmodified copy must pass every pin:\n" + out[-2000:]
    survivors = []
    for name, (rc, out) in sorted(results.items()):
        caught = re.search(r"FAILED \S*test_oracle_pins\.py::(\w+)", out)
        print(f"{name:22s} -> {caught.group(1) if caught else 'NOT CAUGHT'}")
        if rc == 0 or caught is None:
            survivors.append((name, out[-1500:]))
    assert not survivors, "planted mistakes no pin caught: " + ", ".join(n for n, _ in survivors)
