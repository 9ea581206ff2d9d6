"""The oracle's pins must catch plausible mistakes planted in the oracle.

Each case copies the oracle's C source into a temporary tree, plants one
mistake (a swapped index, a wrong sign, a dropped factor, a misplaced bit
field), rebuilds it there, and runs the pin suite against the copy in a
subprocess.  The suite must fail for every planted mistake.  Everything runs
on the CPU; nothing here touches the product library.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "candidate_order": ("{0, 1}, {0, 2}, {0, 3}, {1, 2}, {1, 3}, {2, 3}}",
                        "{0, 1}, {0, 2}, {1, 2}, {0, 3}, {1, 3}, {2, 3}}"),
    "philox_high_halves": ("uint32_t y0 = hi1 ^ x1 ^ k0;", "uint32_t y0 = hi0 ^ x1 ^ k0;"),
    "philox_word3": ("uint32_t y2 = hi0 ^ x3 ^ k1;", "uint32_t y2 = hi0 ^ x1 ^ k1;"),
    "philox_weyl": ("k1 += weyl1;", "k1 += weyl0;"),
    "counter_layout": (
        "uint32_t ctr[4] = {(uint32_t)group, (uint32_t)(group >> 32), step, tensor_id};",
        "uint32_t ctr[4] = {(uint32_t)group, step, (uint32_t)(group >> 32), tensor_id};"),
    "gumbel_sign": ("table[i] = (float)(-log(-log(u)));", "table[i] = (float)(log(-log(u)));"),
    "cell_half": ("uint32_t half = (words[c >> 1] >> (16 * (c & 1))) & 0xFFFFu;",
                  "uint32_t half = (words[c >> 1] >> (16 * (1 - (c & 1)))) & 0xFFFFu;"),
    "cell_bits": ("return (int)(half >> 2);", "return (int)(half & 0x3FFFu);"),
    "noise_sign": ("float s = a + gumbel[c];", "float s = a - gumbel[c];"),
    "softmax_shift": ("if (z[c] > m) m = z[c];", "if (z[c] < m) m = z[c];"),
    "backward_mean": ("r += p[c] * dp[c];", "r += dp[c];"),
    "backward_sign": ("dlogits[c] = dz_dlogit * p[c] * (dp[c] - r);",
                      "dlogits[c] = dz_dlogit * p[c] * (r - dp[c]);"),
    "regulariser_factor": ("+ 2.0 * (double)reg_coeff * x;", "+ (double)reg_coeff * x;"),
    "tie_rule": ("if (best < 0 || logits[c] > logits[best]) best = c;",
                 "if (best < 0 || logits[c] >= logits[best]) best = c;"),
    "meta_position": ("meta[r * (cols / 32) + k / 8] |= code << (4 * (k % 8));",
                      "meta[r * (cols / 32) + k / 8] |= code << (4 * (7 - k % 8));"),
    "meta_code": ("const uint32_t code = (uint32_t)(i | (j << 2));",
                  "const uint32_t code = (uint32_t)(j | (i << 2));"),
    "prior_abs": ("float b = fabsf(orc_bf16_to_float(w[ORC_PAIR[c][1]]));",
                  "float b = orc_bf16_to_float(w[ORC_PAIR[c][1]]);"),
    "bf16_ties": ("double r = nearbyint(q);", "double r = floor(q + 0.5);"),
    "row_sum": ("sq += x * x;", "sq += x;"),
    "dz_dlogit": ("const double dz_dlogit = exact ? (double)kappa / (double)tau",
                  "const double dz_dlogit = exact ? (double)kappa * (double)tau"),
    "storage_bytes": ("return rows * (cols / 2) * elem_bytes + rows * (cols / 4) / 2;",
                      "return rows * (cols / 2) * elem_bytes + rows * (cols / 4);"),
    "code_to_candidate": ("if ((uint32_t)(ORC_PAIR[c][0] | (ORC_PAIR[c][1] << 2)) == code) return c;",
                          "if ((uint32_t)(ORC_PAIR[c][1] | (ORC_PAIR[c][0] << 2)) == code) return c;"),
    "stats_l1": ("for (int j = 0; j < 4; ++j) l1 += orc_candidate_keeps(s, j) != orc_candidate_keeps(q, j);",
                 "for (int j = 0; j < 4; ++j) l1 += orc_candidate_keeps(s, j) != orc_candidate_keeps(s, j);"),
    "stats_maxprob_kappa": ("        float a = kappa * L[c];\n        y[c] = (double)a;",
                            "        float a = L[c];\n        y[c] = (double)a;"),
    "perm_top2": ("  return v[0] + v[1];\n}", "  return v[0] + v[2];\n}"),
    "perm_metric_abs": ("a[j] = fabs(orc_bf16_to_double(W[r * cols + perm[4 * g + j]]));",
                        "a[j] = orc_bf16_to_double(W[r * cols + perm[4 * g + j]]);"),
    "perm_shift_bits": ("return 31 - lr - orc_floor_log2(mx);", "return 32 - lr - orc_floor_log2(mx);"),
    "perm_fixed_round": ("return (uint32_t)floor(ldexp(", "return (uint32_t)nearbyint(ldexp("),
    "perm_tie_rule": ("        if (g > best) {", "        if (g >= best && g > 0) {"),
    "perm_gain_sign": ("  return after - before;", "  return before - after;"),
    "decompress_positions": ("const int i = (int)(code & 3u), j = (int)(code >> 2);",
                             "const int j = (int)(code & 3u), i = (int)(code >> 2);"),
    "perm_swap_restore": ("  perm[b] = perm[a];\n  perm[a] = t;\n  return after",
                          "  perm[a] = t;\n  return after"),
}


def _run_mutant(tmp_root, name, old, new):
    src = open(os.path.join(ROOT, "oracle", "maskllm_oracle.c")).read()
    assert src.count(old) == 1, name
    d = os.path.join(tmp_root, name)
    os.makedirs(os.path.join(d, "oracle"))
    with open(os.path.join(d, "oracle", "maskllm_oracle.c"), "w") as f:
        f.write(src.replace(old, new))
    for fn in ("__init__.py", "_build.py"):
        shutil.copy(os.path.join(ROOT, "oracle", fn), os.path.join(d, "oracle", fn))
    shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(d, "tests"),
                    ignore=shutil.ignore_patterns("__pycache__", "test_oracle_mutations.py"))
    pkg = "semi_structured_sparsity_gb300"
    os.makedirs(os.path.join(d, pkg))
    for fn in ("__init__.py", "workloads.py"):
        shutil.copy(os.path.join(ROOT, pkg, fn), os.path.join(d, pkg, fn))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py", "tests/test_oracle_perm_pins.py",
                        "tests/test_oracle_spmm_pins.py"], cwd=d, capture_output=True, text=True,
                       timeout=600)
    return name, r.returncode, (r.stdout.strip().splitlines() or [""])[-1]


def test_every_planted_mistake_is_caught(tmp_path):
    pytest.importorskip("torch")
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = [ex.submit(_run_mutant, str(tmp_path), n, a, b) for n, (a, b) in MUTATIONS.items()]
        results = [f.result() for f in futs]
    missed = [(n, tail) for n, rc, tail in results if rc == 0]
    assert not missed, missed
