"""Planted mistakes in the oracle must be caught by its pins.

Each case copies oracle.c, plants one plausible mistake (a dropped term, a wrong sign, an
off-by-one index, a transposed operand), builds the copy with the oracle's own flags into a
temporary directory, and runs every pin against it in a child process (so a crash also counts
as caught). A mutant that passes every pin means the pins have a hole. CPU only.
"""
import subprocess
import sys
from pathlib import Path

import pytest

import oracle

ROOT = Path(__file__).resolve().parent.parent
SRC = (ROOT / "oracle" / "oracle.c").read_text()

MUTANTS = {
    "online_no_o_rescale": ("o[c] = o[c] * corr;", "o[c] = o[c];"),
    "online_no_l_rescale": ("l = l * corr;", "l = l;"),
    "online_corr_sign": ("0.0 : exp(m - m_new);", "0.0 : exp(m_new - m);"),
    "online_stale_max_in_p": ("double p = exp(score(q, k + j * d, d, scale) - m_new);",
                              "double p = exp(score(q, k + j * d, d, scale) - m);"),
    "two_pass_no_max_subtraction": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "two_pass_max_starts_at_zero": ("    double m = -INFINITY;\n    for (int64_t j = 0; j < n; ++j)\n        if (s[j] > m)",
                                    "    double m = 0.0;\n    for (int64_t j = 0; j < n; ++j)\n        if (s[j] > m)"),
    "two_pass_no_normalise": ("s[j] = s[j] / l;", "s[j] = s[j];"),
    "scale_dropped": ("return scale * acc;", "return acc;"),
    "key_row_index": ("s[j] = score(q, k + j * d, d, scale);", "s[j] = score(q, k + j, d, scale);"),
    "online_key_row_index": ("double s = score(q, k + j * d, d, scale);",
                             "double s = score(q, k + j * 2, d, scale);"),
    "value_index_transposed": ("o[c] += s[j] * v[j * d + c];", "o[c] += s[j] * v[c * n + j];"),
    "causal_sees_one_more": ("return (i + 1 < nk) ? i + 1 : nk;", "return (i + 2 < nk) ? i + 2 : nk;"),
    "causal_sees_one_less": ("return (i + 1 < nk) ? i + 1 : nk;", "return (i < nk) ? i : nk;"),
    "merge_drops_factor": ("*l_out = l1 * f1 + l2 * f2;", "*l_out = l1 + l2 * f2;"),
    "merge_o_sign": ("o[c] = o1[c] * f1 + o2[c] * f2;", "o[c] = o1[c] * f1 - o2[c] * f2;"),
    "lse_drops_max": ("if (lse) *lse = m + log(l);", "if (lse) *lse = log(l);"),
    "online_lse_drops_log": ("lse[r] = m + log(l);", "lse[r] = m + l;"),
    "rope_sign": ("row[i0] = x0 * c - x1 * sn;", "row[i0] = x0 * c + x1 * sn;"),
    "rope_half_offset": ("const int64_t i1 = (form == 0) ? i + h : 2 * i + 1;",
                         "const int64_t i1 = (form == 0) ? i + h - 1 : 2 * i + 1;"),
    "rope_in_place_overwrite": ("row[i1] = x1 * c + x0 * sn;", "row[i1] = x1 * c + row[i0] * sn;"),
    "bwd_delta_sign": ("const double ds = pij * (dp - delta);", "const double ds = pij * (dp + delta);"),
    "bwd_dq_no_scale": ("dqh[i * d + c] += scale * ds * kh[j * d + c];", "dqh[i * d + c] += ds * kh[j * d + c];"),
    "bwd_dv_uses_dq_row": ("dvh[j * d + c] += pij * doh[i * d + c];", "dvh[j * d + c] += pij * doh[j % nq * d + c];"),
    "bwd_dk_uses_k": ("dkh[j * d + c] += scale * ds * qh[i * d + c];", "dkh[j * d + c] += scale * ds * kh[j * d + c];"),
    "rows_wrong_slice": ("int64_t h = r / nq, i = r % nq;\n            int rc = two_pass_row(q + r * d, k + h * nk * d",
                         "int64_t h = r / nq, i = r % nq;\n            int rc = two_pass_row(q + r * d, k"),
}

CHILD = r"""
import sys
sys.path.insert(0, sys.argv[1])
import oracle
from tests import oracle_pins
failures = oracle_pins.run_all(oracle.Oracle(oracle.load(sys.argv[2])))
print("\n".join(failures[:3]))
sys.exit(1 if failures else 0)
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not unique in oracle.c"
    src = tmp_path / "oracle_mutant.c"
    src.write_text(SRC.replace(old, new))
    lib = oracle.build(src, tmp_path / "liboracle_mutant.so")
    r = subprocess.run([sys.executable, "-c", CHILD, str(ROOT), str(lib)], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout}\n{r.stderr}"
