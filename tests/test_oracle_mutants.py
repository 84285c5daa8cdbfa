"""Mutation check of the oracle's pins (no GPU).

Each case plants one plausible mistake in a copy of the oracle's C source (a
flipped comparison, a dropped term, a wrong index, a transposed operand),
compiles the copy into a temporary directory and runs the pins against it.
At least one pin must fail; otherwise the pins would not notice that mistake
in the real oracle.
"""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sel_oracle.c")

# (name, [(original text, planted text), ...]); each original occurs once.
MUTANTS = [
    ("argmax ties keep the higher index",
     [("if ((double)x[i] > (double)x[best])", "if ((double)x[i] >= (double)x[best])")]),
    ("finite check dropped",
     [("if (!isfinite(x[i]))\n            return 0;", "if (0)\n            return 0;")]),
    ("sort unstable on ties",
     [("if (key[src[b]] > key[src[a]])", "if (key[src[b]] >= key[src[a]])")]),
    ("sort ascending",
     [("if (key[src[b]] > key[src[a]])", "if (key[src[b]] < key[src[a]])")]),
    ("top-k output shifted by one",
     [("oi[j] = ids[j];", "oi[j] = ids[j > 0 ? j - 1 : 0];")]),
    ("temperature dropped in sampling",
     [("z[i] = (double)x[i] / T;", "z[i] = (double)x[i];")]),
    ("top_k ignored",
     [("uint32_t nc = (top_k == 0 || top_k > V) ? V : top_k;", "uint32_t nc = V;")]),
    ("top-p drops the crossing token",
     [("ns = j + 1;\n                break;", "ns = j > 0 ? j : 1;\n                break;")]),
    ("min-p compares absolute probability",
     [("double ratio = (wf[j] / Sf) / pmax;", "double ratio = (wf[j] / Sf);")]),
    ("probability not renormalised after filtering",
     [("        id = order[pick];\n        *prob = wd[pick] / Sd;", "        id = order[pick];\n        *prob = wd[pick] / Sf;")]),
    ("full-row draw in the candidates' order instead of ascending id",
     [("    if (top_k == 0) {\n        /* survivors by ascending id", "    if (0) {\n        /* survivors by ascending id")]),
    ("full-row draw maps u to the neighbouring id",
     [("        id = (uint32_t)(by_id[pick] >> 32);", "        id = (uint32_t)(by_id[pick + 1 < ns ? pick + 1 : pick] >> 32);")]),
    ("inverse CDF picks the next index",
     [("if (pick == ORC_INVALID && u < C)\n            pick = i;",
       "if (pick == ORC_INVALID && u < C)\n            pick = i + 1 < n ? i + 1 : i;")]),
    ("uniform range unchecked",
     [("return u >= 0.0f && u < 1.0f;", "return 1;")]),
    ("accept test compares against q",
     [("if (lhs <= pt)", "if (lhs <= qt)")]),
    ("accept test with p and q transposed",
     [("double lhs = (double)u_acc[n] * qt;", "double lhs = (double)u_acc[n] * pt;"),
      ("if (lhs <= pt)", "if (lhs <= qt)")]),
    ("residual sign flipped",
     [("double d = p[i] - q[i];", "double d = q[i] - p[i];")]),
    ("rejection resamples from p instead of the residual",
     [("if (!(total > 0.0))", "if (1)")]),
    ("bonus drawn from the wrong target row",
     [("softmax_row(target + (size_t)K * V, V, T, p);",
       "softmax_row(target + (size_t)(K - 1) * V, V, T, p);")]),
    ("temperature dropped in acceptance softmax",
     [("p[i] = exp((double)x[i] / T - m);", "p[i] = exp((double)x[i] - m);")]),
    ("argmax rule emits the draft on a mismatch",
     [("emitted[n] = a;", "emitted[n] = n < K ? tokens[n] : a;")]),
    ("argmax rule used for every temperature",
     [("if (T == 0.0)\n        mode = 1;", "mode = 1;")]),
    ("EOG set shifted by one id",
     [("if (excluded[e] == i)", "if (excluded[e] == i + 1)")]),
    ("EOG ties keep the higher index",
     [("if (best == ORC_INVALID || (double)x[i] > (double)x[best])",
       "if (best == ORC_INVALID || (double)x[i] >= (double)x[best])")]),
    ("EOG latch dropped",
     [("!row_is_finite(x, V))\n        return ORC_INVALID;\n    uint32_t best = ORC_INVALID;",
       "0)\n        return ORC_INVALID;\n    uint32_t best = ORC_INVALID;")]),
    ("sampler-match accepts a mismatch",
     [("if (n == K || tokens[n] != drawn)", "if (n == K || tokens[n] == drawn)")]),
    ("sampler-match always samples the first row",
     [("drawn = sample_row(target + (size_t)n * V, V, T,", "drawn = sample_row(target, V, T,")]),
    ("sampler-match ignores bad uniforms",
     [("!uniform_is_valid(u[j]))", "0)")]),
    ("diagnostics take the max for the min",
     [("a += p[i] < q[i] ? p[i] : q[i];", "a += p[i] > q[i] ? p[i] : q[i];")]),
    ("diagnostics square p",
     [("b += p[i] * q[i];", "b += p[i] * p[i];")]),
    ("diagnostics ignore the temperature",
     [("            softmax_row(t, V, T, p);\n            softmax_row(d, V, T, q);",
       "            softmax_row(t, V, 1.0, p);\n            softmax_row(d, V, 1.0, q);")]),
    ("top-n-sigma uses the variance",
     [("double sigma = sqrt(var / (double)V);", "double sigma = var / (double)V;")]),
    ("top-n-sigma measured from the mean",
     [("double thr = (double)x[order[0]] - top_n_sigma * sigma;", "double thr = mean - top_n_sigma * sigma;")]),
    ("typical order reversed",
     [("neg[j] = -score[j];", "neg[j] = score[j];")]),
    ("typical keeps past the crossing",
     [("if (cum >= typical_p) {", "if (cum > typical_p + 0.2) {")]),
    ("typical set not renormalised",
     [("        Sf = S2;\n", "        Sf = Sf;\n")]),
    ("CDF margin measured to the previous step",
     [("double d = fabs(u - c / W);", "double d = fabs(u - (c - w[i]) / W);")]),
    ("CDF margin counts the final step",
     [("if (last_pos != ORC_INVALID && i >= last_pos)", "if (last_pos != ORC_INVALID && i > last_pos)")]),
    ("CDF margin counts steps without mass",
     [("if (w[i] > 0.0) {", "if (1) {")]),
    ("accept margin not scaled by max(p, q)",
     [("double d = fabs(lhs - pt) / scale;", "double d = fabs(lhs - pt);")]),
    ("accept margin scaled by p alone",
     [("double d = fabs(lhs - pt) / scale;", "double d = fabs(lhs - pt) / pt;")]),
    ("top-p margin taken before the prefix's own mass",
     [("            cum += wf[j] / Sf;\n            double d = fabs(cum - top_p);",
       "            double d = fabs(cum - top_p);\n            cum += wf[j] / Sf;")]),
    ("min-p margin on the absolute probability",
     [("double d = fabs(ratio - min_p);", "double d = fabs(wf[j] / Sf - min_p);")]),
    ("top-n-sigma margin not relative to the threshold",
     [("double scale = fabs(thr) > 1.0 ? fabs(thr) : 1.0;", "double scale = 1.0;")]),
    ("typical margin ignores the score gap at the cut",
     [("if (g / sc < *margin)", "if (0)")]),
    ("sampler-match margin keeps only the last draw",
     [("        if (m < *margin)\n            *margin = m;\n        if (n == K || tokens[n] != drawn)",
       "        *margin = m;\n        if (n == K || tokens[n] != drawn)")]),
    ("EOG all-excluded row answers id 0",
     [("    return best;\n}\n\nvoid orc_argmax_excluding(",
       "    return best == ORC_INVALID ? 0 : best;\n}\n\nvoid orc_argmax_excluding(")]),
]


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, edits):
    src = open(SRC).read()
    for orig, planted in edits:
        assert src.count(orig) == 1, f"mutation site not unique/found: {orig!r}"
        src = src.replace(orig, planted)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    lib = oracle.compile_oracle(str(path), str(tmp_path / "libmutant.so"))
    # run the pins in a child: a planted mistake may crash the library
    proc = subprocess.run([sys.executable, oracle_pins.__file__, lib],
                          capture_output=True, text=True, timeout=300)
    assert proc.returncode == 1 and "FAIL pin_" in proc.stdout, (
        f"no pin fails for the planted mistake: {name}\n"
        f"rc={proc.returncode}\n{proc.stdout}\n{proc.stderr[-2000:]}")
