"""Plant plausible slips in copies of the oracle; the pins must reject each one.

Every mutant is a one-token change of ``oracle/ref_reduce.c`` (a wrong sign, a
dropped term, an off-by-one, a wrong index or operand).  Each is compiled to a
temporary library and the pin suite ``test_oracle_pins.py`` is run against it
in a subprocess; the suite must fail.  This is what makes the pins evidence:
they are shown to catch the mistakes they are meant to catch.
"""
import concurrent.futures
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ref_reduce.c")

# (name, text in ref_reduce.c, replacement, which occurrence (0 = first))
MUTANTS = [
    ("causal_off_by_one", "if (causal && j > query[r])", "if (causal && j >= query[r])", 0),
    ("causal_direction", "if (causal && j > query[r])", "if (causal && j < query[r])", 0),
    ("mask_wrong_row", "mask + batch[r] * Tk", "mask + 0 * Tk", 0),
    ("mask_sign", "xr[j] + (mr ? mr[j] : 0.0)", "xr[j] - (mr ? mr[j] : 0.0)", 0),
    ("no_max_shift", "exp(yr[j] - m)", "exp(yr[j])", 0),
    ("no_normalise", "yr[j] = yr[j] / s;", "yr[j] = yr[j];", 0),
    ("softmax_bw_sign", "yr[j] * (dyr[j] - s)", "yr[j] * (dyr[j] + s)", 0),
    ("softmax_bw_drop_sum", "yr[j] * (dyr[j] - s)", "yr[j] * dyr[j]", 0),
    ("softmax_bw_transposed", "s += yr[k] * dyr[k];", "s += yr[k] * yr[k];", 0),
    ("ln_unbiased_var", "var /= (double)N;", "var /= (double)(N - 1);", 0),
    ("ln_eps_outside_root", "1.0 / sqrt(var + eps)", "1.0 / (sqrt(var) + eps)", 0),
    ("ln_gamma_beta_swapped", "rs * gamma[j] + beta[j]", "rs * beta[j] + gamma[j]", 0),
    ("ln_mean_not_subtracted", "yr[j] = (xr[j] - mu) * rs", "yr[j] = xr[j] * rs", 0),
    ("dinp_drop_xhat_term", "rstd[r] * (g - a - xhat * b)", "rstd[r] * (g - a)", 0),
    ("dinp_xhat_sign", "rstd[r] * (g - a - xhat * b)", "rstd[r] * (g - a + xhat * b)", 0),
    ("dinp_drop_mean_g", "rstd[r] * (g - a - xhat * b)", "rstd[r] * (g - xhat * b)", 0),
    ("dinp_gamma_missing", "double g = gamma[j] * dyr[j];", "double g = dyr[j];", 0),
    ("dgamma_no_rstd", "double xhat = (x[r * N + j] - mean[r]) * rstd[r];",
     "double xhat = (x[r * N + j] - mean[r]);", 0),
    ("dgamma_transposed", "dg += dy[r * N + j] * xhat;", "dg += x[r * N + j] * xhat;", 0),
    ("dbeta_weighted", "db += dy[r * N + j];", "db += dy[r * N + j] * xhat;", 0),
    ("one_pass_no_square", "s2 += x[j] * x[j];", "s2 += x[j];", 0),
    ("offset_sign", "if (causal && j > q + offset)", "if (causal && j > q - offset)", 0),
    ("visible_offset_dropped", "if (causal && j > q + offset)\n        return 0;",
     "if (causal && j > q)\n        return 0;", 0),
    ("fw_offset_dropped", "if (causal && j > q + offset)", "if (causal && j > q)", 1),
    ("rms_no_square", "ms += xr[j] * xr[j];", "ms += xr[j];", 0),
    ("rms_eps_outside", "double rs = 1.0 / sqrt(ms + eps);", "double rs = 1.0 / (sqrt(ms) + eps);", 0),
    ("rms_mean_subtracted", "yr[j] = xr[j] * rs * gamma[j];", "yr[j] = (xr[j] - ms) * rs * gamma[j];", 0),
    ("rms_bw_drop_term", "dxr[j] = rstd[r] * (g - xhat * b);", "dxr[j] = rstd[r] * g;", 0),
    ("rms_bw_sign", "dxr[j] = rstd[r] * (g - xhat * b);", "dxr[j] = rstd[r] * (g + xhat * b);", 0),
    ("rms_dgamma_no_rstd", "dg += dy[r * N + j] * (x[r * N + j] * rstd[r]);", "dg += dy[r * N + j] * x[r * N + j];", 0),
    ("ce_no_max_shift", "s += exp(zr[j] - m);", "s += exp(zr[j]);", 0),
    ("ce_lse_drops_max", "lse[r] = m + log(s);", "lse[r] = log(s);", 0),
    ("ce_loss_sign", "loss[r] = lse[r] - zr[t];", "loss[r] = lse[r] + zr[t];", 0),
    ("ce_loss_wrong_class", "loss[r] = lse[r] - zr[t];", "loss[r] = lse[r] - zr[0];", 0),
    ("ce_bw_ignored_row_kept", "if (t < 0)\n                dzr[j] = 0.0;",
     "if (t < -1000)\n                dzr[j] = 0.0;", 0),
    ("ce_bw_onehot_sign", "(exp(zr[j] - lse[r]) - (j == t ? 1.0 : 0.0))",
     "(exp(zr[j] - lse[r]) + (j == t ? 1.0 : 0.0))", 0),
    ("ce_bw_onehot_off_by_one", "(j == t ? 1.0 : 0.0)", "(j == t + 1 ? 1.0 : 0.0)", 0),
    ("ce_bw_no_dloss", "dzr[j] = dloss[r] * (exp(zr[j] - lse[r])", "dzr[j] = 1.0 * (exp(zr[j] - lse[r])", 0),
    ("ce_bw_out_of_range_kept", "else if ((int64_t)t >= V)\n                dzr[j] = NAN;",
     "else if ((int64_t)t >= V + 1)\n                dzr[j] = NAN;", 0),
    ("scaled_fw_scale_dropped", "z = scale * xr[j] + (mr ? mr[j] : 0.0);",
     "z = xr[j] + (mr ? mr[j] : 0.0);", 0),
    ("scaled_fw_scale_on_mask", "z = scale * xr[j] + (mr ? mr[j] : 0.0);",
     "z = scale * (xr[j] + (mr ? mr[j] : 0.0));", 0),
    ("scaled_fw_offset_dropped", "if (!(causal && j > q + offset))", "if (!(causal && j > q))", 0),
    ("scaled_bw_scale_dropped", "scale * yr[j] * (dyr[j] - s)", "yr[j] * (dyr[j] - s)", 0),
    ("scaled_bw_scale_squared", "scale * yr[j] * (dyr[j] - s)", "scale * scale * yr[j] * (dyr[j] - s)", 0),
    ("masked_bw_sum_all_keys", "if (visible(mr, k, q, offset, causal))\n                s += yr[k] * dyr[k];",
     "s += yr[k] * dyr[k];", 0),
    ("masked_bw_no_zeroing", "dxr[j] = visible(mr, j, q, offset, causal) ? yr[j] * (dyr[j] - s) : 0.0;",
     "dxr[j] = yr[j] * (dyr[j] - s);", 0),
]


def _mutate(text, old, new, k):
    pos = -1
    for _ in range(k + 1):
        pos = text.index(old, pos + 1)
    return text[:pos] + new + text[pos + len(old):]


def _run_mutant(tmp, name, old, new, k):
    src = open(SRC, encoding="utf-8").read()
    path_c = os.path.join(tmp, f"{name}.c")
    path_so = os.path.join(tmp, f"{name}.so")
    with open(path_c, "w", encoding="utf-8") as f:
        f.write(_mutate(src, old, new, k))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    path_c, "-o", path_so, "-lm"], check=True)
    env = dict(os.environ, REF_REDUCE_LIB=path_so)
    proc = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle_pins.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, proc.returncode


def test_every_planted_slip_is_caught():
    with tempfile.TemporaryDirectory() as tmp:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            results = list(ex.map(lambda m: _run_mutant(tmp, *m), MUTANTS))
    survived = [name for name, rc in results if rc == 0]
    assert not survived, f"pins did not catch: {survived}"
    # a failing run means failing tests (rc 1), not a crash of the harness
    odd = [(name, rc) for name, rc in results if rc not in (0, 1)]
    assert not odd, f"unexpected pytest exit codes: {odd}"


def test_unmutated_oracle_passes_the_pins():
    with tempfile.TemporaryDirectory() as tmp:
        src = open(SRC, encoding="utf-8").read()
        name, rc = _run_mutant(tmp, "identity", src[:10], src[:10], 0)
    assert rc == 0
