"""Planted mistakes: each mutant is a copy of the oracle's C source with one
plausible error (a wrong mask edge, a dropped term, a wrong index, a
transposed operand, a wrong GQA map), compiled on the CPU.  The independent
pins of test_oracle.py -- everything except the stored-values drift guard,
which is the oracle's own output -- must fail on every mutant and pass on an
unmutated copy built the same way.

Every mutant stays inside the buffers the real oracle reads (it can only see
fewer keys, the same keys in another order, or another in-range head), so a
failing pin is a detection, never a crash.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attn_oracle.c")

# (name, text in attn_oracle.c, replacement)
MUTANTS = [
    ("causal_edge_off_by_one",
     "int64_t last = i + (Sk - Sq);", "int64_t last = i + (Sk - Sq) - 1;"),
    ("causal_top_left_alignment",
     "int64_t last = i + (Sk - Sq);", "int64_t last = i;"),
    ("causal_flag_ignored",
     "if (!causal) return Sk;", "return Sk;"),
    ("fully_masked_row_sees_key0",
     "if (last < 0) return 0;", "if (last < 0) return Sk > 0 ? 1 : 0;"),
    ("scale_dropped",
     "s[j] = scale * acc;", "s[j] = acc;"),
    ("max_not_subtracted",
     "s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    ("exponent_sign_flipped",
     "s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    ("normalisation_dropped",
     "o[d] /= l;", "o[d] /= 1.0;"),
    ("sum_of_squares",
     "l += s[j];", "l += s[j] * s[j];"),
    ("output_accumulates_keys",
     "const double* vj = vbase + j * kstride;", "const double* vj = kbase + j * kstride;"),
    ("keys_reversed",
     "const double* kj = kbase + j * kstride;",
     "const double* kj = kbase + (n_vis - 1 - j) * kstride;"),
    ("dot_product_index_reversed",
     "acc += q[d] * kj[d];", "acc += q[d] * kj[D - 1 - d];"),
    ("gqa_interleaved_prefill",
     "const int64_t kv = h / G;\n    const double* kb = J->k",
     "const int64_t kv = h % J->Hkv;\n    const double* kb = J->k"),
    ("gqa_interleaved_decode",
     "const int64_t kv = h / G;\n      const double* kb = kcache",
     "const int64_t kv = h % Hkv;\n      const double* kb = kcache"),
    ("batch_offset_dropped_for_keys",
     "const double* kb = J->k + (b * J->Sk * J->Hkv + kv) * J->D;",
     "const double* kb = J->k + (kv) * J->D;"),
    ("kv_head_dropped_for_values",
     "const double* vb = J->v + (b * J->Sk * J->Hkv + kv) * J->D;",
     "const double* vb = J->v + (b * J->Sk * J->Hkv) * J->D;"),
    ("decode_valid_length_off_by_one",
     "(int64_t)Hkv * D, L, D,", "(int64_t)Hkv * D, L - 1, D,"),
    ("decode_clamp_below_capacity",
     "if (L > cap) L = cap;", "if (L >= cap) L = cap - 1;"),
    ("probabilities_not_normalised",
     "p_out[j] = s[j] / l;", "p_out[j] = s[j];"),
    ("lse_without_max",
     "if (lse) *lse = m + log(l);", "if (lse) *lse = log(l);"),
    ("lse_log_of_mean",
     "if (lse) *lse = m + log(l);", "if (lse) *lse = m + log(l / (double)n_vis);"),
    ("lse_empty_row_zero",
     "if (lse) *lse = -INFINITY;", "if (lse) *lse = 0.0;"),
    ("bwd_delta_dropped",
     "const double ds = pr[j] * (dp[j] - delta);", "const double ds = pr[j] * dp[j];"),
    ("bwd_key_gradient_unscaled",
     "dkb[j * kstride + d] += J->scale * ds * qi[d];", "dkb[j * kstride + d] += ds * qi[d];"),
    ("bwd_value_gradient_uses_dp",
     "dvb[j * kstride + d] += pr[j] * doi[d];", "dvb[j * kstride + d] += dp[j] * doi[d];"),
    ("bwd_query_gradient_uses_values",
     "dqi[d] += J->scale * ds * kb[j * kstride + d];",
     "dqi[d] += J->scale * ds * vb[j * kstride + d];"),
]

PIN_ARGS = ["-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"), "-x", "-q",
            "-p", "no:cacheprovider", "-m", "not gpu",
            "-k", "not golden_oracle_values"]


def _build_and_run(tmpdir, name, old, new):
    src = open(SRC).read()
    if old is not None:
        assert src.count(old) == 1, f"{name}: mutation site not unique in the oracle"
        src = src.replace(old, new)
    c_path = os.path.join(tmpdir, f"{name}.c")
    so_path = os.path.join(tmpdir, f"lib{name}.so")
    with open(c_path, "w") as f:
        f.write(src)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-w", "-o", so_path, c_path, "-lm"])
    # A pytest plugin, imported before the pins are collected, binds the oracle
    # package to this copy of the library (the oracle itself has no switch).
    plugin = f"mutant_plugin_{name}"
    with open(os.path.join(tmpdir, plugin + ".py"), "w") as f:
        f.write("import oracle\n"
                f"oracle._lib = oracle._bind({so_path!r})\n")
    path = os.pathsep.join([tmpdir, ROOT] + [p for p in [os.environ.get("PYTHONPATH")] if p])
    env = dict(os.environ, PYTHONPATH=path, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable] + PIN_ARGS + ["-p", plugin], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    tmpdir = str(tmp_path_factory.mktemp("oracle_mutants"))
    jobs = [("unmutated", None, None)] + MUTANTS
    workers = max(1, min(8, len(os.sched_getaffinity(0)) // 2))
    with cf.ThreadPoolExecutor(workers) as ex:
        futs = {name: ex.submit(_build_and_run, tmpdir, name, old, new)
                for name, old, new in jobs}
        return {name: f.result() for name, f in futs.items()}


def test_unmutated_copy_passes_the_pins(outcomes):
    rc, out = outcomes["unmutated"]
    assert rc == 0, out


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(outcomes, name):
    rc, out = outcomes[name]
    # pytest exit code 1 = some pin failed (not a crash, not a collection error)
    assert rc == 1, f"mutant {name} survived the pins (exit {rc}):\n{out}"
