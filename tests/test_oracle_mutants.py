"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of oracle/ittt_oracle.c (on the CPU,
in a temporary directory), builds it, and runs the pin suite against that
copy: the suite has to fail.  The same is done for the chunk-by-chunk oracle
(oracle/chunked.py) and its own pins.  The committed oracle is never
modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ittt_oracle.c")
SRC_CHUNKED = os.path.join(ROOT, "oracle", "chunked.py")

# (name, exact text in the oracle, replacement)
MUTANTS = [
    ("silu_drops_gate_sigmoid", "return x / (1.0 + exp(-x));", "return x;"),
    ("conv_taps_flipped",
     "acc += (double)conv_w[c * 3 + (k + 1)] * (double)X0[s * d + c];",
     "acc += (double)conv_w[c * 3 + (1 - k)] * (double)X0[s * d + c];"),
    ("conv_ignores_chunk_edges", "lo = (t / C) * C;\n      hi = lo + C < T ? lo + C : T;",
     "lo = 0;\n      hi = T;"),
    ("target_not_transposed",
     "acc += Xc[t * d + c] * (double)W_target[m * d + c];",
     "acc += Xc[t * d + c] * (double)W_target[c * d + m];"),
    ("update_sign_flipped", "for (int64_t e = 0; e < d * f; ++e) W[e] += eta * dW[e];",
     "for (int64_t e = 0; e < d * f; ++e) W[e] -= eta * dW[e];"),
    ("update_before_apply",
     "      apply_chunk(i * C, Cn, d, f, Z, W, O + b * T * d);         /* apply  */\n"
     "      chunk_delta(i * C, Cn, d, f, Vhat, Z, et, dW);             /* update */\n"
     "      for (int64_t e = 0; e < d * f; ++e) W[e] += eta * dW[e];",
     "      chunk_delta(i * C, Cn, d, f, Vhat, Z, et, dW);\n"
     "      for (int64_t e = 0; e < d * f; ++e) W[e] += eta * dW[e];\n"
     "      apply_chunk(i * C, Cn, d, f, Z, W, O + b * T * d);"),
    ("initial_weight_dropped", "for (int64_t e = 0; e < d * f; ++e) W[e] = (double)W0[e];",
     "for (int64_t e = 0; e < d * f; ++e) W[e] = 0.0;"),
    ("delta_drops_first_token", "for (int64_t t = t0; t < t0 + Cn; ++t)\n        acc += token_rate",
     "for (int64_t t = t0 + 1; t < t0 + Cn; ++t)\n        acc += token_rate"),
    ("delta_uses_Z_for_both_operands", "Vhat[t * d + m] * Z[t * f + j];",
     "Z[t * f + m] * Z[t * f + j];"),
    ("token_rate_ignored", "return eta_tok ? (double)eta_tok[t] : 1.0;", "return 1.0;"),
    ("partial_chunk_dropped", "static int64_t num_chunks(int64_t T, int64_t C) { return (T + C - 1) / C; }",
     "static int64_t num_chunks(int64_t T, int64_t C) { return T / C; }"),
    ("prefix_scan_inclusive",
     "S[i * df + e] = S[(i - 1) * df + e] + dWs[(i - 1) * df + e];",
     "S[i * df + e] = S[(i - 1) * df + e] + dWs[(i < n ? i : n - 1) * df + e];"),
    ("dual_includes_current_chunk", "for (int64_t s = 0; s < i * C; ++s) { /* every token",
     "for (int64_t s = 0; s < (i + 1) * C; ++s) { /* every token"),
    ("l2norm_skipped", "      l2_normalize_rows(d, f, W);\n", "\n"),
    ("l2norm_over_columns",
     "    for (int64_t j = 0; j < f; ++j) ss += W[m * f + j] * W[m * f + j];",
     "    for (int64_t j = 0; j < d; ++j) ss += W[j * f + (m % f)] * W[j * f + (m % f)];"),
    ("l2norm_applied_to_initial_weight",
     "    if (states_out) memcpy(states_out + (b * (n + 1)) * df, W, (size_t)df * sizeof(double));",
     "    l2_normalize_rows(d, f, W);\n"
     "    if (states_out) memcpy(states_out + (b * (n + 1)) * df, W, (size_t)df * sizeof(double));"),
    ("state_entries_skip_eta",
     "out[q * (n + 1) + i + 1] = (double)w0[m * f + j] + eta * sum;",
     "out[q * (n + 1) + i + 1] = (double)w0[m * f + j] + sum;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "ittt_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libittt_oracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", str(lib),
                    str(mutated), "-lm"], check=True)
    env = dict(os.environ, ITTT_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"


# (name, exact text in oracle/chunked.py, replacement)
CHUNKED_MUTANTS = [
    ("silu_drops_sigmoid", "return x / (1.0 + np.exp(-x))", "return x"),
    ("conv_taps_flipped", "pad[:-2] * w[:, 0] + pad[1:-1] * w[:, 1] + pad[2:] * w[:, 2]",
     "pad[:-2] * w[:, 2] + pad[1:-1] * w[:, 1] + pad[2:] * w[:, 0]"),
    ("conv_ignores_chunk_edges",
     "        seg = (lo, hi) if pad_mode == PAD_CHUNK else (0, T)\n        V = conv_rows(X0, conv_w, lo, hi, *seg) @ Wt.T\n        O = Z @ W.T",
     "        seg = (0, T)\n        V = conv_rows(X0, conv_w, lo, hi, *seg) @ Wt.T\n        O = Z @ W.T"),
    ("target_not_transposed", "V = conv_rows(X0, conv_w, lo, hi, *seg) @ Wt.T\n        O = Z @ W.T",
     "V = conv_rows(X0, conv_w, lo, hi, *seg) @ Wt\n        O = Z @ W.T"),
    ("update_sign_flipped", "W_next = W + eta * (Vr.T @ Z)", "W_next = W - eta * (Vr.T @ Z)"),
    ("update_before_apply", "        O = Z @ W.T\n        out = {",
     "        O = Z @ (W + eta * (V.T @ Z)).T\n        out = {"),
    ("initial_weight_dropped", "W = _f64(W0).copy()", "W = 0.0 * _f64(W0)"),
    ("token_rates_ignored", "Vr = V if rates is None else V * rates[lo:hi, None]", "Vr = V"),
    ("apply_uses_Z_for_output", "O = Z @ W.T", "O = Z[:, :W.shape[0]] * 1.0"),
    ("l2norm_skipped", "                W_next = _normalise_rows(W_next)\n", "\n"),
    ("l2norm_over_columns", "norm = np.sqrt((W * W).sum(axis=1))\n    return W / np.maximum(norm, 1e-12)[:, None]",
     "norm = np.sqrt((W * W).sum(axis=0))\n    return W / np.maximum(norm, 1e-12)[None, :]"),
    ("state_grid_skips_eta", "out[i + 1] = out[0] + eta * acc", "out[i + 1] = out[0] + acc"),
    ("state_grid_inclusive", "        acc = acc + V.T @ Z\n        out[i + 1] = out[0] + eta * acc",
     "        acc = acc + V.T @ Z\n        out[i + 1] = out[0] + eta * (acc + V.T @ Z)"),
]


@pytest.mark.parametrize("name,old,new", CHUNKED_MUTANTS, ids=[m[0] for m in CHUNKED_MUTANTS])
def test_chunked_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC_CHUNKED).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "chunked_mutant.py"
    mutated.write_text(src.replace(old, new))
    env = dict(os.environ, ITTT_CHUNKED_ORACLE=str(mutated), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_chunked.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
