"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a temporary copy of oracle.c (a
transposed operand, a dropped term, a wrong sign or index, a missing factor),
builds it, and runs the pin tests against it.  Every mutant must make at
least one pin fail; a mutant that survives means the pins are too weak."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = [
    # (id, original text, mutated text, pin file)
    ("dA_transposed_B", "s += G[m * N + n] * B[k * N + n];", "s += G[m * N + n] * B[n * K + k];",
     "test_oracle_matmul.py"),
    ("Y_dropped_term", "for (int64_t k = 0; k < K; ++k) s += A[m * K + k] * B[k * N + n];",
     "for (int64_t k = 0; k + 1 < K; ++k) s += A[m * K + k] * B[k * N + n];", "test_oracle_matmul.py"),
    ("dB_sign", "dB[k * N + n] = s;", "dB[k * N + n] = -s;", "test_oracle_matmul.py"),
    ("plan_off_by_one", "int64_t size = (r < n_big) ? small + 1 : small;",
     "int64_t size = (r <= n_big) ? small + 1 : small;", "test_oracle_plan.py"),
    ("owner_closed_interval", "if (off[r] <= y && y < off[r + 1]) return r;",
     "if (off[r] <= y && y <= off[r + 1]) return r;", "test_oracle_plan.py"),
    ("gelu_grad_dropped_term", "return cdf + x * pdf;", "return cdf;", "test_oracle_act.py"),
    ("gelu_tanh_coefficient", "return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));",
     "return 0.5 * x * (1.0 + tanh(c * (x + 0.047 * x * x * x)));", "test_oracle_act.py"),
    ("mlp_missing_act_grad", "dz[f] = s * orc_act_grad(act, hp[f]);", "dz[f] = s;", "test_oracle_mlp.py"),
    ("mlp_dW2_wrong_operand", "for (int64_t t = 0; t < T; ++t) s += ha[t] * GY[t * d + c];",
     "for (int64_t t = 0; t < T; ++t) s += dz[t] * GY[t * d + c];", "test_oracle_mlp.py"),
    ("mlp_dX_transposed_W1", "for (int64_t f = 0; f < F; ++f) s += dz[f] * W1[c * F + f];",
     "for (int64_t f = 0; f < F; ++f) s += dz[f] * W1[f * d + c];", "test_oracle_mlp.py"),
    ("ce_onehot_sign", "dz[v] = exp(z[v] - m) / s - (v == y ? 1.0 : 0.0);",
     "dz[v] = exp(z[v] - m) / s + (v == y ? 1.0 : 0.0);", "test_oracle_ce.py"),
    ("ce_loss_missing_max", "if (loss) loss[i] = log(s) + m - z[y];", "if (loss) loss[i] = log(s) - z[y];",
     "test_oracle_ce.py"),
    ("ce_ex_padding_in_softmax", "for (int64_t v = 0; v < vocab_real; ++v) s += exp(z[v] - m);",
     "for (int64_t v = 0; v < V; ++v) s += exp(z[v] - m);", "test_oracle_ce_ex.py"),
    ("ce_ex_mean_gradient_unscaled",
     "dz[v] = (v < vocab_real) ? (exp(z[v] - m) / s - (v == y ? 1.0 : 0.0)) / D : 0.0;",
     "dz[v] = (v < vocab_real) ? (exp(z[v] - m) / s - (v == y ? 1.0 : 0.0)) : 0.0;", "test_oracle_ce_ex.py"),
    ("ce_ex_denominator_counts_ignored", "(count > 0 ? (double)count : 1.0)", "(T > 0 ? (double)T : 1.0)",
     "test_oracle_ce_ex.py"),
    ("silu_grad_dropped_term", "return sg + x * sg * (1.0 - sg);", "return sg;", "test_oracle_act.py"),
    ("glu_gate_and_up_swapped", "double a = orc_act(act, hg[f]) * u[f];", "double a = orc_act(act, u[f]) * hg[f];",
     "test_oracle_glu.py"),
    ("glu_dX_missing_up_branch", "for (int64_t f = 0; f < F; ++f) s += du[f] * Wu[c * F + f];",
     "for (int64_t f = 0; f < F && 0; ++f) s += du[f] * Wu[c * F + f];", "test_oracle_glu.py"),
    ("glu_dHg_missing_up_factor", "dhg[t] = da * u * orc_act_grad(act, hg);", "dhg[t] = da * orc_act_grad(act, hg);",
     "test_oracle_glu.py"),
    ("glu_dWu_wrong_operand", "su += X[t * d + c] * du[t];", "su += X[t * d + c] * dhg[t];", "test_oracle_glu.py"),
    ("heads_replica_index", "for (int32_t r = 0; r < tp; ++r) kv_first[r] = r / rep;",
     "for (int32_t r = 0; r < tp; ++r) kv_first[r] = r % n_kv_heads;", "test_oracle_attn.py"),
    ("heads_uneven_accepted", "if (n_heads % tp != 0) return ORC_ERR_PARTITION;", "", "test_oracle_attn.py"),
    ("attn_dX_missing_branch", "for (int64_t j = 0; j < n[p]; ++j) s += G[p][t * n[p] + j] * W[p][c * n[p] + j];",
     "for (int64_t j = 0; j < n[p] && p < 2; ++j) s += G[p][t * n[p] + j] * W[p][c * n[p] + j];",
     "test_oracle_attn.py"),
    ("attn_dWo_wrong_index", "for (int64_t t = 0; t < T; ++t) s += C[t * nq + j] * GY[t * d + c];",
     "for (int64_t t = 0; t < T; ++t) s += C[t * nq + j] * GY[t * d + (c + 1) % d];", "test_oracle_attn.py"),
    ("ce_sharded_local_max", "for (int64_t j = off[r]; j < off[r + 1]; ++j) sr += exp(z[j] - m);",
     "for (int64_t j = off[r]; j < off[r + 1]; ++j) sr += exp(z[j] - m_r[r]);", "test_oracle_ce.py"),
]


@pytest.mark.parametrize("mid,orig,mut,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, mid, orig, mut, pins):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation site for {mid} not found exactly once"
    msrc = tmp_path / "oracle_mutant.c"
    msrc.write_text(src.replace(orig, mut))
    lib = oracle.compile_oracle(str(msrc), str(tmp_path / "liboracle_mutant.so"))
    env = dict(os.environ, ORACLE_LIB=lib, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", pins)], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {mid} survived the pins in {pins}:\n{r.stdout[-2000:]}"
