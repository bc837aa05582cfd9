"""The oracle pins catch plausible mistakes: each case plants one error in a copy of the oracle
source (on the CPU), builds it, and runs the pin suite against it, which must fail."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gdn_oracle.c")

MUTATIONS = {
    "no_decay": ("  const double decay = exp(g);", "  const double decay = 1.0;"),
    "delta_sign": ("    delta[j] = beta * (v[j] - kv);", "    delta[j] = beta * (v[j] + kv);"),
    "output_before_update": (
        "  for (int i = 0; i < dk; ++i)\n    for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += k[i] * delta[j];",
        "  for (int i = 0; i < 0; ++i)\n    for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += k[i] * delta[j];"),
    "softplus_identity": ("  return log1p(exp(x));", "  return x;"),
    "sigmoid_sign": ("double oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }",
                     "double oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(x)); }"),
    "gqa_modulo": ("    const int hk = h / r; /* repeat_interleave */",
                   "    const int hk = h % d->Hk;"),
    "conv_taps_reversed": (
        "    for (int j = 0; j < K - 1; ++j) acc += w[(size_t)c * K + j] * state[(size_t)j * C + c];",
        "    for (int j = 0; j < K - 1; ++j) acc += w[(size_t)c * K + (K - 2 - j)] * state[(size_t)j * C + c];"),
    "conv_state_not_rolled": ("    if (K > 1) state[(size_t)(K - 2) * C + c] = x[c];", "    (void)0;"),
    "no_q_scale": ("    oracle_l2norm(d->dk, yq + (size_t)hk * d->dk, d->l2_eps, d->q_scale, qn + (size_t)hk * d->dk);",
                   "    oracle_l2norm(d->dk, yq + (size_t)hk * d->dk, d->l2_eps, 1.0, qn + (size_t)hk * d->dk);"),
    "rms_sum_not_mean": ("  const double inv = 1.0 / sqrt(ss / dv + eps);", "  const double inv = 1.0 / sqrt(ss + eps);"),
    "chunk_drop_WS0": ("            for (int f = 0; f < dk; ++f) v += Wm[(size_t)i * dk + f] * S0[(size_t)f * dv + e];\n            Um[(size_t)i * dv + e] -= v;",
                       "            for (int f = 0; f < dk; ++f) v += Wm[(size_t)i * dk + f] * S0[(size_t)f * dv + e];\n            Um[(size_t)i * dv + e] -= 0.0 * v;"),
    "chunk_gamma_sign": ("              v = BETA(i) * exp(gam[i] - gam[j]) * kk;",
                         "              v = BETA(i) * exp(gam[j] - gam[i]) * kk;"),
    "linear_transposed_weight": (
        "      for (int k = 0; k < K; ++k) acc += x[(size_t)m * K + k] * w[(size_t)n * K + k];",
        "      for (int k = 0; k < K; ++k) acc += x[(size_t)m * K + k] * w[(size_t)k * N + n];"),
    "linear_drops_last_term": (
        "      for (int k = 0; k < K; ++k) acc += x[(size_t)m * K + k] * w[(size_t)n * K + k];",
        "      for (int k = 0; k < K - 1; ++k) acc += x[(size_t)m * K + k] * w[(size_t)n * K + k];"),
    "in_proj_b_a_swapped": (
        "    memcpy(b + (size_t)m * Hv, yr + cqkv + zd, sizeof(double) * Hv);",
        "    memcpy(b + (size_t)m * Hv, yr + cqkv + zd + Hv, sizeof(double) * Hv);"),
    "prefill_keeps_state_without_init": (
        "      memset(S, 0, sizeof(double) * rec_slot);\n      memset(cs, 0, sizeof(double) * conv_slot);\n"
        "    }\n    for (int t = t0; t < t1; ++t)",
        "      memset(cs, 0, sizeof(double) * conv_slot);\n    }\n    for (int t = t0; t < t1; ++t)"),
    "chunkwise_keeps_state_without_init": (
        "      memset(S, 0, sizeof(double) * rec_slot);\n      memset(cs, 0, sizeof(double) * conv_slot);\n"
        "    }\n    if (T <= 0) continue;",
        "      memset(cs, 0, sizeof(double) * conv_slot);\n    }\n    if (T <= 0) continue;"),
    "l2norm_eps_outside_root": ("  const double inv = 1.0 / sqrt(ss + eps);",
                                "  const double inv = 1.0 / (sqrt(ss) + eps);"),
    "conv_without_silu": ("    y[c] = oracle_silu(acc);", "    y[c] = acc;"),
    "gate_sigmoid_not_silu": (
        "  for (int j = 0; j < dv; ++j) out[j] = o[j] * inv * w[j] * oracle_silu(z[j]);",
        "  for (int j = 0; j < dv; ++j) out[j] = o[j] * inv * w[j] * oracle_sigmoid(z[j]);"),
    "chunk_output_strict_mask": ("            for (int j = 0; j <= i; ++j) {\n              double qk = 0.0;",
                                 "            for (int j = 0; j < i; ++j) {\n              double qk = 0.0;"),
    "compact_no_snapshot": (
        "    memcpy(rec_state + (size_t)dst[i] * rec_slot_elems, snap_r + (size_t)i * rec_slot_elems,",
        "    memcpy(rec_state + (size_t)dst[i] * rec_slot_elems, rec_state + (size_t)src[i] * rec_slot_elems,"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, source, tmp_path):
    old, new = MUTATIONS[name]
    assert source.count(old) == 1, f"mutation anchor not unique: {name}"
    mutated = tmp_path / "gdn_oracle_mutant.c"
    mutated.write_text(source.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    oracle.compile_to(str(mutated), str(lib))
    env = dict(os.environ, GDN_ORACLE_LIB=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"pins did not catch mutation {name}:\n{res.stdout[-2000:]}"
