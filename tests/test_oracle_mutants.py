"""Plants plausible mistakes in copies of the oracle's C source and checks
that the pins reject every one of them (the pins are not vacuous)."""
import os

import pytest

import oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "psw_oracle.c")

# (name, exact text in the oracle, replacement)
MUTANTS = [
    ("window edge off by one", "(p - j < job->window)", "(p - j <= job->window)"),
    ("gqa modulo mapping", "const int32_t g = h / group;",
     "const int32_t g = h % job->n_kv_heads;"),
    ("scale dropped", "double s = job->scale * dot;", "double s = dot;"),
    ("softcap before scale", "s = job->softcap * tanh(s / job->softcap);",
     "s = job->scale * job->softcap * tanh(dot / job->softcap);"),
    ("softcap not rescaled", "s = job->softcap * tanh(s / job->softcap);",
     "s = tanh(s / job->softcap);"),
    ("slot offset dropped", "return (int64_t)block_table_row[logical_block] * block_size + offset;",
     "return (int64_t)block_table_row[logical_block] * block_size;"),
    ("v read from k pool", "job->k_eq_v ? job->k_pool : job->v_pool", "job->k_pool"),
    ("lse without max", "job->lse[row * job->n_q_heads + h] = m + log(l);",
     "job->lse[row * job->n_q_heads + h] = log(l);"),
    ("cache write skips v", "memcpy(v_pool + slot * row_elems",
     "if (0) memcpy(v_pool + slot * row_elems"),
    ("kv size missing v factor", "return with_v ? 2.0 * one : one;", "return one;"),
    ("rope denominator is the rotated size", "pow(theta, -2.0 * (double)i / (double)hd)",
     "pow(theta, -2.0 * (double)i / (double)(2 * rope_angles))"),
    ("rope sin sign", "y[i] = lo * c - hi * s;", "y[i] = lo * c + hi * s;"),
    ("rope rotates the unrotated dims", "double freq = (i < rope_angles)",
     "double freq = (1)"),
    ("rope adjacent pairs", "double lo = y[i], hi = y[i + half];",
     "double lo = y[i], hi = y[(i + 1) % hd];"),
    ("v rotated", "oracle_norm_rope_row(v + o, hd, eps, v_w, 0,",
     "oracle_norm_rope_row(v + o, hd, eps, v_w, 1,"),
    ("norm eps outside the root", "1.0 / sqrt(ss / (double)hd + eps)",
     "1.0 / (sqrt(ss / (double)hd) + eps)"),
    ("norm over the sum", "1.0 / sqrt(ss / (double)hd + eps)", "1.0 / sqrt(ss + eps)"),
    ("norm weight ignored", "(weight != NULL ? (double)weight[d] : 1.0)", "1.0"),
    ("rope position off by one", "int64_t pos = (int64_t)past_lens[b] + (t - cu_new[b]);\n            for (int32_t h",
     "int64_t pos = (int64_t)past_lens[b] + (t - cu_new[b]) + 1;\n            for (int32_t h"),
    ("bf16 rounding truncates", "double n = nearbyint(ldexp(a, -qexp));",
     "double n = floor(ldexp(a, -qexp));"),
    ("e4m3 exponent bias", "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    ("e4m3 rounds ties away", "double n = nearbyint(ldexp(a, -q)); /* ties to even */",
     "double n = round(ldexp(a, -q));"),
    ("fp8 scale off the code range", "*scale = amax / 448.0f;", "*scale = amax / 240.0f;"),
    ("fp8 scale ignored", "const double s = (double)scale8[r];", "const double s = 1.0;"),
    ("fp8 v read from k codes", "const uint8_t *v8 = job->k_eq_v ? job->k8 : job->v8;",
     "const uint8_t *v8 = job->k8;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, old, new):
    import oracle
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor missing: {old}"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutated), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failures = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failures.append(check.__name__)
    assert failures, f"no pin caught the planted mistake: {name}"
