"""Plants plausible mistakes in a copy of the oracle and checks the pins catch them.

Each mutant is a one-line edit of a private copy of ``oracle/ref_gemm.c``
(built with the oracle's own flags) or of ``oracle/smem_rules.py`` (the
committed oracle is untouched), run against ``test_oracle_pins.py`` in a
child process, so a mutant that reads out of bounds cannot take the test run
down with it.  Every mutant must make the pins fail.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ref_gemm.c")
RULES = os.path.join(ROOT, "oracle", "smem_rules.py")

MUTANTS = {
    "dropped_last_k_term": (
        "for (int64_t k = 0; k < K; ++k) {\n        const double a = (double)A[i * K + k];",
        "for (int64_t k = 0; k + 1 < K; ++k) {\n        const double a = (double)A[i * K + k];"),
    "wrong_sign": ("acc[j] += a * (double)b_row[j];",
                   "acc[j] -= a * (double)b_row[j];"),
    "wrong_leading_dim_b": ("const float *b_row = B + k * N;",
                            "const float *b_row = B + k * K;"),
    "transposed_a_index": ("const double a = (double)A[i * K + k];\n        const float *b_row",
                           "const double a = (double)A[k * M_ + i];\n        const float *b_row"),
    "fp32_accumulation": ("acc[j] += a * (double)b_row[j];",
                          "acc[j] = (float)((float)acc[j] + (float)(a * (double)b_row[j]));"),
    "shifted_output_column": ("c_row[j] = (float)acc[j];",
                              "c_row[j] = (float)acc[j > 0 ? j - 1 : 0];"),
    "w_without_abs": ("wacc[j] += aa * fabs((double)b_row[j]);",
                      "wacc[j] += aa * (double)b_row[j];"),
    "elements_transposed_b": ("const double b = (double)B[k * N + j];",
                              "const double b = (double)B[j * K + k];"),
    # (old, new, occurrence): the fp32 and the 16-bit general forms share
    # these lines; the third field picks which copy is mutated.
    "general_beta_dropped": ("c += beta * c0;", "c += 0.0 * c0;", 0),
    "general_alpha_sign": ("double c = alpha * acc;", "double c = -alpha * acc;", 0),
    "mixed_beta_dropped": ("c += beta * c0;", "c += 0.0 * c0;", 1),
    "mixed_alpha_sign": ("double c = alpha * acc;", "double c = -alpha * acc;", 1),
    "general_trans_b_swapped": ("(trans_b ? B[j * ldb + k] : B[k * ldb + j])",
                                "(trans_b ? B[k * ldb + j] : B[j * ldb + k])", 0),
    "f16_exponent_bias": ("ldexp((double)(1024 + f), e - 25)",
                          "ldexp((double)(1024 + f), e - 24)"),
    "f16_subnormal_as_normal": ("if (e == 0) v = ldexp((double)f, -24);",
                                "if (e == 0) v = ldexp((double)(1024 + f), -25);"),
    "bf16_exponent_bias": ("ldexp((double)(128 + f), e - 134)",
                           "ldexp((double)(128 + f), e - 133)"),
    "mixed_trans_a_ignored": ("value(trans_a ? A[k * lda + i] : A[i * lda + k])",
                              "value(A[i * lda + k])"),
    "general_lda_ignored": ("(trans_a ? A[k * lda + i] : A[i * lda + k])",
                            "(trans_a ? A[k * lda + i] : A[i * K + k])", 0),
    "bias_reversed": ("c += (double)bias[j];", "c += (double)bias[N - 1 - j];", 0),
    "bias_scaled_by_alpha": ("c += (double)bias[j];", "c += alpha * (double)bias[j];", 0),
    "mixed_bias_reversed": ("c += (double)bias[j];", "c += (double)bias[N - 1 - j];", 1),
}


# One-line slips in the shared-memory rules and the bank simulator.
RULE_MUTANTS = {
    "vector_rule_counts_words_not_slots": (
        "distinct = slots // math.gcd(columns // vector_words, slots)",
        "distinct = slots // math.gcd(columns, slots)"),
    "eight_byte_access_in_32_lane_phases": (
        "per_phase = min(32, 128 // width_bytes)\n    total = 0",
        "per_phase = 32 if width_bytes <= 8 else 128 // width_bytes\n    total = 0"),
    "broadcast_not_honoured": (
        "words_in_bank.setdefault(bank(word), set()).add(word)",
        "words_in_bank.setdefault(bank(word), []).append(word)"),
    "padding_rule_not_strict": (
        "return int(simultaneous_rows > distinct_banks(columns))",
        "return int(simultaneous_rows >= distinct_banks(columns))"),
    "bank_of_word_modulo_16": ("return word_offset % NUM_BANKS",
                               "return word_offset % 16"),
}


def _run_pins(env):
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p",
                           "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


def _mutate(name, tmp_path):
    old, new, *which = MUTANTS[name]
    text = open(SRC).read()
    if which:
        assert text.count(old) > which[0], f"mutation site for {name} missing"
        at = -1
        for _ in range(which[0] + 1):
            at = text.index(old, at + 1)
        text = text[:at] + new + text[at + len(old):]
    else:
        assert text.count(old) == 1, f"mutation site for {name} not unique"
        text = text.replace(old, new)
    if "M_" in new:  # the transposed index needs M inside oracle_row
        head = "static void oracle_row(const float *A, const float *B, int64_t N, int64_t K,"
        text = text.replace(head, "static int64_t M_ = 1;\n" + head)
        text = text.replace("if (nrows == 0 || N == 0) return 0;",
                            "if (nrows == 0 || N == 0) return 0;\n    M_ = M;")
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    return oracle.build(force=True, src=str(src), out=str(tmp_path / f"lib{name}.so"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    lib = _mutate(name, tmp_path)
    env = dict(os.environ, MT_ORACLE_LIB=lib, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p",
                        "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


@pytest.mark.parametrize("name", sorted(RULE_MUTANTS))
def test_pins_catch_rule_mutant(name, tmp_path):
    old, new = RULE_MUTANTS[name]
    text = open(RULES).read()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / f"rules_{name}.py"
    src.write_text(text.replace(old, new))
    r = _run_pins(dict(os.environ, MT_ORACLE_RULES=str(src)))
    # A failed pin, not a copy that does not even load.
    assert r.returncode == 1 and " failed" in r.stdout, r.stdout[-2000:]


def test_unmutated_copy_passes(tmp_path):
    # Control: the same procedure without an edit must pass.
    src = tmp_path / "same.c"
    src.write_text(open(SRC).read())
    lib = oracle.build(force=True, src=str(src), out=str(tmp_path / "libsame.so"))
    rules = tmp_path / "rules_same.py"
    rules.write_text(open(RULES).read())
    env = dict(os.environ, MT_ORACLE_LIB=lib, MT_ORACLE_RULES=str(rules),
               OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p",
                        "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
