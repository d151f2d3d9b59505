"""Strength of the oracle's pins: plant a plausible mistake in a copy of the
oracle's C source (a wrong index, a dropped term, a wrong sign, a transposed
operand), build the copy, and check that at least one pin of
tests/test_oracle.py fails against it.  Runs on the CPU only; each mutant runs
in its own process, since a planted indexing mistake may crash it."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pa_oracle.c")

# (name, text in the oracle, planted replacement)
MUTANTS = [
    ("offset_in_block", "(phys * Hkv + kvh) * bs + (j % bs)", "(phys * Hkv + kvh) * bs + ((j + 1) % bs)"),
    ("logical_block", "int64_t phys = bt_row[lb];", "int64_t phys = bt_row[lb > 0 ? lb - 1 : 0];"),
    ("no_max_subtraction", "double p = exp(s[j] - m);", "double p = exp(s[j]);"),
    ("scale_dropped", "s[j] = scale * acc;", "s[j] = acc;"),
    ("no_normalisation", "        o[c] /= l;\n    *m_out", "        (void)0;\n    *m_out"),
    ("k_for_v", "o[c] += p * V[(int64_t)j * d + c];", "o[c] += p * K[(int64_t)j * d + c];"),
    ("gqa_mapping", "int kvh = h / group;", "int kvh = h % Hkv;"),
    ("lse_sign", "double w = pl[p] * exp(pm[p] - M);", "double w = pl[p] * exp(M - pm[p]);"),
    ("lse_combine_weight", "double w = l[(int64_t)k * P + p] * exp(m[(int64_t)k * P + p] - M);",
     "double w = exp(m[(int64_t)k * P + p] - M);"),
    ("scatter_offset", "int64_t blk = s / bs, off = s % bs;", "int64_t blk = s / bs, off = (s + 1) % bs;"),
    ("scatter_head", "key + t * key_stride + (int64_t)h * d", "key + t * key_stride"),
    ("fp16_bias", "v = ldexp((double)(f + 1024), e - 25);", "v = ldexp((double)(f + 1024), e - 24);"),
    ("fp16_subnormal", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("bf16_bias", "v = ldexp((double)(f + 128), e - 134);", "v = ldexp((double)(f + 128), e - 133);"),
    ("partition_start", "int j0 = p * partition_size;", "int j0 = p * partition_size + (p > 0);"),
    ("first_token_dropped", "    for (int j = 0; j < n; ++j) {\n        double p", "    for (int j = 1; j < n; ++j) {\n        double p"),
    ("query_head", "const uint16_t *qrow = query + ((int64_t)i * Hq + h) * d;",
     "const uint16_t *qrow = query + ((int64_t)i * Hq + (h ^ 1) % Hq) * d;"),
    ("e4m3_ties_up", "(frac == 0.5 && fmod(r, 2.0) == 1.0)", "(frac == 0.5)"),
    ("e4m3_bias", "v = ldexp((double)(f + 8), e - 10);", "v = ldexp((double)(f + 8), e - 9);"),
    ("e4m3_late_saturation", "if (a >= 448.0)", "if (a >= 480.0)"),
    ("fp8_k_scale_dropped", "int rc = pa_oracle_gather(K, k_cache, kv_dtype, k_scale,",
     "int rc = pa_oracle_gather(K, k_cache, kv_dtype, 1.0,"),
    ("fp8_scatter_scale", "/ k_scale;", "* k_scale;"),
    ("prefill_not_causal_inclusive", "int n = pos + 1;", "int n = pos;"),
    ("prefill_position", "int pos = ctx - q_len + (row - query_start[i]);",
     "int pos = ctx - q_len + (row - query_start[i]) / 2;"),
    ("prefill_fp8_k_with_v_scale", "rc = pa_oracle_gather(K, k_cache, kv_dtype, k_scale, bt_row, MB, n,",
     "rc = pa_oracle_gather(K, k_cache, kv_dtype, v_scale, bt_row, MB, n,"),
    ("prefill_fp8_v_as_query_type", "rc = pa_oracle_gather(V, v_cache, kv_dtype, v_scale, bt_row, MB, n,",
     "rc = pa_oracle_gather(V, v_cache, dtype, v_scale, bt_row, MB, n,"),
]

RUNNER = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle
oracle._lib = oracle._load(sys.argv[1])
import test_oracle as T
for pin in T.PINS:
    try:
        pin()
    except Exception as e:
        print("CAUGHT", pin.__name__, type(e).__name__)
        sys.exit(3)
print("SURVIVED")
sys.exit(0)
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found in the oracle"
    with tempfile.TemporaryDirectory() as tmp:
        csrc = os.path.join(tmp, "mutant.c")
        so = os.path.join(tmp, "mutant.so")
        open(csrc, "w").write(src.replace(old, new, 1))
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", csrc, "-o", so,
                        "-lm"], check=True)
        runner = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
        r = subprocess.run([sys.executable, "-c", runner, so], capture_output=True, text=True,
                           timeout=600)
    assert r.returncode != 0, f"mutant {name} survived every pin:\n{r.stdout}\n{r.stderr[-2000:]}"
