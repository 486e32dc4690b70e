"""Planted mistakes: each case copies the CPU oracle, plants one plausible slip
in the copy's C source (a swapped nibble, a wrong rounding rule, a dropped or
sign-flipped term, a transposed operand, ...) or in its Python KV-cache layer
(a wrong position, head or query), rebuilds it, and runs the pins
of tests/test_oracle_pins.py that should catch it against the mutant.  The
pins pass on the real oracle (that file's own run); here every mutant must
make at least one of them fail.

The mutant lives in a temporary directory and is imported as ``oracle`` by a
child pytest process started there, with that directory ahead of the
repository on its path (checked before the run); the real oracle is never
modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")

# (name, original text in gq_oracle.c, planted text, -k selection of the pins)
MUTANTS = [
    ("q4_0 nibble order swapped",
     "blk[2 + j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));",
     "blk[2 + j] = (uint8_t)(c[2 * j + 1] | (c[2 * j] << 4));",
     "q4_0_worked_example"),
    ("q4_0 scale max/8 instead of max/7",
     "uint16_t dh = or_f16_rn(amax / 7.0f);",
     "uint16_t dh = or_f16_rn(amax / 8.0f);",
     "q4_0_worked_example"),
    ("codes rounded half to even",
     "static float rha(float v) { return roundf(v); }",
     "static float rha(float v) { return rintf(v); }",
     "ties or rounding_illustration"),
    ("fp16 scale ties rounded away from zero",
     "round_up = rem > half || (rem == half && (q & 1));",
     "round_up = rem >= half;",
     "f16_rn_sweep"),
    ("q4_k min added instead of subtracted",
     "out[e] = d * (double)f[j] * (double)q - dmin * (double)f[8 + j];",
     "out[e] = d * (double)f[j] * (double)q + dmin * (double)f[8 + j];",
     "q4_k_handmade"),
    ("q4_k min term of the product sign-flipped",
     "double t2 = -(dx * dmin * (double)s[1]);",
     "double t2 = (dx * dmin * (double)s[1]);",
     "bruteforce"),
    ("q4_k min term dropped from the integer sums",
     "S2 += (int32_t)f[8 + j] * (int32_t)t;",
     "S2 += 0;",
     "integer_special_case_q4_k"),
    ("q4_k 6-bit fields packed MSB-first",
     "if ((f[k] >> b) & 1) out[bit / 8] |= (uint8_t)(1u << (bit % 8));",
     "if ((f[k] >> (5 - b)) & 1) out[bit / 8] |= (uint8_t)(1u << (bit % 8));",
     "q4_k_handmade"),
    ("q8_k sub-block sums over the wrong elements",
     "for (int i = 0; i < 32; i++) s += q[32 * j + i];",
     "for (int i = 0; i < 32; i++) s += q[8 * j + i];",
     "roundtrip_symmetric"),
    ("q6_k top bits in reversed order",
     "for (int k = 0; k < 4; k++) h |= (c[4 * l + k] >> 4) << (2 * k);",
     "for (int k = 0; k < 4; k++) h |= (c[4 * l + k] >> 4) << (6 - 2 * k);",
     "q6_k_handmade"),
    ("q6_k scale max/32 instead of max/31",
     "uint16_t dh = or_f16_rn(amax / 31.0f);",
     "uint16_t dh = or_f16_rn(amax / 32.0f);",
     "q6_k_handmade"),
    ("q6_k code offset 31 in the integer dot",
     "s += (q6_k_code(w, e) - 32) * (int8_t)a[4 + e];",
     "s += (q6_k_code(w, e) - 31) * (int8_t)a[4 + e];",
     "integer_special_case_q6_k"),
    ("q6_k activation scale read as fp16",
     "double dw = or_f16_to_f32(get_u16(w));\n        double dx = get_f32(a);\n        double t = dw",
     "double dw = or_f16_to_f32(get_u16(w));\n        double dx = or_f16_to_f32(get_u16(a));\n        double t = dw",
     "bruteforce"),
    ("q5_k fifth bits packed in the wrong bit positions",
     "if (q[e] >> 4) blk[144 + 4 * j + i] |= (uint8_t)(1u << (2 * t + p));",
     "if (q[e] >> 4) blk[144 + 4 * j + i] |= (uint8_t)(1u << (t + 4 * p));",
     "q5_k_handmade"),
    ("q5_k fit with 30 code steps instead of 31",
     "k_asym_fit(x, 31.0f, &dh, &dminh, fields, q);",
     "k_asym_fit(x, 30.0f, &dh, &dminh, fields, q);",
     "q5_k_handmade"),
    ("q5_k fifth bit weighted 8 instead of 16 when read",
     "q |= ((blk[144 + 4 * j + i] >> (2 * t + p)) & 1) << 4;",
     "q |= ((blk[144 + 4 * j + i] >> (2 * t + p)) & 1) << 3;",
     "integer_special_case_q5_k"),
    ("error-minimizing search window of zero",
     "#define EM_WINDOW 4",
     "#define EM_WINDOW 0",
     "errmin"),
    ("error-minimizing search scores absolute instead of squared errors",
     "acc = acc + e * e;",
     "acc = acc + fabsf(e);",
     "errmin_window_bruteforce"),
    ("error-minimizing search keeps the last candidate tried",
     "if (e < best) {",
     "if (1) {",
     "errmin"),
    ("q8_0 scale max/128 instead of max/127",
     "uint16_t dh = or_f16_rn(amax / 127.0f);",
     "uint16_t dh = or_f16_rn(amax / 128.0f);",
     "q8_0_ties"),
    ("q8_k scale rounded to fp16",
     "float d = amax / 127.0f;",
     "float d = or_f16_to_f32(or_f16_rn(amax / 127.0f));",
     "rounding_illustration or roundtrip_symmetric"),
    ("q4_k dmin rounded to nearest instead of up",
     "uint16_t dminh = or_f16_ru(neg_lo_max / 63.0f);",
     "uint16_t dminh = or_f16_rn(neg_lo_max / 63.0f);",
     "q4_k"),
    ("product written transposed (batch and rows swapped)",
     "y[b * rows + r] = acc;",
     "y[r * batch + b] = acc;",
     "bruteforce"),
]


# Slips in the oracle's Python layer (the KV-cache functions over the C codec).
PY_MUTANTS = [
    ("kv append writes the next position",
     "cache[h, pos] = quantize(t, x[h]).reshape(-1)",
     "cache[h, min(pos + 1, cache.shape[1] - 1)] = quantize(t, x[h]).reshape(-1)",
     "kv_append"),
    ("kv append quantizes every head with head 0's values",
     "cache[h, pos] = quantize(t, x[h]).reshape(-1)",
     "cache[h, pos] = quantize(t, x[0]).reshape(-1)",
     "kv_append"),
    ("kv scores pair every head's keys with head 0's query",
     "qq = quantize(Q8_0, q[h:h + 1])",
     "qq = quantize(Q8_0, q[0:1])",
     "kv_scores"),
    ("kv scores skip the first position",
     "y, tt = matmul_ref(t, cache[h, :n_pos], qq, n_pos, head_dim, 1)",
     "y, tt = matmul_ref(t, cache[h, 1:n_pos + 1], qq, n_pos, head_dim, 1)",
     "kv_scores"),
]


@pytest.mark.parametrize("name,orig,planted,pins,layer",
                         [m + ("c",) for m in MUTANTS] + [m + ("py",) for m in PY_MUTANTS],
                         ids=[m[0] for m in MUTANTS + PY_MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, orig, planted, pins, layer):
    c_src = open(os.path.join(ORACLE, "gq_oracle.c"), encoding="utf-8").read()
    py_src = open(os.path.join(ORACLE, "__init__.py"), encoding="utf-8").read()
    src = c_src if layer == "c" else py_src
    assert src.count(orig) == 1, f"mutation site not unique or missing: {orig!r}"
    if layer == "c":
        c_src = c_src.replace(orig, planted)
    else:
        py_src = py_src.replace(orig, planted)
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(py_src, encoding="utf-8")
    (pkg / "gq_oracle.c").write_text(c_src, encoding="utf-8")
    # the mutant must compile (a build error must not pass for a caught mistake)
    (pkg / "_build").mkdir()
    cc = subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-std=c11",
                         "-shared", "-fPIC", str(pkg / "gq_oracle.c"), "-o", str(pkg / "_build" / "liboracle.so"),
                         "-lm"], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([str(tmp_path), ROOT]))
    # and it must be the oracle the child processes import
    where = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__)"], cwd=tmp_path, env=env,
                           capture_output=True, text=True)
    assert where.stdout.strip().startswith(str(tmp_path)), where.stdout + where.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-k", pins],
                       cwd=tmp_path, env=env, capture_output=True, text=True, timeout=600)
    out = r.stdout + r.stderr
    assert r.returncode == 1 and " failed" in out, f"planted mistake not caught: {name}\n{out[-2000:]}"
