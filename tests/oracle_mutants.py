"""Deliberate mistakes to plant in a copy of the oracle's C source (never in
the oracle itself), one at a time: each is (name, exact source text, its
replacement).  tests/test_oracle_mutations.py builds every copy and checks
that the oracle's pins fail on it -- evidence that the pins would catch that
kind of slip (a dropped term, a wrong sign, index, bias or rounding rule, a
transposed operand)."""

MUTANTS = [
    # number formats
    ("e2m1 exponent bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)"),
    ("e2m1 subnormal step", "(e == 0) ? 0.5 * m :", "(e == 0) ? 1.0 * m :"),
    ("e4m3 exponent bias", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    ("e4m3 subnormal exponent", "ldexp(m / 8.0, -6)", "ldexp(m / 8.0, -7)"),
    ("e4m3 ties to odd", "(d == bestd && (b & 1) == 0 && (best & 1) == 1)",
     "(d == bestd && (b & 1) == 1 && (best & 1) == 0)"),
    ("e4m3 saturates to NaN", "return 0x7E; /* saturate", "return 0x7F; /* saturate"),
    ("e2m1 ties to odd", "(d == bestd && (c & 1) == 0 && (best & 1) == 1)",
     "(d == bestd && (c & 1) == 1 && (best & 1) == 0)"),
    ("e2m1 drops the sign of zero", "return best | (signbit(q) ? 8 : 0);",
     "return best | ((signbit(q) && best) ? 8 : 0);"),
    ("bf16 truncates", "rint(ldexp(v, -qexp))", "trunc(ldexp(v, -qexp))"),
    # quantiser
    ("absmax of signed values", "if (ax > amax)\n            amax = ax;", "if (x > amax)\n            amax = x;"),
    ("global scale divisor", "return amax / 2688.0f;", "return amax / 2689.0f;"),
    ("block amax of signed values", "if (fabsf(x[i]) > amax_b)\n                    amax_b = fabsf(x[i]);",
     "if (x[i] > amax_b)\n                    amax_b = x[i];"),
    ("block scale drops the 6", "float t = amax_b / six_g;", "float t = amax_b / g;"),
    ("decode step drops g", "float d = (float)oracle_e4m3_value(s) * g;",
     "float d = (float)oracle_e4m3_value(s);"),
    ("quotient by a reciprocal", "float q = x[i] / d;", "float q = x[i] * (1.0f / d);"),
    ("fp8 quotient by a reciprocal", "const float q = v / s; /* binary32 division */",
     "const float q = v * (1.0f / s);"),
    ("e2m1 saturates to 4", "return 7 | (signbit(q) ? 8 : 0); /* saturate */",
     "return 6 | (signbit(q) ? 8 : 0); /* saturate */"),
    ("zero step gives nonzero codes", "if (d == 0.0f) {\n                    codes[i] = 0;",
     "if (d == 0.0f) {\n                    codes[i] = 8;"),
    ("e4m3 ties to the larger code", "if (d < bestd || (d == bestd && (b & 1) == 0 && (best & 1) == 1)) {",
     "if (d <= bestd) {"),
    ("e4m3 search skips 448", "for (int b = 1; b <= 0x7E; ++b) {", "for (int b = 1; b < 0x7E; ++b) {"),
    ("block stride 8", "x[i] = oracle_bf16_to_float(row[b * 16 + i]);", "x[i] = oracle_bf16_to_float(row[b * 8 + i]);"),
    ("bf16 subnormal floor", "if (qexp < -133)\n        qexp = -133;", "if (qexp < -126)\n        qexp = -126;"),
    ("codes packed high nibble first", "(uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));",
     "(uint8_t)(codes[2 * j + 1] | (codes[2 * j] << 4));"),
    # dequantisation
    ("dequant nibble order", "int code = (i & 1) ? (byte >> 4) : (byte & 15);",
     "int code = (i & 1) ? (byte & 15) : (byte >> 4);"),
    ("dequant scale index", "int s = scales[row * (k / 16) + i / 16];",
     "int s = scales[row * (k / 16) + i / 32];"),
    ("dequant drops g", "return (double)g * oracle_e4m3_value(s) * oracle_e2m1_value(code);",
     "return oracle_e4m3_value(s) * oracle_e2m1_value(code);"),
    # RMSNorm
    ("rmsnorm sum instead of mean", "sqrt(ss / (double)ks + (double)eps)", "sqrt(ss + (double)eps)"),
    ("rmsnorm eps outside the root", "1.0 / sqrt(ss / (double)ks + (double)eps)",
     "1.0 / (sqrt(ss / (double)ks) + (double)eps)"),
    ("rmsnorm ignores gamma", "* r *\n                   (double)oracle_bf16_to_float(gamma[i]);", "* r;"),
    ("rmsnorm offset gamma", "* r *\n                   (double)oracle_bf16_to_float(gamma[i]);",
     "* r *\n                   (1.0 + (double)oracle_bf16_to_float(gamma[i]));"),
    # GEMV / GEMM
    ("gemv ignores the row offset", "dequant_one(packed, scales, g, k, n0 + j, i);\n                acc += p;",
     "dequant_one(packed, scales, g, k, j, i);\n                acc += p;"),
    ("gemv signed error scale", "acc += p;\n                aacc += fabs(p);\n            }\n            y[r * nn + j] = acc;\n"
     "            sabs[r * nn + j] = aacc;\n        }\n    }\n}\n\n/* Greedy",
     "acc += p;\n                aacc += p;\n            }\n            y[r * nn + j] = acc;\n"
     "            sabs[r * nn + j] = aacc;\n        }\n    }\n}\n\n/* Greedy"),
    ("dequant in binary32", "return (double)g * oracle_e4m3_value(s) * oracle_e2m1_value(code);",
     "return (double)(g * (float)oracle_e4m3_value(s) * (float)oracle_e2m1_value(code));"),
    ("gemv accumulates in binary32", "double acc = 0.0, aacc = 0.0;\n            for (int64_t i = 0; i < k; ++i) {\n"
     "                double p = (double)oracle_bf16_to_float(a[r * lda + i]) *\n                           dequant_one",
     "float acc = 0.0, aacc = 0.0;\n            for (int64_t i = 0; i < k; ++i) {\n"
     "                double p = (double)oracle_bf16_to_float(a[r * lda + i]) *\n                           dequant_one"),
    ("gemm transposed operand", "dequant_one(packed, scales, g, k, cols[p], i);",
     "dequant_one(packed, scales, g, k, rows[p], i);"),
    ("gemm activation row", "A[rows[p] * lda + i]", "A[cols[p] * lda + i]"),
    # argmax, mask, log-probability
    ("argmax ties to the highest index", "        if (y[i] > bestv) {\n            bestv = y[i];\n            best = i;\n"
     "        }\n    }\n    return best;",
     "        if (y[i] >= bestv) {\n            bestv = y[i];\n            best = i;\n"
     "        }\n    }\n    return best;"),
    ("masked argmax bit order", "if (word >= nwords || ((mask[word] >> (i % 32)) & 1) == 0)\n                continue;\n"
     "        }\n        any = 1;\n        if (y[i] > bestv)",
     "if (word >= nwords || ((mask[word] >> (31 - i % 32)) & 1) == 0)\n                continue;\n"
     "        }\n        any = 1;\n        if (y[i] > bestv)"),
    ("masked argmax reads words past the mask", "if (word >= nwords || ((mask[word] >> (i % 32)) & 1) == 0)\n"
     "                continue;\n        }\n        any = 1;\n        if (y[i] > bestv)",
     "if (word < nwords && ((mask[word] >> (i % 32)) & 1) == 0)\n"
     "                continue;\n        }\n        any = 1;\n        if (y[i] > bestv)"),
    ("log-prob sums disallowed tokens", "    double s = 0.0;\n    for (int64_t i = 0; i < n; ++i) {\n        if (mask != NULL) {",
     "    double s = 0.0;\n    for (int64_t i = 0; i < n; ++i) {\n        if (0) {"),
    ("log-prob drops the shift", "return y[idx] - (mx + log(s));", "return y[idx] - log(s);"),
    ("argmax lets NaN win", "        if (y[i] > bestv) {\n            bestv = y[i];\n            best = i;\n"
     "        }\n    }\n    return best;",
     "        if (!(y[i] <= bestv)) {\n            bestv = y[i];\n            best = i;\n"
     "        }\n    }\n    return best;"),
    ("log-prob uses log1p", "return y[idx] - (mx + log(s));", "return y[idx] - (mx + log1p(s));"),
    # FP8 weights
    ("fp8 scale divisor", "const float s = amax / 448.0f;", "const float s = amax / 240.0f;"),
    ("fp8 drops the sign of zero", "(signbit(v) ? 0x80 : 0)", "(v < 0.0f ? 0x80 : 0)"),
    ("fp8 decode drops the sign", "return (byte & 0x80) ? -v : v;", "return v;"),
    ("fp8 drops the sign", "codes[r * k + i] = (uint8_t)(mag | (signbit(v) ? 0x80 : 0));",
     "codes[r * k + i] = (uint8_t)mag;"),
    ("fp8 zero row codes", "if (s == 0.0f) {\n                codes[r * k + i] = 0;",
     "if (s == 0.0f) {\n                codes[r * k + i] = 0x80;"),
    ("fp8 gemv drops the row scale", "(oracle_fp8_value(codes[(n0 + j) * k + i]) * s);",
     "(oracle_fp8_value(codes[(n0 + j) * k + i]));"),
]
