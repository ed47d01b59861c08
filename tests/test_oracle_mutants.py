"""Plant plausible mistakes in copies of the oracle; the pins must catch each.

Every mutant is a textual edit of oracle.c compiled into a temporary library
on the CPU.  The product library is not involved.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pin_checks as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, mutated text); each original must occur in oracle.c
MUTANTS = [
    ("bias_sign", "if (b) z += (double)b[n];", "if (b) z -= (double)b[n];"),
    ("dropped_last_k", "for (int64_t k = 0; k < K; ++k) s += (double)x[k] * (double)w[k];",
     "for (int64_t k = 0; k + 1 < K; ++k) s += (double)x[k] * (double)w[k];"),
    ("gelu_scale", "erf(z / sqrt(2.0))", "erf(z / 2.0)"),
    ("gelu_tanh_form", "return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));",
     "return 0.5 * z * (1.0 + tanh(0.7978845608028654 * (z + 0.044715 * z * z * z)));"),
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("bf16_7_bits", "ldexp(nearbyint(ldexp(m, 8)), e - 8)", "ldexp(nearbyint(ldexp(m, 7)), e - 7)"),
    ("bf16_truncate", "ldexp(nearbyint(ldexp(m, 8)), e - 8)", "ldexp(floor(ldexp(m, 8)), e - 8)"),
    ("column_shard_offset", "const float* Wi = W + (int64_t)i * ns * ldw;",
     "const float* Wi = W + (int64_t)i * ns;"),
    ("column_concat_offset", "double* Yi = Y + (int64_t)i * ns;", "double* Yi = Y;"),
    ("row_input_slice", "int rc = orc_linear(M, ks, N, X + (int64_t)i * ks, ldx,",
     "int rc = orc_linear(M, ks, N, X, ldx,"),
    ("row_bias_per_shard", "W + (int64_t)i * ks, ldw, NULL, ORC_ACT_NONE, part, N);",
     "W + (int64_t)i * ks, ldw, b, ORC_ACT_NONE, part, N);"),
    ("qkv_kv_group", "(int64_t)H * hd + (int64_t)i * hk * hd,", "(int64_t)H * hd,"),
    ("swiglu_swapped", "Y[m * ldy + n] = orc_silu(g) * u;", "Y[m * ldy + n] = orc_silu(u) * g;"),
    ("h_not_rounded", "if (round_h) h[j] = orc_round_bf16(h[j]);", "(void)round_h;"),
    ("ring_direction", "const int r = (c + s) % tp;", "const int r = (c + tp - s) % tp;"),
    ("ring_no_hop_rounding", "acc = wire_bf16 ? orc_round_bf16(acc) : orc_round_f32(acc);", ";"),
    ("ring_chunk_start_rank0", "double acc = part[(int64_t)c * L + e];", "double acc = part[e];"),
    ("e4m3_3_bits", "r = ldexp(nearbyint(ldexp(m, 4)), e - 4);", "r = ldexp(nearbyint(ldexp(m, 3)), e - 3);"),
    ("e4m3_no_saturation", "if (r > 448.0) r = 448.0;", ";"),
    ("fp8_scale_e5m2_max", "const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;",
     "const float sc = amax > 0.0f ? amax / 57344.0f : 1.0f;"),
    ("fp8_row_scale_shard0", "y += (double)S[(int64_t)i * N + n] *", "y += (double)S[n] *"),
    ("fp8_column_scale_dropped", "double z = (double)S[n] * dot(K, X + m * ldx, Q + n * ldq);",
     "double z = dot(K, X + m * ldx, Q + n * ldq);"),
    ("ring_partial_not_rounded",
     "for (int64_t e = 0; e < L; ++e) pi[e] = wire_bf16 ? orc_round_bf16(pi[e]) : orc_round_f32(pi[e]);",
     ";"),
    # the fp32 wire of the ring kept in fp64
    ("round_f32_identity", "double orc_round_f32(double x) { return (double)(float)x; }",
     "double orc_round_f32(double x) { return x; }"),
    # the FP8 quotient W / s taken in fp64 instead of fp32
    ("fp8_quotient_fp64", "const float v = W[r * ldw + c] / sc; /* fp32 division */",
     "const double v = (double)W[r * ldw + c] / (double)sc;"),
    # the FP8 row scale one fp32 ulp off
    ("fp8_scale_one_ulp", "const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;",
     "const float sc = amax > 0.0f ? nextafterf(amax / 448.0f, 1e30f) : 1.0f;"),
    # the sampled-rows ring: chunk of the sampled row's own index, not the full call's
    ("ring_rows_local_chunk", "const int64_t e = rows[r] * N + n;", "const int64_t e = r * N + n;"),
    ("ring_rows_no_hop_rounding",
     "        acc += p[(c + s) % tp];\n        acc = wire_bf16 ? orc_round_bf16(acc) : orc_round_f32(acc);",
     "        acc += p[(c + s) % tp];"),
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, orig, mut):
    src = open(SRC).read()
    assert orig in src, f"mutation site for {name} not found"
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(src.replace(orig, mut, 1))
    lib = tmp_path / f"liboracle_{name}.so"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                    str(path), "-o", str(lib), "-lm"], check=True)
    res = pins.run_all(oracle.Oracle(str(lib)))
    failed = [k for k, v in res.items() if v is not None]
    assert failed, f"mutant {name} passed every pin"
