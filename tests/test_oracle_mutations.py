"""Plant one plausible mistake at a time in a copy of the oracle (on the CPU)
and require that at least one pin catches it: the pins have teeth.

Each mutation is a textual substitution in the oracle's C source, compiled
with the oracle's own flags into a temporary library.
"""
import pytest

import oracle
import pins

# (name, original text, planted text, pins expected to catch it)
MUTATIONS = [
    ("philox multiplier 1 changed", "#define PHILOX_M1 0xCD9E8D57u", "#define PHILOX_M1 0xCD9E8453u",
     ["philox"]),
    ("philox key raised before the first round", "if (round > 0) {", "if (round >= 0) {",
     ["philox"]),
    ("philox products swapped", "uint32_t n0 = hi1 ^ c1 ^ k0;", "uint32_t n0 = hi0 ^ c1 ^ k0;",
     ["philox"]),
    ("philox key words swapped", "uint32_t n2 = hi0 ^ c3 ^ k1;", "uint32_t n2 = hi0 ^ c3 ^ k0;",
     ["philox"]),
    ("philox nine rounds", "round < 10;", "round < 9;", ["philox"]),
    ("element takes the wrong word", "return w[i & 3];", "return w[(i + 1) & 3];", ["mapping"]),
    ("step in counter word 3", "{ (uint32_t)q, (uint32_t)(q >> 32), step, 0u }",
     "{ (uint32_t)q, (uint32_t)(q >> 32), 0u, step }", ["mapping"]),
    ("counter is i not i>>2", "uint64_t q = i >> 2;", "uint64_t q = i;", ["mapping"]),
    ("sr uses the high random half", "uint32_t sum = u + (r & 0xFFFFu);",
     "uint32_t sum = u + (r >> 16);", ["sr"]),
    ("sr adds one bit too many", "uint32_t sum = u + (r & 0xFFFFu);",
     "uint32_t sum = u + (r & 0x1FFFFu);", ["sr"]),
    ("sr without the NaN rule", "    if (f32_is_nan_bits(u))\n        return (uint16_t)((u >> 16) | 0x0040u);\n    uint32_t sum = u + (r",
     "    uint32_t sum = u + (r", ["nan"]),
    ("rne ties away from zero", "uint32_t sum = u + 0x7FFFu + keep_lsb;", "uint32_t sum = u + 0x8000u;",
     ["rne"]),
    ("eps dropped", "float den = dq + ep;", "float den = dq;", ["adamw_special"]),
    ("eps inside the square root", "float rt = sqrtf(v1);", "float rt = sqrtf(v1 + ep);",
     ["adamw_special"]),
    ("first bias correction dropped", "out[6] = (float)(lr / (1.0 - pow(beta1, t)));", "out[6] = (float)lr;",
     ["adamw", "adamw_special"]),
    ("second bias correction dropped", "out[7] = (float)sqrt(1.0 - pow(beta2, t));", "out[7] = 1.0f;",
     ["adamw", "adamw_special"]),
    ("bias correction at t-1", "double t = (double)step;", "double t = (double)step + 1.0;",
     ["adamw", "adamw_special"]),
    ("weight decay with the wrong sign", "out[3] = (float)(1.0 - lr * wd);", "out[3] = (float)(1.0 + lr * wd);",
     ["adamw", "adamw_special"]),
    ("weight decay dropped", "float p1 = p * decay;", "float p1 = p;", ["adamw", "adamw_special"]),
    ("betas swapped in the first moment", "float bm = b1 * m;", "float bm = b2 * m;",
     ["adamw", "adamw_special"]),
    ("update added instead of subtracted", "float pn = p1 - upd;", "float pn = p1 + upd;",
     ["adamw", "adamw_special"]),
    ("gradient not squared", "float gg = g * g;", "float gg = g;", ["adamw", "adamw_special"]),
    ("old first moment written back", "exp_avg[j] = m1;", "exp_avg[j] = m;", ["adamw", "adamw_special"]),
    ("gemm reads B transposed", "(double)bf16_to_f32(b[j * k + t])", "(double)bf16_to_f32(b[t * n + j])",
     ["gemm"]),
    ("gemm drops the last product", "for (uint64_t t = 0; t < k; ++t)", "for (uint64_t t = 0; t + 1 < k; ++t)",
     ["gemm"]),
    ("gemm accumulates in binary32", "            double s = 0.0;", "            float s = 0.0f;", ["gemm"]),
    ("gemm keys by the slice row", "oracle_element_word((row0 + i) * n + j, step, seed)",
     "oracle_element_word(i * n + j, step, seed)", ["gemm"]),
    ("gemm keys by column-major index", "oracle_element_word((row0 + i) * n + j, step, seed)",
     "oracle_element_word(j * (row0 + m) + row0 + i, step, seed)", ["gemm"]),
    ("base_index ignored", "oracle_element_word(base_index + j, step, seed));\n            ((uint16_t",
     "oracle_element_word(j, step, seed));\n            ((uint16_t", ["dtype", "shards"]),
    ("betas swapped in the second moment", "float bv = b2 * v;", "float bv = b1 * v;",
     ["adamw", "adamw_special"]),
    ("old second moment written back", "exp_avg_sq[j] = v1;", "exp_avg_sq[j] = v;", ["adamw", "adamw_special"]),
    ("bias correction multiplied in", "float dq = rt / bc2s;", "float dq = rt * bc2s;", ["adamw", "adamw_special"]),
    ("rounding modes swapped", "uint16_t h = rounding == 1", "uint16_t h = rounding == 0", ["dtype"]),
]


def _run_pins(o, which, philox_ref):
    """Run the named pin groups; return the first AssertionError (or None)."""
    groups = {
        "philox": [lambda: pins.pin_philox_matches_reference(o, *philox_ref)],
        "mapping": [lambda: pins.pin_element_mapping(o, *philox_ref)],
        "sr": [lambda: pins.pin_sr_exhaustive(o, n_random=200)],
        "nan": [lambda: pins.pin_sr_inf_nan(o)],
        "rne": [lambda: pins.pin_rne_matches_torch(o)],
        "adamw": [lambda: pins.pin_adamw_textbook(o)],
        "adamw_special": [lambda: pins.pin_adamw_special_cases(o),
                          lambda: pins.pin_adamw_one_step_tight(o)],
        "dtype": [lambda: pins.pin_adamw_dtype_paths(o)],
        "shards": [lambda: pins.pin_shard_invariance(o)],
        "gemm": [lambda: pins.pin_gemm_exact_small(o), lambda: pins.pin_gemm_closed_forms(o)],
    }
    for g in which:
        for f in groups[g]:
            try:
                f()
            except AssertionError as e:
                return e
    return None


@pytest.mark.parametrize("name,old,new,catch", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, catch, tmp_path, philox_ref):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for '{name}' not found exactly once"
    o = oracle.compile_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    err = _run_pins(o, catch, philox_ref)
    assert err is not None, f"planted mistake '{name}' passed every pin in {catch}"
