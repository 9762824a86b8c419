"""Plant plausible mistakes in copies of the oracle source and check that the
pins in test_oracle.py catch each one (CPU only; the real oracle is untouched)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gemm_oracle.c")

MUTATIONS = {
    "B read as if never transposed": ("J->transB ? j * J->ldb + k : k * J->ldb + j",
                                      "J->transB ? k * J->ldb + j : k * J->ldb + j"),
    "A index transposed": ("J->transA ? k * J->lda + i : i * J->lda + k",
                           "J->transA ? i * J->lda + k : k * J->lda + i"),
    "last k term dropped": ("for (int64_t k = 0; k < J->K; ++k)", "for (int64_t k = 0; k + 1 < J->K; ++k)"),
    "beta term sign flipped": ("rv += J->beta * c0;", "rv -= J->beta * c0;"),
    "alpha dropped": ("double rv = J->alpha * s;", "double rv = s;"),
    "fp16 exponent bias off by one": ("e - 15);", "e - 16);"),
    "bf16 fraction width wrong": ("1.0 + (double)f / 128.0", "1.0 + (double)f / 256.0"),
    "C0 leading dimension ignored": ("i * J->ldc + j", "i * J->N + j"),
    "E4M3 exponent bias off by one": ("e - 7);", "e - 8);"),
    "E4M3 NaN rule too wide": ("e == 0xF && f == 0x7", "e == 0xF"),
    "E5M2 fraction width wrong": ("1.0 + (double)f / 4.0", "1.0 + (double)f / 8.0"),
    "E5M2 subnormal scale wrong": ("(double)f / 4.0, -14)", "(double)f / 4.0, -15)"),
    "B decoded with A's type": ("in_value(J->b_type, J->B", "in_value(J->a_type, J->B"),
    "GELU argument not divided by sqrt 2": ("erf(z / sqrt(2.0))", "erf(z)"),
    "ReLU passes negatives": ("d = z > 0.0 ? z : 0.0;", "d = z > 0.0 ? z : -z;"),
    "bias indexed by row": ("z += (double)bias[j];", "z += (double)bias[i % N];"),
    "output scale dropped": ("R[i * ldr + j] = scale * d;", "R[i * ldr + j] = d;"),
    "B batch stride ignored": ("(const char*)B + b * strideB * eb", "(const char*)B"),
    "C0 batch offset ignored": ("(const char*)C0 + b * strideC * ec", "(const char*)C0"),
    "group weights not advanced": ("(const char*)B + g * strideB * eb", "(const char*)B"),
    "group rows not offset": ("(const char*)A + off * lda * ea", "(const char*)A"),
    "fp32 read at the 16-bit width": ("in_type == ORACLE_IN_F32 ? 4 : 2", "in_type == ORACLE_IN_F32 ? 2 : 2"),
    "scale block size doubled": ("k / J->block]", "k / (2 * J->block)]"),
    "FP4 nibble order swapped": ("(idx & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF)",
                                 "(idx & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4)"),
    "E8M0 bias off by one": ("ldexp(1.0, (int)x - 127)", "ldexp(1.0, (int)x - 128)"),
    "E2M1 exponent bias dropped": ("ldexp(1.0 + (double)f / 2.0, e - 1)", "ldexp(1.0 + (double)f / 2.0, e)"),
    "UE4M3 sign bit kept": ("oracle_e4m3_value((uint8_t)(x & 0x7F))", "oracle_e4m3_value(x)"),
    "B scaled by A's factors": ("J->SFB[j * J->ld_sfb", "J->SFA[i * J->ld_sfa"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, repo_tmp):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation site not found: %s" % old
    mutated = repo_tmp / "mut.c"
    mutated.write_text(src.replace(old, new))
    lib = repo_tmp / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", str(mutated),
                    "-o", str(lib), "-lpthread", "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True)
    assert r.returncode != 0, "the pins did not catch: %s" % name
