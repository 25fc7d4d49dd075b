"""Each plausible mistake planted in a copy of the oracle's C source (on the
CPU) must fail at least one pin: the pins are strong enough to notice it."""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle
import oracle_pins as pins

# (name, text in pgemm_oracle.c, replacement, which occurrence (0-based))
MUTANTS = [
    ("f32 rows drop first k", "for (int k = 0; k < K; ++k)", "for (int k = 1; k < K; ++k)", 0),
    ("f32 rows drop last k (missing epilogue tile)", "for (int k = 0; k < K; ++k)",
     "for (int k = 0; k < K - 1; ++k)", 0),
    ("bf16 rows transposed A", "bf16_bits_to_double(A[(size_t)i * K + k])",
     "bf16_bits_to_double(A[(size_t)k * M + i])", 0),
    ("f32 rows wrong B column", "(double)B[(size_t)k * N + j]", "(double)B[(size_t)k * N + (N - 1 - j)]", 0),
    ("f32 entries B indexed with A's leading dimension", "(double)B[(size_t)k * N + j]",
     "(double)B[((size_t)k * K + j) % ((size_t)K * N)]", 1),
    ("f32 rows beta sign", "out += b * (double)C_in", "out -= b * (double)C_in", 0),
    ("bf16 entries beta dropped", "if (beta != 0.0f) o += b *", "if (0) o += b *", 1),
    ("f32 rows reads C when beta == 0", "if (beta != 0.0f) out += b *", "out += b *", 0),
    ("i8 rows alpha ignored", "uint64_t out = (uint64_t)(int64_t)alpha * (uint64_t)s;",
     "uint64_t out = (uint64_t)s;", 0),
    ("i8 entries int8 read as unsigned", "s += (int64_t)A[(size_t)i * K + k]",
     "s += (int64_t)(uint8_t)A[(size_t)i * K + k]", 1),
    ("i8 saturates instead of wrapping", "uint32_t lo = (uint32_t)(v & 0xffffffffu);",
     "int64_t sv = (int64_t)v; uint32_t lo = (uint32_t)(sv > 2147483647LL ? 2147483647LL : "
     "(sv < -2147483648LL ? -2147483648LL : sv));", 0),
    ("f32 rows float accumulator", "double s = 0.0;", "float s = 0.0f;", 0),
    ("bf16 widening wrong shift", "((uint32_t)h) << 16", "((uint32_t)h) << 8", 0),
    ("f32 entries alpha applied to C too", "double o = a * s;\n        if (beta != 0.0f) o += b *",
     "double o = a * s;\n        if (beta != 0.0f) o += a * b *", 0),
    ("f32 output truncated toward zero",
     "C_out[(size_t)i * N + j] = (float)out;",
     "{ float f_ = (float)out; if ((double)f_ != out && ((double)f_ > out) == (out > 0)) "
     "f_ = nextafterf(f_, 0.0f); C_out[(size_t)i * N + j] = f_; }", 0),
]


def _plant(src: str, old: str, new: str, which: int) -> str:
    pos = -1
    for _ in range(which + 1):
        pos = src.find(old, pos + 1)
        assert pos >= 0, f"oracle source no longer contains occurrence {which} of {old!r}"
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name,old,new,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, which):
    with open(oracle.SOURCE) as f:
        src = f.read()
    mutated = _plant(src, old, new, which)
    if "nextafterf" in mutated:
        mutated = "#include <math.h>\n" + mutated
    with tempfile.TemporaryDirectory() as d:
        c_path = os.path.join(d, "mutant.c")
        with open(c_path, "w") as f:
            f.write(mutated)
        lib = oracle.compile_oracle(c_path, os.path.join(d, "libmutant.so"), extra=("-lm",))
        # run the pins in a child process: a mutant may crash (e.g. read a NULL C),
        # which counts as caught
        here = os.path.dirname(os.path.abspath(__file__))
        code = ("import sys; sys.path[:0] = [%r, %r]\n"
                "import oracle, oracle_pins as pins\n"
                "bad = pins.run_all(oracle.Oracle(%r))\n"
                "print(sorted(bad)); sys.exit(3 if bad else 0)\n"
                % (here, os.path.dirname(here), lib))
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                           timeout=600)
    # 3: at least one pin failed; negative: the mutant crashed the child
    assert r.returncode == 3 or r.returncode < 0, \
        f"no pin noticed the planted mistake: {name} (rc={r.returncode})\n{r.stdout}{r.stderr}"
