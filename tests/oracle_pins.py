"""Pins for the CPU oracle: facts fixed by mathematics, not by the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` handle and returns a list
of failure strings (empty = pinned).  They are run against the real oracle in
``test_oracle.py`` and against deliberately broken copies of it in
``test_oracle_mutants.py``, which shows that a plausible mistake anywhere in
the oracle (a dropped term, a wrong sign or index, a transposed operand, a
wrong rounding or wrap) fails at least one pin.

The operation pinned is C_out = alpha * A @ B + beta * C_in with row-major
A (MxK), B (KxN), C (MxN), the kernel signature and output update of
"Double Buffering: Software Pipelining the K-Loop" (section "The Kernel").
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

BF16_ONE = np.uint16(0x3F80)


def _as_operand(dtype, x):
    """Exactly representable values -> operand array of the oracle's dtype."""
    x = np.asarray(x)
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "bf16":
        return si.to_bf16_bits(x.astype(np.float32))
    return x.astype(np.int8)


def _out_t(dtype):
    return np.int32 if dtype == "i8" else np.float32


def _all_paths(orc, dtype, A, B, C, alpha, beta):
    """Evaluate through every oracle entry point: full rows, a row sub-range
    stitched together, and entry-by-entry.  Returns the list of results."""
    M, N = A.shape[0], B.shape[1]
    res = [orc.gemm(dtype, A, B, C, alpha, beta)]
    if M >= 2:
        h = M // 2
        top = orc.gemm(dtype, A, B, C, alpha, beta, rows=(0, h))
        bot = orc.gemm(dtype, A, B, C, alpha, beta, rows=(h, M))
        res.append(np.concatenate([top, bot], axis=0))
    if M * N:
        ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        res.append(orc.entries(dtype, A, B, C, alpha, beta, ii.ravel(), jj.ravel()).reshape(M, N))
    return res


def _expect_equal(fails, tag, results, expected):
    expected = np.asarray(expected)
    for p, r in enumerate(results):
        if r.shape != expected.shape:
            fails.append(f"{tag}[path {p}]: shape {r.shape} != {expected.shape}")
            continue
        same = (r == expected) | (np.isnan(r) & np.isnan(expected)) if r.dtype.kind == "f" else r == expected
        if not np.all(same):
            bad = np.argwhere(~same)[0]
            fails.append(f"{tag}[path {p}]: first mismatch at {tuple(bad)}: "
                         f"{r[tuple(bad)]} != {expected[tuple(bad)]}")


# ----------------------------------------------------------------- pins ----
def pin_identity(orc):
    """A = I gives C = alpha*B (+ beta*C); B = I gives C = alpha*A.  Exact for
    alpha a power of two."""
    fails = []
    for dtype in ("f32", "bf16", "i8"):
        for (M, N) in ((5, 7), (16, 3)):
            K = M
            if dtype == "i8":
                Bv = si.uniform_i8((K, N), 11).astype(np.int64)
                Av = si.uniform_i8((M, 9), 12).astype(np.int64)
            else:
                Bv = si.uniform_f32((K, N), 11).astype(np.float64)
                Av = si.uniform_f32((M, 9), 12).astype(np.float64)
                if dtype == "bf16":
                    Bv = si.bf16_bits_to_f32(si.to_bf16_bits(Bv.astype(np.float32))).astype(np.float64)
                    Av = si.bf16_bits_to_f32(si.to_bf16_bits(Av.astype(np.float32))).astype(np.float64)
            I = np.eye(K)
            r = _all_paths(orc, dtype, _as_operand(dtype, I), _as_operand(dtype, Bv), None, 2, 0)
            _expect_equal(fails, f"identity-A {dtype} {M}x{N}", r, (2 * Bv).astype(_out_t(dtype)))
            I9 = np.eye(9)
            r = _all_paths(orc, dtype, _as_operand(dtype, Av), _as_operand(dtype, I9), None, 1, 0)
            _expect_equal(fails, f"identity-B {dtype} {M}x9", r, Av.astype(_out_t(dtype)))
    return fails


def pin_selection(orc):
    """A selection matrix (one 1 per row, at column s[i]) copies rows of B:
    C[i,:] = B[s[i],:]; a selection B (one 1 per column, at row t[j]) copies
    columns of A: C[:,j] = A[:,t[j]].  Non-square shapes, so a transposed
    operand or a swapped leading dimension cannot pass."""
    fails = []
    M, K, N = 6, 11, 4
    rng = np.random.default_rng(5)
    s = rng.integers(0, K, size=M)
    t = rng.integers(0, K, size=N)
    Asel = np.zeros((M, K))
    Asel[np.arange(M), s] = 1
    Bsel = np.zeros((K, N))
    Bsel[t, np.arange(N)] = 1
    for dtype in ("f32", "bf16", "i8"):
        if dtype == "i8":
            Bv = si.uniform_i8((K, N), 21).astype(np.int64)
            Av = si.uniform_i8((M, K), 22).astype(np.int64)
        else:
            Bv = si.small_int_f32((K, N), 21, -100, 100).astype(np.float64) / 8
            Av = si.small_int_f32((M, K), 22, -100, 100).astype(np.float64) / 8
        r = _all_paths(orc, dtype, _as_operand(dtype, Asel), _as_operand(dtype, Bv), None, 1, 0)
        _expect_equal(fails, f"select-rows {dtype}", r, Bv[s].astype(_out_t(dtype)))
        r = _all_paths(orc, dtype, _as_operand(dtype, Av), _as_operand(dtype, Bsel), None, 1, 0)
        _expect_equal(fails, f"select-cols {dtype}", r, Av[:, t].astype(_out_t(dtype)))
    return fails


def pin_all_ones(orc):
    """A = B = 1, alpha = 1, beta = 0: every entry equals K exactly."""
    fails = []
    for dtype in ("f32", "bf16", "i8"):
        for (M, N, K) in ((3, 4, 1), (7, 5, 33), (2, 3, 1000)):
            A = _as_operand(dtype, np.ones((M, K)))
            B = _as_operand(dtype, np.ones((K, N)))
            r = _all_paths(orc, dtype, A, B, None, 1, 0)
            _expect_equal(fails, f"all-ones {dtype} K={K}", r, np.full((M, N), K, _out_t(dtype)))
    return fails


def pin_alpha_beta(orc):
    """Closed forms of the output update on A = B = 1 (sum = K):
    alpha*K + beta*c, with c exactly representable so the result is exact;
    beta = 0 must not read C (a NaN there must not leak); K = 0 gives beta*c."""
    fails = []
    M, N, K = 4, 6, 8
    c = si.small_int_f32((M, N), 31, -50, 50).astype(np.float64)
    for dtype in ("f32", "bf16", "i8"):
        A = _as_operand(dtype, np.ones((M, K)))
        B = _as_operand(dtype, np.ones((K, N)))
        Cin = c.astype(_out_t(dtype))
        for alpha, beta in ((1, 1), (3, -2), (-1, 5), (0, 1), (2, 0)):
            r = _all_paths(orc, dtype, A, B, Cin, alpha, beta)
            _expect_equal(fails, f"alpha-beta {dtype} a={alpha} b={beta}", r,
                          (alpha * K + beta * c).astype(_out_t(dtype)))
        if dtype != "i8":
            nanC = np.full((M, N), np.nan, np.float32)
            r = _all_paths(orc, dtype, A, B, nanC, 1.0, 0.0)
            _expect_equal(fails, f"beta=0 ignores C {dtype}", r, np.full((M, N), K, np.float32))
            half = _all_paths(orc, dtype, A, B, Cin, 1.0, 0.5)
            _expect_equal(fails, f"beta=0.5 {dtype}", half, (K + 0.5 * c).astype(np.float32))
        # K = 0: the sum is empty
        A0 = _as_operand(dtype, np.zeros((M, 0)))
        B0 = _as_operand(dtype, np.zeros((0, N)))
        r = _all_paths(orc, dtype, A0, B0, Cin, 7, 3)
        _expect_equal(fails, f"K=0 {dtype}", r, (3 * c).astype(_out_t(dtype)))
    return fails


def pin_small_integers(orc):
    """Integer-valued operands: every partial sum is an integer far below 2^24,
    so the exact result is order independent and equals the int64 matrix
    product (numpy integer matmul, a library routine on exact integers)."""
    fails = []
    for dtype in ("f32", "bf16", "i8"):
        for (M, N, K, seed) in ((9, 13, 40, 41), (17, 16, 257, 42)):
            Ai = si.small_int_f32((M, K), seed, -4, 4).astype(np.int64)
            Bi = si.small_int_f32((K, N), seed + 1, -4, 4).astype(np.int64)
            Ci = si.small_int_f32((M, N), seed + 2, -9, 9).astype(np.int64)
            exact = 3 * (Ai @ Bi) - 2 * Ci
            r = _all_paths(orc, dtype, _as_operand(dtype, Ai), _as_operand(dtype, Bi),
                           Ci.astype(_out_t(dtype)), 3, -2)
            _expect_equal(fails, f"small-int {dtype} {M}x{N}x{K}", r, exact.astype(_out_t(dtype)))
    return fails


def _exact_float_case(dtype, M, N, K, seed):
    Af = si.uniform_f32((M, K), seed)
    Bf = si.uniform_f32((K, N), seed + 1)
    Cf = si.uniform_f32((M, N), seed + 2)
    if dtype == "bf16":
        A = si.to_bf16_bits(Af)
        B = si.to_bf16_bits(Bf)
        Av, Bv = si.bf16_bits_to_f32(A), si.bf16_bits_to_f32(B)
    else:
        A, B, Av, Bv = Af, Bf, Af, Bf
    return A, B, Cf, Av, Bv


def pin_exact_rational(orc):
    """Tiny brute force in exact rational arithmetic (Python Fractions): the
    oracle must be within half an fp32 ulp of the exact value of
    alpha*sum_k a_ik b_kj + beta*c_ij, plus the fp64 summation error bound
    (K+2) * 2^-52 * (|alpha| sum_k |a_ik b_kj| + |beta c_ij|)."""
    fails = []
    alpha, beta = np.float32(0.7109375), np.float32(-1.25)
    shapes = [(1, 1, 1), (2, 3, 5), (3, 7, 2), (5, 1, 17), (7, 16, 3), (16, 5, 16), (3, 2, 64)]
    for dtype in ("f32", "bf16"):
        for n, (M, N, K) in enumerate(shapes):
            A, B, C, Av, Bv = _exact_float_case(dtype, M, N, K, 100 + n)
            got_all = _all_paths(orc, dtype, A, B, C, float(alpha), float(beta))
            Fa, Fb = Fraction(float(alpha)), Fraction(float(beta))
            for i in range(M):
                for j in range(N):
                    terms = [Fraction(float(Av[i, k])) * Fraction(float(Bv[k, j])) for k in range(K)]
                    exact = Fa * sum(terms, Fraction(0)) + Fb * Fraction(float(C[i, j]))
                    mag = abs(Fa) * sum(abs(t) for t in terms) + abs(Fb * Fraction(float(C[i, j])))
                    slack = float(mag) * (K + 2) * 2.0 ** -52
                    ulp = float(np.spacing(np.float32(abs(float(exact)))))
                    for p, got in enumerate(got_all):
                        err = abs(Fraction(float(got[i, j])) - exact)
                        if float(err) > 0.5 * ulp + slack:
                            fails.append(f"exact {dtype} {M}x{N}x{K} path {p} at ({i},{j}): "
                                         f"|{float(got[i, j])} - {float(exact)}| = {float(err)}")
    return fails


def pin_bf16_widening(orc):
    """Known bf16 bit patterns on the diagonal of A, B = I: C holds the values."""
    fails = []
    bits = np.array([0x3F80, 0xC000, 0x3E80, 0x4049, 0xBF00, 0x4780, 0x0000, 0x3C00], np.uint16)
    vals = np.array([1.0, -2.0, 0.25, 3.140625, -0.5, 65536.0, 0.0, 2.0 ** -7], np.float32)
    n = bits.size
    A = np.zeros((n, n), np.uint16)
    A[np.arange(n), np.arange(n)] = bits
    B = np.zeros((n, n), np.uint16)
    B[np.arange(n), np.arange(n)] = BF16_ONE
    r = _all_paths(orc, "bf16", A, B, None, 1.0, 0.0)
    _expect_equal(fails, "bf16 widening", r, np.diag(vals).astype(np.float32))
    return fails


def pin_int8_extremes(orc):
    """All -128 times all -128 gives K*2^14 per entry; mixed -128/127 with a
    large alpha wraps modulo 2^32 (closed forms, Python integers)."""
    fails = []

    def wrap(v):
        v &= 0xFFFFFFFF
        return v - (1 << 32) if v >= (1 << 31) else v

    for (K, a, b, alpha, beta, c) in ((4096, -128, -128, 1, 0, 0),
                                      (4096, -128, 127, 100, 0, 0),
                                      (1000, 127, 127, 2 ** 31 - 1, -(2 ** 31), 12345),
                                      (3, -1, 1, -7, 1, -(2 ** 31))):
        M, N = 3, 5
        A = np.full((M, K), a, np.int8)
        B = np.full((K, N), b, np.int8)
        C = np.full((M, N), c, np.int32)
        exp = wrap(alpha * K * a * b + beta * c)
        r = _all_paths(orc, "i8", A, B, C, alpha, beta)
        _expect_equal(fails, f"int8 extreme K={K} a={a} b={b} alpha={alpha}", r,
                      np.full((M, N), exp, np.int32))
    return fails


def pin_textbook_example(orc):
    """The hand-computed example in tests/golden/textbook_2x3x2.txt."""
    fails = []
    fx = load_textbook_golden()
    for dtype in ("f32", "bf16", "i8"):
        A = _as_operand(dtype, fx["A"])
        B = _as_operand(dtype, fx["B"])
        r = _all_paths(orc, dtype, A, B, None, 1, 0)
        _expect_equal(fails, f"textbook AB {dtype}", r, fx["AB"].astype(_out_t(dtype)))
        C = fx["C"].astype(_out_t(dtype))
        r = _all_paths(orc, dtype, A, B, C, int(fx["alpha"]), int(fx["beta"]))
        _expect_equal(fails, f"textbook update {dtype}", r, fx["out"].astype(_out_t(dtype)))
    return fails


def load_textbook_golden():
    """Parse tests/golden/textbook_2x3x2.txt (``name: rows separated by ;``)."""
    out = {}
    with open(os.path.join(GOLDEN, "textbook_2x3x2.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            rows = [r.split() for r in val.split(";")]
            arr = np.array([[float(x) for x in r] for r in rows])
            out[key.strip()] = arr if arr.size > 1 else arr.item()
    return out


ALL_PINS = [pin_identity, pin_selection, pin_all_ones, pin_alpha_beta, pin_small_integers,
            pin_exact_rational, pin_bf16_widening, pin_int8_extremes, pin_textbook_example]


def run_all(orc):
    """Run every pin; return {pin name: [failures]} for the pins that failed."""
    bad = {}
    for pin in ALL_PINS:
        try:
            f = pin(orc)
        except Exception as e:  # a crash of the oracle under test is a failure too
            f = [f"raised {type(e).__name__}: {e}"]
        if f:
            bad[pin.__name__] = f
    return bad
