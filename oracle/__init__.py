"""CPU reference oracle for the pipelined GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product (``software_pipelined_tiled_loop_gb300``) never imports it, and this
package imports nothing from the product: the two share no code.

The arithmetic lives in ``pgemm_oracle.c`` (plain C, fp64 accumulation for
float operands, int64 for int8), built with gcc into ``_build/liboracle.so``.
It evaluates the plain definition

    C_out = alpha * A @ B + beta * C_in      (row-major A: MxK, B: KxN, C: MxN)

from "Double Buffering: Software Pipelining the K-Loop", section "The Kernel"
(kernel signature and the alpha/beta output update), which the third page
("GPU-Kernel pipelinen", Schritt 5) says pipelining leaves unchanged.

Every function here is pinned by ``tests/test_oracle.py`` (identity,
permutation, all-ones, exact small-integer results, exact rational brute force,
int8 extremes) and the pins are shown to catch planted mistakes by
``tests/test_oracle_mutants.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pgemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None


def compile_oracle(source: str = SOURCE, out: str = LIB_PATH, extra: tuple = ()) -> str:
    """Compile an oracle source file to a shared library with gcc (-O2 -fopenmp).

    ``-ffp-contract=off`` keeps every multiply and add a separately rounded
    double operation, exactly as written in the C source.
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", *extra, source, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build ``_build/liboracle.so`` if it is missing or older than its source."""
    if force or not os.path.exists(LIB_PATH) or \
            os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE):
        compile_oracle()
    return LIB_PATH


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    i32, i64, f32, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
    rows = [i32, i32, i32, None, vp, vp, None, vp, vp, i32, i32]
    ents = [i32, i32, i32, None, vp, vp, None, vp, i64, vp, vp, vp]
    for name, scal in (("f32", f32), ("bf16", f32), ("i8", ctypes.c_int32)):
        fr = getattr(lib, f"oracle_gemm_{name}_rows")
        a = list(rows)
        a[3] = a[6] = scal
        fr.argtypes, fr.restype = a, i32
        fe = getattr(lib, f"oracle_gemm_{name}_entries")
        b = list(ents)
        b[3] = b[6] = scal
        fe.argtypes, fe.restype = b, i32
    lib.oracle_num_threads.argtypes, lib.oracle_num_threads.restype = [], i32
    lib.oracle_set_num_threads.argtypes, lib.oracle_set_num_threads.restype = [i32], None
    return lib


class Oracle:
    """ctypes handle over one compiled oracle library (the real one or a test mutant)."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        self.lib = _declare(ctypes.CDLL(lib_path))

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _ptr(a):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.lib.oracle_set_num_threads(int(n))

    # -- full / row-range evaluation --------------------------------------
    def gemm(self, dtype: str, A, B, C=None, alpha=1, beta=0, rows=None):
        """Return alpha*A@B + beta*C (rows ``rows=(r0, r1)`` only, if given).

        dtype: "f32" (A, B float32), "bf16" (A, B uint16 bf16 bits, C float32)
        or "i8" (A, B int8, C int32).  The result has shape (r1-r0, N).
        """
        A, B = np.ascontiguousarray(A), np.ascontiguousarray(B)
        M, K = A.shape
        K2, N = B.shape
        if K2 != K:
            raise ValueError("inner dimensions differ")
        r0, r1 = (0, M) if rows is None else rows
        out_t = np.int32 if dtype == "i8" else np.float32
        if C is not None:
            C = np.ascontiguousarray(C, dtype=out_t)
            if C.shape != (M, N):
                raise ValueError("C shape mismatch")
        elif beta != 0:
            raise ValueError("beta != 0 needs C")
        _check_dtypes(dtype, A, B)
        if not (0 <= r0 <= r1 <= M):
            raise ValueError("row range out of bounds")
        out = np.empty((r1 - r0, N), dtype=out_t)
        # the C entry point writes rows r0..r1-1 of an M x N row-major buffer;
        # hand it a base pointer r0 rows before ``out`` so only r1-r0 rows are held
        base = ctypes.c_void_p(out.ctypes.data - r0 * N * out.itemsize) if r1 > r0 \
            else self._ptr(out)
        fn = getattr(self.lib, f"oracle_gemm_{dtype}_rows")
        rc = fn(M, N, K, alpha, self._ptr(A), self._ptr(B), beta, self._ptr(C),
                base, r0, r1)
        if rc != 0:
            raise ValueError(f"oracle_gemm_{dtype}_rows rejected its arguments")
        return out

    def entries(self, dtype: str, A, B, C, alpha, beta, ii, jj):
        """Return the entries C_out[ii[t], jj[t]] one by one."""
        A, B = np.ascontiguousarray(A), np.ascontiguousarray(B)
        M, K = A.shape
        N = B.shape[1]
        _check_dtypes(dtype, A, B)
        out_t = np.int32 if dtype == "i8" else np.float32
        if C is not None:
            C = np.ascontiguousarray(C, dtype=out_t)
        elif beta != 0:
            raise ValueError("beta != 0 needs C")
        ii = np.ascontiguousarray(ii, dtype=np.int64)
        jj = np.ascontiguousarray(jj, dtype=np.int64)
        out = np.empty(ii.shape[0], dtype=out_t)
        fn = getattr(self.lib, f"oracle_gemm_{dtype}_entries")
        rc = fn(M, N, K, alpha, self._ptr(A), self._ptr(B), beta, self._ptr(C),
                ii.shape[0], self._ptr(ii), self._ptr(jj), self._ptr(out))
        if rc != 0:
            raise ValueError(f"oracle_gemm_{dtype}_entries rejected its arguments")
        return out


def _check_dtypes(dtype, A, B):
    want = {"f32": np.float32, "bf16": np.uint16, "i8": np.int8}[dtype]
    if A.dtype != want or B.dtype != want:
        raise TypeError(f"{dtype} oracle wants {np.dtype(want).name} operands")


def get() -> Oracle:
    """The oracle built from ``pgemm_oracle.c`` (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
        return _lib
