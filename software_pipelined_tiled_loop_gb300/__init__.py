"""Python binding of libpipegemm, the software-pipelined GEMM library for GB300.

Argument marshalling only: every function here forwards to the C ABI declared
in ``include/pgemm.h`` (same names), and all arithmetic runs in the library's
CUDA kernels.  There is no fallback: if ``libpipegemm.so`` has not been built,
``lib()`` raises.

Operands may be given as torch tensors (CUDA, contiguous, row-major) or as raw
device pointers (ints).  ``stream`` defaults to torch's current stream when
torch is importable, else the legacy default stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "PgemmError", "lib", "library_path", "gemm_f32", "gemm_bf16", "gemm_i8", "gemm_f32_ex",
    "gemm_bf16_ex", "gemm_i8_ex", "pgemm_default_config", "pgemm_list_configs",
    "pgemm_kernel_attrs", "pgemm_get_device_status", "pgemm_selftest_wait_timeout",
    "pgemm_status_string", "pgemm_version", "gemm_i8_noalloc", "NOALLOC_SCRATCH_BYTES",
    "pgemm_stage_reuse_demo", "pgemm_schedule", "pgemm_stream_k_plan", "pgemm_trim_scratch",
    "DTYPES", "STATUS", "EXPORTED", "PRODUCERS", "ENGINES",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpipegemm.so")

STATUS = {
    0: "PGEMM_OK", 1: "PGEMM_ERR_INVALID_VALUE", 2: "PGEMM_ERR_MISALIGNED",
    3: "PGEMM_ERR_UNSUPPORTED_DEVICE", 4: "PGEMM_ERR_CUDA", 5: "PGEMM_ERR_TIMEOUT",
    6: "PGEMM_ERR_UNSUPPORTED_CONFIG", 7: "PGEMM_ERR_TOO_LARGE",
}
# Size of the fixed device array gemm_i8_noalloc widens its operands into.
NOALLOC_SCRATCH_BYTES = 32 << 20
DTYPES = {"f32": 0, "bf16": 1, "i8": 2}
# pgemm_producer: who fills the shared-memory stages
PRODUCERS = {"tma": 0, "registers": 1, "staged": 2, "widen_in_kernel": 3}
# pgemm_engine: which multiply-accumulate consumes the stages
ENGINES = {"default": 0, "mma_sync": 1}
# Every function include/pgemm.h declares.
EXPORTED = [
    "gemm_f32", "gemm_bf16", "gemm_i8", "gemm_f32_ex", "gemm_bf16_ex", "gemm_i8_ex",
    "pgemm_default_config", "pgemm_list_configs", "pgemm_kernel_attrs",
    "pgemm_get_device_status", "pgemm_selftest_wait_timeout", "pgemm_status_string",
    "pgemm_version", "gemm_i8_noalloc", "pgemm_stage_reuse_demo", "pgemm_schedule",
    "pgemm_stream_k_plan", "pgemm_trim_scratch",
]


class PgemmError(RuntimeError):
    """A non-OK pgemm_status."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class Config(ctypes.Structure):
    """pgemm_config.  A tuple (bm, bn, bk, stages[, max_k_parts[, producer[,
    engine[, group_m]]]]) converts to it."""
    _fields_ = [("bm", ctypes.c_int), ("bn", ctypes.c_int), ("bk", ctypes.c_int),
                ("stages", ctypes.c_int), ("max_k_parts", ctypes.c_int),
                ("producer", ctypes.c_int), ("engine", ctypes.c_int), ("group_m", ctypes.c_int)]

    def as_tuple(self):
        """The kernel the configuration names: (bm, bn, bk, stages), with
        (..., max_k_parts, producer, engine) appended when the producer or
        the engine is not the default, and group_m after them when set."""
        if self.group_m:
            return (self.bm, self.bn, self.bk, self.stages, self.max_k_parts, self.producer,
                    self.engine, self.group_m)
        if self.producer or self.engine:
            return (self.bm, self.bn, self.bk, self.stages, self.max_k_parts, self.producer,
                    self.engine)
        return (self.bm, self.bn, self.bk, self.stages)


_lock = threading.Lock()
_lib = None


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    i, f, vp, i32 = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_int32
    ll = ctypes.c_longlong
    cfgp = ctypes.POINTER(Config)
    ip = ctypes.POINTER(ctypes.c_int)
    llp = ctypes.POINTER(ctypes.c_longlong)
    sig = {
        "gemm_f32": [i, i, i, f, vp, vp, f, vp, vp],
        "gemm_bf16": [i, i, i, f, vp, vp, f, vp, vp],
        "gemm_i8": [i, i, i, i32, vp, vp, i32, vp, vp],
        "gemm_i8_noalloc": [i, i, i, i32, vp, vp, i32, vp, vp],
        "gemm_f32_ex": [i, i, i, f, vp, vp, f, vp, cfgp, vp],
        "gemm_bf16_ex": [i, i, i, f, vp, vp, f, vp, cfgp, vp],
        "gemm_i8_ex": [i, i, i, i32, vp, vp, i32, vp, cfgp, vp],
        "pgemm_default_config": [i, i, i, i, cfgp],
        "pgemm_list_configs": [i, cfgp, i],
        "pgemm_kernel_attrs": [i, cfgp, ip, ip, ip, ip],
        "pgemm_get_device_status": [vp],
        "pgemm_selftest_wait_timeout": [i, vp],
        "pgemm_status_string": [i],
        "pgemm_version": [],
        "pgemm_stage_reuse_demo": [vp, i, i, vp, vp, i, i, ctypes.c_uint, vp, i, vp],
        "pgemm_schedule": [i, cfgp, i, i, i, llp, ip, llp, ip, llp],
        "pgemm_stream_k_plan": [ll, i, i, i, llp, ip, ip, llp],
        "pgemm_trim_scratch": [],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.pgemm_status_string.restype = ctypes.c_char_p
    return L


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise RuntimeError(
                    f"{library_path} is missing: build it with "
                    "`python -m software_pipelined_tiled_loop_gb300.build` (needs nvcc)")
            _lib = _declare(ctypes.CDLL(library_path))
        return _lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_cuda:
            raise ValueError("operands must be CUDA tensors (or raw device pointers)")
        if not x.is_contiguous():
            raise ValueError("operands must be contiguous row-major tensors")
        return int(x.data_ptr())
    raise TypeError(f"cannot take a device pointer from {type(x).__name__}")


def _stream(s) -> int:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available():
                return int(torch.cuda.current_stream().cuda_stream)
        except ImportError:
            pass
        return 0
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(code: int, where: str) -> None:
    if code != 0:
        raise PgemmError(code, where)


def _cfg(config):
    if config is None:
        return None
    if isinstance(config, Config):
        return ctypes.byref(config)
    return ctypes.byref(Config(*config))


def gemm_f32(M, N, K, alpha, A, B, beta, C, stream=None):
    """C <- alpha*A@B + beta*C, fp32 (FFMA).  Asynchronous on ``stream``."""
    _check(lib().gemm_f32(M, N, K, alpha, _ptr(A), _ptr(B), beta, _ptr(C), _stream(stream)),
           "gemm_f32")


def gemm_bf16(M, N, K, alpha, A, B, beta, C, stream=None):
    """C (fp32) <- alpha*A@B + beta*C with bf16 A, B (tcgen05).  Asynchronous."""
    _check(lib().gemm_bf16(M, N, K, alpha, _ptr(A), _ptr(B), beta, _ptr(C), _stream(stream)),
           "gemm_bf16")


def gemm_i8(M, N, K, alpha, A, B, beta, C, stream=None):
    """C (int32) <- alpha*A@B + beta*C with int8 A, B, exact modulo 2^32.  Asynchronous."""
    _check(lib().gemm_i8(M, N, K, int(alpha), _ptr(A), _ptr(B), int(beta), _ptr(C),
                         _stream(stream)), "gemm_i8")


def gemm_i8_noalloc(M, N, K, alpha, A, B, beta, C, stream=None):
    """gemm_i8 that allocates no device memory: for callers whose memory is
    owned by their own allocator or budget, or who may not call an allocator
    on this path.  Operands are widened into one fixed 32 MiB device array
    shared by all calls (calls overlapping on the GPU race); larger problems
    raise PgemmError(PGEMM_ERR_TOO_LARGE).  The first call on a device looks
    up that array's address and should come before any stream capture."""
    _check(lib().gemm_i8_noalloc(M, N, K, int(alpha), _ptr(A), _ptr(B), int(beta), _ptr(C),
                                 _stream(stream)), "gemm_i8_noalloc")


def gemm_f32_ex(M, N, K, alpha, A, B, beta, C, config=None, stream=None):
    _check(lib().gemm_f32_ex(M, N, K, alpha, _ptr(A), _ptr(B), beta, _ptr(C), _cfg(config),
                             _stream(stream)), "gemm_f32_ex")


def gemm_bf16_ex(M, N, K, alpha, A, B, beta, C, config=None, stream=None):
    _check(lib().gemm_bf16_ex(M, N, K, alpha, _ptr(A), _ptr(B), beta, _ptr(C), _cfg(config),
                              _stream(stream)), "gemm_bf16_ex")


def gemm_i8_ex(M, N, K, alpha, A, B, beta, C, config=None, stream=None):
    _check(lib().gemm_i8_ex(M, N, K, int(alpha), _ptr(A), _ptr(B), int(beta), _ptr(C),
                            _cfg(config), _stream(stream)), "gemm_i8_ex")


def pgemm_stage_reuse_demo(X, rows, cols, perm, out, check_reuse, delay_warp=-1, delay_ns=0,
                           trace=None, trace_cap=0, stream=None):
    """The two-stage copy-and-reduce hazard experiment (with or without the
    consume-before-reuse wait).  X: rows x cols fp32, perm: int32 row order,
    out: rows fp32 (zeroed by the caller); trace: optional uint64 buffer."""
    _check(lib().pgemm_stage_reuse_demo(_ptr(X), rows, cols, _ptr(perm), _ptr(out),
                                        int(check_reuse), int(delay_warp), int(delay_ns),
                                        _ptr(trace), int(trace_cap), _stream(stream)),
           "pgemm_stage_reuse_demo")


def pgemm_schedule(dtype: str, M: int, N: int, K: int, config=None):
    """The persistent schedule of a call on the current device: a dict with
    tiles, slots (units running at once), split_tiles and parts (split along
    K), and half_tiles (tiles run as two half-width units)."""
    t, sl, st, p = ctypes.c_longlong(), ctypes.c_int(), ctypes.c_longlong(), ctypes.c_int()
    ht = ctypes.c_longlong()
    _check(lib().pgemm_schedule(DTYPES[dtype], _cfg(config), M, N, K, ctypes.byref(t),
                                ctypes.byref(sl), ctypes.byref(st), ctypes.byref(p),
                                ctypes.byref(ht)),
           "pgemm_schedule")
    return {"tiles": t.value, "slots": sl.value, "split_tiles": st.value, "parts": p.value,
            "half_tiles": ht.value}


def pgemm_stream_k_plan(tiles: int, slots: int, k_tiles: int, max_parts: int = 0):
    """The stream-K rule (host only): a dict with sk_tiles, sk_slots,
    max_pieces and share (K-iterations per slot)."""
    st, gs, mp, sh = ctypes.c_longlong(), ctypes.c_int(), ctypes.c_int(), ctypes.c_longlong()
    _check(lib().pgemm_stream_k_plan(tiles, slots, k_tiles, max_parts, ctypes.byref(st),
                                     ctypes.byref(gs), ctypes.byref(mp), ctypes.byref(sh)),
           "pgemm_stream_k_plan")
    return {"sk_tiles": st.value, "sk_slots": gs.value, "max_pieces": mp.value,
            "share": sh.value}


def pgemm_default_config(dtype: str, M: int, N: int, K: int):
    c = Config()
    _check(lib().pgemm_default_config(DTYPES[dtype], M, N, K, ctypes.byref(c)),
           "pgemm_default_config")
    return c.as_tuple()


def pgemm_list_configs(dtype: str):
    n = lib().pgemm_list_configs(DTYPES[dtype], None, 0)
    arr = (Config * max(n, 1))()
    lib().pgemm_list_configs(DTYPES[dtype], arr, n)
    return [arr[i].as_tuple() for i in range(n)]


def pgemm_kernel_attrs(dtype: str, config):
    out = [ctypes.c_int(0) for _ in range(4)]
    _check(lib().pgemm_kernel_attrs(DTYPES[dtype], _cfg(config), *[ctypes.byref(o) for o in out]),
           "pgemm_kernel_attrs")
    return {"smem_bytes": out[0].value, "regs_per_thread": out[1].value,
            "threads_per_block": out[2].value, "blocks_per_sm": out[3].value}


def pgemm_get_device_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device status code."""
    return int(lib().pgemm_get_device_status(_stream(stream)))


def pgemm_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    return int(lib().pgemm_selftest_wait_timeout(int(limit_us), _stream(stream)))


def pgemm_status_string(code: int) -> str:
    return lib().pgemm_status_string(int(code)).decode()


def pgemm_version() -> int:
    return int(lib().pgemm_version())


def pgemm_trim_scratch() -> None:
    """Synchronise the current device and give the library's unused scratch
    memory back (the pool otherwise keeps it between calls)."""
    _check(lib().pgemm_trim_scratch(), "pgemm_trim_scratch")
