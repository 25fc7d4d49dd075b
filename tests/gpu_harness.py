"""Helpers for the GPU parity tests: upload seeded host operands, call the
library through its C ABI binding, read the result back, and compare with the
oracle on the same host operands."""
from __future__ import annotations

import math

import numpy as np

import software_pipelined_tiled_loop_gb300 as pg


def torch_mod():
    import torch
    return torch


def to_device(x: np.ndarray):
    torch = torch_mod()
    if x.dtype == np.uint16:  # bf16 bit patterns travel as int16
        x = x.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda")


def from_device(t, dtype) -> np.ndarray:
    return t.cpu().numpy().view(dtype)


def run_gpu(dtype: str, A, B, C, alpha, beta, config=None, repeat: int = 1):
    """Run C <- alpha*A@B + beta*C on the GPU; return (result, device status)."""
    torch = torch_mod()
    M, K = A.shape
    N = B.shape[1]
    out_t = np.int32 if dtype == "i8" else np.float32
    dA, dB = to_device(A), to_device(B)
    dC = to_device(np.ascontiguousarray(C, dtype=out_t))
    fn = {"f32": pg.gemm_f32_ex, "bf16": pg.gemm_bf16_ex, "i8": pg.gemm_i8_ex}[dtype]
    for _ in range(repeat):
        fn(M, N, K, alpha, dA, dB, beta, dC, config=config)
    torch.cuda.synchronize()
    status = pg.pgemm_get_device_status()
    return from_device(dC, out_t), status


def float_bound(A, B, K, dtype) -> float:
    """1e-4 * sqrt(K) * max|A| * max|B| over the operand values."""
    if K == 0:
        return 0.0
    if dtype == "bf16":
        import seeded_inputs as si
        a = np.abs(si.bf16_bits_to_f32(A)).max()
        b = np.abs(si.bf16_bits_to_f32(B)).max()
    else:
        a, b = np.abs(A).max(), np.abs(B).max()
    return 1e-4 * math.sqrt(K) * float(a) * float(b)


def compare(dtype, got, ref, A, B, K, exact=False):
    """Assert parity: bit-exact for int8 (and for exact float cases), else the bound."""
    assert got.shape == ref.shape
    if dtype == "i8" or exact:
        bad = np.argwhere(got != ref) if dtype == "i8" else np.argwhere(
            ~((got == ref) | (np.isnan(got) & np.isnan(ref))))
        assert bad.size == 0, (f"{len(bad)} mismatches, first at {tuple(bad[0])}: "
                               f"{got[tuple(bad[0])]} vs {ref[tuple(bad[0])]}")
        return 0.0
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    err = float(np.max(np.abs(got.astype(np.float64) - ref.astype(np.float64)))) if got.size else 0.0
    bound = float_bound(A, B, K, dtype)
    assert err <= bound, f"max |C - C_ref| = {err:g} > bound {bound:g}"
    return err
