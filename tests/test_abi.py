"""The C ABI: the library loads, exports every function include/pgemm.h
declares, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

import software_pipelined_tiled_loop_gb300 as pg
from software_pipelined_tiled_loop_gb300 import build as pgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pgemm.h")


@pytest.fixture(scope="module")
def L():
    pgbuild.build()
    return pg.lib()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"PGEMM_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(pg.EXPORTED)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_no_stray_exports(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", pg.library_path], capture_output=True,
                         text=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert exported == declared_functions()


def test_status_strings(L):
    for code in range(8):
        assert pg.pgemm_status_string(code)
    assert pg.pgemm_version() >= 100


def test_list_configs(L):
    f32 = pg.pgemm_list_configs("f32")
    bf16 = pg.pgemm_list_configs("bf16")
    i8 = pg.pgemm_list_configs("i8")
    # stage counts 2..6 are built for every dtype (the stage sweep), plus the
    # S = 1 unpipelined comparator
    for cfgs in (f32, bf16, i8):
        assert {c[3] for c in cfgs} == {1, 2, 3, 4, 5, 6}
    assert {c[3] for c in bf16 if c[1] == 128} == {1, 2, 3, 4, 5, 6}
    # 128 x 256 single-CTA tiles fit four stages; the CTA pair's 256 x 256 six
    assert {c[3] for c in bf16 if c[1] == 256 and c[0] == 128} == {1, 2, 3, 4}
    assert {c[3] for c in bf16 if c[0] == 256 and c[2] == 64} == {4, 5, 6}
    # the pair also with stages of 128 K columns (two 64-column sub-tiles
    # landed under one barrier), TMA producer, for both tensor-core dtypes
    for cfgs in (bf16, i8):
        wide = [c for c in cfgs if c[0] == 256 and c[2] == 128]
        assert {c[3] for c in wide} == {2, 3}
        assert all(len(c) <= 5 or c[5] == pg.PRODUCERS["tma"] for c in wide)
    # the register-staged comparator: fp32 only, two buffers, named by its producer
    regs = [c for c in f32 if len(c) > 5 and c[5] == pg.PRODUCERS["registers"]]
    assert {(c[0], c[1], c[3]) for c in regs} == {(128, 128, 2), (128, 64, 2)}
    assert not [c for c in bf16 if len(c) > 5 and c[5] != pg.PRODUCERS["tma"]]
    # int8 on the CTA pair also with the register-staged producer (int8 read
    # and widened in registers by the GEMM itself)
    i8_regs = [c for c in i8 if len(c) > 5 and c[5] == pg.PRODUCERS["registers"]]
    assert {(c[0], c[1], c[3]) for c in i8_regs} == {(256, 256, 4), (256, 256, 5), (256, 256, 6)}
    # int8 on the CTA pair with int8 stages by TMA widened in shared memory
    # (`stages` = depth of the int8 ring)
    i8_staged = [c for c in i8 if len(c) > 5 and c[5] == pg.PRODUCERS["staged"]]
    assert {(c[0], c[1], c[3]) for c in i8_staged} == {(256, 256, 4), (256, 256, 5), (256, 256, 6)}
    assert not [c for c in f32 + bf16 if len(c) > 5 and c[5] == pg.PRODUCERS["staged"]]
    # int8 on the CTA pair with the widening inside the GEMM
    i8_wik = [c for c in i8 if len(c) > 5 and c[5] == pg.PRODUCERS["widen_in_kernel"]]
    assert {(c[0], c[1], c[3]) for c in i8_wik} == {(256, 256, 4), (256, 256, 5)}
    # the mma.sync int8 engine: 128 x 128 tiles, K-tiles of 128 int8
    imma = [c for c in i8 if len(c) > 6 and c[6] == pg.ENGINES["mma_sync"]]
    assert {(c[0], c[1], c[2]) for c in imma} == {(128, 128, 128)}
    assert {c[3] for c in imma} == {2, 3, 4, 6}
    assert not [c for c in f32 + bf16 if len(c) > 6 and c[6] != pg.ENGINES["default"]]


@pytest.mark.parametrize("fn", ["gemm_f32", "gemm_bf16", "gemm_i8", "gemm_i8_noalloc"])
def test_host_validation_without_gpu(L, fn):
    # gemm_i8_noalloc checks its arguments before it looks up its device array
    f = getattr(L, fn)
    a = 1 if fn.startswith("gemm_i8") else 1.0
    good = 1 << 20  # never dereferenced: validation fails or the call is a no-op first
    # negative dimensions
    assert f(-1, 4, 4, a, good, good, 0 * a, good, None) == 1
    assert f(4, -1, 4, a, good, good, 0 * a, good, None) == 1
    assert f(4, 4, -1, a, good, good, 0 * a, good, None) == 1
    # empty output: nothing to do
    assert f(0, 4, 4, a, None, None, 0 * a, None, None) == 0
    assert f(4, 0, 4, a, None, None, 0 * a, None, None) == 0
    # NULL operands with work to do
    assert f(4, 4, 4, a, None, good, 0 * a, good, None) == 1
    assert f(4, 4, 4, a, good, good, 0 * a, None, None) == 1
    # misaligned base pointers
    assert f(4, 4, 4, a, good + 4, good, 0 * a, good, None) == 2
    assert f(4, 4, 4, a, good, good + 2, 0 * a, good, None) == 2
    assert f(4, 4, 4, a, good, good, 0 * a, good + 8, None) == 2


def test_binding_rejects_host_tensors(L):
    torch = pytest.importorskip("torch")
    x = torch.zeros(4, 4)
    with pytest.raises(ValueError):
        pg.gemm_f32(4, 4, 4, 1.0, x, x, 0.0, x)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import importlib
    monkeypatch.setattr(pg, "library_path", str(tmp_path / "nope.so"))
    monkeypatch.setattr(pg, "_lib", None)
    with pytest.raises(RuntimeError):
        pg.lib()


def test_stage_reuse_demo_validation_without_gpu(L):
    good = 1 << 20
    f = L.pgemm_stage_reuse_demo
    assert f(good, 4, 3, good, good, 1, -1, 0, None, 0, None) == 1      # cols % 4
    assert f(good, 4, 16384, good, good, 1, -1, 0, None, 0, None) == 1  # too wide for 2 stages
    assert f(good, 4, 16, good, good, 1, 7, 0, None, 0, None) == 1      # no such warp
    assert f(good + 4, 4, 16, good, good, 1, -1, 0, None, 0, None) == 2  # misaligned X
    assert f(good, 0, 16, None, None, 1, -1, 0, None, 0, None) == 0      # nothing to do


def test_config_struct_matches_the_header():
    # the binding's pgemm_config has the header's fields, in the header's order
    src = open(HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} pgemm_config;", src, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = []
    for decl in body.split(";"):
        decl = decl.strip()
        if decl:
            assert decl.startswith("int "), decl
            names += [n.strip() for n in decl[4:].split(",")]
    assert [f[0] for f in pg.Config._fields_] == names
    assert ctypes.sizeof(pg.Config) == 4 * len(names)
