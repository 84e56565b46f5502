"""The C-ABI library without a GPU: it loads, exports every function that
include/dqd.h declares, and rejects bad arguments on the host (status +
message) before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dqd.h")


@pytest.fixture(scope="module")
def lib():
    from memory_bound_decode_dq_gb300 import build
    path = build.build()
    L = ctypes.CDLL(path)
    return L


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"DQD_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_four_operations():
    names = set(declared_functions())
    assert {"dq_gemm", "gqa_decode_attn", "pack_int4_g128", "quant_fp8_rowwise"} <= names
    assert len(names) >= 10


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


class WeightDesc(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int32), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("data", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zeros", ctypes.c_void_p)]


OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA = range(5)


def _msg(lib):
    lib.dqd_last_error.restype = ctypes.c_char_p
    return lib.dqd_last_error().decode()


def test_status_strings_and_version(lib):
    lib.dqd_status_string.restype = ctypes.c_char_p
    names = [lib.dqd_status_string(i).decode() for i in range(5)]
    assert names == ["DQD_OK", "DQD_ERR_INVALID_ARG", "DQD_ERR_UNSUPPORTED", "DQD_ERR_WORKSPACE", "DQD_ERR_CUDA"]
    assert lib.dqd_status_string(99) is not None
    lib.dqd_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.dqd_version()


def test_pack_bytes(lib):
    f = lib.pack_int4_g128_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    assert f(1024, 1024, 0) == 64 * 8 * 1024
    assert f(1024, 1024, 1) == 64 * 8 * 32
    assert f(1024, 1024, 2) == 64 * 8 * 8
    assert f(17, 128, 0) == 2 * 1024          # ragged n rounds up to 16-row tiles
    assert f(16, 100, 0) == 0 and f(0, 128, 0) == 0 and f(16, 128, 3) == 0


def _gemm(lib, desc, x=None, m=1, y=0x1000, ws=None, wsb=0):
    f = lib.dq_gemm
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    return f(ctypes.byref(desc) if desc is not None else None, x, m, y, ws, wsb, None)


@pytest.mark.parametrize("wtype,n,k,data,scales,zeros,m,status,fragment", [
    (7, 16, 128, 0x1000, 0x1000, 0x1000, 1, INVALID, "unknown weight type"),
    (2, 16, 100, 0x1000, 0x1000, 0x1000, 1, INVALID, "k % 128"),
    (0, 16, 12, 0x1000, None, None, 1, INVALID, "k % 8"),
    (1, 16, 24, 0x1000, 0x1000, None, 1, INVALID, "k % 16"),
    (1, 16, 32, 0x1000, None, None, 1, INVALID, "row scales"),
    (2, 16, 128, 0x1000, None, 0x1000, 1, INVALID, "packed scales"),
    (0, 16, 128, 0x1008, None, None, 1, INVALID, "16-byte aligned"),
    (0, 16, 128, None, None, None, 1, INVALID, "16-byte aligned"),
    (0, -1, 128, 0x1000, None, None, 1, INVALID, "negative"),
    (0, 16, 128, 0x1000, None, None, 65537, UNSUPPORTED, "m must be"),
    (0, 16, 128, 0x1000, None, None, -1, UNSUPPORTED, "m must be"),
])
def test_dq_gemm_host_checks(lib, wtype, n, k, data, scales, zeros, m, status, fragment):
    d = WeightDesc(wtype, n, k, data, scales, zeros)
    assert _gemm(lib, d, x=0x2000, m=m) == status
    assert fragment in _msg(lib)


def test_dq_gemm_null_descriptor_and_outputs(lib):
    assert _gemm(lib, None) == INVALID
    d = WeightDesc(0, 16, 128, 0x1000, None, None)
    assert _gemm(lib, d, x=0x2000, y=None) == INVALID
    assert _gemm(lib, d, x=None) == INVALID
    assert _gemm(lib, d, x=0x2004) == INVALID
    # m == 0 and n == 0 are no-ops that succeed without any CUDA call
    assert _gemm(lib, d, x=0x2000, m=0) == OK
    assert _gemm(lib, WeightDesc(0, 0, 128, None, None, None), x=0x2000) == OK


def test_quant_and_pack_host_checks(lib):
    q = lib.quant_fp8_rowwise
    q.restype = ctypes.c_int
    q.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert q(0x1000, 4, 24, 0x2000, 0x3000, None) == INVALID
    assert q(0x1000, 0, 32, 0x2000, 0x3000, None) == INVALID
    assert q(None, 4, 32, 0x2000, 0x3000, None) == INVALID
    assert q(0x1000, 4, 32, 0x2001, 0x3000, None) == INVALID
    p = lib.pack_int4_g128
    p.restype = ctypes.c_int
    p.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 2 + [ctypes.c_void_p] * 4
    assert p(0x1000, 0x1000, 0x1000, 16, 64, 0x1000, 0x1000, 0x1000, None) == INVALID
    assert p(0x1000, 0x1000, None, 16, 128, 0x1000, 0x1000, 0x1000, None) == INVALID
    assert p(0x1000, 0x1000, 0x1000, 0, 128, 0x1000, 0x1000, 0x1000, None) == INVALID


def _attn(lib, b=1, w=1, hq=8, hkv=2, d=128, max_context=64, max_blocks=4, num_blocks=4,
          scale=0.088, q=0x1000, kp=0x1000, vp=0x1000, table=0x1000, ctx=0x1000, out=0x1000):
    f = lib.gqa_decode_attn
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p] + \
                 [ctypes.c_int32] * 6 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.c_void_p]
    return f(q, kp, vp, num_blocks, table, max_blocks, ctx, max_context, b, w, hq, hkv, d, scale, out,
             None, 0, None)


@pytest.mark.parametrize("kw,status,fragment", [
    (dict(d=64), UNSUPPORTED, "head_dim"),
    (dict(w=17), UNSUPPORTED, "verify width"),
    (dict(hq=6, hkv=4), INVALID, "hq % hkv"),
    (dict(b=0), INVALID, ">= 1"),
    (dict(max_context=65), INVALID, "exceeds 16"),
    (dict(num_blocks=0), INVALID, "num_blocks"),
    (dict(scale=float("nan")), INVALID, "finite"),
    (dict(q=None), INVALID, "aligned"),
    (dict(out=0x1002), INVALID, "aligned"),
    (dict(table=0x1002), INVALID, "4-byte"),
])
def test_attn_host_checks(lib, kw, status, fragment):
    assert _attn(lib, **kw) == status
    assert fragment in _msg(lib)


def test_binding_refuses_to_run_without_library(tmp_path, monkeypatch):
    """The Python binding has no fallback: with the library absent it raises."""
    import importlib.util
    src = os.path.join(ROOT, "memory_bound_decode_dq_gb300", "dqd.py")
    fake_pkg = tmp_path / "pkg"
    fake_pkg.mkdir()
    (fake_pkg / "dqd.py").write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("dqd_probe", fake_pkg / "dqd.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "dqd.h"

int main(void) {
  /* host-only calls: no device is touched */
  const char* v = dqd_version();
  const char* s = dqd_status_string(DQD_ERR_WORKSPACE);
  size_t codes = pack_int4_g128_bytes(256, 1024, 0);
  dqd_weight w;
  memset(&w, 0, sizeof w);
  w.type = DQD_W_INT4_G128;
  w.n = 64;
  w.k = 100; /* not a multiple of 128: refused on the host */
  size_t ws = 0;
  dqd_status st = dq_gemm_workspace_bytes(&w, 1, &ws);
  printf("%s|%s|%zu|%d\n", v ? v : "", s ? s : "", codes, (int)st);
  return 0;
}
"""


@pytest.mark.parametrize("std", ["c99", "c11"])
def test_header_is_plain_c_and_links(lib, tmp_path, std):
    """A C program includes the header under a strict C standard, links
    against libdqd.so and makes host-only calls."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    from memory_bound_decode_dq_gb300 import build
    libdir = os.path.dirname(build.build())
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    r = subprocess.run([gcc, f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), f"-L{libdir}", "-ldqd", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    version, status, codes, st = out.stdout.strip().split("|")
    assert version and status
    assert int(codes) == 256 * 1024 // 2
    assert int(st) == 1  # DQD_ERR_INVALID_ARG
