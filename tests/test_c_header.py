"""include/attn.h from plain C, and the binding against the header (no GPU).

The boundary is a C ABI, so the header must compile as C (not only as the
C++ the library is built from), a C program must link against libattn.so
and get its argument errors back without any GPU, and the Python binding's
ctypes signatures must match the header's parameter lists type by type: a
size_t passed as an int, or a dropped argument, would otherwise shift every
later argument in the call without any error.
"""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from exact_io_aware_attn_gb300 import _lib, build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def libpath():
    build_mod.build()
    _lib.lib()
    return _lib.LIB_PATH


def header_declarations():
    """{name: (return type, [parameter types])} for every function attn.h
    declares, types normalised ("const" dropped, single spaces, '*' attached)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"#[^\n]*", "", text)

    def norm(t):
        t = re.sub(r"\bconst\b", "", t)
        t = re.sub(r"\s*\*\s*", "*", t)
        return " ".join(t.split())

    decls = {}
    for m in re.finditer(r"([A-Za-z_][\w \t\*]*?)\b(attn_[a-z_]+)\s*\(([^)]*)\)\s*;", text):
        ret, name, params = norm(m.group(1)), m.group(2), m.group(3).strip()
        types = []
        if params and params != "void":
            for p in params.split(","):
                p = " ".join(p.split())
                p = re.sub(r"\s*\*\s*", "*", p)
                types.append(norm(re.sub(r"\b\w+$", "", p)))  # drop the parameter name
        decls[name] = (ret, types)
    return decls


RET = {"attn_status_t": ctypes.c_int, "int": ctypes.c_int, "size_t": ctypes.c_size_t,
       "char*": ctypes.c_char_p}
ARG = {"int": ctypes.c_int, "float": ctypes.c_float, "size_t": ctypes.c_size_t,
       "unsigned int": ctypes.c_uint, "unsigned int*": ctypes.POINTER(ctypes.c_uint)}


def ctype_of_param(t):
    if t in ARG:
        return ARG[t]
    assert t.endswith("*"), f"unmapped parameter type {t!r}"
    return ctypes.c_void_p  # every other pointer is an address the binding passes through


def test_header_parses_to_every_declared_function():
    decls = header_declarations()
    assert len(decls) == len(_lib.SIGNATURES) >= 20
    assert decls["attn_fwd"] == ("attn_status_t", ["void*"] * 3 + ["void*", "float*"] +
                                 ["int"] * 5 + ["float", "int", "int", "void*"])


def test_binding_signatures_match_the_header():
    for name, (ret, params) in header_declarations().items():
        res, args = _lib.SIGNATURES[name]
        assert res is RET[ret], f"{name}: return {ret} bound as {res}"
        assert len(args) == len(params), f"{name}: {len(params)} parameters, {len(args)} bound"
        for i, (t, a) in enumerate(zip(params, args)):
            assert a is ctype_of_param(t) or a == ctype_of_param(t), \
                f"{name}: parameter {i} is {t}, bound as {a}"


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "attn.h"

/* Every call below fails validation or only computes a size, so nothing
   touches a GPU. Exits non-zero on the first unexpected result. */
int main(void) {
  char buf[64];
  attn_status_t st;
  if (attn_abi_version() != ATTN_ABI_VERSION) return 1;
  if (strcmp(attn_status_string(ATTN_ERR_WORKSPACE), "ATTN_ERR_WORKSPACE") != 0) return 2;
  /* d = 96 is outside the supported set */
  st = attn_fwd((const void*)0x1000, (const void*)0x2000, (const void*)0x3000, (void*)0x4000,
                (float*)0x5000, 1, 1, 8, 8, 96, 0.125f, 0, ATTN_BF16, NULL);
  if (st != ATTN_ERR_UNSUPPORTED) return 3;
  /* a null q */
  st = attn_fwd(NULL, (const void*)0x2000, (const void*)0x3000, (void*)0x4000, (float*)0x5000,
                1, 1, 8, 8, 64, 0.125f, 0, ATTN_F16, NULL);
  if (st != ATTN_ERR_INVALID_ARG) return 4;
  /* an empty problem is a valid no-op */
  st = attn_fwd(NULL, NULL, NULL, NULL, NULL, 0, 4, 8, 8, 64, 0.125f, 1, ATTN_BF16, NULL);
  if (st != ATTN_OK) return 5;
  /* decode workspace: one partial of d + 4 floats per (b, h, split) */
  if (attn_workspace_bytes(2, 3, 1, 1000, 64, 16) != (size_t)2 * 3 * 16 * 68 * 4) return 6;
  if (attn_bwd_workspace_bytes(1, 2, 100, 100, 64) != (size_t)8 * 2 * 128) return 7;
  /* the allocation-free decode rejects partials beyond its fixed scratch
     (4096 x 32 heads x 64 splits x 132 floats); fake addresses 2^36 apart so
     that no tensor overlaps another */
  st = attn_fwd_decode_noalloc((const void*)(1ull << 36), (const void*)(2ull << 36),
                               (const void*)(3ull << 36), (void*)(4ull << 36),
                               (float*)(5ull << 36), 4096, 32, 1000, 128, 0.088f, ATTN_BF16,
                               64, NULL);
  if (st != ATTN_ERR_WORKSPACE) return 8;
  snprintf(buf, sizeof buf, "%s", attn_status_string(12345));
  if (strcmp(buf, "ATTN_ERR_UNKNOWN") != 0) return 9;
  printf("ok\n");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_is_plain_c_and_links(libpath, tmp_path):
    src = tmp_path / "abi_check.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi_check"
    libdir = os.path.dirname(libpath)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
           libpath, f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    # no GPU visible: every call here must return before touching CUDA, so a
    # regression that moved a check after a launch fails with ATTN_ERR_CUDA
    # instead of launching kernels on the fake addresses
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
