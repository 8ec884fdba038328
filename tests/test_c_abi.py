"""The C ABI from plain C: include/int8kv.h compiles as C99 (warnings as
errors), and a C program linked against libint8kv.so calls the host-only
entry points (the split geometry, workspace sizes, the prefill split rule,
status names) and agrees with the ctypes binding.  No device is touched."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")
LIBDIR = os.path.join(ROOT, "int8_kv_cache_gb300")

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")

C_SRC = r"""
#include "int8kv.h"
#include <stdio.h>

int main(void) {
  int32_t ns = 0, chunk = 0;
  i8kv_status st = split_geometry(2048, 16, 152, 64, 128, 32, I8KV_GEOM_POW2_TILES, 0, &ns,
                                  &chunk);
  printf("%d %d %d\n", (int)st, (int)ns, (int)chunk);
  st = split_geometry(4096, 32, 608, 16, 128, 32, I8KV_GEOM_WAVE, 0, &ns, &chunk);
  printf("%d %d %d\n", (int)st, (int)ns, (int)chunk);
  printf("%lu\n", (unsigned long)split_workspace_bytes(16, 8, 12, 256));
  printf("%d\n", (int)dsa_prefill_auto_splits(128, 24, 2, 152));
  printf("%lu\n", (unsigned long)dsa_prefill_workspace_bytes(16, 24, 2, 256, 300, 100, 3));
  printf("%s\n", i8kv_status_string(I8KV_EWORKSPACE));
  printf("%d\n", (int)i8kv_version());
  return 0;
}
"""


def test_header_compiles_as_c99_and_links(tmp_path):
    lib_path = os.path.join(LIBDIR, "libint8kv.so")
    if not os.path.exists(lib_path):
        pytest.skip("libint8kv.so not built")
    src = tmp_path / "abi.c"
    src.write_text(C_SRC)
    exe = tmp_path / "abi"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INC,
                        str(src), "-L", LIBDIR, "-lint8kv", f"-Wl,-rpath,{LIBDIR}", "-o",
                        str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, run.stderr
    lines = run.stdout.strip().split("\n")

    lib = ctypes.CDLL(lib_path)
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    geo = lib.split_geometry
    geo.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32),
                    ctypes.POINTER(i32)]
    geo.restype = i32

    def geometry(*args):
        ns, ch = i32(), i32()
        st = geo(*args, ctypes.byref(ns), ctypes.byref(ch))
        return f"{st} {ns.value} {ch.value}"
    assert lines[0] == geometry(2048, 16, 152, 64, 128, 32, 1, 0)
    assert lines[1] == geometry(4096, 32, 608, 16, 128, 32, 0, 0)
    lib.split_workspace_bytes.restype = ctypes.c_size_t
    lib.split_workspace_bytes.argtypes = [i32] * 4
    assert int(lines[2]) == lib.split_workspace_bytes(16, 8, 12, 256)
    lib.dsa_prefill_auto_splits.restype = i32
    lib.dsa_prefill_auto_splits.argtypes = [i32] * 4
    assert int(lines[3]) == lib.dsa_prefill_auto_splits(128, 24, 2, 152) == 6
    lib.dsa_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.dsa_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32, i64, i32, i32]
    assert int(lines[4]) == lib.dsa_prefill_workspace_bytes(16, 24, 2, 256, 300, 100, 3) > 0
    assert "workspace" in lines[5]
    assert int(lines[6]) == 300
