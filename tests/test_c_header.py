"""The public header is plain C: a C99 program that includes only
include/lioncub.h compiles with -std=c99 -pedantic -Werror, links against
liblioncub.so, sees the documented struct sizes, and gets the documented
codes from calls that fail validation before touching the device."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include "lioncub.h"
#include <stdio.h>
#include <string.h>

static int fails = 0;
#define CHECK(c) do { if (!(c)) { printf("failed: %s\n", #c); ++fails; } } while (0)

int main(void)
{
    lioncub_t h = 0;
    lioncub_tensor bad[2] = {{0, 40, 0}, {40, 24, 0}};
    void* p = (void*)1;
    CHECK(sizeof(lioncub_tensor) == 24);
    CHECK(sizeof(lioncub_diag) == 48);
    CHECK(lioncub_create(&h, 100, 0, NULL, 0, 0.9f, 0.99f, 1e-4f, 0.1f, LIONCUB_MODE_SIGN_MAJORITY, 1,
                         LIONCUB_GRAD_BF16, 0) == LIONCUB_ERR_ARG);
    CHECK(strstr(lioncub_last_error(NULL), "W=0") != NULL);
    CHECK(lioncub_create(&h, 64, 2, bad, 2, 0.9f, 0.99f, 1e-4f, 0.1f, LIONCUB_MODE_L1_INTSUM, 4,
                         LIONCUB_GRAD_F32, 1) == LIONCUB_ERR_ALIGN);
    CHECK(h == NULL);
    CHECK(lioncub_step(NULL, NULL, NULL) == LIONCUB_ERR_ARG);
    CHECK(lioncub_wire_words(NULL) == -1);
    CHECK(lioncub_host_alloc(&p, 0) == LIONCUB_OK && p == NULL);
    CHECK(strcmp(lioncub_strerror(LIONCUB_ERR_OOM), "LIONCUB_ERR_OOM") == 0);
    lioncub_destroy(NULL);
    lioncub_host_free(NULL);
    printf("%s\n", fails ? "FAIL" : "OK");
    return fails != 0;
}
"""


def test_header_is_c99_and_links(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from communication_compressed_sign_gb300 import build
    lib = build.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib)
    r = subprocess.run([cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", f"-I{ROOT}/include", str(src),
                        f"-L{libdir}", "-llioncub", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr
