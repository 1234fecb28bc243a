"""include/wq4.h is a C header. A C11 program that includes it compiles with gcc under -Wall
-Wextra -pedantic -Werror, links against libwq4.so and calls the entry points that need no GPU:
the sizes, the status texts, the build flag and the argument rules, which reject bad calls before
any CUDA work. The C example in README.md compiles against it too. Runs without a GPU."""
import os
import shutil
import subprocess

import pytest

import weight_only_quantized_wq4_gb300 as wq4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUT = os.path.join(ROOT, "weight_only_quantized_wq4_gb300", "_build", "c_header")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "wq4.h"

#define EXPECT(cond) do { if (!(cond)) { printf("failed: %s\n", #cond); return 1; } } while (0)

int main(void) {
    const void* X = (const void*)0x10000;   /* 16-byte aligned stand-ins, never dereferenced */
    const void* W = (const void*)0x20000;
    void* Y = (void*)0x30000;
    int rec[4] = {1, 1, 1, 1};
    size_t ws = 1;
    EXPECT(wq4_version() >= 100);
    EXPECT(strcmp(wq4_status_string(WQ4_OK), "ok") == 0);
    EXPECT(strcmp(wq4_status_string(WQ4_ERR_BOUNDS), "unknown status") != 0);
    /* a blob: a 256-byte header, then per 128 x 128 tile one 8448-byte record (8192 bytes of
       4-bit codes, 256 bytes of bf16 scales) */
    EXPECT(wq4_prepacked_bytes(4096, 4096, 128, WQ4_U4B8) == 256 + (size_t)32 * 32 * 8448);
    EXPECT(wq4_prepacked_bytes(100, 4096, 128, WQ4_U4B8) == 0);
    EXPECT(wq4_debug_checks() == 0);
    EXPECT(wq4_last_violation(rec) == 0 && rec[0] == 0 && rec[3] == 0);
    EXPECT(wq4_last_violation(NULL) == WQ4_ERR_INVALID);
    EXPECT(wq4_mm(X, W, Y, -1, 128, 128, 128, WQ4_BF16, WQ4_U4B8, NULL, 0, NULL) == WQ4_ERR_INVALID);
    EXPECT(wq4_mm(NULL, W, Y, 8, 128, 128, 128, WQ4_BF16, WQ4_U4B8, NULL, 0, NULL) == WQ4_ERR_INVALID);
    EXPECT(wq4_mm(X, W, Y, 8, 100, 128, 128, WQ4_BF16, WQ4_U4B8, NULL, 0, NULL) == WQ4_ERR_UNSUPPORTED);
    EXPECT(wq4_mm(X, W, Y, 0, 128, 128, 128, WQ4_BF16, WQ4_U4B8, NULL, 0, NULL) == WQ4_OK);
    EXPECT(wq4_workspace_bytes(-1, 128, 128, 128, &ws) == WQ4_ERR_INVALID);
    EXPECT(wq4_set_option(-12345, 0) == WQ4_ERR_INVALID);
    printf("ok\n");
    return 0;
}
"""


@pytest.fixture(scope="module")
def built():
    return wq4.build()


def test_c_program_compiles_links_and_runs(built):
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("no gcc")
    os.makedirs(OUT, exist_ok=True)
    src = os.path.join(OUT, "use_wq4.c")
    exe = os.path.join(OUT, "use_wq4")
    with open(src, "w") as f:
        f.write(PROGRAM)
    libdir = os.path.dirname(built)
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        src, "-o", exe, "-L", libdir, "-l:libwq4.so", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_readme_c_example_compiles():
    """The C example in README.md compiles against wq4.h and the CUDA runtime header."""
    import re
    gcc, cuda_inc = shutil.which("gcc"), "/usr/local/cuda/include"
    if not gcc or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("no gcc or CUDA headers")
    with open(os.path.join(ROOT, "README.md")) as f:
        blocks = re.findall(r"```c\n(.*?)```", f.read(), flags=re.S)
    assert len(blocks) == 1
    os.makedirs(OUT, exist_ok=True)
    src = os.path.join(OUT, "readme_example.c")
    with open(src, "w") as f:
        f.write(blocks[0])
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only", "-I", cuda_inc,
                        "-I", os.path.join(ROOT, "include"), src], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
