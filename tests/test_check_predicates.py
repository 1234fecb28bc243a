"""The debug build's bounds predicates (csrc/wq4_check.h), compiled for the host with g++ and
checked at their boundaries against the rules they state:
  - a tiled tensor copy's innermost coordinate times the element size is a multiple of 16 bytes,
    and its box lies inside the tensor;
  - a byte range lies inside its buffer;
  - a scheduled tile holds at least one token, its 128 weight rows lie inside N, and its group
    range is non-empty and inside K.
Also checked: in a release build the check macro is the constant true, with its condition never
evaluated. Runs without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "weight_only_quantized_wq4_gb300", "csrc")
OUT = os.path.join(ROOT, "weight_only_quantized_wq4_gb300", "_build", "check_host")

DRIVER = r"""
#include <cstdio>
#include <cstring>
#include "wq4_check.h"
using namespace wq4::check;
int main() {
    char op[16];
    while (std::scanf("%15s", op) == 1) {
        long long v[8] = {0};
        if (!std::strcmp(op, "tma")) {
            std::scanf("%lld %lld %lld %lld", v, v + 1, v + 2, v + 3);
            std::printf("%d\n", tma_x_ok(v[0], (int)v[1], (int)v[2], v[3]) ? 1 : 0);
        } else if (!std::strcmp(op, "span")) {
            std::scanf("%lld %lld %lld %lld", v, v + 1, v + 2, v + 3);
            std::printf("%d\n", span_ok(v[0], v[1], v[2], v[3]) ? 1 : 0);
        } else if (!std::strcmp(op, "al")) {
            std::scanf("%lld", v);
            std::printf("%d\n", aligned16((unsigned long long)v[0]) ? 1 : 0);
        } else if (!std::strcmp(op, "tile")) {
            for (int i = 0; i < 8; ++i) std::scanf("%lld", v + i);
            std::printf("%d\n", tile_ok((int)v[0], (int)v[1], (int)v[2], (int)v[3], (int)v[4], (int)v[5], (int)v[6],
                                        (int)v[7]) ? 1 : 0);
        } else if (!std::strcmp(op, "macro")) {
            int evaluated = 0;
            const bool r = WQ4_CHECK((++evaluated, false), nullptr, nullptr, kSiteTile, 0, 0, 0);
            std::printf("%d %d %d\n", r ? 1 : 0, evaluated, wq4::kDebugChecks ? 1 : 0);
        }
    }
    return 0;
}
"""

# (case, expected): expected answers from the rules above, worked out by hand
CASES = [
    # TMA innermost coordinate: 16-bit elements need x % 8 == 0, 8-bit x % 16, 32-bit x % 4, 64-bit x % 2
    ("tma 0 2 128 4096", 1), ("tma 8 2 64 4096", 1), ("tma 4 2 64 4096", 0), ("tma 64 2 64 128", 1),
    ("tma 4 4 64 4096", 1), ("tma 2 4 64 4096", 0), ("tma 2 8 2 4096", 1), ("tma 1 8 1 4096", 0),
    ("tma 16 1 16 4096", 1), ("tma 8 1 16 4096", 0), ("tma -8 2 64 4096", 0),
    # the box inside the tensor: [4032, 4096) fits a 4096-wide tensor, [4040, 4104) does not
    ("tma 4032 2 64 4096", 1), ("tma 4040 2 64 4096", 0), ("tma 4096 2 64 4096", 0), ("tma 0 2 128 64", 0),
    # byte ranges
    ("span 0 8448 0 8448", 1), ("span 1 8448 0 8448", 0), ("span -16 16 0 100", 0), ("span 100 0 0 100", 1),
    ("span 0 -1 0 100", 0), ("span 8448 8448 0 270336", 1), ("span 261888 8448 0 270336", 1),
    ("span 261904 8448 0 270336", 0),
    # 16-byte alignment
    ("al 0", 1), ("al 4096", 1), ("al 4104", 0), ("al 65537", 0), ("al 48", 1),
    # tiles: m-tile mt of NT tokens holds a token iff mt * NT < rows; n-tile nt fits iff (nt + 1) * 128 <= N;
    # groups [g0, g1) non-empty inside [0, k_groups)
    ("tile 0 128 1 0 128 0 32 32", 1), ("tile 1 128 128 0 128 0 32 32", 0), ("tile 1 128 129 0 128 0 32 32", 1),
    ("tile 2 192 385 2 384 0 8 8", 1), ("tile 0 192 100 3 384 0 8 8", 0), ("tile -1 16 100 0 128 0 1 1", 0),
    ("tile 0 16 100 -1 128 0 1 1", 0), ("tile 0 16 100 0 128 3 3 8", 0), ("tile 0 16 100 0 128 7 8 8", 1),
    ("tile 0 16 100 0 128 7 9 8", 0), ("tile 0 16 100 0 128 -1 2 8", 0), ("tile 0 16 0 0 128 0 8 8", 0),
]


@pytest.fixture(scope="module")
def driver():
    gxx = shutil.which("g++")
    if not gxx:
        pytest.skip("no g++")
    os.makedirs(OUT, exist_ok=True)
    src = os.path.join(OUT, "check_driver.cpp")
    exe = os.path.join(OUT, "check_driver")
    with open(src, "w") as f:
        f.write(DRIVER)
    r = subprocess.run([gxx, "-std=c++17", "-O1", "-Wall", "-I", CSRC, src, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def run(exe, lines):
    r = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    return r.stdout.split("\n")


def test_predicates_at_their_boundaries(driver):
    got = run(driver, [c for c, _ in CASES])
    for (case, want), g in zip(CASES, got):
        assert int(g) == want, "%s: got %s, want %d" % (case, g, want)


def test_release_macro_is_true_and_unevaluated(driver):
    assert run(driver, ["macro"])[0].split() == ["1", "0", "0"]
