"""Host check of the CTA-pair kernel's token tiling (pair_tile_width / pair_tile_count in csrc/internal.h), compiled
with the host compiler: for every member count up to 70,000 the tiles cover the rows exactly, each holds at most 256
rows in a multiple of 32, there are ceil(rows / 256) of them, and never more than the single-CTA kernel's 128-row
tiles (the workspace's tile-list capacity is sized for those)."""

import os
import shutil
import subprocess

import pytest

from conftest import ROOT

SRC = r"""
#include "internal.h"
#include <cstdio>
using namespace moe;
int main() {
  for (int rows = 0; rows <= 70000; ++rows) {
    const int w = pair_tile_width(rows), c = pair_tile_count(rows);
    if (rows == 0) { if (w != 0 || c != 0) { printf("rows 0: %d %d\n", w, c); return 1; } continue; }
    if (w <= 0 || w > 256 || w % 32) { printf("width %d for %d rows\n", w, rows); return 1; }
    if (c * w < rows || (c - 1) * w >= rows) { printf("cover %d rows: %d x %d\n", rows, c, w); return 1; }
    if (c != (rows + 255) / 256) { printf("count %d for %d rows\n", c, rows); return 1; }
    if (c > (rows + 127) / 128) { printf("capacity %d for %d rows\n", c, rows); return 1; }
  }
  printf("ok\n");
  return 0;
}
"""


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda.h")):
            return os.path.join(d, "include")
    return None


def test_pair_token_tiles_cover_rows(tmp_path):
    inc = _cuda_include()
    cxx = shutil.which("g++")
    if inc is None or cxx is None:
        pytest.skip("needs g++ and the CUDA headers")
    src = tmp_path / "tiles.cpp"
    src.write_text(SRC)
    exe = tmp_path / "tiles"
    csrc = os.path.join(ROOT, "expert_major_chunked_gb300", "csrc")
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-I", csrc, "-I", inc, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
