"""The chunk scorer's work split (host code, no GPU): every CTA gets an even
share of the visible key tiles, the ranges cover every visible tile once, and
each range starts on a visible tile. A chunk query t at pos0 sees
min((pos0 + t + 1) // 4, n_comp) compressed rows ("【#3】ds4.c を読み解く" §3:
chunks keep absolute positions); a query group's tiles are those with a row
visible to its last query."""
import pathlib
import shutil
import subprocess

import pytest

ROOT = pathlib.Path(__file__).resolve().parents[1]
CSRC = ROOT / "compressed_kv_sparse_gb300" / "csrc"

PROG = r"""
#include <cstdio>
#include <cstdlib>
#include "split.h"
int main(int argc, char **argv) {
  const uint32_t batch = atoi(argv[1]), T = atoi(argv[2]), qg = atoi(argv[3]);
  const uint32_t pos0 = atoi(argv[4]), n_comp = atoi(argv[5]), grid = atoi(argv[6]);
  const uint32_t rows = 128, n_groups = (T + qg - 1) / qg;
  const uint32_t vis_max = std::min((pos0 + T) / 4, n_comp);
  const uint32_t tiles_per = (vis_max + rows - 1) / rows;
  std::vector<uint32_t> start(grid + 1);
  ds4a::split_visible_tiles(batch, T, qg, pos0, n_comp, rows, n_groups, tiles_per, grid,
                            start.data());
  printf("%u %u\n", n_groups, tiles_per);
  for (uint32_t j = 0; j <= grid; ++j) printf("%u\n", start[j]);
  return 0;
}
"""


@pytest.fixture(scope="module")
def prog(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    d = tmp_path_factory.mktemp("split")
    src, exe = d / "split.cpp", d / "split"
    src.write_text(PROG)
    subprocess.run([cxx, "-O1", "-std=c++17", "-I", str(CSRC), str(src), "-o", str(exe)],
                   check=True)
    return exe


def visible(tile, g, T, qg, pos0, n_comp):
    last = min(T, (g + 1) * qg) - 1
    vis = min((pos0 + last + 1) // 4, n_comp)
    return tile * 128 < vis


@pytest.mark.parametrize("batch,T,qg,pos0,n_comp,grid", [
    (1, 4096, 4, 28672, 8192, 152),    # the benchmarked chunk
    (1, 4096, 4, 0, 1024, 152),        # a first chunk: visible rows grow from 0
    (2, 37, 4, 3001, 760, 152),        # ragged group count, more CTAs than tiles
    (3, 1000, 4, 123, 281, 7),         # few CTAs
    (1, 4096, 4, 28672, 7500, 152),    # rows capped by the cache
])
def test_split_even_and_complete(prog, batch, T, qg, pos0, n_comp, grid):
    out = subprocess.run([str(prog), *map(str, (batch, T, qg, pos0, n_comp, grid))],
                         check=True, capture_output=True, text=True).stdout.split()
    n_groups, tiles_per = int(out[0]), int(out[1])
    start = [int(x) for x in out[2:]]
    total = batch * n_groups * tiles_per
    assert len(start) == grid + 1 and start[0] == 0 and start[-1] == total
    assert all(a <= b for a, b in zip(start, start[1:]))

    def is_vis(item):
        tile = item % tiles_per
        g = (item // tiles_per) % n_groups
        return visible(tile, g, T, qg, pos0, n_comp)

    counts = [sum(1 for it in range(a, b) if is_vis(it)) for a, b in zip(start, start[1:])]
    n_vis = sum(1 for it in range(total) if is_vis(it))
    assert sum(counts) == n_vis                          # every visible tile once
    assert max(counts) - min(counts) <= 1                # an even share
    for a, b in zip(start, start[1:]):
        if a < b and a < total:
            assert is_vis(a)                             # ranges start on a visible tile
