"""Host logic of the prompt-chunk attention's key splits: how many CTAs of a
cluster share the key tiles of one (row tile, KV head) pair.  Compiled as
plain C++ against csrc/kvq_key_splits.h and driven with made-up SM counts
and resident-cluster counts, no GPU involved.  Each expected count is worked
out by hand from the cost (waves of clusters) x (tiles per split) + 2 below
its case."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "quantized_kv_cache_append_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "kvq_key_splits.h"
static int calls = 0;
static int cap = 8;   // cluster sizes above cap cannot be resident
// an idealised GPU of 152 SMs: floor(152 / ns) clusters of ns CTAs at once
static int maxc(int ns) { ++calls; return ns > cap ? 0 : 152 / ns; }
static void show(long long base, int n_all, int sms) {
  calls = 0;
  const int s = kvq::choose_key_splits(base, n_all, sms, maxc);
  printf("%d %d\n", s, calls);
}
int main() {
  show(152, 4096, 152);  // as many pairs as SMs: no split, no query
  show(64, 1024, 0);     // unknown SM count: no split
  show(64, 7, 152);      // 7 tiles: no split keeps four tiles each
  show(64, 1024, 152);
  show(16, 1024, 152);
  cap = 4;
  show(16, 1024, 152);   // clusters above 4 cannot be resident
  cap = 8;
  show(16, 20, 152);     // at most 5 splits of four tiles
  show(100, 64, 152);
  return 0;
}
"""

EXPECTED = [
    (1, 0),
    (1, 0),
    (1, 0),
    # base 64, 1024 tiles: unsplit 1 wave x 1024 = 1024; ns 2: 76 clusters,
    # 1 wave x 512 + 2 = 514; ns 3: 50, 2 x 342 + 2 = 686; ns 4: 38,
    # 2 x 256 + 2 = 514; ns 5: 30, 3 x 205 + 2; ns 6: 25, 3 x 171 + 2 = 515;
    # ns 7: 21, 4 x 147 + 2; ns 8: 19, 4 x 128 + 2 = 514: 2 (ties keep the
    # smaller count), 7 queries
    (2, 7),
    # base 16: every ns fits in one wave, 1024 / ns + 2 falls with ns: 8
    (8, 7),
    # ns 5..8 cannot be resident: the best of 2..4 is 4 (256 + 2)
    (4, 7),
    # 20 tiles: ns up to 5; ns 5: 1 x 4 + 2 = 6 against ns 4: 1 x 5 + 2 = 7
    (5, 4),
    # base 100, 64 tiles: unsplit 64; ns 2: 2 x 32 + 2 = 66; ns 3: 50
    # clusters, 2 x 22 + 2 = 46; ns 4: 3 x 16 + 2 = 50; ns 5: 4 x 13 + 2 = 54;
    # ns 6: 4 x 11 + 2 = 46 (not below); ns 7: 5 x 10 + 2 = 52;
    # ns 8: 6 x 8 + 2 = 50: 3
    (3, 7),
]


def test_key_split_choice(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "ks.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "ks"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = [tuple(int(x) for x in ln.split()) for ln in out if ln.strip()]
    assert got == EXPECTED
