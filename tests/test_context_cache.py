"""Host logic of the per-(device, context) cache behind the library's
one-time kernel setup (shared-memory limits, occupancy) and the static
scratch address: compiled as plain C++ against csrc/kvq_context_cache.h and
driven with made-up device numbers and context ids, no GPU involved."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "quantized_kv_cache_append_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "kvq_context_cache.h"
using kvq::ContextCache;
static int calls = 0;
static unsigned long long after = 0;
static bool ok_setup = true;
static int next_value = 100;
static int get(ContextCache<int>& c, int dev, unsigned long long ctx) {
  int v = -1;
  const bool ok = c.get(dev, ctx, &v,
                        [](int* out) { ++calls; if (!ok_setup) return false; *out = next_value++; return true; },
                        [] { return after; });
  return ok ? v : -1;
}
static void show(int v) { printf("%d %d\n", v, calls); }
int main() {
  ContextCache<int> c;
  after = 7;
  show(get(c, 0, 7));      // first use: setup
  show(get(c, 0, 7));      // same context: cached
  after = 9;
  show(get(c, 0, 9));      // new context (a reset): setup again
  show(get(c, 0, 9));
  after = 11;
  show(get(c, 1, 11));     // another device: its own slot
  show(get(c, 0, 9));      // device 0 still cached
  after = 0;
  show(get(c, 2, 0));      // unknown context: never cached
  show(get(c, 2, 0));
  after = 5;
  show(get(c, 3, 0));      // no context before, one made by the setup
  show(get(c, 3, 5));      // then cached under it
  ok_setup = false;
  show(get(c, 4, 5));      // failed setup: error, nothing stored
  ok_setup = true;
  show(get(c, 4, 5));
  show(get(c, -1, 5));     // out-of-range devices are refused
  show(get(c, 64, 5));
  return 0;
}
"""

EXPECTED = [(100, 1), (100, 1), (101, 2), (101, 2), (102, 3), (101, 3), (103, 4), (104, 5),
            (105, 6), (105, 6), (-1, 7), (106, 8), (-1, 8), (-1, 8)]


def test_context_cache_logic(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "cc.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "cc"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe), "-pthread"],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = [tuple(int(x) for x in ln.split()) for ln in out if ln.strip()]
    assert got == EXPECTED
