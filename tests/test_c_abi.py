"""The C ABI from plain C: include/kvq.h compiles as strict C99 (gcc
-std=c99 -pedantic -Werror), a C program links libkvq.so, and its host-only
calls give what the binding gives (sizes), refuse what they must before any
launch, and plan a streamed pool's residency (no GPU involved)."""
import os
import shutil
import subprocess

import pytest

import quantized_kv_cache_append_gb300 as kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    kvq.build()
    lib = kvq.LIB_PATH
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_host")
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_host.c"),
                    lib, "-Wl,-rpath," + os.path.dirname(lib), "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return dict(line.split(" ", 1) for line in out.strip().splitlines())


def test_sizes_match_the_binding(program):
    got = [int(x) for x in program["block_bytes"].split()]
    want = [kvq.kvq_block_bytes(kvq.KVQ_F16, 8, 128, 256), kvq.kvq_block_bytes(kvq.KVQ_Q8, 8, 128, 256),
            kvq.kvq_block_bytes(kvq.KVQ_K8V4, 2, 256, 256)]
    assert got == want
    # K8V4 at 2 KV heads of 256 dims: 816 bytes a cell
    assert got[2] == 816 * 256


def test_refusals_before_any_launch(program):
    assert int(program["append"]) == kvq.KVQ_ERR_ARG
    assert int(program["decode"]) == kvq.KVQ_ERR_ARG
    assert int(program["workspace"]) == 0


def test_residency_plan_from_c(program):
    assert program["plan"].split() == ["0", "fetch", "3", "hits", "0"]
    # misses take the free slots in first-use order
    assert program["pairs"].split() == ["4:0", "1:1", "5:2"]
    # the row's entries: blocks 4, 1, 5 in slots 0, 1, 2; block 2 not resident
    assert program["slots"].split() == ["0", "1", "2", "-1"]
    assert program["again"].split() == ["0", "fetch", "0", "hits", "3"]


def test_e2e_host_program_builds_and_refuses_bad_arguments(tmp_path):
    """tests/e2e_host.c (the bench's end-to-end step from plain C) compiles
    against the header and the library; without arguments it prints its
    usage and exits 1 before touching a device."""
    import importlib
    kb = importlib.import_module("quantized_kv_cache_append_gb300.build")   # the module, not build()
    if not os.path.exists(kb._nvcc()):
        pytest.skip("no nvcc")
    kvq.build()
    exe = str(tmp_path / "e2e_host")
    subprocess.run([kb._nvcc(), "-O2", "-o", exe, os.path.join(ROOT, "tests", "e2e_host.c"), "-I",
                    kb.INCLUDE, "-L", kb.BUILD_DIR, "-lkvq", "-Xlinker", f"-rpath,{kb.BUILD_DIR}"],
                   check=True, capture_output=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 1 and "usage" in r.stderr
    r = subprocess.run([exe, "0", "1", "1"], capture_output=True, text=True)
    assert r.returncode == 1
