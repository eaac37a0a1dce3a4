"""The boundary is a C ABI: include/kvattn.h compiles as strict C99 and as
C++, and a plain C program links against the library and drives its
host-side calls (version, status strings, the block allocator, the
multi-layer cache arithmetic) with no Python involved.  CPU only: nothing
here launches a kernel."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")
LIBDIR = os.path.join(ROOT, "kv_cache_attention_rope_gb300")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "kvattn.h"

int main(void)
{
    kvattn_allocator* a = NULL;
    int32_t ids[4], row[4] = {-1, -1, -1, -1}, child[4] = {-1, -1, -1, -1}, src = 0, dst = 0;
    kvattn_config cfg = {32, 8, 128, KVATTN_BF16, 10000.0f, 0.0f};
    kvattn_cache layer;
    if (kvattn_version() != KVATTN_VERSION) return 1;
    if (strcmp(kvattn_status_string(KVATTN_ERR_OUT_OF_BLOCKS), "out of KV blocks") != 0) return 2;
    if (kvattn_allocator_create(8, &a) != KVATTN_OK) return 3;
    if (kvattn_alloc_blocks(a, 4, ids) != KVATTN_OK || kvattn_allocator_num_free(a) != 4) return 4;
    if (kvattn_alloc_blocks(a, 5, ids) != KVATTN_ERR_OUT_OF_BLOCKS || kvattn_allocator_num_failures(a) != 1) return 5;
    if (kvattn_free_blocks(a, ids, 4) != KVATTN_OK || kvattn_allocator_num_free(a) != 8) return 6;
    /* a 20-token sequence, a fork of it, and an append that copies the shared partial block */
    if (kvattn_table_grow(a, row, 4, 16, 0, 20) != KVATTN_OK) return 7;
    if (kvattn_table_fork(a, row, child, 4, 16, 20) != KVATTN_OK || kvattn_allocator_refcount(a, row[1]) != 2) return 8;
    if (kvattn_table_prepare_append(a, child, 4, 16, 20, 21, &src, &dst) != KVATTN_OK) return 9;
    if (src != row[1] || dst != child[1] || kvattn_allocator_refcount(a, row[1]) != 1) return 10;
    if (kvattn_table_release(a, child, 4, 16, 21) != KVATTN_OK) return 11;
    if (kvattn_table_release(a, row, 4, 16, 20) != KVATTN_OK || kvattn_allocator_num_free(a) != 8) return 12;
    kvattn_allocator_destroy(a);
    /* layer 3 of a 4-layer cache: regions 6 and 7 of the allocation */
    if (kvattn_layer_cache(&cfg, (void*)(size_t)0x10000, 4, 100, 16, 3, &layer) != KVATTN_OK) return 13;
    if ((size_t)layer.k_pool != 0x10000 + 6u * 100u * 8u * 16u * 128u * 2u) return 14;
    if (kvattn_layered_cache_bytes(&cfg, 4, 100, 16) != 8u * 100u * 8u * 16u * 128u * 2u) return 15;
    printf("ok\n");
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None or shutil.which("g++") is None, reason="no C compiler")
def test_header_is_strict_c_and_cxx():
    for cmd in (["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only", "-x", "c"],
                ["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-x", "c++"]):
        r = subprocess.run(cmd + [os.path.join(INC, "kvattn.h")], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_plain_c_program_drives_the_host_calls(tmp_path):
    if not os.path.exists(os.path.join(LIBDIR, "libkvattn.so")):
        pytest.skip("library not built")
    src = tmp_path / "prog.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "prog"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", INC, str(src), "-o", str(exe),
                        "-L", LIBDIR, "-lkvattn", "-Wl,-rpath," + LIBDIR], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
