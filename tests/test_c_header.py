"""The boundary is a C ABI: include/gbattn.h must compile as plain C99 on its own, and a C
program must link every declared entry point against libgbattn.so.  The program also runs
the calls that need no GPU (version, status strings, size and plan queries, argument
checks)."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import streaming_attention_flashattention_gb300 as gb  # noqa: E402

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "gbattn.h"

typedef void (*any_fn)(void);

int main(void) {
    /* every entry point is a C symbol the program can take the address of */
    any_fn fns[] = {
        (any_fn)attn_fwd, (any_fn)attn_fwd_counted, (any_fn)attn_fwd_host_workspace_size, (any_fn)attn_fwd_host,
        (any_fn)attn_prefill_kvcache, (any_fn)attn_decode_workspace_size,
        (any_fn)attn_decode_workspace_bytes,
        (any_fn)attn_decode_splitkv, (any_fn)attn_decode_multitoken_workspace_size,
        (any_fn)attn_decode_multitoken, (any_fn)attn_decode_splitkv_noalloc,
        (any_fn)attn_decode_plan, (any_fn)attn_prefill_plan, (any_fn)attn_last_device_error,
        (any_fn)attn_selftest_bounded_wait, (any_fn)attn_status_string, (any_fn)attn_version};
    for (size_t i = 0; i < sizeof fns / sizeof fns[0]; ++i)
        if (!fns[i]) return 10;
    if (attn_version() < 100) return 11;
    if (strcmp(attn_status_string(GBATTN_OK), "ok") != 0) return 12;
    /* host-only queries */
    if (attn_decode_workspace_bytes(4, 64, 8, 1, 32768, 128, 16, 152) == 0) return 13;
    int plan[7];
    if (attn_decode_plan(4, 64, 8, 1, 32768, 128, 16, 152, plan) != GBATTN_OK) return 14;
    if (plan[0] != 16 || plan[1] != 0 || plan[3] != 1024 || plan[6] != 2) return 15;
    int pp[4];
    if (attn_prefill_plan(1, 64, 8, 8192, 8192, 1, 152, pp) != GBATTN_OK) return 16;
    if (pp[0] != 0 || pp[1] != 2048 || pp[3] != 4096) return 17;
    /* argument checks come before any device work */
    if (attn_fwd(0, 0, 0, 0, 0, 1, 2, 1, 128, 128, 128, 0.1f, 0, GBATTN_BF16, 0)
        != GBATTN_ERR_INVALID_ARG) return 18;
    if (attn_fwd_counted((void*)0x10000, (void*)0x10000, (void*)0x10000, (void*)0x20000, 0, 1, 2,
                         1, 128, 128, 128, 0.1f, 0, 0, 0) != GBATTN_ERR_INVALID_ARG) return 19;
    printf("c abi ok\n");
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    from streaming_attention_flashattention_gb300 import build
    build.build()
    gb.load_library()
    return gb.LIBRARY_PATH


def test_header_is_c99_and_links(tmp_path, lib_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_gbattn.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "use_gbattn"
    libdir = os.path.dirname(lib_path)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-l:libgbattn.so", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    assert "c abi ok" in run.stdout
