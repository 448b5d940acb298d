"""The boundary from a plain C caller (no GPU, no Python in the call path).

A C99 program includes include/gqa_attn.h, links libgqa_attn.so and, without a
device, calls the entry points that answer on the host: the version and status
strings, the size queries, and refusals of bad arguments. It also takes the
address of every function the header declares, so the link fails if one is
missing. This shows the header is valid C and the library is usable without
torch.
"""
import os
import re
import shutil
import subprocess

import pytest

import gqa_causal_attention_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_attn.h")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "gqa_attn.h"

typedef void (*any_fn)(void);
static any_fn all_fns[] = { %(fns)s };

int main(void) {
    int bad = 0;
    for (size_t i = 0; i < sizeof(all_fns) / sizeof(all_fns[0]); ++i)
        if (!all_fns[i]) bad |= 1;
    if (strcmp(attn_status_string(ATTN_OK), "ok") != 0) bad |= 2;
    attn_rope_params rp;
    memset(&rp, 0, sizeof rp);
    rp.theta = 10000.0;
    rp.max_positions = 100;
    /* 100 positions x 8 pairs x (cos, sin) x 4 bytes at D = 16 */
    if (attn_rope_table_bytes(&rp, 16) != 100 * 8 * 2 * 4) bad |= 4;
    if (gqa_attn_prefill_workspace_size(1, 2, 16, 64) < 2 * 64 * 16 * 4) bad |= 8;
    /* refused on the host before anything could be launched */
    if (gqa_attn_prefill(NULL, NULL, NULL, NULL, 1, 4, 2, 16, 64, 0, 0.f, 0.f, NULL, 0, NULL,
                         NULL) != ATTN_ERR_NULL) bad |= 16;
    if (gqa_attn_prefill((const float*)16, (const float*)16, (const float*)16, (float*)16,
                         1, 6, 4, 16, 64, 0, 0.f, 0.f, NULL, 0, NULL, NULL) != ATTN_ERR_SHAPE)
        bad |= 32;
    if (attn_selftest_wait_timeout(NULL, NULL) != ATTN_ERR_NULL) bad |= 64;
    printf("%%s %%d\n", attn_version(), bad);
    return bad;
}
"""


def _declared():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_plain_c_program_links_and_calls_the_library(tmp_path):
    lib = g.library_path()
    g.load()                                           # builds the library if needed
    src = tmp_path / "caller.c"
    fns = ", ".join(f"(any_fn){n}" for n in _declared())
    src.write_text(PROGRAM % {"fns": fns})
    exe = tmp_path / "caller"
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-Wno-pedantic",
                    "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
                    "-L", libdir, "-lgqa_attn", "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.split()[-1] == "0" and run.stdout.count(".") == 2
