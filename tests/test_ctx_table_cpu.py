"""The per-context address table behind pcp_attn_varlen_noalloc.

The scratch array's device address belongs to one CUDA context; a device
reset ends that context and the next one may place the array elsewhere. The
table (``csrc/ctx_table.h``, plain C++) keys the address by the context's
process-unique ID. This test compiles a small program against the header with
g++ on the CPU: an ID never seen gives nothing (a new context looks the address
up again), an entry is replaced in place, and a full table drops its oldest
entry.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "context_prefill_attention_gb300", "csrc")

PROGRAM = r"""
#include <stdio.h>
#include "ctx_table.h"
int main() {
    pcp::CtxTable<4> t;
    int a = 0, b = 0, c = 0;
    if (t.find(1) != nullptr) return 1;
    t.put(1, &a);
    if (t.find(1) != &a) return 2;
    if (t.find(2) != nullptr) return 3;          /* a later context: not found */
    t.put(2, &b);
    if (t.find(2) != &b || t.find(1) != &a) return 4;
    t.put(1, &c);                                 /* same context: replaced */
    if (t.find(1) != &c) return 5;
    t.put(3, &a);
    t.put(4, &a);
    t.put(5, &b);                                 /* full: the oldest slot (ID 1) goes */
    if (t.find(1) != nullptr) return 6;
    if (t.find(5) != &b || t.find(2) != &b || t.find(3) != &a || t.find(4) != &a) return 7;
    puts("ok");
    return 0;
}
"""


def test_ctx_table_keys_by_context_id(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    src = tmp_path / "t.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "t"
    subprocess.check_call([gxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, str(src), "-o", str(exe)])
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout)
