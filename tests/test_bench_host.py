"""Host-side logic of bench.py that needs no GPU: the kernel-source hash that keys the
committed ncu traffic table."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_only_drops_comments_not_code():
    src = ('int a = 1;  // trailing\n/* block\n comment */ const char* s = "x//y/*z*/";\n'
           "char q = '\"';\nint b = 2; /* inline */ int c = 3;\n")
    out = bench.code_only(src)
    assert "trailing" not in out and "block" not in out and "inline" not in out
    assert '"x//y/*z*/"' in out  # comment markers inside a string are code
    assert "char q = '\"';" in out
    assert out.startswith("int a = 1; ") and out.endswith("int c = 3;")


def test_comment_edits_keep_the_hash_code_edits_change_it():
    base = "int f(int x) {\n    return x + 1;  // add one\n}\n"
    assert bench.code_only(base) == bench.code_only(base.replace("add one", "increment"))
    assert bench.code_only(base) == bench.code_only("int f(int x) { return x + 1; }")
    assert bench.code_only(base) != bench.code_only(base.replace("x + 1", "x + 2"))


def test_traffic_table_is_keyed_by_a_current_hash_or_reads_null():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        table = json.load(f)
    h = bench.kernel_hash()
    assert len(h) == 16 and all(c in "0123456789abcdef" for c in h)
    for workload, row in table.items():
        got = bench.load_traffic(workload)
        if row["kernel_hash"] == h:
            assert got == row["traffic_bytes_per_launch"]
        else:
            assert got is None
