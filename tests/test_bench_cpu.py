"""Host-side pieces of bench.py that decide what the JSON line reports.

The DRAM traffic of the dominant kernel comes from a recorded ncu capture and
is reported only while the kernel sources still hash to the key recorded with
it.  The hash ignores comments and whitespace (an edit to either leaves the
kernels, and their counters, as they were) and changes with any code.
"""
import json
import os

import bench


def test_code_only_drops_comments_and_whitespace():
    src = 'int a = 1; // one\n/* block\n comment */ float  b=2.0f;\n'
    assert bench._code_only(src) == "inta=1;floatb=2.0f;"


def test_code_only_keeps_string_and_char_literals():
    # comment markers inside literals are code, not comments (whitespace goes
    # everywhere, inside literals too: the result is only ever hashed)
    src = 'const char *s = "a // b /* c */"; char q = \'/\'; // tail\n'
    assert bench._code_only(src) == 'constchar*s="a//b/*c*/";charq=\'/\';'
    # an escaped quote does not end the literal
    assert bench._code_only('x = "a\\"//b"; // c') == 'x="a\\"//b";'


def test_code_only_separates_code_edits_from_comment_edits():
    a = "int f(int x) { return x + 1; }  // add one\n"
    comment_edit = "int f(int x) {\n    return x + 1;   /* plus one */\n}\n"
    code_edit = "int f(int x) { return x + 2; }  // add one\n"
    assert bench._code_only(a) == bench._code_only(comment_edit)
    assert bench._code_only(a) != bench._code_only(code_edit)


def test_traffic_reported_only_for_the_recorded_sources(monkeypatch):
    """A traffic record counts only while the kernel sources hash to its key:
    the bench reports the recorded bytes then, and null once the code changed."""
    with open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json"), encoding="utf-8") as fh:
        rec = json.load(fh)
    for k in ("tc_cols", "tc_fused"):
        monkeypatch.setattr(bench, "kernel_src_sha", lambda: rec[k]["kernel_src_sha"])
        assert bench.ncu_traffic(k) == rec[k]["bytes_per_launch"]
        monkeypatch.setattr(bench, "kernel_src_sha", lambda: "0" * 16)
        assert bench.ncu_traffic(k) is None
    assert bench.ncu_traffic("no_such_kernel") is None
