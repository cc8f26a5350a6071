"""The stamp that ties a traffic capture to the step kernel's sources hashes
their code only: comments and blank lines do not change it, code does, and
string and character literals are kept whole."""
from precision_states_gb300 import build as b


def test_code_only_drops_comments_keeps_literals():
    src = ('int a = 1; // note\n/* block\n comment */ const char* s = "x//y/*z*/";\n'
           "char q = '/';  \n\n\tb++;\n")
    assert b.code_only(src) == 'int a = 1;\n const char* s = "x//y/*z*/";\nchar q = \'/\';\n\tb++;'


def test_comment_edits_keep_the_stamp_and_code_edits_change_it(tmp_path, monkeypatch):
    f = tmp_path / "k.cuh"
    monkeypatch.setattr(b, "CSRC", str(tmp_path))
    f.write_text("// header\nint f(int x) { return x + 1; }\n")
    s0 = b.source_stamp(["k.cuh"])
    f.write_text("// a longer header\n\n/* and a block */\nint f(int x) { return x + 1; }  // trailing\n")
    assert b.source_stamp(["k.cuh"]) == s0
    f.write_text("// header\nint f(int x) { return x + 2; }\n")
    assert b.source_stamp(["k.cuh"]) != s0


def test_committed_traffic_records_match_the_current_sources():
    """profiles/traffic.json holds DRAM counters for the step kernel as it
    was when they were taken; the bench reports them only while the stamp
    matches.  A source change without a new capture must show here, not as
    a silently null figure in the bench line."""
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles", "traffic.json")
    with open(path) as fh:
        records = json.load(fh)
    assert records
    want = b.source_stamp(b.STEP_KERNEL_SOURCES)
    for name, rec in records.items():
        assert rec["source_stamp"] == want, name
