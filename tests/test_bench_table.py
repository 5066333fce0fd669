"""The ncu traffic table in profiles/ stays attached to a kernel only while
the kernel's code is unchanged: bench.code_hash ignores comments, trailing
blanks and empty lines, and nothing else. A row whose code hash no longer
matches its source yields no traffic figure rather than a stale one."""
import os

import bench


def _hash(tmp_path, name, text):
    p = tmp_path / name
    p.write_text(text)
    return bench.code_hash(str(p))


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    base = 'int f(int x) {\n  return x + 1;  // one\n}\n'
    same = '/* header\n   comment */\nint f(int x) {\n\n  return x + 1;   \n}\n// trailing\n'
    assert _hash(tmp_path, "a.cu", base) == _hash(tmp_path, "b.cu", same)


def test_code_hash_sees_code_and_string_changes(tmp_path):
    base = 'const char* s = "a // not a comment";\nint f(int x) { return x + 1; }\n'
    code = 'const char* s = "a // not a comment";\nint f(int x) { return x + 2; }\n'
    text = 'const char* s = "a // changed";\nint f(int x) { return x + 1; }\n'
    h = _hash(tmp_path, "a.cu", base)
    assert h != _hash(tmp_path, "b.cu", code)
    assert h != _hash(tmp_path, "c.cu", text)


def test_traffic_rows_resolve_only_while_the_code_matches():
    with open(bench.TRAFFIC_TABLE) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert rows
    for r in rows:
        path = os.path.join(bench.ROOT, "jagged_attention_recsys_gdpa_gb300", "csrc", r[2])
        match = bench.code_hash(path)[:12] == r[3]
        # scaled by algorithmic bytes: the captured case itself gets its own count back
        assert bench.ncu_traffic(r[0], r[1], float(r[5])) == (float(r[4]) if match else None), r[:4]
