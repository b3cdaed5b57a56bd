"""The committed DRAM-traffic record that bench.py reports beside the roofline:
it is keyed on the kernel's code (comments and blank lines ignored), so an edit
of the commentary keeps it and any code change drops it (traffic: null)."""

import os

import bench


def _write(tmp_path, name, text):
    p = os.path.join(tmp_path, name)
    with open(p, "w") as f:
        f.write(text)
    return p


def test_code_digest_ignores_comments_only(tmp_path):
    base = 'int f(int x) {  // doubles\n  return 2 * x;  /* twice */\n}\nconst char* s = "a // b";\n'
    a = _write(tmp_path, "a.cu", base)
    b = _write(tmp_path, "b.cu", "// header\n\n" + base.replace("// doubles", "// times two") + "\n/* tail\n */\n")
    c = _write(tmp_path, "c.cu", base.replace("2 * x", "3 * x"))
    d = _write(tmp_path, "d.cu", base.replace('"a // b"', '"a // c"'))  # inside a string: code
    assert bench.code_digest([a]) == bench.code_digest([b])
    assert bench.code_digest([a]) != bench.code_digest([c])
    assert bench.code_digest([a]) != bench.code_digest([d])

