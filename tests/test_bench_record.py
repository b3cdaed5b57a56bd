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



def test_reference_config_matches_library_group():
    """Both arms print the same workload config: the reference arm computes the
    group's size from the oracle planner with the library's member alignment,
    and it equals what the library's own group placement gives."""
    import argparse

    import block_quant_gb300 as bq
    import workloads as W

    args = argparse.Namespace(members=None, muon=True, workload=bench.WORKLOAD)
    ref = bench.reference_config(args, 1)
    cfg = W.config(bench.WORKLOAD)
    lays = [bq.plan(u.tensors, cfg.V, cfg.alpha, cfg.start_align) for u in cfg.units]
    g = bq.Group([(lays[u], cfg.dev_lo, cfg.dev_hi) for u, unit in enumerate(cfg.units) for _ in range(unit.repeat)])
    assert ref["members"] == len(g.place) == 82
    assert ref["elements"] + ref["padding_elements"] == g.info["elems"]
    tabs = [W.Table(lay.export()) for lay in lays]
    assert ref["elements"] == sum(int(t.dev_intervals(0, 1)[:, 3].sum()) * u.repeat for t, u in zip(tabs, cfg.units))
