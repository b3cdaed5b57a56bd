"""Planner study on model-shaped tensor groups, with the library's planner:

* padding of one layer unit against the row granularity (1x, 16x, 128x rows)
  across FSDP sizes, on a GPT-OSS-120B layer (experts fused into one tensor) and
  a DeepSeek-V3-671B MoE layer (the two models of the walkthrough's padding
  figure, paper section 6.4: below 3% at 1x / 16x rows, step-like spikes up to
  about 18% for GPT-OSS at 128x rows);
* the three placement orders the walkthrough names (paper section 5: given,
  by block size, by shape) on every configuration's units.

Shapes only (synthetic): GPT-OSS d = 2880, 64 query / 8 key-value heads of 64,
128 experts of width 2880; DeepSeek-V3 d = 7168, multi-head latent attention
(q rank 1536, kv rank 512, 128 heads of 128 + 64 rotary), 256 routed experts of
width 2048 plus one shared, each expert its own gate / up / down tensors (the
pages single out GPT-OSS for fusing its experts into one tensor).  2-D tensors
take exactly rows x cols granularity, 1-D tensors 32 elements.

    python -m workloads.planner_study            # markdown tables
"""

import time

import numpy as np

from . import TensorSpec, config, _gptoss_layer


def gptoss_layer():
    return _gptoss_layer(2880, 64, 8, 64, 128, 2880, 256, False)


def deepseek_v3_moe_layer():
    d, heads, qr, kvr, nope, rope, vd, ne, fe = 7168, 128, 1536, 512, 128, 64, 128, 256, 2048
    T = lambda n, r, c: TensorSpec(n, r, c, 1, 0, False)  # noqa: E731 (g set by the sweep)
    return [
        T("attn_norm", 1, d),
        T("q_a", qr, d), T("q_a_norm", 1, qr), T("q_b", heads * (nope + rope), qr),
        T("kv_a", kvr + rope, d), T("kv_a_norm", 1, kvr), T("kv_b", heads * (nope + vd), kvr),
        T("o", d, heads * vd),
        T("mlp_norm", 1, d),
        T("router", ne, d), T("router_bias", 1, ne),
    ] + [t for e in range(ne) for t in (T(f"e{e}_gate", fe, d), T(f"e{e}_up", fe, d), T(f"e{e}_down", d, fe))] + [
        T("shared_gate", fe, d), T("shared_up", fe, d), T("shared_down", d, fe),
    ]


def padding_sweep(tensors, rows_gran, Vs, alpha=128, start_align=16):
    """[(V, S, padding fraction, plan seconds)] with 2-D granularity rows_gran rows."""
    import block_quant_gb300 as bq

    # exact row granularity: placement ignores the optimizer kind, and the Muon
    # kind accepts any g for 2-D tensors; 1-D tensors take 32-element blocks
    descs = [(t.rows, t.cols, 32, 3, 0) if t.rows == 1 else (t.rows, t.cols, rows_gran * t.cols, 2, 0)
             for t in tensors]
    total = sum(t.rows * t.cols for t in tensors)
    out = []
    for V in Vs:
        t0 = time.perf_counter()
        L = bq.plan(descs, V, alpha, start_align)
        dt = time.perf_counter() - t0
        S = L.info()["S"]
        out.append((V, S, 1 - total / (V * S), dt))
    return out


def order_study(names):
    """{(config, unit, order): padding fraction}."""
    import block_quant_gb300 as bq

    res = {}
    for name in names:
        c = config(name)
        for u in c.units:
            total = sum(t.numel for t in u.tensors)
            for order in (0, 1, 2):
                S = bq.plan(u.tensors, c.V, c.alpha, c.start_align, order).info()["S"]
                res[(name, u.name, order)] = 1 - total / (c.V * S)
    return res


def main():
    Vs = [8, 16, 32, 64, 128, 256, 512, 1024]
    print("| layer | rows | " + " | ".join(f"V={v}" for v in Vs) + " | max | max plan s |")
    print("|---|---|" + "---|" * (len(Vs) + 2))
    for lname, ts in (("GPT-OSS-120B", gptoss_layer()), ("DeepSeek-V3", deepseek_v3_moe_layer())):
        for rows in (1, 16, 128):
            r = padding_sweep(ts, rows, Vs)
            cells = " | ".join(f"{100 * p:.2f}%" for _, _, p, _ in r)
            print(f"| {lname} | {rows}x | {cells} | {100 * max(p for _, _, p, _ in r):.2f}% | "
                  f"{max(t for *_, t in r):.3f} |")
    print()
    names = ["toy", "llama3-8b-layer", "llama3-70b-rank0", "gpt-oss-120b-rank0", "llama3-8b-layer-tile32"]
    res = order_study(names)
    print("| config / unit | given | by block size | by shape |")
    print("|---|---|---|---|")
    for (name, unit, order), p in res.items():
        if order == 0:
            print(f"| {name} / {unit} | " + " | ".join(f"{100 * res[(name, unit, o)]:.3f}%" for o in (0, 1, 2)) + " |")


if __name__ == "__main__":
    main()
