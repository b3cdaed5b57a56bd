"""Plain CPU oracle for the DBuffer step — TEST INFRASTRUCTURE ONLY.

This package restates, slowly and literally, what the veScale-FSDP pages say the
data-parallel hot path computes, so that the CUDA path can be checked against it.
It is not part of the product: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  It
shares no code with ``block_quant_gb300`` (neither package imports the other).

Modules
-------
planner   RaggedShard layout problem: earliest-fit feasibility, the prefix /
          binary-search heuristic, brute-force optimum, invariants, derived
          interval and scale-slot tables, flat export format.
codecs    bf16 round-to-nearest-even, OCP FP8 E4M3 encode/decode, linear absmax
          int8 / uint8 block quantisers.
pack      group-level pre-communication add / scale / zero / copy into the DBuffer.
adam8     block-wise 8-bit Adam step (dequantise, fp32 update, requantise), in the
          operation order the kernels reproduce bit for bit (the contract leg).
fp8       128x128 block FP8 requantisation of the updated parameters (contract leg).
plain     the same Adam step and FP8 requantisation in the plainest operation order
          (every fp32 operation separate, division by the scales and the bias
          corrections): the textbook definition the kernels are measured against.
muon      Newton-Schulz orthogonalisation in fp64.

Sources (cited per function): "veScale-FSDP: Flexible and High-Performance FSDP at
Scale" (bud-325.pages.dev summary: TL;DR, Key claims, Method), the feynmanwiki
walkthrough "veScale-FSDP: Flexible, Structure-Aware Sharding at 10K-GPU Scale"
(paper sections 4-6 in prose), the mlsanity abstract page.  Where those pages are
silent the reading taken is stated in the function's docstring.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against
brute force, closed forms or a library routine; none is "parity unpinned".
"""

from . import codecs, planner, pack, adam8, fp8, muon, plain  # noqa: F401
