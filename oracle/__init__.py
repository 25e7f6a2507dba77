"""Plain, slow CPU oracle for one EAGLE / EAGLE-2 draft-and-verify round.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code, header, table or constant generator with the CUDA library
under ``eagle_feature_level_gb300/``; the two meet only in the seeded inputs
of ``eagle_synth``.

Floating point runs in fp64 (numpy), from bf16 weights converted exactly.
Discrete decisions that the method leaves to sampling use exact integer
arithmetic (Python ints), so that a decision never depends on summation
order.  Each function cites the passage of the three source pages it
follows:

  * Page A: "EAGLE 推测解码为什么比 Medusa 快？（含 EAGLE-2 动态草稿树）"
    (zzszmyf.github.io notes, chapter 04)
  * Page B: "eagle-feature-level-speculative-decoding"
    (charlestar.github.io, 2026-06-09)
  * Page C: "EAGLE 完全拆解：特征级草稿模型如何把投机解码推到 3 倍以上"
    (pinghaoyang.com.cn)

Functions whose result is a reading of a silent passage rather than a
checked definition say "parity unpinned" in their docstring.  Unpinned:
the decoder layer's internal conventions beyond what the parameter-count
table fixes (RMSNorm eps, rotate-half RoPE with theta 10000, norm placement)
and the static tree templates.
"""
