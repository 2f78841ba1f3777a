"""CPU oracle for the DeepSeek Sparse Attention (MLA) forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, helpers or tables) and never
takes an input or an expected value from it.

Modules:
  dsa_oracle  the definition of the forward, written out in float64 (numpy):
              gather, full (non-online) softmax, weighted sum, lse.
  emu         the pages' blockwise online-softmax algorithm with skip-scale,
              emulated step by step in float32 with the bf16 cast of S.
  formats     bit-level decoders of bf16, FP8-e4m3 and FP4-e2m1 and of the
              656-byte FP8 and 448-byte FP4 KV rows.
  paged       logical positions of a sequence -> rows of a paged KV pool
              through a block table (the forward itself is unchanged).
  out_proj    the output projection with residual that follows the
              attention, y = O . W_o + x, in float64.

Every function is pinned by ``tests/test_oracle*.py`` against values fixed by
the pages or by mathematics (closed forms, invariants, brute force, library
routines reached by an independent route).
"""
