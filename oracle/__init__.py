"""CPU oracle for the W4A16 single-token decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or call
anything in this package.  The product library never routes through it, and the
oracle never imports the product package: the two share no code.

What it computes is the plain definition of each step, in float64 NumPy, written
from the source pages:

* "How to build your own LLM runtime from scratch (Towards Data Science)" -- the
  wiki summary of the build-log; section "What it actually builds" names
  symmetric group-wise INT4 weights (group 128), the paged KV cache of 16 tokens
  per 4 KiB page, the fused Q/K/V/O and gate/up/down GEMVs and greedy sampling.
* "How To Build Your Own LLM Runtime From Scratch | daily.dev" -- section
  "Questions this post answers", second question: softmax must stay correct at
  partial KV tail pages.
* "Build Crude Implementations for Learning" -- section "Paged KV cache": a
  request's tokens live in non-contiguous blocks reached through a block table.

Module map:

* ``quant``  -- symmetric group-128 quantisation, the packed nibble format, unpack.
* ``gemv``   -- dequantise-then-matvec in float64.
* ``paged``  -- KV append into pages, and attention by gathering pages into a
  contiguous array followed by a two-pass softmax.
* ``model``  -- RMSNorm, RoPE, SwiGLU, the Qwen2-style decode step, argmax, and
  the prompt pass (the decode step over each prompt token in turn).
* ``w4a8``   -- the INT8-activation variant the pages measured and dropped
  (activations quantised per 128-group, exact integer group dots).

Pins (``tests/test_oracle_*.py``) tie every function to values fixed by the
pages or by mathematics: hand-worked packed words, closed forms, brute force on
tiny inputs and invariants.  The end-to-end decode step is the composition of
pinned ops, and is itself pinned by two symmetries (relabelled hidden groups;
relabelled KV heads with their query groups) that a misrouted, transposed or
misgrouped projection breaks, by an identity (layers with zero output and
down projections leave the embedding -> final norm -> LM head path), which a
dropped residual breaks, by a closed gate that silences the MLP exactly,
which gate and up swapped breaks, and by a cancellation (attention built to add
exactly minus the embedding zeroes every logit), which a sign-flipped residual
breaks.  No published logits exist to compare the composed step with.
"""

from . import quant, gemv, paged, model  # noqa: F401
