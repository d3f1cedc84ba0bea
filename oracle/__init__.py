"""fp64 CPU oracle for exact softmax attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import or call it. It shares no code with the CUDA path in
``online_softmax_09_gb300/`` and imports nothing from it.

Sources (web pages, cited by title and section):

* [P1] "FlashAttention Implementation > How FlashAttention Uses Tiling"
  (mbrenndoerfer.com): "The Running Statistics", "Why the Correction Factor
  Works", and the memory bound M_flash = O(n d + B_r B_c).
* [P2] "FlashAttention - Compute attention in tiles" (divagr.pages.dev,
  attention-lab): "Tiling and online softmax", "Numerical accuracy".
* [P3] "LLM Architecture Refresh [3]: Flash Attention Is Exact, and Here's the
  Proof" (bearbearyu1223.github.io): section 1 (standard attention), section 2
  (online softmax), section 3 (partial softmaxes compose), section 4 (tiled
  attention), section 5 (causal mask), section 7 (causal skipping), section 8
  (FLOP and byte counters; backward by recomputation).

Every function in :mod:`oracle.attention` is pinned by a ``-m "not gpu"`` test
against something other than itself (printed values of the pages, closed
forms, a library routine, brute force, finite differences). The one quantity
the pages print but whose input data they do not give -- the "2 of 31 blocks
rescaled" count for a real 2,048-logit row -- is "parity unpinned"; its counter
is pinned only on synthetic rows with known answers.
"""

from .attention import (  # noqa: F401
    algorithmic_flops,
    attention_backward,
    attention_backward_head,
    attention_backward_rows,
    attention_forward,
    attention_forward_head,
    attention_probs,
    attention_query_block,
    attention_rows,
    attention_split_forward_head,
    brute_force_attention,
    causal_tile_counts,
    naive_counts,
    online_softmax,
    tile_schedule_counts,
    tiled_attention,
)
