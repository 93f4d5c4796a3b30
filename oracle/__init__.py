"""CPU oracle for the ring-attention forward.

THIS PACKAGE IS TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (``context_ring_attention_gb300``) never imports, calls or links
anything in here, and nothing in here imports the product: the two share no code.

Everything is plain numpy in float64, written from the method's definition on the
source pages:

* "Module 23: Distributed Training" (learnllm.pages.dev), sections "The Math: One
  Block at a Time", "Exact by Construction", "The Causal Imbalance — and the
  Striped Fix";
* "Explain ring attention and how it enables very long contexts across multiple
  devices?" (Transformer Architecture Q&A), sections "The ring" and "The
  causal-mask problem";
* "3.6 Distributed Training II: Tensor, Pipeline, Sequence & Expert Parallelism",
  section "Ring Attention".

Functions and what pins each one (tests in ``tests/test_oracle_pins.py``):

==========================  ===============================================================
``layout_positions``        the per-device causal pair counts printed in "The Causal
                            Imbalance" (contiguous and striped, exact integers); bijection;
                            zigzag's exact balance (the reading of "paired up
                            block-by-block").
``causal_pair_counts``      the same printed counts (golden fixture).
``to_natural``              inverts the layout map (round trips for every layout; the contiguous
                            layout is the identity).
``full_attention``          scipy.special.softmax / logsumexp on small cases; closed forms
                            (one key, identical keys, causal row 0); row sums of 1;
                            GQA head mapping against per-head single-head calls.
``full_attention_rows``     equals ``full_attention`` row by row.
``attention_rows``          equals ``full_attention`` row by row (causal, by position).
``ring_sim``                the Q&A page's 4-device toy (seed 1) equals ordinary attention;
                            Module 23's (2,4,96,32) example, full and causal, within the
                            page's 1e-5; layout invariance after un-permuting.
``ring_partials``           merging them reproduces ``full_attention``.
``pass_blocks``,            after t exchanges slot p holds the block that started in slot
``held_blocks``             (p - t) mod N (labelled rows); N exchanges are the identity;
                            attention over the held block equals ``ring_partials`` entry t.
``attention_backward``      central finite differences of ``full_attention`` (float64) on tiny
                            cases, causal and not, with grouped heads; a single key gives
                            dV = dO and dQ = dK = 0; the rows of dK sum to zero; row blocks
                            give the same gradients as the whole.
``attention_backward_rows`` through ``attention_backward`` (which is built from it) the finite
                            differences above; on its own, a subset of query rows gives
                            those rows' dQ, and the key-row parts of all query rows split
                            into subsets add up to dK and dV.
``ring_backward``           equals ``attention_backward`` for every layout, causal and not.
``ulysses_seq_to_head``,    labelled rows land on the device of their head at their position;
``ulysses_head_to_seq``     the two exchanges are inverse; exchange, per-device attention,
                            exchange back equals attention over the whole sequence.
``merge_partials``          splitting the keys into halves and merging reproduces
                            ``full_attention``; -inf parts are ignored.
``tile_counts``             brute force over every (q, k) pair of every tile on small
                            shapes; closed forms at 128x128 tiles.
==========================  ===============================================================

No function here is "parity unpinned".
"""

from .layouts import CONTIGUOUS, STRIPED, ZIGZAG, LAYOUTS, layout_positions, causal_pair_counts, to_natural
from .attention import attention_rows, full_attention, full_attention_rows
from .ring import ring_sim, ring_partials, pass_blocks, held_blocks
from .merge import merge_partials
from .backward import attention_backward, attention_backward_rows, ring_backward
from .ulysses import ulysses_seq_to_head, ulysses_head_to_seq
from .tiles import tile_counts, tile_classes_bruteforce

__all__ = [
    "CONTIGUOUS", "STRIPED", "ZIGZAG", "LAYOUTS",
    "layout_positions", "causal_pair_counts", "to_natural",
    "full_attention", "full_attention_rows", "attention_rows",
    "ring_sim", "ring_partials", "pass_blocks", "held_blocks", "merge_partials",
    "attention_backward", "attention_backward_rows", "ring_backward", "ulysses_seq_to_head", "ulysses_head_to_seq",
    "tile_counts", "tile_classes_bruteforce",
]
