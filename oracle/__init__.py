"""Reference oracle for context-parallel blockwise attention -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct CPU restatement (numpy, float64) of what the
per-rank hot path computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it.  The library in ``context_blockwise_attention_gb300`` never
imports, calls or links anything here, and nothing here imports the library: the two share no
code.  Inputs for both sides come from the seeded generators in
``context_blockwise_attention_gb300.workloads`` (random numbers only, none of the method).

Sources (pages are cited by title and section):

* "FCP: from a fixed ring to a free topology" (lqnn.cn/news/264049), section 3.3
  "attention computation re-ordering": scores are ``q . k^T / sqrt(head_dim)``, softmax
  normalised by the running maximum and sum, output = accumulator / sum; the result must not
  depend on the order in which KV blocks arrive.
* "PCP and DCP sequence parallelism guide" (hmyw.cn/news/122838), section 2.3 (numerical
  stability: global max, then local exp, then global sum, then normalise), section 4.2
  (``global_softmax``), section 3.5 (``split_sequence_for_cp``: rank ``r`` takes the contiguous
  block starting at ``r * local_len``; positions stay global).
* "Zig-Zag Ring Attention" article (intelliparadigm.com, article 2133809), section 4.2:
  with 4 GPUs, GPU 0 takes tokens 0, 4, 8, ... and GPU 1 takes 1, 5, 9, ...
* "Halo context parallelism (CP + Ulysses attention)" (sheratonhq.com/news/191935), section
  "Ulysses attention: three all-to-alls for one exact computation": each rank holds S/cp tokens
  of all heads; the exchange gives it all S tokens of H/cp heads; exact because heads are
  independent.  Example: cp=4, 64 Q heads / 8 KV heads -> 16 Q heads per rank.  The backward
  pass runs the same exchanges in reverse; the guide above (section 2.3, gradient handling)
  reduce-scatters the gradients of the split sequence.  ``backward.py`` writes out the chain
  rule of the attention definition, whole and per KV chunk.

Pins (what the oracle is checked against, in ``tests/test_oracle_pins.py``): pure-Python
brute force on tiny inputs (softmax computed without max-subtraction, and the FCP article's
blockwise online accumulation with shuffled block order), closed forms (Q = 0, constant V,
causal row 0, K = 0), central finite differences of the brute-force forward for the gradients,
the sum over chunks of the per-chunk gradients, a library special case (``torch.nn.functional.scaled_dot_product_attention``
in float64), merge invariants (permutation, associativity) and the worked layout examples the
pages print (``tests/golden/``).  Planted-mistake tests show each pin family fails on a
plausible bug.
"""

from .layouts import shard_positions, sub_chunk_positions, visible_pair_count
from .attention import attention, merge
from .backward import attention_backward, chunk_backward
from .ulysses import seq_to_head, head_to_seq

__all__ = [
    "shard_positions",
    "sub_chunk_positions",
    "visible_pair_count",
    "attention",
    "merge",
    "attention_backward",
    "chunk_backward",
    "seq_to_head",
    "head_to_seq",
]
