"""Oracle: global token positions held by a context-parallel rank -- test infrastructure only.

Contiguous split: "PCP and DCP sequence parallelism guide", section 3.5
(``split_sequence_for_cp``): the sequence length must divide evenly by the CP size, each rank
keeps ``local_len = seq_len // cp_size`` tokens starting at ``cp_rank * local_len``, and the
positions a rank sees stay global (same section, on position encodings).

Strided ("zig-zag") split: "Zig-Zag Ring Attention" article, section 4.2: instead of
consecutive blocks, GPU 0 takes tokens 0, 4, 8, ... and GPU 1 takes 1, 5, 9, ... (4 GPUs), so
rank ``r`` holds ``r, r + cp, r + 2 cp, ...``.

Two-block split: the same article (sections 4.2 and 5.2) states the aim of the zig-zag
assignment -- every GPU gets both early and late tokens, so causal work is even.  The
block-granular way to meet it (not printed on the pages; offered as an extra layout): cut the
sequence into ``2 cp`` equal blocks and give rank ``r`` block ``r`` and block ``2 cp - 1 - r``,
in that (ascending) order.

Work-balanced contiguous split: "PCP and DCP sequence parallelism guide", section 2.3 (load
balancing): an even split by token count leaves causal work uneven, since early tokens see
only their prefix and late tokens see everything; DCP splits by the actual distribution of
work instead.  Reading taken (the page gives no formula): contiguous blocks whose causal work is
even at token granularity.  With ``W(b) = b (b + 1) / 2`` causal pairs among the first ``b``
tokens, rank ``r`` holds ``[b_r, b_{r+1})`` where ``b_r`` is the smallest ``b`` with
``W(b) >= r W(S) / cp`` (``b_0 = 0``, ``b_cp = S``); shards then have different lengths.
"""

import math

import numpy as np

CONTIGUOUS = "contiguous"
STRIDED = "strided"
TWO_BLOCK = "two_block"
BALANCED = "balanced"


def balanced_bounds(seq_len: int, cp: int) -> list:
    """Boundaries ``[b_0, ..., b_cp]`` of the work-balanced contiguous split (see the module
    docstring).  Integer arithmetic: ``b_r`` is the smallest ``b`` with
    ``b (b + 1) cp >= r S (S + 1)``."""
    if cp <= 0 or seq_len <= 0:
        raise ValueError("seq_len and cp must be positive")
    total = seq_len * (seq_len + 1)
    bounds = [0]
    for r in range(1, cp):
        need = r * total  # compare b (b + 1) cp against this
        b = math.isqrt(need // cp)
        while b > 0 and (b - 1) * b * cp >= need:
            b -= 1
        while b * (b + 1) * cp < need:
            b += 1
        bounds.append(b)
    bounds.append(seq_len)
    if any(bounds[i] >= bounds[i + 1] for i in range(cp)):
        raise ValueError("the work-balanced split leaves a rank without tokens (seq_len too small for cp)")
    return bounds


def shard_positions(seq_len: int, cp: int, rank: int, kind: str) -> np.ndarray:
    """Global positions (int64, ascending) of the tokens rank ``rank`` holds, in local order."""
    if cp <= 0 or seq_len <= 0:
        raise ValueError("seq_len and cp must be positive")
    if not 0 <= rank < cp:
        raise ValueError("rank out of range")
    if kind == BALANCED:
        bounds = balanced_bounds(seq_len, cp)
        return np.arange(bounds[rank], bounds[rank + 1], dtype=np.int64)
    if seq_len % cp != 0:
        # the guide asserts divisibility; padding is the data pipeline's job
        raise ValueError("seq_len must be a multiple of cp")
    local_len = seq_len // cp
    if kind == CONTIGUOUS:
        start = rank * local_len
        return np.arange(start, start + local_len, dtype=np.int64)
    if kind == STRIDED:
        # every cp-th token, starting at the rank's own index
        return np.array([rank + cp * i for i in range(local_len)], dtype=np.int64)
    if kind == TWO_BLOCK:
        if seq_len % (2 * cp) != 0:
            raise ValueError("the two-block split needs seq_len to be a multiple of 2 * cp")
        block = seq_len // (2 * cp)
        early = [rank * block + i for i in range(block)]
        late = [(2 * cp - 1 - rank) * block + i for i in range(block)]
        return np.array(early + late, dtype=np.int64)
    raise ValueError(f"unknown layout kind {kind!r}")


def sub_chunk_positions(positions: np.ndarray, index: int, length: int) -> np.ndarray:
    """Positions of the ``index``-th run of ``length`` consecutive local tokens of a shard.

    A shard is sent as KV chunks of a fixed token count ("FCP" article, section 4.3, chunks of
    about 4K tokens); chunk ``index`` is local rows ``[index*length, (index+1)*length)``.
    """
    lo = index * length
    hi = lo + length
    if lo < 0 or hi > len(positions):
        raise ValueError("sub-chunk out of range")
    return np.asarray(positions[lo:hi], dtype=np.int64)


def visible_pair_count(q_pos: np.ndarray, k_pos: np.ndarray, causal: bool) -> int:
    """Number of (query, key) pairs with ``k_pos <= q_pos`` (all pairs when not causal).

    Counted by sorting the key positions and binary-searching each query position.
    """
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    if not causal:
        return int(len(q_pos) * len(k_pos))
    ks = np.sort(k_pos)
    return int(np.searchsorted(ks, q_pos, side="right").sum())
