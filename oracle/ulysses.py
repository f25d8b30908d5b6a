"""Oracle: the Ulysses sequence <-> head reshard as an index formula -- test infrastructure only.

"Halo context parallelism (CP + Ulysses attention)", section "Ulysses attention: three
all-to-alls for one exact computation": before the exchange each of the ``cp`` ranks holds
``S/cp`` tokens of every head; after it, rank ``r`` holds all ``S`` tokens of ``H/cp`` heads.
Q is exchanged once, K and V once (fused), the output once more in the reverse direction.

Reading taken where the page is silent: rank ``r`` receives heads ``[r*H/cp, (r+1)*H/cp)``
(with contiguous GQA groups this keeps each Q group with its KV head -- the page's example,
cp=4 with 64 Q / 8 KV heads, gives 16 Q heads and 2 KV heads per rank), and a token lands at
row = its global position, so the result is in global sequence order for any shard layout.

    seq -> head:  Y_r[pos_s(i), j, :] = X_s[i, r*H/cp + j, :]
    head -> seq:  X_s[i, r*H/cp + j, :] = Y_r[pos_s(i), j, :]
"""

import numpy as np


def seq_to_head(x_shards, positions):
    """x_shards: cp arrays [S/cp, H, D]; positions: cp int arrays of global positions.

    Returns cp arrays [S, H/cp, D].
    """
    cp = len(x_shards)
    if cp == 0 or len(positions) != cp:
        raise ValueError("need one position array per shard")
    local, heads, d = x_shards[0].shape
    if heads % cp != 0:
        raise ValueError("head count must be a multiple of cp")
    hl = heads // cp
    seq = local * cp
    out = [np.zeros((seq, hl, d), dtype=x_shards[0].dtype) for _ in range(cp)]
    for r in range(cp):
        for s in range(cp):
            out[r][np.asarray(positions[s])] = x_shards[s][:, r * hl:(r + 1) * hl, :]
    return out


def head_to_seq(y_shards, positions):
    """y_shards: cp arrays [S, H/cp, D]; positions as in ``seq_to_head``.

    Returns cp arrays [S/cp, H, D].
    """
    cp = len(y_shards)
    if cp == 0 or len(positions) != cp:
        raise ValueError("need one position array per shard")
    seq, hl, d = y_shards[0].shape
    local = seq // cp
    out = [np.zeros((local, hl * cp, d), dtype=y_shards[0].dtype) for _ in range(cp)]
    for s in range(cp):
        pos = np.asarray(positions[s])
        for r in range(cp):
            out[s][:, r * hl:(r + 1) * hl, :] = y_shards[r][pos]
    return out
