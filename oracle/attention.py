"""Oracle: exact softmax attention and the (O, LSE) merge in float64 -- test infrastructure only.

The method is exact, so the oracle is the plain definition, not the blockwise algorithm.

Attention ("FCP" article, section 3.3; "PCP and DCP" guide, section 4.2): for query row ``i``
with global position ``p_i`` and head ``h``, the visible key set is every key when not causal
and the keys with global position ``p_k <= p_i`` when causal.  With ``s_j = scale * q . k_j``
(``scale = 1/sqrt(head_dim)``):

    M   = max_j s_j
    Z   = sum_j exp(s_j - M)
    O   = sum_j exp(s_j - M) v_j / Z
    LSE = M + ln Z                    (natural log)

Query head ``h`` reads KV head ``h // (Hq // Hkv)`` (native GQA: "Halo" article, Ulysses
section; the grouping itself is not printed on the pages -- contiguous groups are the reading
taken).  A row with no visible key has ``O = 0`` and ``LSE = -inf`` (the pages do not cover it;
the pseudocode read literally would divide 0 by 0).

Merge ("PCP and DCP" guide, section 2.3 numerical stability and section 4.2 ``global_softmax``):
global maximum first, then the exponentials against it and their global sum, then normalise.
In terms of partials ``(O_i, LSE_i)``:

    M   = max_i LSE_i
    w_i = exp(LSE_i - M)
    O   = sum_i w_i O_i / sum_i w_i
    LSE = M + ln sum_i w_i

A partial with ``LSE_i = -inf`` has weight 0; if every partial is ``-inf`` the result is
``O = 0``, ``LSE = -inf``.
"""

import math

import numpy as np

_ROW_BLOCK = 64


def _as_f64(x):
    if hasattr(x, "detach"):  # torch tensor (any dtype) -> exact widening
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def attention(q, k, v, q_pos, k_pos, causal=True, scale=None, rows=None):
    """Exact attention of (a subset of) the query rows against one key set.

    q: [Sq, Hq, D]; k, v: [Skv, Hkv, D]; q_pos: [Sq]; k_pos: [Skv] (global positions).
    rows: optional 1-D array of query row indices (default: all rows).
    Returns (O [n, Hq, D] float64, LSE [n, Hq] float64).
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    sq, hq, d = q.shape
    skv, hkv, dk = k.shape
    if v.shape != k.shape or dk != d:
        raise ValueError("k and v must be [Skv, Hkv, D] with the query's D")
    if hq % hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if len(q_pos) != sq or len(k_pos) != skv:
        raise ValueError("position arrays must match the token counts")
    group = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rows = np.arange(sq) if rows is None else np.asarray(rows, dtype=np.int64)
    n = len(rows)
    out = np.zeros((n, hq, d), dtype=np.float64)
    lse = np.full((n, hq), -np.inf, dtype=np.float64)
    if skv == 0 or n == 0:
        return out, lse
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        for h in range(hq):
            kh = k[:, h // group, :]
            vh = v[:, h // group, :]
            for b0 in range(0, n, _ROW_BLOCK):
                rr = rows[b0:b0 + _ROW_BLOCK]
                s = scale * (q[rr, h, :] @ kh.T)  # [b, Skv]
                if causal:
                    visible = k_pos[None, :] <= q_pos[rr][:, None]
                    s = np.where(visible, s, -np.inf)
                m = s.max(axis=1)
                has = np.isfinite(m)
                e = np.exp(s - np.where(has, m, 0.0)[:, None])  # masked keys -> exp(-inf) = 0
                z = e.sum(axis=1)
                o = (e @ vh) / np.where(has, z, 1.0)[:, None]
                out[b0:b0 + len(rr), h, :] = np.where(has[:, None], o, 0.0)
                lse[b0:b0 + len(rr), h] = np.where(has, m + np.log(np.where(has, z, 1.0)), -np.inf)
    return out, lse


def merge(o_parts, lse_parts):
    """Combine partials (O_i [.., D], LSE_i [..]) over the same query rows into exact attention."""
    if len(o_parts) == 0 or len(o_parts) != len(lse_parts):
        raise ValueError("need matching, non-empty lists of partials")
    o = np.stack([_as_f64(x) for x in o_parts])      # [P, ..., D]
    lse = np.stack([_as_f64(x) for x in lse_parts])  # [P, ...]
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        m = lse.max(axis=0)                           # global max
        has = np.isfinite(m)
        w = np.exp(lse - np.where(has, m, 0.0)[None])  # exp against the global max; -inf -> 0
        z = w.sum(axis=0)                             # global sum
        num = np.where(w[..., None] > 0, w[..., None] * o, 0.0).sum(axis=0)
        out = np.where(has[..., None], num / np.where(has, z, 1.0)[..., None], 0.0)
        out_lse = np.where(has, m + np.log(np.where(has, z, 1.0)), -np.inf)
    return out, out_lse
