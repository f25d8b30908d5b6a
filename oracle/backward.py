"""Oracle: gradients of exact attention in float64 -- test infrastructure only.

The pages fix only where the backward pass sits: in training the sequence is split across
cards, so the gradients are split the same way and reduced across cards ("PCP and DCP
sequence parallelism guide", section 2.3, gradient handling: a reduce-scatter), and the Ulysses
exchange runs its three steps in reverse for the backward pass ("Halo context parallelism"
article, Ulysses section).  What is differentiated is the forward definition the attention
oracle implements; the gradients below are its chain rule, written out.

For one head, with ``s_ij = scale * q_i . k_j`` over the visible pairs and
``P_ij = exp(s_ij - LSE_i)`` (the softmax), given ``dO`` (the gradient of a loss with respect to
the output ``O = P V``):

    dV_j  = sum_i P_ij dO_i
    dP_ij = dO_i . v_j
    dS_ij = P_ij (dP_ij - sum_l P_il dP_il)        (softmax Jacobian)
    dQ_i  = scale * sum_j dS_ij k_j
    dK_j  = scale * sum_i dS_ij q_i

GQA: a KV head's dK and dV are sums over the Q heads that read it.  Rows with no visible key
contribute nothing.

Per chunk (what one rank computes when its query rows meet one KV chunk): the same formulas
restricted to the chunk's keys, with ``P_ij = exp(s_ij - LSE_i)`` taken against the FINAL
(merged) ``LSE_i`` of the row and ``sum_l P_il dP_il`` over every key of the row, which equals
``D_i = dO_i . O_i`` for the final output ``O_i``.  Summing the per-chunk ``dQ`` over a row's
chunks, and each chunk's ``dK``/``dV`` over the query ranks that saw it (the reduce-scatter of
the guide), gives the gradients of the unsharded attention.
"""

import math

import numpy as np


def _as_f64(x):
    if hasattr(x, "detach"):  # torch tensor (any dtype) -> exact widening
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _check_shapes(q, k, v, d_o, q_pos, k_pos):
    sq, hq, d = q.shape
    skv, hkv, dk = k.shape
    if v.shape != k.shape or dk != d or d_o.shape != q.shape:
        raise ValueError("q/dO [Sq, Hq, D] and k/v [Skv, Hkv, D] with one D")
    if hq % hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if len(q_pos) != sq or len(k_pos) != skv:
        raise ValueError("position arrays must match the token counts")


def attention_backward(q, k, v, d_o, q_pos, k_pos, causal=True, scale=None):
    """dQ, dK, dV of exact attention (the forward oracle's definition) for a given dO.

    q, d_o: [Sq, Hq, D]; k, v: [Skv, Hkv, D]; positions as in ``attention``.
    Returns (dQ [Sq, Hq, D], dK [Skv, Hkv, D], dV [Skv, Hkv, D]) in float64.
    """
    q, k, v, d_o = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(d_o)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    _check_shapes(q, k, v, d_o, q_pos, k_pos)
    sq, hq, d = q.shape
    hkv = k.shape[1]
    group = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    if k.shape[0] == 0 or sq == 0:
        return dq, dk, dv
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        for h in range(hq):
            g = h // group
            s = scale * (q[:, h, :] @ k[:, g, :].T)  # [Sq, Skv]
            if causal:
                s = np.where(k_pos[None, :] <= q_pos[:, None], s, -np.inf)
            m = s.max(axis=1)
            has = np.isfinite(m)
            e = np.exp(s - np.where(has, m, 0.0)[:, None])
            p = e / np.where(has, e.sum(axis=1), 1.0)[:, None]
            p = np.where(has[:, None], p, 0.0)  # softmax; rows that see nothing have no P
            dv[:, g, :] += p.T @ d_o[:, h, :]
            dp = d_o[:, h, :] @ v[:, g, :].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[:, h, :] = scale * (ds @ k[:, g, :])
            dk[:, g, :] += scale * (ds.T @ q[:, h, :])
    return dq, dk, dv


def chunk_backward(q, k, v, d_o, o, lse, q_pos, k_pos, causal=True, scale=None):
    """One KV chunk's share of the gradients, given the rows' final output ``o`` and ``lse``.

    q, d_o, o: [Sq, Hq, D]; lse: [Sq, Hq] (natural log, -inf for rows that see no key at all);
    k, v: [Skv, Hkv, D] of the chunk.  Returns (dQ share [Sq, Hq, D], dK [Skv, Hkv, D],
    dV [Skv, Hkv, D]).
    """
    q, k, v, d_o, o = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(d_o), _as_f64(o)
    lse = _as_f64(lse)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    _check_shapes(q, k, v, d_o, q_pos, k_pos)
    sq, hq, d = q.shape
    hkv = k.shape[1]
    group = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    if k.shape[0] == 0 or sq == 0:
        return dq, dk, dv
    delta = (d_o * o).sum(axis=2)  # [Sq, Hq]: sum over all of the row's keys of P dP
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        for h in range(hq):
            g = h // group
            s = scale * (q[:, h, :] @ k[:, g, :].T)
            if causal:
                s = np.where(k_pos[None, :] <= q_pos[:, None], s, -np.inf)
            finite = np.isfinite(lse[:, h])
            p = np.exp(s - np.where(finite, lse[:, h], 0.0)[:, None])
            p = np.where(finite[:, None], p, 0.0)
            dv[:, g, :] += p.T @ d_o[:, h, :]
            dp = d_o[:, h, :] @ v[:, g, :].T
            ds = p * (dp - delta[:, h][:, None])
            dq[:, h, :] = scale * (ds @ k[:, g, :])
            dk[:, g, :] += scale * (ds.T @ q[:, h, :])
    return dq, dk, dv
