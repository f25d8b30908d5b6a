"""Independent checks that pin the oracle to something other than itself.

Each ``check_*`` takes an oracle-like module (``attention``, ``merge``, ``shard_positions``,
``seq_to_head``, ``head_to_seq``) and raises AssertionError when it disagrees with a pin.  The
same checks run against the real oracle (they must pass) and against copies of the oracle with a
planted mistake (they must fail), in ``test_oracle_pins.py``.

Pins used:
  * brute force on tiny inputs, in pure Python floats: softmax as exp(s_j) / sum_k exp(s_k) with
    no max-subtraction (inputs are small, nothing overflows);
  * the blockwise online accumulation of the "FCP" article (section 3.3), in pure Python, over a
    shuffled block order -- a different algorithm that reaches the same result;
  * closed forms: Q = 0, constant V, causal global row 0, K = 0;
  * a library special case: torch.nn.functional.scaled_dot_product_attention in float64, with
    GQA expressed through torch.repeat_interleave of the KV heads, and torch.logsumexp;
  * worked examples printed on the pages (tests/golden/);
  * merge invariants: any order of partials, associativity, extreme LSE spreads;
  * gradients: central finite differences of the brute-force forward for every element, torch
    autograd through SDPA in float64, the sum of per-chunk gradients over a sharded sequence,
    softmax-Jacobian invariants and closed forms.
"""

import math
import os
import random

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- brute force (pure Python)

def brute_attention(q, k, v, q_pos, k_pos, causal, scale):
    """Softmax attention by explicit loops; q/k/v nested lists [S][H][D] of floats."""
    sq, hq, d = len(q), len(q[0]), len(q[0][0])
    skv, hkv = len(k), len(k[0]) if len(k) else 1
    group = hq // hkv
    out = [[[0.0] * d for _ in range(hq)] for _ in range(sq)]
    lse = [[-math.inf] * hq for _ in range(sq)]
    for i in range(sq):
        for h in range(hq):
            g = h // group
            weights = []
            for j in range(skv):
                if causal and k_pos[j] > q_pos[i]:
                    continue
                s = scale * sum(q[i][h][t] * k[j][g][t] for t in range(d))
                weights.append((math.exp(s), j))
            if not weights:
                continue
            z = sum(w for w, _ in weights)
            for t in range(d):
                out[i][h][t] = sum(w * v[j][g][t] for w, j in weights) / z
            lse[i][h] = math.log(z)
    return np.array(out), np.array(lse)


def fcp_blockwise(q_row, keys, vals, scale, block, rng):
    """The FCP article's section 3.3 accumulation for one query row, blocks in shuffled order.

    keys/vals: lists of visible key / value vectors.  Returns (output, lse).
    """
    idx = list(range(len(keys)))
    blocks = [idx[b:b + block] for b in range(0, len(idx), block)]
    rng.shuffle(blocks)
    running_max = -math.inf
    running_sum = 0.0
    acc = [0.0] * len(q_row)
    for blk in blocks:
        scores = [scale * sum(a * b for a, b in zip(q_row, keys[j])) for j in blk]
        new_max = max(running_max, max(scores))
        c = math.exp(running_max - new_max) if running_max != -math.inf else 0.0
        acc = [a * c for a in acc]
        running_sum = running_sum * c
        p = [math.exp(s - new_max) for s in scores]
        for pj, j in zip(p, blk):
            acc = [a + pj * x for a, x in zip(acc, vals[j])]
        running_sum += sum(p)
        running_max = new_max
    return [a / running_sum for a in acc], running_max + math.log(running_sum)


def _tiny_case(seed, sq, skv, hq, hkv, d, q_pos, k_pos, mag=0.7):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((sq, hq, d)) * mag
    k = rng.standard_normal((skv, hkv, d)) * mag
    v = rng.standard_normal((skv, hkv, d))
    return q, k, v, np.asarray(q_pos, np.int64), np.asarray(k_pos, np.int64)


TINY_CASES = [
    # (seed, sq, skv, hq, hkv, d, q_pos, k_pos, causal)
    (1, 5, 7, 2, 2, 4, range(5), range(7), False),
    (2, 6, 6, 4, 2, 3, range(6), range(6), True),                       # GQA, aligned causal
    (3, 4, 8, 4, 1, 5, [3, 7, 11, 15], [0, 2, 4, 6, 8, 10, 12, 14], True),  # strided shards
    (4, 5, 4, 2, 1, 4, [0, 1, 2, 3, 4], [2, 3, 4, 5], True),            # rows 0,1 see nothing
    (5, 3, 9, 6, 3, 2, [20, 21, 22], range(9), True),                   # whole chunk in the past
    (6, 7, 3, 2, 2, 6, [1, 9, 17, 25, 33, 41, 49], [8, 24, 40], True),
]


def check_brute_force(orc):
    for seed, sq, skv, hq, hkv, d, qp, kp, causal in TINY_CASES:
        q, k, v, qpos, kpos = _tiny_case(seed, sq, skv, hq, hkv, d, qp, kp)
        scale = 1.0 / math.sqrt(d)
        o_ref, l_ref = brute_attention(q.tolist(), k.tolist(), v.tolist(), qpos.tolist(),
                                       kpos.tolist(), causal, scale)
        o, l = orc.attention(q, k, v, qpos, kpos, causal=causal)
        assert np.allclose(o, o_ref, atol=1e-12, rtol=0), f"O differs from brute force, case {seed}"
        assert np.array_equal(np.isinf(l), np.isinf(l_ref)), f"empty rows differ, case {seed}"
        fin = np.isfinite(l_ref)
        assert np.allclose(l[fin], l_ref[fin], atol=1e-12, rtol=0), f"LSE differs, case {seed}"


def check_fcp_blockwise(orc):
    bound = float(golden_rows("fcp_error_bound.txt")[0][0])
    rng = random.Random(7)
    for seed, sq, skv, hq, hkv, d, qp, kp, causal in TINY_CASES:
        q, k, v, qpos, kpos = _tiny_case(seed, sq, skv, hq, hkv, d, qp, kp)
        scale = 1.0 / math.sqrt(d)
        o, l = orc.attention(q, k, v, qpos, kpos, causal=causal)
        group = hq // hkv
        for i in range(sq):
            for h in range(hq):
                vis = [j for j in range(skv) if not causal or kpos[j] <= qpos[i]]
                if not vis:
                    continue
                keys = [k[j, h // group].tolist() for j in vis]
                vals = [v[j, h // group].tolist() for j in vis]
                out, lse = fcp_blockwise(q[i, h].tolist(), keys, vals, scale, 2, rng)
                err = max(abs(a - b) for a, b in zip(out, o[i, h]))
                assert err < 1e-12 and err < bound, f"blockwise accumulation differs (case {seed})"
                assert abs(lse - l[i, h]) < 1e-12


def check_closed_forms(orc):
    rng = np.random.default_rng(11)
    sq = skv = 9
    hq, hkv, d = 4, 2, 8
    pos = np.arange(sq)
    # Q = 0: uniform weights over the visible keys
    q = np.zeros((sq, hq, d))
    k = rng.standard_normal((skv, hkv, d))
    v = rng.standard_normal((skv, hkv, d))
    o, l = orc.attention(q, k, v, pos, pos, causal=True)
    for i in range(sq):
        for h in range(hq):
            g = h // (hq // hkv)
            assert np.allclose(o[i, h], v[:i + 1, g].mean(axis=0), atol=1e-12)
            assert abs(l[i, h] - math.log(i + 1)) < 1e-12
    # K = 0, non-causal: column mean of V, LSE = ln Skv
    q = rng.standard_normal((sq, hq, d))
    o, l = orc.attention(q, np.zeros_like(k), v, pos, pos, causal=False)
    for h in range(hq):
        g = h // (hq // hkv)
        assert np.allclose(o[:, h], v[:, g].mean(axis=0)[None], atol=1e-12)
    assert np.allclose(l, math.log(skv), atol=1e-12)
    # every V row equal to c -> O = c
    c = rng.standard_normal(d)
    vc = np.broadcast_to(c, (skv, hkv, d)).copy()
    o, l = orc.attention(q, k, vc, pos, pos, causal=True)
    assert np.allclose(o, np.broadcast_to(c, o.shape), atol=1e-12)
    # causal global row 0 sees exactly key 0: O = v_0, LSE = scale * q_0 . k_0
    o, l = orc.attention(q, k, v, pos, pos, causal=True)
    for h in range(hq):
        g = h // (hq // hkv)
        assert np.allclose(o[0, h], v[0, g], atol=1e-12)
        assert abs(l[0, h] - float(q[0, h] @ k[0, g]) / math.sqrt(d)) < 1e-12


def check_sdpa(orc):
    """torch SDPA (float64) with GQA via repeat_interleave of KV heads; LSE via torch.logsumexp."""
    rng = np.random.default_rng(5)
    for causal in (False, True):
        s, hq, hkv, d = 24, 6, 2, 16
        q = rng.standard_normal((s, hq, d))
        k = rng.standard_normal((s, hkv, d))
        v = rng.standard_normal((s, hkv, d))
        pos = np.arange(s)
        o, l = orc.attention(q, k, v, pos, pos, causal=causal)
        tq = torch.from_numpy(q).permute(1, 0, 2)[None]
        tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)[None]
        tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
        ref = ref[0].permute(1, 0, 2).numpy()
        assert np.allclose(o, ref, atol=1e-12), "O differs from torch SDPA"
        scores = (tq @ tk.transpose(-1, -2)) / math.sqrt(d)
        if causal:
            scores = scores.masked_fill(torch.ones(s, s, dtype=torch.bool).triu(1), -math.inf)
        lref = torch.logsumexp(scores, dim=-1)[0].T.numpy()
        assert np.allclose(l, lref, atol=1e-12), "LSE differs from torch.logsumexp"


def check_merge(orc):
    rng = np.random.default_rng(3)
    s, hq, hkv, d, n = 32, 4, 2, 8, 4
    q = rng.standard_normal((s, hq, d))
    k = rng.standard_normal((s * n, hkv, d))
    v = rng.standard_normal((s * n, hkv, d))
    qpos = np.arange(s) * n + 1  # strided shard, rank 1 of 4
    kpos = np.arange(s * n)
    full_o, full_l = orc.attention(q, k, v, qpos, kpos, causal=True)
    chunks = [np.arange(c * s, (c + 1) * s) for c in range(n)]
    parts = [orc.attention(q, k[ix], v[ix], qpos, kpos[ix], causal=True) for ix in chunks]
    order_rng = np.random.default_rng(9)
    for _ in range(6):
        perm = order_rng.permutation(n)
        o, l = orc.merge([parts[i][0] for i in perm], [parts[i][1] for i in perm])
        assert np.allclose(o, full_o, atol=1e-12) and np.allclose(l, full_l, atol=1e-12)
    ab = orc.merge([parts[0][0], parts[1][0]], [parts[0][1], parts[1][1]])
    abc = orc.merge([ab[0], parts[2][0], parts[3][0]], [ab[1], parts[2][1], parts[3][1]])
    assert np.allclose(abc[0], full_o, atol=1e-12) and np.allclose(abc[1], full_l, atol=1e-12)
    # one partial: identity
    o, l = orc.merge([parts[2][0]], [parts[2][1]])
    assert np.allclose(o, parts[2][0]) and np.array_equal(np.isinf(l), np.isinf(parts[2][1]))
    # equal LSEs: plain average, LSE + ln 2
    a = rng.standard_normal((3, d))
    b = rng.standard_normal((3, d))
    la = np.array([0.5, -2.0, 7.0])
    o, l = orc.merge([a, b], [la, la])
    assert np.allclose(o, (a + b) / 2, atol=1e-12) and np.allclose(l, la + math.log(2), atol=1e-12)
    # extreme spreads: no overflow, dominated by the largest LSE
    lx = np.array([-800.0, 0.0, 700.0])
    ly = np.array([-800.0, 750.0, -700.0])
    o, l = orc.merge([a, b], [lx, ly])
    assert np.allclose(o[0], (a[0] + b[0]) / 2, atol=1e-12)
    assert abs(l[0] - (-800.0 + math.log(2))) < 1e-9
    assert np.allclose(o[1], b[1], atol=1e-12) and abs(l[1] - 750.0) < 1e-9
    assert np.allclose(o[2], a[2], atol=1e-12) and abs(l[2] - 700.0) < 1e-9
    # all partials empty
    o, l = orc.merge([a, b], [np.full(3, -np.inf), np.full(3, -np.inf)])
    assert np.all(o == 0) and np.all(np.isneginf(l))


def check_layouts(orc):
    for cp, rank, first in golden_rows("zigzag_cp4.txt"):
        cp, rank = int(cp), int(rank)
        want = [int(x) for x in first.split(",")]
        got = orc.shard_positions(64, cp, rank, "strided")
        assert list(got[:len(want)]) == want, "zig-zag example from the page not reproduced"
    for seq_len, cp, local_len in golden_rows("contiguous_split.txt"):
        seq_len, cp, local_len = int(seq_len), int(cp), int(local_len)
        for r in range(cp):
            got = orc.shard_positions(seq_len, cp, r, "contiguous")
            assert len(got) == local_len and got[0] == r * local_len
            assert np.all(np.diff(got) == 1)
    # two-block split, written out by hand for S=16, cp=2 and S=24, cp=3
    assert list(orc.shard_positions(16, 2, 0, "two_block")) == [0, 1, 2, 3, 12, 13, 14, 15]
    assert list(orc.shard_positions(16, 2, 1, "two_block")) == [4, 5, 6, 7, 8, 9, 10, 11]
    assert list(orc.shard_positions(24, 3, 1, "two_block")) == [4, 5, 6, 7, 16, 17, 18, 19]
    # its point: every rank's causal work against the whole sequence is the same, in closed form
    # b^2 (2cp - 1) + b (b + 1) for blocks of b = S / (2 cp) tokens
    for seq_len, cp in ((64, 4), (48, 8), (96, 3)):
        b = seq_len // (2 * cp)
        for r in range(cp):
            work = orc.visible_pair_count(orc.shard_positions(seq_len, cp, r, "two_block"),
                                          np.arange(seq_len), True)
            assert work == b * b * (2 * cp - 1) + b * (b + 1), "two-block split is not balanced"
    # work-balanced contiguous split: brute force over b (linear scan of the causal pair count
    # W(b) = 1 + 2 + ... + b), and the balance it buys
    for seq_len, cp in ((64, 4), (100, 3), (1000, 8), (4097, 5)):
        total = seq_len * (seq_len + 1) // 2
        bounds = [0]
        for r in range(1, cp):
            b, w = 0, 0
            while w * cp < r * total:
                b += 1
                w += b
            bounds.append(b)
        bounds.append(seq_len)
        for r in range(cp):
            got = orc.shard_positions(seq_len, cp, r, "balanced")
            assert list(got) == list(range(bounds[r], bounds[r + 1])), "balanced split differs from brute force"
            work = orc.visible_pair_count(got, np.arange(seq_len), True)
            assert abs(work - total / cp) <= seq_len, "balanced split is not balanced"
    for kind in ("contiguous", "strided", "two_block", "balanced"):
        for seq_len, cp in ((64, 4), (48, 8), (7, 7), (14, 7), (32768, 8)):
            if kind == "two_block" and seq_len % (2 * cp):
                continue
            if kind == "balanced" and seq_len < 4 * cp:
                continue
            allpos = np.concatenate([orc.shard_positions(seq_len, cp, r, kind) for r in range(cp)])
            assert np.array_equal(np.sort(allpos), np.arange(seq_len)), "layout is not a cover"
            # every rank's causal pairs against every chunk add up to S(S+1)/2
            tot = sum(orc.visible_pair_count(orc.shard_positions(seq_len, cp, r, kind),
                                             orc.shard_positions(seq_len, cp, c, kind), True)
                      for r in range(cp) for c in range(cp))
            assert tot == seq_len * (seq_len + 1) // 2


def check_ulysses(orc):
    (cp, hq, hkv, per_rank), = [tuple(int(x) for x in r) for r in golden_rows("ulysses_cp4.txt")]
    rng = np.random.default_rng(21)
    seq, d = 32, 4
    for kind in ("contiguous", "strided", "two_block"):
        pos = [orc.shard_positions(seq, cp, r, kind) for r in range(cp)]
        q_full = rng.standard_normal((seq, hq, d))
        k_full = rng.standard_normal((seq, hkv, d)) * 0.3
        v_full = rng.standard_normal((seq, hkv, d))
        qs = [q_full[p] for p in pos]
        ks = [k_full[p] for p in pos]
        vs = [v_full[p] for p in pos]
        qh = orc.seq_to_head(qs, pos)
        kh = orc.seq_to_head(ks, pos)
        vh = orc.seq_to_head(vs, pos)
        assert qh[0].shape == (seq, per_rank, d), "head split differs from the page's example"
        assert kh[0].shape == (seq, hkv // cp, d)
        # exactness: attention on the head-sharded tensors equals the heads' slice of attention
        # on the unsharded sequence (heads are independent)
        ref_o, _ = orc.attention(q_full, k_full, v_full, np.arange(seq), np.arange(seq), True)
        outs = []
        for r in range(cp):
            o_r, _ = orc.attention(qh[r], kh[r], vh[r], np.arange(seq), np.arange(seq), True)
            assert np.allclose(o_r, ref_o[:, r * per_rank:(r + 1) * per_rank], atol=1e-12)
            outs.append(o_r)
        back = orc.head_to_seq(outs, pos)
        for s in range(cp):
            assert np.allclose(back[s], ref_o[pos[s]], atol=1e-12)
        # round trip is the identity, bit for bit
        rt = orc.head_to_seq(qh, pos)
        for s in range(cp):
            assert np.array_equal(rt[s], qs[s])


# ---------------------------------------------------------------- gradients

def _brute_loss(q, k, v, d_o, qpos, kpos, causal, scale):
    """sum(dO * O) with O from the pure-Python brute force: its gradient is the backward pass."""
    o, _ = brute_attention(q.tolist(), k.tolist(), v.tolist(), qpos.tolist(), kpos.tolist(),
                           causal, scale)
    return float((np.asarray(o) * d_o).sum())


def check_backward_finite_differences(orc):
    """Every gradient element against a central difference of the brute-force forward."""
    eps = 1e-6
    for seed, sq, skv, hq, hkv, d, qp, kp, causal in TINY_CASES[:4]:
        q, k, v, qpos, kpos = _tiny_case(seed, sq, skv, hq, hkv, d, qp, kp)
        d_o = np.random.default_rng(seed + 100).standard_normal(q.shape)
        scale = 1.0 / math.sqrt(d)
        dq, dk, dv = orc.attention_backward(q, k, v, d_o, qpos, kpos, causal=causal)
        for name, x, g in (("dQ", q, dq), ("dK", k, dk), ("dV", v, dv)):
            for idx in np.ndindex(x.shape):
                xp = x.copy()
                xm = x.copy()
                xp[idx] += eps
                xm[idx] -= eps
                args_p = [xp if y is x else y for y in (q, k, v)]
                args_m = [xm if y is x else y for y in (q, k, v)]
                fd = (_brute_loss(*args_p, d_o, qpos, kpos, causal, scale) -
                      _brute_loss(*args_m, d_o, qpos, kpos, causal, scale)) / (2 * eps)
                assert abs(fd - g[idx]) < 1e-7, f"{name}{idx} differs from finite differences (case {seed})"


def check_backward_autograd(orc):
    """torch autograd through SDPA in float64 (GQA via repeat_interleave, which sums the
    group's gradients back onto each KV head)."""
    rng = np.random.default_rng(9)
    for causal in (False, True):
        s, hq, hkv, d = 20, 6, 2, 8
        q = rng.standard_normal((s, hq, d))
        k = rng.standard_normal((s, hkv, d))
        v = rng.standard_normal((s, hkv, d))
        d_o = rng.standard_normal((s, hq, d))
        pos = np.arange(s)
        dq, dk, dv = orc.attention_backward(q, k, v, d_o, pos, pos, causal=causal)
        tq = torch.from_numpy(q).requires_grad_()
        tk = torch.from_numpy(k).requires_grad_()
        tv = torch.from_numpy(v).requires_grad_()
        g = hq // hkv
        out = torch.nn.functional.scaled_dot_product_attention(
            tq.permute(1, 0, 2)[None], tk.permute(1, 0, 2).repeat_interleave(g, dim=0)[None],
            tv.permute(1, 0, 2).repeat_interleave(g, dim=0)[None], is_causal=causal)
        out[0].permute(1, 0, 2).backward(torch.from_numpy(d_o))
        assert np.allclose(dq, tq.grad.numpy(), atol=1e-11), "dQ differs from autograd"
        assert np.allclose(dk, tk.grad.numpy(), atol=1e-11), "dK differs from autograd"
        assert np.allclose(dv, tv.grad.numpy(), atol=1e-11), "dV differs from autograd"


def check_backward_chunks(orc):
    """Per-chunk gradients (against the final O and LSE) add up to the unsharded gradients, in
    any chunk order; closed forms and invariants of the softmax Jacobian."""
    rng = np.random.default_rng(13)
    seq, cp, hq, hkv, d = 32, 4, 4, 2, 6
    q = rng.standard_normal((seq, hq, d))
    k = rng.standard_normal((seq, hkv, d))
    v = rng.standard_normal((seq, hkv, d))
    d_o = rng.standard_normal((seq, hq, d))
    full = np.arange(seq)
    dq_ref, dk_ref, dv_ref = orc.attention_backward(q, k, v, d_o, full, full, causal=True)
    # the gradients do not depend on how the sequence is sharded (strided query shards here,
    # contiguous KV chunks), chunk order shuffled
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o_all, lse_all = orc.attention(q, k, v, full, full, causal=True)
    for r in range(cp):
        qpos = np.arange(r, seq, cp)
        order = rng.permutation(cp)
        for c in order:
            kpos = np.arange(c * seq // cp, (c + 1) * seq // cp)
            a, b, e = orc.chunk_backward(q[qpos], k[kpos], v[kpos], d_o[qpos], o_all[qpos],
                                         lse_all[qpos], qpos, kpos, causal=True)
            dq[qpos] += a
            dk[kpos] += b  # the reduce-scatter: each chunk's owner sums every rank's share
            dv[kpos] += e
    assert np.allclose(dq, dq_ref, atol=1e-12), "chunked dQ differs from the unsharded gradient"
    assert np.allclose(dk, dk_ref, atol=1e-12), "chunked dK differs"
    assert np.allclose(dv, dv_ref, atol=1e-12), "chunked dV differs"
    # invariants: each row's dS sums to 0, so the dK of every KV head sums to 0 over keys; each
    # row's P sums to 1, so the dV of every KV head sums to its group's dO
    assert np.allclose(dk_ref.sum(axis=0), 0.0, atol=1e-12)
    for g in range(hkv):
        grp = d_o[:, g * (hq // hkv):(g + 1) * (hq // hkv), :].sum(axis=(0, 1))
        assert np.allclose(dv_ref[:, g].sum(axis=0), grp, atol=1e-12)
    # constant V: O does not depend on Q or K at all
    vc = np.broadcast_to(rng.standard_normal(d), v.shape).copy()
    a, b, _ = orc.attention_backward(q, k, vc, d_o, full, full, causal=True)
    assert np.allclose(a, 0.0, atol=1e-12) and np.allclose(b, 0.0, atol=1e-12)
    # causal row 0 sees one key: its softmax is the constant 1, so its dQ is 0
    assert np.allclose(dq_ref[0], 0.0, atol=1e-12)


ALL_CHECKS = [check_brute_force, check_fcp_blockwise, check_closed_forms, check_sdpa,
              check_merge, check_layouts, check_ulysses, check_backward_finite_differences,
              check_backward_autograd, check_backward_chunks]
