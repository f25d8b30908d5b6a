"""Seeded random sweeps of the partial, fused chunk-list and backward kernels against the oracle.

The hand-picked cases elsewhere cover the named edge cases; these draw many more shapes at random
(ragged row and key counts, GQA groups up to 8, both head dims, both input dtypes, affine position
maps with strides 1..8 and offsets on either side of the queries, causal or not, default or
explicit softmax scale), so that a tile-boundary or indexing slip that only shows for some
combination has many chances to be caught.  Every draw comes from a fixed seed, and every case
prints its parameters when it fails.
"""

import numpy as np
import pytest
import torch

import helpers
import oracle
from helpers import TOL_BF16_LSE, TOL_BF16_O, TOL_F32, TOL_GRAD_BF16, TOL_GRAD_F32, compare_grad, compare_partial

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    helpers.ensure_built()

import context_blockwise_attention_gb300 as cpa  # noqa: E402
from context_blockwise_attention_gb300 import PosMap  # noqa: E402
from context_blockwise_attention_gb300 import workloads as wl  # noqa: E402

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _pos(m: PosMap, n):
    return m.base + m.stride * np.arange(n, dtype=np.int64)


def _draw_maps(rng, sq):
    """A query map and a generator of KV maps placed before, across or after the queries."""
    qs = int(rng.choice([1, 1, 2, 4, 8]))
    qb = int(rng.integers(0, 3000))
    q_end = qb + qs * max(sq - 1, 0)

    def kv_map():
        ks = int(rng.choice([1, 1, 2, 4, 8]))
        kb = int(rng.integers(max(0, qb - 1500), q_end + 200))
        return PosMap(kb, ks)

    return PosMap(qb, qs), kv_map


def _draw_heads(rng, d):
    hkv = int(rng.choice([1, 2, 4]))
    group = int(rng.choice([1, 2, 4, 8]))
    if d == 128 and hkv * group > 8:
        group = max(1, 8 // hkv)
    return hkv * group, hkv


def _draw_case(rng):
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    d = int(rng.choice([64, 128]))
    hq, hkv = _draw_heads(rng, d)
    sq = int(rng.integers(1, 600))
    causal = bool(rng.random() < 0.75)
    scale = 0.0 if rng.random() < 0.7 else float(rng.uniform(0.03, 0.2))
    qm, kv_map = _draw_maps(rng, sq)
    return dict(dtype=dtype, d=d, hq=hq, hkv=hkv, sq=sq, causal=causal, scale=scale, qm=qm, kv_map=kv_map)


def _tols(dtype):
    return (TOL_F32, TOL_F32) if dtype == torch.float32 else (TOL_BF16_O, TOL_BF16_LSE)


N_PARTIAL = 40


@pytest.mark.parametrize("i", range(N_PARTIAL), ids=[f"p{i}" for i in range(N_PARTIAL)])
def test_random_partial(i):
    rng = np.random.default_rng(5000 + i)
    c = _draw_case(rng)
    skv = int(rng.integers(1, 800))
    km = c["kv_map"]()
    seed = 7000 + 10 * i
    q = wl.normal((c["sq"], c["hq"], c["d"]), c["dtype"], seed + 1, 0.5, device=DEV)
    k = wl.normal((skv, c["hkv"], c["d"]), c["dtype"], seed + 2, 0.5, device=DEV)
    v = wl.normal((skv, c["hkv"], c["d"]), c["dtype"], seed + 3, 1.0, device=DEV)
    o = torch.full((c["sq"], c["hq"], c["d"]), float("nan"), device=DEV)
    lse = torch.full((c["sq"], c["hq"]), float("nan"), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    cpa.partial_attn(q, k, v, c["qm"], km, causal=c["causal"], o=o, lse=lse, status=status, scale=c["scale"])
    torch.cuda.synchronize()
    assert status.item() == 0
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), _pos(c["qm"], c["sq"]), _pos(km, skv),
                                    causal=c["causal"], scale=c["scale"] if c["scale"] > 0 else None)
    tol_o, tol_l = _tols(c["dtype"])
    what = f"partial {i}: {({k_: c[k_] for k_ in c if k_ != 'kv_map'})} skv={skv} kv={km}"
    compare_partial(o.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, tol_o, tol_l, what)


N_FUSED = 16


@pytest.mark.parametrize("i", range(N_FUSED), ids=[f"f{i}" for i in range(N_FUSED)])
def test_random_fused_chunks(i):
    """One chunk-list call over 1..6 chunks (some empty) in a random arrival order."""
    rng = np.random.default_rng(6000 + i)
    c = _draw_case(rng)
    n = int(rng.integers(1, 7))
    seed = 8000 + 100 * i
    q = wl.normal((c["sq"], c["hq"], c["d"]), c["dtype"], seed, 0.5, device=DEV)
    chunks = []
    for j in range(n):
        skv = 0 if rng.random() < 0.1 else int(rng.integers(1, 500))
        k = wl.normal((skv, c["hkv"], c["d"]), c["dtype"], seed + 10 * j + 1, 0.5, device=DEV)
        v = wl.normal((skv, c["hkv"], c["d"]), c["dtype"], seed + 10 * j + 2, 1.0, device=DEV)
        chunks.append((k, v, c["kv_map"]()))
    order = [int(x) for x in rng.permutation(n)]
    o = torch.full((c["sq"], c["hq"], c["d"]), float("nan"), device=DEV)
    lse = torch.full((c["sq"], c["hq"]), float("nan"), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    cpa.partial_attn_chunks(q, [chunks[j] for j in order], c["qm"], causal=c["causal"], o=o, lse=lse,
                            status=status, scale=c["scale"])
    torch.cuda.synchronize()
    assert status.item() == 0
    k_all = torch.cat([ch[0].cpu() for ch in chunks])
    v_all = torch.cat([ch[1].cpu() for ch in chunks])
    pos = np.concatenate([_pos(ch[2], ch[0].shape[0]) for ch in chunks])
    o_ref, l_ref = oracle.attention(q.cpu(), k_all, v_all, _pos(c["qm"], c["sq"]), pos, causal=c["causal"],
                                    scale=c["scale"] if c["scale"] > 0 else None)
    tol_o, tol_l = _tols(c["dtype"])
    what = (f"fused {i}: {({k_: c[k_] for k_ in c if k_ != 'kv_map'})} order={order} "
            f"chunks={[(ch[0].shape[0], ch[2]) for ch in chunks]}")
    compare_partial(o.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, tol_o, tol_l, what)


N_BWD = 16


@pytest.mark.parametrize("i", range(N_BWD), ids=[f"b{i}" for i in range(N_BWD)])
def test_random_backward(i):
    """Backward of one (query shard, chunk) pair whose rows' softmax also covers a second chunk,
    against the oracle's chain rule with the final O and LSE over both chunks."""
    rng = np.random.default_rng(9000 + i)
    c = _draw_case(rng)
    skv = int(rng.integers(1, 600))
    km = c["kv_map"]()
    oskv = int(rng.integers(0, 300))
    okm = c["kv_map"]()
    seed = 9500 + 10 * i
    dt, sq, hq, hkv, d = c["dtype"], c["sq"], c["hq"], c["hkv"], c["d"]
    q = wl.normal((sq, hq, d), dt, seed + 1, 0.5, device=DEV)
    k = wl.normal((skv, hkv, d), dt, seed + 2, 0.5, device=DEV)
    v = wl.normal((skv, hkv, d), dt, seed + 3, 1.0, device=DEV)
    d_o = wl.normal((sq, hq, d), dt, seed + 4, 1.0, device=DEV)
    k2 = wl.normal((oskv, hkv, d), dt, seed + 5, 0.5)
    v2 = wl.normal((oskv, hkv, d), dt, seed + 6, 1.0)
    scale = c["scale"] if c["scale"] > 0 else None
    qp = _pos(c["qm"], sq)
    o_ref, l_ref = oracle.attention(q.cpu(), torch.cat([k.cpu(), k2]), torch.cat([v.cpu(), v2]), qp,
                                    np.concatenate([_pos(km, skv), _pos(okm, oskv)]), causal=c["causal"], scale=scale)
    o32 = torch.from_numpy(o_ref).float()
    l32 = torch.from_numpy(l_ref).float()
    aux = cpa.attn_bwd_prep(o32.to(DEV), d_o, l32.to(DEV))
    poison = 0.25
    dq = torch.full(q.shape, poison, device=DEV)
    dk = torch.full(k.shape, poison, device=DEV)
    dv = torch.full(v.shape, poison, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    cpa.partial_attn_bwd(q, k, v, d_o, aux, c["qm"], km, dq, dk, dv, causal=c["causal"], scale=c["scale"],
                         status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = oracle.chunk_backward(q.cpu(), k.cpu(), v.cpu(), d_o.cpu(), o32, l32, qp, _pos(km, skv),
                                causal=c["causal"], scale=scale)
    tol = TOL_GRAD_BF16 if dt == torch.bfloat16 else TOL_GRAD_F32
    what = f"bwd {i}: {({k_: c[k_] for k_ in c if k_ != 'kv_map'})} skv={skv} kv={km} other=({oskv}, {okm})"
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        compare_grad(g.cpu().double().numpy() - poison, r, tol, f"{name} {what}")


# head-count extremes the random draws do not reach: MQA with many query heads, wide GQA at D=128
_HEAD_CASES = [(64, 1, 64), (16, 1, 128), (64, 8, 128), (1, 1, 128)]


@pytest.mark.parametrize("hq,hkv,d", _HEAD_CASES, ids=[f"h{a}_{b}_d{c}" for a, b, c in _HEAD_CASES])
def test_head_extremes(hq, hkv, d):
    sq, skv = 200, 333
    qm, km, km2 = PosMap(100, 3), PosMap(0, 2), PosMap(1, 2)
    q = wl.normal((sq, hq, d), torch.bfloat16, 11, 0.5, device=DEV)
    k = wl.normal((skv, hkv, d), torch.bfloat16, 12, 0.5, device=DEV)
    v = wl.normal((skv, hkv, d), torch.bfloat16, 13, 1.0, device=DEV)
    k2 = wl.normal((150, hkv, d), torch.bfloat16, 14, 0.5, device=DEV)
    v2 = wl.normal((150, hkv, d), torch.bfloat16, 15, 1.0, device=DEV)
    d_o = wl.normal((sq, hq, d), torch.bfloat16, 16, 1.0, device=DEV)
    qp = _pos(qm, sq)
    # forward, one chunk
    o, lse = cpa.partial_attn(q, k, v, qm, km, causal=True)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), qp, _pos(km, skv), causal=True)
    compare_partial(o.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, TOL_BF16_O, TOL_BF16_LSE, f"partial {hq}/{hkv}")
    # forward over both chunks in one call
    o2, l2 = cpa.partial_attn_chunks(q, [(k2, v2, km2), (k, v, km)], qm, causal=True)
    kall, vall = torch.cat([k.cpu(), k2.cpu()]), torch.cat([v.cpu(), v2.cpu()])
    kp = np.concatenate([_pos(km, skv), _pos(km2, 150)])
    o2_ref, l2_ref = oracle.attention(q.cpu(), kall, vall, qp, kp, causal=True)
    compare_partial(o2.cpu().numpy(), l2.cpu().numpy(), o2_ref, l2_ref, TOL_BF16_O, TOL_BF16_LSE, f"chunks {hq}/{hkv}")
    # backward of the first chunk against the final (two-chunk) O and LSE
    o32, l32 = torch.from_numpy(o2_ref).float(), torch.from_numpy(l2_ref).float()
    aux = cpa.attn_bwd_prep(o32.to(DEV), d_o, l32.to(DEV))
    dq = torch.zeros(q.shape, device=DEV)
    dk = torch.zeros(k.shape, device=DEV)
    dv = torch.zeros(v.shape, device=DEV)
    cpa.partial_attn_bwd(q, k, v, d_o, aux, qm, km, dq, dk, dv, causal=True)
    torch.cuda.synchronize()
    ref = oracle.chunk_backward(q.cpu(), k.cpu(), v.cpu(), d_o.cpu(), o32, l32, qp, _pos(km, skv), causal=True)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        compare_grad(g.cpu().numpy(), r, TOL_GRAD_BF16, f"{name} {hq}/{hkv} d={d}")


def test_positions_near_the_limit():
    """Positions up to just below the checked limit (2e9) with strides in the millions: the
    kernels' position arithmetic (products of a stride and a row index near 2^31, differences of
    large positions) matches the oracle on the same int64 positions, in the partial, the chunk
    list and the backward."""
    sq, hq, hkv, d = 333, 4, 2, 128
    qm = PosMap(7, 6_000_000)
    specs = [(300, PosMap(3, 6_000_000)), (257, PosMap(1_794_000_005, 777))]
    q = wl.normal((sq, hq, d), torch.bfloat16, 41, 0.5, device=DEV)
    d_o = wl.normal((sq, hq, d), torch.bfloat16, 42, 1.0, device=DEV)
    ks = [wl.normal((n, hkv, d), torch.bfloat16, 43 + i, 0.5, device=DEV) for i, (n, _) in enumerate(specs)]
    vs = [wl.normal((n, hkv, d), torch.bfloat16, 53 + i, 1.0, device=DEV) for i, (n, _) in enumerate(specs)]
    qp = _pos(qm, sq)
    kp = [_pos(m, n) for n, m in specs]
    assert qp.max() > 1.99e9 and max(k.max() for k in kp) < 2e9 and qp.max() < 2e9
    o1, l1 = cpa.partial_attn(q, ks[1], vs[1], qm, specs[1][1], causal=True)
    r1 = oracle.attention(q.cpu(), ks[1].cpu(), vs[1].cpu(), qp, kp[1], causal=True)
    compare_partial(o1.cpu().numpy(), l1.cpu().numpy(), *r1, TOL_BF16_O, TOL_BF16_LSE, "partial, positions near 2e9")
    o, lse = cpa.partial_attn_chunks(q, [(ks[i], vs[i], specs[i][1]) for i in (1, 0)], qm, causal=True)
    ref_o, ref_l = oracle.attention(q.cpu(), torch.cat([k.cpu() for k in ks]), torch.cat([v.cpu() for v in vs]),
                                    qp, np.concatenate(kp), causal=True)
    compare_partial(o.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, TOL_BF16_O, TOL_BF16_LSE, "chunks, positions near 2e9")
    o32, l32 = torch.from_numpy(ref_o).float(), torch.from_numpy(ref_l).float()
    aux = cpa.attn_bwd_prep(o32.to(DEV), d_o, l32.to(DEV))
    dq = torch.zeros(q.shape, device=DEV)
    dks = [torch.zeros(k.shape, device=DEV) for k in ks]
    dvs = [torch.zeros(k.shape, device=DEV) for k in ks]
    cpa.partial_attn_bwd_chunks(q, d_o, aux, qm, [(ks[i], vs[i], specs[i][1], dks[i], dvs[i]) for i in (0, 1)], dq)
    torch.cuda.synchronize()
    dq_ref = np.zeros((sq, hq, d))
    for i in range(2):
        a, bk, bv = oracle.chunk_backward(q.cpu(), ks[i].cpu(), vs[i].cpu(), d_o.cpu(), o32, l32, qp, kp[i], causal=True)
        dq_ref += a
        compare_grad(dks[i].cpu().numpy(), bk, TOL_GRAD_BF16, f"dK {i}, positions near 2e9")
        compare_grad(dvs[i].cpu().numpy(), bv, TOL_GRAD_BF16, f"dV {i}, positions near 2e9")
    compare_grad(dq.cpu().numpy(), dq_ref, TOL_GRAD_BF16, "dQ, positions near 2e9")


def test_chunk_lists_at_the_maximum():
    """CP_MAX_CHUNKS = 64 small chunks (ragged, some empty, strided positions) in one forward call,
    and the same 64 in one backward call, which the library splits into launches of at most 32
    chunks (the 32-chunk and the 8-chunk table sizes both run)."""
    sq, hq, hkv, d = 260, 4, 2, 64
    rng = np.random.default_rng(77)
    qm = PosMap(5, 8)
    specs = []
    for i in range(cpa.api.CP_MAX_CHUNKS):
        n = 0 if i % 8 in (1, 4, 6) else int(rng.integers(1, 40))  # 40 live chunks: 32 + 8 per launch
        specs.append((n, PosMap(int(rng.integers(0, 2400)), int(rng.choice([1, 4, 8])))))
    q = wl.normal((sq, hq, d), torch.bfloat16, 61, 0.5, device=DEV)
    d_o = wl.normal((sq, hq, d), torch.bfloat16, 62, 1.0, device=DEV)
    ks = [wl.normal((n, hkv, d), torch.bfloat16, 1000 + i, 0.5, device=DEV) for i, (n, _) in enumerate(specs)]
    vs = [wl.normal((n, hkv, d), torch.bfloat16, 2000 + i, 1.0, device=DEV) for i, (n, _) in enumerate(specs)]
    qp = _pos(qm, sq)
    kp = np.concatenate([_pos(m, n) for n, m in specs])
    o, lse = cpa.partial_attn_chunks(q, [(ks[i], vs[i], specs[i][1]) for i in range(len(specs))], qm, causal=True)
    ref_o, ref_l = oracle.attention(q.cpu(), torch.cat([k.cpu() for k in ks]), torch.cat([v.cpu() for v in vs]),
                                    qp, kp, causal=True)
    compare_partial(o.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, TOL_BF16_O, TOL_BF16_LSE, "64-chunk forward")
    o32, l32 = torch.from_numpy(ref_o).float(), torch.from_numpy(ref_l).float()
    aux = cpa.attn_bwd_prep(o32.to(DEV), d_o, l32.to(DEV))
    dq = torch.zeros(q.shape, device=DEV)
    dks = [torch.zeros(k.shape, device=DEV) for k in ks]
    dvs = [torch.zeros(k.shape, device=DEV) for k in ks]
    cpa.partial_attn_bwd_chunks(q, d_o, aux, qm, [(ks[i], vs[i], specs[i][1], dks[i], dvs[i]) for i in range(len(specs))],
                                dq)
    torch.cuda.synchronize()
    dq_ref = np.zeros((sq, hq, d))
    for i, (n, m) in enumerate(specs):
        if n == 0:
            continue  # an empty chunk adds nothing
        a, bk, bv = oracle.chunk_backward(q.cpu(), ks[i].cpu(), vs[i].cpu(), d_o.cpu(), o32, l32, qp, _pos(m, n),
                                          causal=True)
        dq_ref += a
        compare_grad(dks[i].cpu().numpy(), bk, TOL_GRAD_BF16, f"64-chunk dK {i}")
        compare_grad(dvs[i].cpu().numpy(), bv, TOL_GRAD_BF16, f"64-chunk dV {i}")
    compare_grad(dq.cpu().numpy(), dq_ref, TOL_GRAD_BF16, "64-chunk dQ")


def test_empty_query_shard_everywhere():
    """A rank with no query rows (sq = 0): every call succeeds, launches nothing harmful and
    leaves the other operands untouched -- partial, chunk list, merge, backward prep, backward of
    one chunk and of a chunk list (whose dK, dV must stay as they were)."""
    hq, hkv, d = 4, 2, 128
    q = torch.empty((0, hq, d), dtype=torch.bfloat16, device=DEV)
    k = wl.normal((200, hkv, d), torch.bfloat16, 81, 0.5, device=DEV)
    v = wl.normal((200, hkv, d), torch.bfloat16, 82, 1.0, device=DEV)
    qm, km = PosMap(0, 1), PosMap(0, 1)
    o, lse = cpa.partial_attn(q, k, v, qm, km, causal=True)
    assert o.shape == (0, hq, d) and lse.shape == (0, hq)
    o2, l2 = cpa.partial_attn_chunks(q, [(k, v, km), (k, v, PosMap(500, 1))], qm, causal=True)
    assert o2.shape == (0, hq, d)
    om, lm = cpa.merge_partials([o, o], [lse, lse])
    assert om.shape == (0, hq, d)
    aux = cpa.attn_bwd_prep(o, q, lse)
    dq = torch.zeros((0, hq, d), device=DEV)
    dk = torch.full(k.shape, 0.5, device=DEV)
    dv = torch.full(v.shape, 0.5, device=DEV)
    cpa.partial_attn_bwd(q, k, v, q, aux, qm, km, dq, dk, dv, causal=True)
    cpa.partial_attn_bwd_chunks(q, q, aux, qm, [(k, v, km, dk, dv)], dq)
    torch.cuda.synchronize()
    assert torch.all(dk == 0.5) and torch.all(dv == 0.5)


@pytest.mark.parametrize("d", [64, 128])
def test_large_logits(d):
    """Scores with a spread of tens (q, k ~ N(0, 6^2)): the running maximum jumps often, so the
    lazy rescale of O and l runs many times, and most probabilities underflow -- the result must
    still match the oracle (forward per chunk and over a chunk list, and the backward)."""
    sq, hq, hkv = 300, 4, 2
    qm, km1, km2 = PosMap(300, 1), PosMap(0, 1), PosMap(150, 2)
    q = wl.normal((sq, hq, d), torch.bfloat16, 91, 6.0, device=DEV)
    k1 = wl.normal((400, hkv, d), torch.bfloat16, 92, 6.0, device=DEV)
    v1 = wl.normal((400, hkv, d), torch.bfloat16, 93, 1.0, device=DEV)
    k2 = wl.normal((200, hkv, d), torch.bfloat16, 94, 6.0, device=DEV)
    v2 = wl.normal((200, hkv, d), torch.bfloat16, 95, 1.0, device=DEV)
    d_o = wl.normal((sq, hq, d), torch.bfloat16, 96, 1.0, device=DEV)
    qp, kp1, kp2 = _pos(qm, sq), _pos(km1, 400), _pos(km2, 200)
    o, lse = cpa.partial_attn(q, k1, v1, qm, km1, causal=True)
    ro, rl = oracle.attention(q.cpu(), k1.cpu(), v1.cpu(), qp, kp1, causal=True)
    compare_partial(o.cpu().numpy(), lse.cpu().numpy(), ro, rl, TOL_BF16_O, TOL_BF16_LSE, f"large logits d={d}")
    o2, l2 = cpa.partial_attn_chunks(q, [(k2, v2, km2), (k1, v1, km1)], qm, causal=True)
    ro2, rl2 = oracle.attention(q.cpu(), torch.cat([k1.cpu(), k2.cpu()]), torch.cat([v1.cpu(), v2.cpu()]), qp,
                                np.concatenate([kp1, kp2]), causal=True)
    compare_partial(o2.cpu().numpy(), l2.cpu().numpy(), ro2, rl2, TOL_BF16_O, TOL_BF16_LSE, f"large logits chunks d={d}")
    o32, l32 = torch.from_numpy(ro2).float(), torch.from_numpy(rl2).float()
    aux = cpa.attn_bwd_prep(o32.to(DEV), d_o, l32.to(DEV))
    dq = torch.zeros(q.shape, device=DEV)
    dk = torch.zeros(k1.shape, device=DEV)
    dv = torch.zeros(v1.shape, device=DEV)
    cpa.partial_attn_bwd(q, k1, v1, d_o, aux, qm, km1, dq, dk, dv, causal=True)
    torch.cuda.synchronize()
    ref = oracle.chunk_backward(q.cpu(), k1.cpu(), v1.cpu(), d_o.cpu(), o32, l32, qp, kp1, causal=True)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        compare_grad(g.cpu().numpy(), r, TOL_GRAD_BF16, f"large logits {name} d={d}")


@pytest.mark.parametrize("d", [64, 128])
def test_score_jumps_inside_tiles(d):
    """Every 128-key tile after the first raises the row maximum twice: keys 0..63 sit 7.9 (log2
    units) above the previous tiles' maximum and keys 64..127 10.5 above it, each group with a
    row sum of thousands, so the second half of a tile outgrows a reference that the first half
    still fits and O and l are rescaled between the two halves' contributions.  Both halves carry
    weight in the result (the first about a sixth of the second), so a contribution dropped or
    scaled twice shows in O and LSE.  Checked against the oracle per chunk and over a chunk list."""
    sq, hq, hkv, n = 1024, 2, 1, 1024
    scale = 1.0 / np.sqrt(d)
    u = np.full(d, 1.0 / np.sqrt(d))
    level = np.zeros(n)
    for t in range(1, n // 128):
        base = 10.5 * (t - 1)
        level[128 * t: 128 * t + 64] = base + 7.9
        level[128 * t + 64: 128 * (t + 1)] = base + 10.5
    a = level / (scale * np.log2(np.e))  # q = u, k_j = a_j u  =>  score_j * log2(e) = level_j
    rng = np.random.default_rng(7)
    q = torch.from_numpy(np.tile(u, (sq, hq, 1))).to(torch.bfloat16)
    k = torch.from_numpy((a[:, None] * u[None, :])[:, None, :].repeat(hkv, axis=1)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((n, hkv, d))).to(torch.bfloat16)
    qm, km = PosMap(0, 1), PosMap(0, 1)
    qp, kp = _pos(qm, sq), _pos(km, n)
    ro, rl = oracle.attention(q, k, v, qp, kp, causal=True)
    o, lse = cpa.partial_attn(q.to(DEV), k.to(DEV), v.to(DEV), qm, km, causal=True)
    compare_partial(o.cpu().numpy(), lse.cpu().numpy(), ro, rl, TOL_BF16_O, TOL_BF16_LSE, f"score jumps d={d}")
    half = n // 2
    chunks = [(k[:half].to(DEV), v[:half].to(DEV), PosMap(0, 1)), (k[half:].to(DEV), v[half:].to(DEV), PosMap(half, 1))]
    o2, l2 = cpa.partial_attn_chunks(q.to(DEV), chunks, qm, causal=True)
    compare_partial(o2.cpu().numpy(), l2.cpu().numpy(), ro, rl, TOL_BF16_O, TOL_BF16_LSE, f"score jumps chunks d={d}")
