"""GPU parity at small sizes: every kernel through the C ABI against the CPU oracle.

Sizes span several 128-row tiles and ragged tails while the oracle finishes in seconds.
Outputs are poisoned with NaN before each call so an unwritten row cannot pass.
"""

import time

import numpy as np
import pytest
import torch

import helpers
import oracle
from helpers import TOL_BF16_LSE, TOL_BF16_O, TOL_F32, compare_partial

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    helpers.ensure_built()

import context_blockwise_attention_gb300 as cpa  # noqa: E402
from context_blockwise_attention_gb300 import PosMap  # noqa: E402
from context_blockwise_attention_gb300 import api  # noqa: E402
from context_blockwise_attention_gb300 import workloads as wl  # noqa: E402

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _pos(m: PosMap, n):
    return m.base + m.stride * np.arange(n, dtype=np.int64)


def _run_partial(sq, skv, hq, hkv, d, causal, qm, km, dtype, o_dtype=torch.float32, flags=0,
                 seed=0, scale=0.0):
    q = wl.normal((sq, hq, d), dtype, seed * 10 + 1, 0.5, device=DEV)
    k = wl.normal((skv, hkv, d), dtype, seed * 10 + 2, 0.5, device=DEV)
    v = wl.normal((skv, hkv, d), dtype, seed * 10 + 3, 1.0, device=DEV)
    o = torch.full((sq, hq, d), float("nan"), dtype=o_dtype, device=DEV)
    lse = torch.full((sq, hq), float("nan"), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    cpa.partial_attn(q, k, v, qm, km, causal=causal, o=o, lse=lse, flags=flags, status=status,
                     scale=scale)
    torch.cuda.synchronize()
    assert status.item() == 0
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), _pos(qm, sq), _pos(km, skv),
                                    causal=causal, scale=scale if scale > 0 else None)
    return o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref


# (sq, skv, hq, hkv, d, causal, q map, kv map)
TC_CASES = [
    (256, 256, 2, 2, 128, False, PosMap(0, 1), PosMap(0, 1)),
    (256, 256, 2, 2, 64, False, PosMap(0, 1), PosMap(0, 1)),
    (384, 384, 4, 2, 128, True, PosMap(0, 1), PosMap(0, 1)),
    (300, 777, 4, 1, 64, True, PosMap(3, 4), PosMap(0, 1)),
    (513, 200, 8, 2, 128, True, PosMap(0, 1), PosMap(300, 1)),   # rows < 300 see nothing
    (1024, 1024, 8, 2, 128, True, PosMap(7, 8), PosMap(2, 8)),    # strided shard vs chunk
    (640, 1280, 4, 4, 64, True, PosMap(5, 8), PosMap(0, 4)),
    (1, 1, 1, 1, 64, True, PosMap(0, 1), PosMap(0, 1)),
    (129, 129, 2, 1, 128, False, PosMap(0, 1), PosMap(0, 1)),
    (200, 300, 2, 2, 128, True, PosMap(0, 1), PosMap(1000, 1)),   # whole chunk in the future
]


@pytest.mark.parametrize("case", TC_CASES, ids=[f"tc{i}" for i in range(len(TC_CASES))])
def test_tc_partial_parity(case):
    sq, skv, hq, hkv, d, causal, qm, km = case
    o, l, o_ref, l_ref = _run_partial(sq, skv, hq, hkv, d, causal, qm, km, torch.bfloat16,
                                      seed=sq + skv)
    compare_partial(o, l, o_ref, l_ref, TOL_BF16_O, TOL_BF16_LSE, f"tc {case}")


@pytest.mark.parametrize("case", [TC_CASES[3], TC_CASES[5], TC_CASES[6]], ids=["r3", "r5", "r6"])
def test_tc_descending_tile_order(case):
    # visiting the chunk's KV tiles last-to-first gives the same partial
    sq, skv, hq, hkv, d, causal, qm, km = case
    o, l, o_ref, l_ref = _run_partial(sq, skv, hq, hkv, d, causal, qm, km, torch.bfloat16,
                                      flags=api.CP_FLAG_KV_DESCENDING, seed=3)
    compare_partial(o, l, o_ref, l_ref, TOL_BF16_O, TOL_BF16_LSE, "descending")


def test_tc_bf16_output_and_scale():
    sq, skv, hq, hkv, d = 384, 512, 4, 2, 128
    o, l, o_ref, l_ref = _run_partial(sq, skv, hq, hkv, d, True, PosMap(128, 1), PosMap(0, 1),
                                      torch.bfloat16, o_dtype=torch.bfloat16, seed=9, scale=0.2)
    compare_partial(o, l, o_ref, l_ref, TOL_BF16_O, TOL_BF16_LSE, "bf16 out")


def test_tc_empty_chunk():
    q = wl.normal((100, 2, 64), torch.bfloat16, 1, device=DEV)
    k = torch.empty((0, 2, 64), dtype=torch.bfloat16, device=DEV)
    o, l = cpa.partial_attn(q, k, k, PosMap(0, 1), PosMap(0, 1))
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(l))


SIMT_CASES = [
    (128, 128, 2, 2, 64, False, PosMap(0, 1), PosMap(0, 1)),
    (200, 333, 4, 2, 128, True, PosMap(1, 3), PosMap(0, 1)),
    (64, 64, 2, 1, 64, True, PosMap(0, 1), PosMap(32, 1)),
    (1, 5, 1, 1, 64, True, PosMap(4, 1), PosMap(0, 1)),
]


@pytest.mark.parametrize("case", SIMT_CASES, ids=[f"simt{i}" for i in range(len(SIMT_CASES))])
def test_simt_partial_parity(case):
    sq, skv, hq, hkv, d, causal, qm, km = case
    o, l, o_ref, l_ref = _run_partial(sq, skv, hq, hkv, d, causal, qm, km, torch.float32, seed=5)
    compare_partial(o, l, o_ref, l_ref, TOL_F32, TOL_F32, f"simt {case}")


def test_simt_descending():
    sq, skv, hq, hkv, d, causal, qm, km = SIMT_CASES[1]
    o, l, o_ref, l_ref = _run_partial(sq, skv, hq, hkv, d, causal, qm, km, torch.float32,
                                      flags=api.CP_FLAG_KV_DESCENDING, seed=6)
    compare_partial(o, l, o_ref, l_ref, TOL_F32, TOL_F32, "simt descending")


# ------------------------------------------------------------------------------- layout

@pytest.mark.parametrize("kind", ["contiguous", "strided"])
def test_layout_positions_bit_exact(kind):
    for seq, cp in ((64, 4), (32768, 8), (262144, 8), (131072, 4), (7, 7)):
        for r in range(cp):
            m, pos = cpa.shard_layout(seq, cp, r, kind, positions=True)
            ref = oracle.shard_positions(seq, cp, r, kind)
            assert np.array_equal(pos.cpu().numpy().astype(np.int64), ref)
            assert np.array_equal(_pos(m, len(ref)), ref)


def test_segments_positions_bit_exact():
    for kind in ("contiguous", "strided", "two_block", "balanced"):
        for seq, cp in ((64, 4), (32768, 8), (131072, 4), (16, 8)):
            if kind == "balanced" and seq < 4 * cp:
                continue
            for r in range(cp):
                segs, pos = cpa.shard_segments(seq, cp, r, kind, positions=True)
                ref = oracle.shard_positions(seq, cp, r, kind)
                assert np.array_equal(pos.cpu().numpy().astype(np.int64), ref)
                assert np.array_equal(np.concatenate([_pos(m, n) for m, n in segs]), ref)


@pytest.mark.parametrize("d", [64, 128])
def test_two_block_layout_attention(d):
    # every rank of a two-block split: each query segment against every rank's KV segments,
    # fused (one call per query segment) and as partials + merge; the union over ranks is the
    # unsharded causal attention
    seq, cp, hq, hkv = 2048, 4, 4, 2
    qf = wl.normal((seq, hq, d), torch.bfloat16, 501, 0.5, device=DEV)
    kf = wl.normal((seq, hkv, d), torch.bfloat16, 502, 0.5, device=DEV)
    vf = wl.normal((seq, hkv, d), torch.bfloat16, 503, 1.0, device=DEV)
    o_ref, l_ref = oracle.attention(qf.cpu(), kf.cpu(), vf.cpu(), np.arange(seq), np.arange(seq),
                                    causal=True)
    segs = [cpa.shard_segments(seq, cp, r, "two_block") for r in range(cp)]
    kv_chunks = []
    for r in range(cp):
        for m, n in segs[r]:
            kv_chunks.append((kf[m.base:m.base + n].contiguous(), vf[m.base:m.base + n].contiguous(), m))
    order = np.random.default_rng(5).permutation(len(kv_chunks))
    for r in range(cp):
        pos = np.concatenate([_pos(m, n) for m, n in segs[r]])
        q = qf[torch.from_numpy(pos).to(DEV)].contiguous()
        o_fused = torch.full((len(pos), hq, d), float("nan"), device=DEV)
        l_fused = torch.full((len(pos), hq), float("nan"), device=DEV)
        parts = []
        row = 0
        for m, n in segs[r]:
            cpa.partial_attn_chunks(q[row:row + n], [kv_chunks[i] for i in order], m,
                                    o=o_fused[row:row + n], lse=l_fused[row:row + n])
            row += n
        for i in order:
            k, v, km = kv_chunks[i]
            o_p = torch.full((len(pos), hq, d), float("nan"), device=DEV)
            l_p = torch.full((len(pos), hq), float("nan"), device=DEV)
            row = 0
            for m, n in segs[r]:
                cpa.partial_attn(q[row:row + n], k, v, m, km, o=o_p[row:row + n], lse=l_p[row:row + n])
                row += n
            parts.append((o_p, l_p))
        o_m, l_m = cpa.merge_partials([p[0] for p in parts], [p[1] for p in parts],
                                      out_dtype=torch.float32)
        torch.cuda.synchronize()
        for o, l, what in ((o_fused, l_fused, "fused"), (o_m, l_m, "partials+merge")):
            compare_partial(o.cpu().numpy(), l.cpu().numpy(), o_ref[pos], l_ref[pos],
                            TOL_BF16_O, TOL_BF16_LSE, f"two-block rank {r} {what} d={d}")


# ------------------------------------------------------------------------------- merge

def _random_partials(n, sq, h, d, seed, empty_frac=0.3, spread=4.0):
    rng = np.random.default_rng(seed)
    os_ = [rng.standard_normal((sq, h, d)).astype(np.float32) for _ in range(n)]
    ls = [(rng.standard_normal((sq, h)) * spread).astype(np.float32) for _ in range(n)]
    for i in range(n):
        mask = rng.random((sq, h)) < empty_frac
        ls[i][mask] = -np.inf
        os_[i][mask] = 0.0
    return os_, ls


@pytest.mark.parametrize("n,d", [(1, 64), (3, 128), (8, 128), (64, 64), (128, 32), (5, 256)])
def test_merge_parity(n, d):
    sq, h = 77, 3
    os_, ls = _random_partials(n, sq, h, d, seed=n * d)
    ls[0][0, 0] = 80.0  # extreme spread in one row
    for i in range(n):  # one row empty in every partial
        ls[i][1, 1] = -np.inf
        os_[i][1, 1] = 0.0
    o_ref, l_ref = oracle.merge(os_, ls)
    og = [torch.from_numpy(x).to(DEV) for x in os_]
    lg = [torch.from_numpy(x).to(DEV) for x in ls]
    for out_dtype, tol in ((torch.float32, 1e-5), (torch.bfloat16, 2e-2)):
        o = torch.full((sq, h, d), float("nan"), dtype=out_dtype, device=DEV)
        lse = torch.full((sq, h), float("nan"), device=DEV)
        cpa.merge_partials(og, lg, o=o, lse=lse)
        torch.cuda.synchronize()
        compare_partial(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, tol, 1e-5,
                        f"merge n={n} d={d} {out_dtype}")


def test_merge_order_independent_and_associative():
    n, sq, h, d = 8, 64, 4, 128
    os_, ls = _random_partials(n, sq, h, d, seed=1)
    og = [torch.from_numpy(x).to(DEV) for x in os_]
    lg = [torch.from_numpy(x).to(DEV) for x in ls]
    base_o, base_l = cpa.merge_partials(og, lg, out_dtype=torch.float32)
    rng = np.random.default_rng(0)
    for _ in range(8):
        perm = rng.permutation(n)
        o, l = cpa.merge_partials([og[i] for i in perm], [lg[i] for i in perm],
                                  out_dtype=torch.float32)
        assert torch.allclose(o, base_o, atol=1e-5, rtol=0)
        assert torch.allclose(l, base_l, atol=1e-5, rtol=0, equal_nan=False) or \
            torch.equal(torch.isneginf(l), torch.isneginf(base_l))
    a_o, a_l = cpa.merge_partials(og[:3], lg[:3], out_dtype=torch.float32)
    b_o, b_l = cpa.merge_partials([a_o] + og[3:], [a_l] + lg[3:], out_dtype=torch.float32)
    torch.cuda.synchronize()
    fin = torch.isfinite(base_l)
    assert torch.allclose(b_o, base_o, atol=1e-5, rtol=0)
    assert torch.allclose(b_l[fin], base_l[fin], atol=1e-5, rtol=0)


# ------------------------------------------------------------------------------- reshard

@pytest.mark.parametrize("kind", ["contiguous", "strided", "two_block"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_reshard_bit_exact(kind, dtype):
    seq, cp, d = 512, 4, 64
    heads = (16, 8, 8)  # Q, and K|V fused in one launch
    w = wl.Workload(0, "t", "bf16", True, 16, 8, d, seq, cp, kind)
    shards = [[wl.normal((seq // cp, hh, d), dtype, 100 * t + r, device=DEV) for r in range(cp)]
              for t, hh in enumerate(heads)]
    pos = [oracle.shard_positions(seq, cp, r, kind) for r in range(cp)]
    (yq,) = cpa.ulysses_reshard("seq_to_head", [shards[0]], cp, seq, kind)
    yk, yv = cpa.ulysses_reshard("seq_to_head", [shards[1], shards[2]], cp, seq, kind)
    torch.cuda.synchronize()
    for t, ys in ((0, yq), (1, yk), (2, yv)):
        ref = oracle.seq_to_head([x.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy()
                                  for x in shards[t]], pos)
        for r in range(cp):
            got = ys[r].cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy()
            assert np.array_equal(got, ref[r])
    (xb,) = cpa.ulysses_reshard("head_to_seq", [yq], cp, seq, kind)
    torch.cuda.synchronize()
    for r in range(cp):
        assert torch.equal(xb[r], shards[0][r])
    del w


# ------------------------------------------------------------------------------- fault

@pytest.mark.parametrize("d", [64, 128])
def test_bounded_wait_reports_timeout_and_context_survives(d):
    # both head dims: the bounded waits and the MMA issue take a different form at each
    sq, skv, hq, hkv = 512, 512, 4, 2
    q = wl.normal((sq, hq, d), torch.bfloat16, 1, device=DEV)
    k = wl.normal((skv, hkv, d), torch.bfloat16, 2, device=DEV)
    v = wl.normal((skv, hkv, d), torch.bfloat16, 3, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.time()
    cpa.partial_attn(q, k, v, PosMap(0, 1), PosMap(0, 1), causal=True, status=status,
                     flags=api.CP_FLAG_TEST_STALL, wait_timeout_ms=50)
    torch.cuda.synchronize()
    dt = time.time() - t0
    st = status.item()
    assert st & 0xff == api.CP_ERR_TIMEOUT, st
    # the site of whichever bounded wait expired first: the injected one (9) or a wait that
    # depends on it (the stalled MMA warp starves the S/P/O handshakes and the TMA ring)
    assert (st >> 8) in range(1, 10), st
    assert dt < 10.0
    # the context is still usable and a normal call is correct
    o, l, o_ref, l_ref = _run_partial(sq, skv, hq, hkv, d, True, PosMap(0, 1), PosMap(0, 1),
                                      torch.bfloat16, seed=77)
    compare_partial(o, l, o_ref, l_ref, TOL_BF16_O, TOL_BF16_LSE, "after fault")


# ------------------------------------------------------------------------------- fused chunk list

# (sq, hq, hkv, d, causal, q map, [(skv, kv map)], dtype)
FUSED_CASES = [
    (384, 4, 2, 128, True, PosMap(7, 8),
     [(256, PosMap(0, 8)), (300, PosMap(2, 8)), (0, PosMap(5, 8)), (129, PosMap(3, 8))], torch.bfloat16),
    (300, 4, 1, 64, True, PosMap(3, 4), [(777, PosMap(0, 1)), (128, PosMap(5000, 1))], torch.bfloat16),
    (256, 2, 2, 64, False, PosMap(0, 1), [(100, PosMap(0, 1)), (200, PosMap(100, 1)), (50, PosMap(300, 1))],
     torch.bfloat16),
    (513, 8, 2, 128, True, PosMap(0, 1), [(200, PosMap(300, 1)), (300, PosMap(0, 1))], torch.bfloat16),
    (200, 4, 2, 128, True, PosMap(1, 3), [(333, PosMap(0, 1)), (64, PosMap(2, 5))], torch.float32),
]


def _fused_inputs(case, seed):
    sq, hq, hkv, d, causal, qm, chunk_specs, dtype = case
    q = wl.normal((sq, hq, d), dtype, seed, 0.5, device=DEV)
    chunks = []
    for i, (skv, km) in enumerate(chunk_specs):
        k = wl.normal((skv, hkv, d), dtype, seed + 10 * i + 1, 0.5, device=DEV)
        v = wl.normal((skv, hkv, d), dtype, seed + 10 * i + 2, 1.0, device=DEV)
        chunks.append((k, v, km))
    return q, chunks


def _fused_oracle(case, q, chunks):
    sq, hq, hkv, d, causal, qm, _, _ = case
    k_all = torch.cat([c[0].cpu() for c in chunks])
    v_all = torch.cat([c[1].cpu() for c in chunks])
    pos = np.concatenate([_pos(c[2], c[0].shape[0]) for c in chunks])
    return oracle.attention(q.cpu(), k_all, v_all, _pos(qm, sq), pos, causal=causal)


@pytest.mark.parametrize("case", FUSED_CASES, ids=[f"fused{i}" for i in range(len(FUSED_CASES))])
def test_fused_chunks_parity_and_order(case):
    sq, hq, hkv, d, causal, qm, _, dtype = case
    q, chunks = _fused_inputs(case, 31)
    o_ref, l_ref = _fused_oracle(case, q, chunks)
    tol_o, tol_l = (TOL_F32, TOL_F32) if dtype == torch.float32 else (TOL_BF16_O, TOL_BF16_LSE)
    for order in (list(range(len(chunks))), list(range(len(chunks)))[::-1]):
        o = torch.full((sq, hq, d), float("nan"), dtype=torch.float32, device=DEV)
        lse = torch.full((sq, hq), float("nan"), device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        cpa.partial_attn_chunks(q, [chunks[i] for i in order], qm, causal=causal, o=o, lse=lse,
                                status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        compare_partial(o.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, tol_o, tol_l,
                        f"fused {case[:6]} order {order}")


def test_fused_matches_partials_plus_merge():
    case = FUSED_CASES[0]
    sq, hq, hkv, d, causal, qm, _, _ = case
    q, chunks = _fused_inputs(case, 77)
    o_f, l_f = cpa.partial_attn_chunks(q, chunks, qm, causal=causal, o_dtype=torch.bfloat16)
    parts = [cpa.partial_attn(q, k, v, qm, km, causal=causal) for k, v, km in chunks if k.shape[0] > 0]
    o_m, l_m = cpa.merge_partials([p[0] for p in parts], [p[1] for p in parts], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    fin = torch.isfinite(l_m)
    assert torch.equal(torch.isneginf(l_f), torch.isneginf(l_m))
    assert (o_f.float() - o_m.float()).abs().max().item() <= TOL_BF16_O
    assert (l_f[fin] - l_m[fin]).abs().max().item() <= TOL_BF16_LSE


def test_fused_all_chunks_empty():
    q = wl.normal((50, 2, 64), torch.bfloat16, 1, device=DEV)
    e = torch.empty((0, 2, 64), dtype=torch.bfloat16, device=DEV)
    o, l = cpa.partial_attn_chunks(q, [(e, e, PosMap(0, 1)), (e, e, PosMap(9, 1))], PosMap(0, 1))
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(l))


@pytest.mark.parametrize("kind", ["contiguous", "strided", "two_block"])
@pytest.mark.parametrize("cp", [1, 64])
def test_reshard_extreme_cp_and_four_tensors(cp, kind):
    # the API's extremes: one rank, and 64 ranks with one head each (a 128-byte run per token);
    # four tensors in one launch, both directions, bit-exact against the oracle's index formula
    seq, d = 1024, 64
    heads = (64, 64, 128, 64)
    shards = [[wl.normal((seq // cp, hh, d), torch.bfloat16, 700 + 10 * t + r, device=DEV) for r in range(cp)]
              for t, hh in enumerate(heads)]
    pos = [oracle.shard_positions(seq, cp, r, kind) for r in range(cp)]
    ys = cpa.ulysses_reshard("seq_to_head", shards, cp, seq, kind)
    torch.cuda.synchronize()
    for t in range(4):
        ref = oracle.seq_to_head([x.cpu().view(torch.int16).numpy() for x in shards[t]], pos)
        for r in range(cp):
            assert np.array_equal(ys[t][r].cpu().view(torch.int16).numpy(), ref[r]), (t, r)
    back = cpa.ulysses_reshard("head_to_seq", ys, cp, seq, kind)
    torch.cuda.synchronize()
    for t in range(4):
        for r in range(cp):
            assert torch.equal(back[t][r], shards[t][r]), (t, r)
