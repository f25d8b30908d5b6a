"""GPU parity of the backward pass (prep kernel, fp32 CUDA-core and bf16 tensor-core partial
backward) against the float64 oracle's chain rule.

The final O and LSE a backward call needs come from the oracle (rounded to fp32), so a
backward test measures the backward kernels alone; the end-to-end test at the bottom runs the
forward on the GPU too.  Gradient buffers are poisoned with a known value first: the kernels
ACCUMULATE, so what they add is read as the difference.
"""

import time

import numpy as np
import pytest
import torch

import helpers
import oracle
from helpers import TOL_GRAD_BF16, TOL_GRAD_F32, compare_grad

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    helpers.ensure_built()

import context_blockwise_attention_gb300 as cpa  # noqa: E402
from context_blockwise_attention_gb300 import PosMap  # noqa: E402
from context_blockwise_attention_gb300 import workloads as wl  # noqa: E402

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None
LOG2E = 1.4426950408889634


def _pos(m: PosMap, n):
    return m.base + m.stride * np.arange(n, dtype=np.int64)


def test_prep_matches_definition():
    for dt_o, dt_do in ((torch.float32, torch.float32), (torch.bfloat16, torch.bfloat16),
                        (torch.bfloat16, torch.float32)):
        for sq, hq, d in ((300, 3, 128), (128, 2, 64), (1, 1, 64)):
            o = wl.normal((sq, hq, d), dt_o, 1, device=DEV)
            d_o = wl.normal((sq, hq, d), dt_do, 2, device=DEV)
            lse = wl.normal((sq, hq), torch.float32, 3, 4.0, device=DEV)
            lse[0, 0] = float("-inf")
            aux = torch.full((cpa.bwd_aux_floats(sq, hq),), float("nan"), device=DEV)
            cpa.attn_bwd_prep(o, d_o, lse, aux=aux)
            torch.cuda.synchronize()
            pad = (sq + 127) // 128 * 128
            a = aux.cpu().numpy().reshape(2, hq, pad)
            ln = lse.cpu().double().numpy()
            want_nl = np.where(np.isneginf(ln), -np.inf, -ln * LOG2E).T
            want_nd = -(o.cpu().double() * d_o.cpu().double()).sum(-1).numpy().T
            assert np.array_equal(np.isneginf(a[0, :, :sq]), np.isneginf(want_nl))
            fin = np.isfinite(want_nl)
            assert np.allclose(a[0, :, :sq][fin], want_nl[fin], rtol=1e-6, atol=1e-6)
            assert np.allclose(a[1, :, :sq], want_nd, rtol=1e-5, atol=1e-4)
            assert np.all(np.isneginf(a[0, :, sq:])) and np.all(a[1, :, sq:] == 0)


def _case_inputs(sq, skv, hq, hkv, d, causal, qm, km, dtype, seed, other_skv=0, other_km=None):
    """Query shard, one chunk and (optionally) a second chunk that shares the rows' softmax; the
    final O and LSE over both chunks come from the oracle."""
    q = wl.normal((sq, hq, d), dtype, seed + 1, 0.5, device=DEV)
    k = wl.normal((skv, hkv, d), dtype, seed + 2, 0.5, device=DEV)
    v = wl.normal((skv, hkv, d), dtype, seed + 3, 1.0, device=DEV)
    d_o = wl.normal((sq, hq, d), dtype, seed + 4, 1.0, device=DEV)
    k_all, v_all, pos_all = k.cpu(), v.cpu(), _pos(km, skv)
    if other_skv:
        k2 = wl.normal((other_skv, hkv, d), dtype, seed + 5, 0.5)
        v2 = wl.normal((other_skv, hkv, d), dtype, seed + 6, 1.0)
        k_all = torch.cat([k_all, k2])
        v_all = torch.cat([v_all, v2])
        pos_all = np.concatenate([pos_all, _pos(other_km, other_skv)])
    o_ref, l_ref = oracle.attention(q.cpu(), k_all, v_all, _pos(qm, sq), pos_all, causal=causal)
    o32 = torch.from_numpy(o_ref).float()
    l32 = torch.from_numpy(l_ref).float()
    return q, k, v, d_o, o32, l32


def _run_bwd(q, k, v, d_o, o32, l32, qm, km, causal, poison=0.25):
    aux = cpa.attn_bwd_prep(o32.to(DEV), d_o, l32.to(DEV))
    dq = torch.full(q.shape, poison, device=DEV)
    dk = torch.full(k.shape, poison, device=DEV)
    dv = torch.full(v.shape, poison, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    cpa.partial_attn_bwd(q, k, v, d_o, aux, qm, km, dq, dk, dv, causal=causal, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return (dq.cpu().double().numpy() - poison, dk.cpu().double().numpy() - poison,
            dv.cpu().double().numpy() - poison)


# (sq, skv, hq, hkv, d, causal, q map, kv map, other chunk (skv, map) or None)
BWD_CASES = [
    (256, 256, 2, 2, 128, False, PosMap(0, 1), PosMap(0, 1), None),
    (256, 256, 2, 2, 64, False, PosMap(0, 1), PosMap(0, 1), None),
    (384, 384, 4, 2, 128, True, PosMap(0, 1), PosMap(0, 1), None),
    (300, 777, 4, 1, 64, True, PosMap(3, 4), PosMap(0, 1), None),
    (513, 200, 8, 2, 128, True, PosMap(0, 1), PosMap(300, 1), (300, PosMap(0, 1))),  # early rows see nothing here
    (1024, 512, 8, 2, 128, True, PosMap(7, 8), PosMap(2, 8), (512, PosMap(4098, 8))),  # strided, second chunk
    (640, 1280, 4, 4, 64, True, PosMap(5, 8), PosMap(0, 4), None),
    (129, 129, 2, 1, 128, False, PosMap(0, 1), PosMap(0, 1), (64, PosMap(500, 1))),
    (200, 300, 2, 2, 128, True, PosMap(0, 1), PosMap(1000, 1), (200, PosMap(0, 1))),  # chunk in the future
    (1, 1, 1, 1, 64, True, PosMap(0, 1), PosMap(0, 1), None),
    (700, 390, 16, 2, 64, False, PosMap(0, 1), PosMap(0, 1), (100, PosMap(390, 1))),  # GQA 8, ragged, non-causal
    (257, 257, 1, 1, 128, True, PosMap(0, 1), PosMap(0, 1), None),                    # one head, ragged tails
    (512, 1024, 8, 8, 128, True, PosMap(3, 2), PosMap(0, 1), (256, PosMap(2048, 1))),  # MHA, strided queries
]


def _oracle_bwd(q, k, v, d_o, o32, l32, qm, km, causal):
    return oracle.chunk_backward(q.cpu(), k.cpu(), v.cpu(), d_o.cpu(), o32, l32, _pos(qm, q.shape[0]),
                                 _pos(km, k.shape[0]), causal=causal)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16_tc", "f32_simt"])
@pytest.mark.parametrize("case", BWD_CASES, ids=[f"bwd{i}" for i in range(len(BWD_CASES))])
def test_partial_bwd_parity(case, dtype):
    sq, skv, hq, hkv, d, causal, qm, km, other = case
    oskv, okm = other if other else (0, None)
    q, k, v, d_o, o32, l32 = _case_inputs(sq, skv, hq, hkv, d, causal, qm, km, dtype, 17, oskv, okm)
    got = _run_bwd(q, k, v, d_o, o32, l32, qm, km, causal)
    ref = _oracle_bwd(q, k, v, d_o, o32, l32, qm, km, causal)
    tol = TOL_GRAD_BF16 if dtype == torch.bfloat16 else TOL_GRAD_F32
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        compare_grad(g, r, tol, f"{name} {case[:6]} {dtype}")


def test_bwd_accumulates_and_empty_chunk_is_noop():
    sq, skv, hq, hkv, d = 256, 256, 4, 2, 128
    qm = km = PosMap(0, 1)
    q, k, v, d_o, o32, l32 = _case_inputs(sq, skv, hq, hkv, d, True, qm, km, torch.bfloat16, 5)
    aux = cpa.attn_bwd_prep(o32.to(DEV), d_o, l32.to(DEV))
    dq = torch.zeros(q.shape, device=DEV)
    dk = torch.zeros(k.shape, device=DEV)
    dv = torch.zeros(v.shape, device=DEV)
    cpa.partial_attn_bwd(q, k, v, d_o, aux, qm, km, dq, dk, dv)
    once = [t.clone() for t in (dq, dk, dv)]
    cpa.partial_attn_bwd(q, k, v, d_o, aux, qm, km, dq, dk, dv)
    e = torch.empty((0, hkv, d), dtype=torch.bfloat16, device=DEV)
    ez = torch.empty((0, hkv, d), device=DEV)
    cpa.partial_attn_bwd(q, e, e, d_o, aux, qm, PosMap(0, 1), dq, ez, ez)
    torch.cuda.synchronize()
    for a, b in zip((dq, dk, dv), once):
        assert torch.allclose(a, 2 * b, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16_tc", "f32_simt"])
def test_chunked_backward_equals_unsharded_gradient(dtype):
    # every rank of a strided cp=4 split, each against the 4 chunks (2 sub-chunks per shard) in a
    # seeded order: dQ summed over a rank's chunks, dK/dV summed into the chunk owner's buffers
    # over every query rank (the pages' reduce-scatter) = the gradient of unsharded attention
    seq, cp, hq, hkv, d = 1024, 4, 4, 2, 128
    qf = wl.normal((seq, hq, d), dtype, 61, 0.5)
    kf = wl.normal((seq, hkv, d), dtype, 62, 0.5)
    vf = wl.normal((seq, hkv, d), dtype, 63, 1.0)
    dof = wl.normal((seq, hq, d), dtype, 64, 1.0)
    full = np.arange(seq)
    o_ref, l_ref = oracle.attention(qf, kf, vf, full, full, causal=True)
    dq_ref, dk_ref, dv_ref = oracle.attention_backward(qf, kf, vf, dof, full, full, causal=True)
    shards = [oracle.shard_positions(seq, cp, r, "strided") for r in range(cp)]
    maps = [cpa.shard_layout(seq, cp, r, "strided") for r in range(cp)]
    local = seq // cp
    kd = [kf[torch.from_numpy(p)].contiguous().to(DEV) for p in shards]
    vd = [vf[torch.from_numpy(p)].contiguous().to(DEV) for p in shards]
    dk = [torch.zeros((local, hkv, d), device=DEV) for _ in range(cp)]
    dv = [torch.zeros((local, hkv, d), device=DEV) for _ in range(cp)]
    dq = np.zeros((seq, hq, d))
    half = local // 2
    for r in range(cp):
        idx = torch.from_numpy(shards[r])
        q = qf[idx].contiguous().to(DEV)
        d_o = dof[idx].contiguous().to(DEV)
        aux = cpa.attn_bwd_prep(torch.from_numpy(o_ref[shards[r]]).float().to(DEV), d_o,
                                torch.from_numpy(l_ref[shards[r]]).float().to(DEV))
        dq_r = torch.zeros((local, hq, d), device=DEV)
        for c in np.random.default_rng(r).permutation(2 * cp):
            src, sub = divmod(int(c), 2)
            sl = slice(sub * half, (sub + 1) * half)
            cpa.partial_attn_bwd(q, kd[src][sl], vd[src][sl], d_o, aux, maps[r],
                                 cpa.sub_chunk_map(maps[src], sub, half), dq_r, dk[src][sl], dv[src][sl])
        torch.cuda.synchronize()
        dq[shards[r]] = dq_r.cpu().double().numpy()
    tol = TOL_GRAD_BF16 if dtype == torch.bfloat16 else TOL_GRAD_F32
    compare_grad(dq, dq_ref, tol, "dQ (all ranks)")
    for r in range(cp):
        compare_grad(dk[r].cpu().numpy(), dk_ref[shards[r]], tol, f"dK shard {r}")
        compare_grad(dv[r].cpu().numpy(), dv_ref[shards[r]], tol, f"dV shard {r}")


def test_end_to_end_forward_then_backward():
    # forward on the GPU (partials + merge), then the backward from its own O and LSE
    seq, cp, r, hq, hkv, d = 2048, 4, 3, 8, 2, 64
    w_q = wl.normal((seq, hq, d), torch.bfloat16, 71, 0.5)
    w_k = wl.normal((seq, hkv, d), torch.bfloat16, 72, 0.5)
    w_v = wl.normal((seq, hkv, d), torch.bfloat16, 73, 1.0)
    w_do = wl.normal((seq, hq, d), torch.bfloat16, 74, 1.0)
    full = np.arange(seq)
    qpos = oracle.shard_positions(seq, cp, r, "contiguous")
    qm = cpa.shard_layout(seq, cp, r, "contiguous")
    q = w_q[torch.from_numpy(qpos)].contiguous().to(DEV)
    d_o = w_do[torch.from_numpy(qpos)].contiguous().to(DEV)
    chunks = []
    for c in range(r + 1):  # contiguous layout: later chunks are entirely in the future
        p = oracle.shard_positions(seq, cp, c, "contiguous")
        chunks.append((w_k[torch.from_numpy(p)].contiguous().to(DEV), w_v[torch.from_numpy(p)].contiguous().to(DEV),
                       cpa.shard_layout(seq, cp, c, "contiguous")))
    o, lse = cpa.partial_attn_chunks(q, chunks, qm, o_dtype=torch.bfloat16)
    aux = cpa.attn_bwd_prep(o, d_o, lse)
    dq = torch.zeros(q.shape, device=DEV)
    grads = []
    for k, v, km in chunks:
        dk = torch.zeros(k.shape, device=DEV)
        dv = torch.zeros(k.shape, device=DEV)
        cpa.partial_attn_bwd(q, k, v, d_o, aux, qm, km, dq, dk, dv)
        grads.append((dk, dv))
    torch.cuda.synchronize()
    # reference: this rank's share of the unsharded gradient = the gradient of its own rows' loss
    kk = torch.cat([c[0].cpu() for c in chunks])
    vv = torch.cat([c[1].cpu() for c in chunks])
    kpos = full[:len(kk)]
    dq_ref, dk_ref, dv_ref = oracle.attention_backward(q.cpu(), kk, vv, d_o.cpu(), qpos, kpos, causal=True)
    compare_grad(dq.cpu().numpy(), dq_ref, TOL_GRAD_BF16, "e2e dQ")
    n = seq // cp
    for c, (dk, dv) in enumerate(grads):
        compare_grad(dk.cpu().numpy(), dk_ref[c * n:(c + 1) * n], TOL_GRAD_BF16, f"e2e dK chunk {c}")
        compare_grad(dv.cpu().numpy(), dv_ref[c * n:(c + 1) * n], TOL_GRAD_BF16, f"e2e dV chunk {c}")


def test_ulysses_backward_three_steps_in_reverse():
    # Ulysses: forward = reshard Q and K|V seq->head, full-sequence attention per head-rank,
    # reshard O head->seq; backward = the same three steps in reverse: dO seq->head, the
    # backward per head-rank, dQ and dK|dV head->seq (fp32).  Compared with the gradients of
    # unsharded attention.
    seq, cp, hq, hkv, d = 1024, 4, 8, 4, 64
    full = PosMap(0, 1)
    qf = wl.normal((seq, hq, d), torch.bfloat16, 81, 0.5)
    kf = wl.normal((seq, hkv, d), torch.bfloat16, 82, 0.5)
    vf = wl.normal((seq, hkv, d), torch.bfloat16, 83, 1.0)
    dof = wl.normal((seq, hq, d), torch.bfloat16, 84, 1.0)
    local = seq // cp
    shard = lambda x: [x[r * local:(r + 1) * local].contiguous().to(DEV) for r in range(cp)]  # noqa: E731
    (yq,) = cpa.ulysses_reshard("seq_to_head", [shard(qf)], cp, seq)
    yk, yv = cpa.ulysses_reshard("seq_to_head", [shard(kf), shard(vf)], cp, seq)
    (ydo,) = cpa.ulysses_reshard("seq_to_head", [shard(dof)], cp, seq)
    dqh, dkh, dvh = [], [], []
    for r in range(cp):
        o, lse = cpa.partial_attn(yq[r], yk[r], yv[r], full, full, o_dtype=torch.bfloat16)
        aux = cpa.attn_bwd_prep(o, ydo[r], lse)
        dq = torch.zeros(yq[r].shape, device=DEV)
        dk = torch.zeros(yk[r].shape, device=DEV)
        dv = torch.zeros(yv[r].shape, device=DEV)
        cpa.partial_attn_bwd(yq[r], yk[r], yv[r], ydo[r], aux, full, full, dq, dk, dv)
        dqh.append(dq)
        dkh.append(dk)
        dvh.append(dv)
    (dqs,) = cpa.ulysses_reshard("head_to_seq", [dqh], cp, seq)
    dks, dvs = cpa.ulysses_reshard("head_to_seq", [dkh, dvh], cp, seq)
    torch.cuda.synchronize()
    pos = np.arange(seq)
    dq_ref, dk_ref, dv_ref = oracle.attention_backward(qf, kf, vf, dof, pos, pos, causal=True)
    for r in range(cp):
        sl = slice(r * local, (r + 1) * local)
        # the forward's O is bf16 here, so D = dO.O carries O's rounding; an error e in D_i enters
        # the whole dQ row as -e * scale * sum_j P_ij k_j, which does not cancel the way the
        # row's exact value does: dQ is held to the tensor-wide bound only
        compare_grad(dqs[r].cpu().numpy(), dq_ref[sl], TOL_GRAD_BF16, f"Ulysses dQ shard {r}", rows=False)
        compare_grad(dks[r].cpu().numpy(), dk_ref[sl], TOL_GRAD_BF16, f"Ulysses dK shard {r}")
        compare_grad(dvs[r].cpu().numpy(), dv_ref[sl], TOL_GRAD_BF16, f"Ulysses dV shard {r}")


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_bounded_wait_reports_timeout_and_context_survives(d):
    # block 0's MMA warp waits on a barrier nothing completes: its bounded wait expires, the
    # kernel records CP_ERR_TIMEOUT with the site, every CTA leaves, and the next call is correct
    # (both head dims: their waits and MMA issue take different forms)
    sq, skv, hq, hkv = 512, 512, 4, 2
    qm = km = PosMap(0, 1)
    q, k, v, d_o, o32, l32 = _case_inputs(sq, skv, hq, hkv, d, True, qm, km, torch.bfloat16, 9)
    aux = cpa.attn_bwd_prep(o32.to(DEV), d_o, l32.to(DEV))
    dq = torch.zeros(q.shape, device=DEV)
    dk = torch.zeros(k.shape, device=DEV)
    dv = torch.zeros(v.shape, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.time()
    cpa.partial_attn_bwd(q, k, v, d_o, aux, qm, km, dq, dk, dv, status=status, wait_timeout_ms=200,
                         flags=cpa.api.CP_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert time.time() - t0 < 20
    st = int(status.item())
    assert st & 0xff == cpa.api.CP_ERR_TIMEOUT and (st >> 8) >= 1, hex(st)
    got = _run_bwd(q, k, v, d_o, o32, l32, qm, km, True)
    ref = _oracle_bwd(q, k, v, d_o, o32, l32, qm, km, True)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        compare_grad(g, r, TOL_GRAD_BF16, f"{name} after a timed-out call")



@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16_tc", "f32_simt"])
def test_bwd_chunk_list_matches_oracle(dtype):
    # one call over a list of chunks (ragged, one empty, one entirely in the future, different
    # strides) = the sum of the chunks' shares
    sq, hq, hkv, d = 333, 4, 2, 128
    qm = PosMap(5, 3)
    specs = [(200, PosMap(0, 2)), (0, PosMap(0, 1)), (129, PosMap(400, 1)), (64, PosMap(5000, 1)),
             (300, PosMap(1, 3))]
    q = wl.normal((sq, hq, d), dtype, 91, 0.5, device=DEV)
    d_o = wl.normal((sq, hq, d), dtype, 92, 1.0, device=DEV)
    ks = [wl.normal((n, hkv, d), dtype, 93 + i, 0.5, device=DEV) for i, (n, _) in enumerate(specs)]
    vs = [wl.normal((n, hkv, d), dtype, 103 + i, 1.0, device=DEV) for i, (n, _) in enumerate(specs)]
    kpos = np.concatenate([_pos(m, n) for n, m in specs])
    o_ref, l_ref = oracle.attention(q.cpu(), torch.cat([k.cpu() for k in ks]), torch.cat([v.cpu() for v in vs]),
                                    _pos(qm, sq), kpos, causal=True)
    o32, l32 = torch.from_numpy(o_ref).float(), torch.from_numpy(l_ref).float()
    aux = cpa.attn_bwd_prep(o32.to(DEV), d_o, l32.to(DEV))
    dq = torch.zeros(q.shape, device=DEV)
    dks = [torch.zeros(k.shape, device=DEV) for k in ks]
    dvs = [torch.zeros(k.shape, device=DEV) for k in ks]
    cpa.partial_attn_bwd_chunks(q, d_o, aux, qm, [(k, v, m, dk, dv) for k, v, (_, m), dk, dv in
                                                   zip(ks, vs, specs, dks, dvs)], dq)
    torch.cuda.synchronize()
    tol = TOL_GRAD_BF16 if dtype == torch.bfloat16 else TOL_GRAD_F32
    dq_ref = np.zeros((sq, hq, d))
    for i, (n, m) in enumerate(specs):
        a, bk, bv = oracle.chunk_backward(q.cpu(), ks[i].cpu(), vs[i].cpu(), d_o.cpu(), o32, l32, _pos(qm, sq),
                                          _pos(m, n), causal=True)
        dq_ref += a
        compare_grad(dks[i].cpu().numpy(), bk, tol, f"chunk-list dK {i}")
        compare_grad(dvs[i].cpu().numpy(), bv, tol, f"chunk-list dV {i}")
    compare_grad(dq.cpu().numpy(), dq_ref, tol, "chunk-list dQ")


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_chunk_list_blocked_order(d):
    # enough units (KV tiles x chunks x heads >= 16 per SM) for the kernel to deal them in its
    # blocked order -- 16 KV tiles of a head together -- with chunks of 20 KV tiles (so blocks
    # run past a chunk's end), a ragged last tile, a chunk in the future and GQA 4
    sq, hq, hkv = 300, 16, 4
    qm = PosMap(20000, 7)
    specs = [(2560, PosMap(j, 8)) for j in range(7)] + [(2500, PosMap(7, 8)), (2560, PosMap(10 ** 6, 1))]
    assert sum(-(-n // 128) for n, _ in specs[:8]) * hq >= 16 * 152
    q = wl.normal((sq, hq, d), torch.bfloat16, 191, 0.5, device=DEV)
    d_o = wl.normal((sq, hq, d), torch.bfloat16, 192, 1.0, device=DEV)
    ks = [wl.normal((n, hkv, d), torch.bfloat16, 193 + i, 0.5, device=DEV) for i, (n, _) in enumerate(specs)]
    vs = [wl.normal((n, hkv, d), torch.bfloat16, 213 + i, 1.0, device=DEV) for i, (n, _) in enumerate(specs)]
    kpos = np.concatenate([_pos(m, n) for n, m in specs])
    o_ref, l_ref = oracle.attention(q.cpu(), torch.cat([k.cpu() for k in ks]), torch.cat([v.cpu() for v in vs]),
                                    _pos(qm, sq), kpos, causal=True)
    o32, l32 = torch.from_numpy(o_ref).float(), torch.from_numpy(l_ref).float()
    aux = cpa.attn_bwd_prep(o32.to(DEV), d_o, l32.to(DEV))
    dq = torch.zeros(q.shape, device=DEV)
    dks = [torch.zeros(k.shape, device=DEV) for k in ks]
    dvs = [torch.zeros(k.shape, device=DEV) for k in ks]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    cpa.partial_attn_bwd_chunks(q, d_o, aux, qm, [(k, v, m, dk, dv) for k, v, (_, m), dk, dv in
                                                   zip(ks, vs, specs, dks, dvs)], dq, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    dq_ref = np.zeros((sq, hq, d))
    for i, (n, m) in enumerate(specs):
        a, bk, bv = oracle.chunk_backward(q.cpu(), ks[i].cpu(), vs[i].cpu(), d_o.cpu(), o32, l32, _pos(qm, sq),
                                          _pos(m, n), causal=True)
        dq_ref += a
        compare_grad(dks[i].cpu().numpy(), bk, TOL_GRAD_BF16, f"blocked dK {i}")
        compare_grad(dvs[i].cpu().numpy(), bv, TOL_GRAD_BF16, f"blocked dV {i}")
    compare_grad(dq.cpu().numpy(), dq_ref, TOL_GRAD_BF16, "blocked dQ")
