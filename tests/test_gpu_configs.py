"""GPU parity at the benchmark workloads' full sizes, in the launch sequence bench.py times.

Workloads 1 and 2: every row and head of every partial and of the merged output.
Workloads 3-5: a seeded sample of 256 query rows per rank (always including row 0, the last
row, the rows on both sides of the first 128-row tile boundaries and, for workload 5, the first
visible row of every chunk and the row just before it), all heads; every partial on the same
rows.  Workload 4: 256 rows per head-rank.  The Ulysses reshards of workload 4 are compared bit
for bit in full.
"""

import numpy as np
import pytest
import torch

import helpers
import oracle
from helpers import TOL_BF16_LSE, TOL_BF16_O, TOL_F32, TOL_GRAD_BF16, compare_grad, compare_partial

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    helpers.ensure_built()

import bench  # noqa: E402
from context_blockwise_attention_gb300 import workloads as wl  # noqa: E402

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _rows_for(w, n_rows, sample, local=None):
    local = w.local_len if local is None else local
    if sample is None:
        return np.arange(local)
    must = [0, local - 1, 127, 128, 255, 256, 383, 384]
    if w.chunks_per_shard > 1:
        for c in range(w.chunks_per_shard):
            must += [c * w.chunk_len, c * w.chunk_len - 1]
    return wl.sample_rows(local, sample, seed=n_rows, must=must)


def _check_rank_workload(cfg, layout, sample, query_ranks=None):
    w = wl.WORKLOADS[cfg]
    tol_o, tol_l = (TOL_F32, TOL_F32) if w.dtype == "f32" else (TOL_BF16_O, TOL_BF16_LSE)
    steps = []
    for qr in (query_ranks or [None]):
        step = bench.Step(cfg, DEV, query_rank=qr, layout=layout)
        for kw in step.attn_calls:  # poison outputs so unwritten rows cannot pass
            kw["o"].fill_(float("nan"))
            kw["lse"].fill_(float("nan"))
        for _, _, out, lse in step.rank_plans:
            out.fill_(float("nan"))
            lse.fill_(float("nan"))
        step.run()
        torch.cuda.synchronize()
        steps.append(step)
    kv_cpu = {r: (k.cpu(), v.cpu()) for r, (k, v) in steps[0].kv.items()}
    shard_pos = {r: oracle.shard_positions(w.seq_len, w.cp, r, layout) for r in range(w.cp)}
    all_k = torch.cat([kv_cpu[r][0] for r in range(w.cp)])
    all_v = torch.cat([kv_cpu[r][1] for r in range(w.cp)])
    all_pos = np.concatenate([shard_pos[r] for r in range(w.cp)])
    worst = [0.0, 0.0]
    for step in steps:
        for qr, q, out, lse in step.rank_plans:
            qpos = shard_pos[qr]
            rows = _rows_for(w, w.local_len + qr, sample, local=q.shape[0])
            q_cpu = q.cpu()
            # every partial on the sampled rows of its query block; positions from the oracle's
            # own layout, cut to the call's row ranges
            for i, (cqr, row, nq, src, lo, nk) in enumerate(step.call_meta):
                if cqr != qr:
                    continue
                kw = step.attn_calls[i]
                sel = rows[(rows >= row) & (rows < row + nq)]
                if len(sel) == 0:
                    continue
                o_ref, l_ref = oracle.attention(q_cpu[sel], kv_cpu[src][0][lo:lo + nk],
                                                kv_cpu[src][1][lo:lo + nk], qpos[sel],
                                                shard_pos[src][lo:lo + nk], causal=w.causal)
                idx = torch.from_numpy(sel - row).to(DEV)
                eo, el = compare_partial(kw["o"][idx].float().cpu().numpy(), kw["lse"][idx].cpu().numpy(),
                                         o_ref, l_ref, tol_o, tol_l,
                                         f"cfg{cfg} rank{qr} rows {row}+ chunk({src},{lo})")
                worst = [max(worst[0], eo), max(worst[1], el)]
            # merged output against unsharded attention over every key
            o_ref, l_ref = oracle.attention(q_cpu[rows], all_k, all_v, qpos[rows], all_pos,
                                            causal=w.causal)
            idx = torch.from_numpy(rows).to(DEV)
            eo, el = compare_partial(out[idx].float().cpu().numpy(), lse[idx].cpu().numpy(), o_ref,
                                     l_ref, tol_o, tol_l, f"cfg{cfg} rank{qr} merged")
            worst = [max(worst[0], eo), max(worst[1], el)]
    return worst


def test_cfg1_fp32_all_ranks_full():
    # fp32 non-causal MHA S=512 CP=4: all 4 ranks, 4 chunks each in seeded random order
    worst = _check_rank_workload(1, "contiguous", None)
    assert worst[0] <= TOL_F32


def test_cfg2_rank7_full():
    # every row and head: 8 partials and the merged output
    _check_rank_workload(2, "strided", None)


def test_cfg2_rank0_sampled():
    _check_rank_workload(2, "strided", 256, query_ranks=[0])


@pytest.mark.parametrize("layout", ["strided", "contiguous", "two_block", "balanced"])
def test_cfg3_all_ranks_sampled(layout):
    _check_rank_workload(3, layout, 256)


def test_cfg5_rank7_sampled_outliers():
    _check_rank_workload(5, "strided", 256)


def _check_fused(cfg, layout, sample):
    w = wl.WORKLOADS[cfg]
    step = bench.Step(cfg, DEV, layout=layout, fused=True)
    for _, _, out, lse in step.rank_plans:
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    kv_cpu = {r: (k.cpu(), v.cpu()) for r, (k, v) in step.kv.items()}
    all_k = torch.cat([kv_cpu[r][0] for r in range(w.cp)])
    all_v = torch.cat([kv_cpu[r][1] for r in range(w.cp)])
    all_pos = np.concatenate([oracle.shard_positions(w.seq_len, w.cp, r, layout) for r in range(w.cp)])
    for qr, q, out, lse in step.rank_plans:
        qpos = oracle.shard_positions(w.seq_len, w.cp, qr, layout)
        rows = _rows_for(w, w.local_len + qr, sample, local=q.shape[0])
        idx = torch.from_numpy(rows).to(DEV)
        o_ref, l_ref = oracle.attention(q[idx].cpu(), all_k, all_v, qpos[rows], all_pos, causal=w.causal)
        compare_partial(out[idx].float().cpu().numpy(), lse[idx].cpu().numpy(), o_ref, l_ref,
                        TOL_BF16_O, TOL_BF16_LSE, f"cfg{cfg} fused rank{qr}")


def test_cfg2_fused_full():
    # one launch consumes the 8 chunks in arrival order; every row and head
    _check_fused(2, "strided", None)


@pytest.mark.parametrize("layout", ["strided", "contiguous"])
def test_cfg3_fused_sampled(layout):
    # every rank's query shard in one launch over its 8 chunks (contiguous: the chunks in the
    # shard's future are not issued)
    _check_fused(3, layout, 256)


def test_cfg3_balanced_fused_sampled():
    # shards of equal causal work and unequal length, each query shard in one launch
    _check_fused(3, "balanced", 256)


def test_cfg3_two_block_fused_sampled():
    # two query blocks per rank, each one launch over the 16 KV blocks visible to it
    _check_fused(3, "two_block", 256)


def test_cfg5_fused_sampled():
    # 64 chunks with K outliers in one launch
    _check_fused(5, "strided", 256)


def test_cfg4_ulysses():
    w = wl.WORKLOADS[4]
    cp, S = w.cp, w.seq_len
    step = bench.Step(4, DEV)
    for t in step.yo + step.ylse + step.xo:
        t.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    pos = [oracle.shard_positions(S, cp, r, w.layout) for r in range(cp)]
    i16 = torch.int16

    def ints(ts):
        return [t.cpu().view(i16).numpy() for t in ts]
    # seq -> head reshards, bit for bit
    for src, dst in ((step.qs, step.yq), (step.ks, step.yk), (step.vs, step.yv)):
        ref = oracle.seq_to_head(ints(src), pos)
        for r in range(cp):
            assert np.array_equal(dst[r].cpu().view(i16).numpy(), ref[r])
    # head -> seq reshard, bit for bit, on generated data in the step's own buffers
    hl, kl = w.hq // cp, w.hkv // cp
    gen = [wl.normal((S, hl, w.d), torch.bfloat16, 900 + r, device=DEV) for r in range(cp)]
    for r in range(cp):
        step.yo[r].copy_(gen[r])
    import context_blockwise_attention_gb300 as cpa
    cpa.ulysses_reshard("head_to_seq", [step.yo], cp, S, w.layout, out=[step.xo])
    torch.cuda.synchronize()
    back = oracle.head_to_seq(ints(gen), pos)
    for s in range(cp):
        assert np.array_equal(step.xo[s].cpu().view(i16).numpy(), back[s])
    # the whole step again, then attention on 256 sampled rows against the unsharded inputs:
    # per head-rank O and LSE (head-sharded), and the final sequence-sharded O.  (The path's final
    # product is O; LSE stays head-sharded, where the backward's three reversed exchanges use it.)
    for t in step.yo + step.ylse + step.xo:
        t.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    q_full = torch.cat([x.cpu() for x in step.qs])  # contiguous layout: global order
    k_full = torch.cat([x.cpu() for x in step.ks])
    v_full = torch.cat([x.cpu() for x in step.vs])
    gpos = np.arange(S)
    rows = wl.sample_rows(S, 256, seed=4, must=[0, 1, 127, 128, S - 1, S // 2])
    idx = torch.from_numpy(rows).to(DEV)
    local = S // cp
    for r in range(cp):
        o_ref, l_ref = oracle.attention(q_full[rows][:, r * hl:(r + 1) * hl], k_full[:, r * kl:(r + 1) * kl],
                                        v_full[:, r * kl:(r + 1) * kl], rows, gpos, causal=True)
        compare_partial(step.yo[r][idx].float().cpu().numpy(), step.ylse[r][idx].cpu().numpy(), o_ref,
                        l_ref, TOL_BF16_O, TOL_BF16_LSE, f"cfg4 head-rank {r}")
        final = np.stack([step.xo[t // local][t % local, r * hl:(r + 1) * hl].float().cpu().numpy()
                          for t in rows])
        assert helpers.max_abs(final, o_ref) <= TOL_BF16_O, f"cfg4 final output, heads of rank {r}"


def test_cfg2_backward_sampled():
    # the backward of workload 2 (rank 7, 8 chunks) as the bench times it: GPU forward (fused),
    # prep, one partial backward per chunk.  The oracle computes the rows' final O and LSE itself
    # (all rows, all keys), then the exact gradients on samples: dQ on sampled rows (against
    # every chunk), dK and dV on sampled keys of every shard (against every row)
    w = wl.WORKLOADS[2]
    fstep = bench.Step(2, DEV, fused=True)
    bstep = bench.BwdStep(fstep)
    bstep.run()
    torch.cuda.synchronize()
    assert len(fstep.blocks) == 1
    qr, qb, _, _, _, _ = fstep.blocks[0]
    layout = w.layout
    qpos = oracle.shard_positions(w.seq_len, w.cp, qr, layout)
    q_cpu = qb.cpu()
    d_o = bstep.preps[0]["d_o"].cpu()
    kv_cpu = {r: (k.cpu(), v.cpu()) for r, (k, v) in fstep.kv.items()}
    spos = {r: oracle.shard_positions(w.seq_len, w.cp, r, layout) for r in range(w.cp)}
    k_all = torch.cat([kv_cpu[r][0] for r in range(w.cp)])
    v_all = torch.cat([kv_cpu[r][1] for r in range(w.cp)])
    o_ref, l_ref = oracle.attention(q_cpu, k_all, v_all, qpos, np.concatenate([spos[r] for r in range(w.cp)]),
                                    causal=True)
    rows = _rows_for(w, w.local_len + qr, 256)
    ri = torch.from_numpy(rows)
    dq_ref = np.zeros((len(rows), w.hq, w.d))
    for r in range(w.cp):
        dq_ref += oracle.chunk_backward(q_cpu[ri], kv_cpu[r][0], kv_cpu[r][1], d_o[ri], o_ref[rows],
                                        l_ref[rows], qpos[rows], spos[r], causal=True)[0]
    compare_grad(bstep.dqs[0].cpu().numpy()[rows], dq_ref, TOL_GRAD_BF16, "cfg2 dQ (sampled rows)")
    keys = wl.sample_rows(w.local_len, 64, seed=3, must=[0, 127, 128, w.local_len - 1])
    ki = torch.from_numpy(keys)
    for r in range(w.cp):
        _, dk_ref, dv_ref = oracle.chunk_backward(q_cpu, kv_cpu[r][0][ki], kv_cpu[r][1][ki], d_o, o_ref, l_ref,
                                                  qpos, spos[r][keys], causal=True)
        compare_grad(bstep.dk[r].cpu().numpy()[keys], dk_ref, TOL_GRAD_BF16, f"cfg2 dK shard {r} (sampled keys)")
        compare_grad(bstep.dv[r].cpu().numpy()[keys], dv_ref, TOL_GRAD_BF16, f"cfg2 dV shard {r} (sampled keys)")



def test_cfg4_backward_sampled():
    # the Ulysses backward at full size as the bench times it (dO seq->head, 4 head-rank backward
    # calls over the whole sequence, dQ and dK|dV head->seq).  dQ exact on sampled rows (the
    # oracle computes the rows' O and LSE itself); dK, dV through identities of the softmax
    # Jacobian that hold at any size: per KV head, sum_j dV_j = sum_i (group's dO_i) and
    # sum_j dK_j = 0
    w = wl.WORKLOADS[4]
    cp, S = w.cp, w.seq_len
    hl, kl = w.hq // cp, w.hkv // cp
    bstep = bench.UlyssesBwdStep(bench.Step(4, DEV))
    bstep.run()
    torch.cuda.synchronize()
    f = bstep.fwd
    q_full = torch.cat([x.cpu() for x in f.qs])  # contiguous layout: global order
    k_full = torch.cat([x.cpu() for x in f.ks])
    v_full = torch.cat([x.cpu() for x in f.vs])
    do_full = torch.cat([x.cpu() for x in bstep.xdo])
    dq = torch.cat([x.cpu() for x in bstep.dqs]).numpy()
    dk = torch.cat([x.cpu() for x in bstep.dks]).double().numpy()
    dv = torch.cat([x.cpu() for x in bstep.dvs]).double().numpy()
    gpos = np.arange(S)
    rows = wl.sample_rows(S, 48, seed=6, must=[0, 1, 128, S - 1])
    ri = torch.from_numpy(rows)
    for r in range(cp):
        qh = q_full[:, r * hl:(r + 1) * hl]
        kh = k_full[:, r * kl:(r + 1) * kl]
        vh = v_full[:, r * kl:(r + 1) * kl]
        doh = do_full[:, r * hl:(r + 1) * hl]
        o_ref, l_ref = oracle.attention(qh[ri], kh, vh, rows, gpos, causal=True)
        dq_ref = oracle.chunk_backward(qh[ri], kh, vh, doh[ri], o_ref, l_ref, rows, gpos, causal=True)[0]
        # the forward's O is bf16 (the path's final output), so D = dO.O carries O's rounding into
        # whole dQ rows: dQ is held to the tensor-wide bound only
        compare_grad(dq[rows][:, r * hl:(r + 1) * hl], dq_ref, TOL_GRAD_BF16, f"cfg4 dQ head-rank {r}", rows=False)
    group = w.hq // w.hkv
    do64 = do_full.double().numpy()
    for g in range(w.hkv):
        want = do64[:, g * group:(g + 1) * group].sum(axis=(0, 1))
        got = dv[:, g].sum(axis=0)
        assert np.abs(got - want).max() <= 1e-2 * max(1.0, np.abs(want).max()), f"cfg4 sum dV, KV head {g}"
        ksum = np.abs(dk[:, g].sum(axis=0)).max()
        assert ksum <= 1e-2 * max(1.0, np.abs(dk[:, g]).sum(axis=0).max()), f"cfg4 sum dK, KV head {g}"


def test_e2e_overlapped_copies_match_resident_step():
    # the bench's end-to-end step copies each chunk on a second stream and lets every partial
    # wait only for its own chunk: with the device inputs wiped first, its merged output must be
    # the same bits as the step run on resident inputs
    step = bench.Step(2, DEV, host_copy=True)
    step.run()
    torch.cuda.synchronize()
    ref = [t.clone() for t in step._output_tensors]
    for _, d in step.host_inputs:
        d.fill_(float("nan"))
    step.run_e2e()
    torch.cuda.synchronize()
    for (d, h), r in zip(step.host_outputs, ref):
        assert torch.equal(d, r)
        assert torch.equal(h.to(DEV), r)
