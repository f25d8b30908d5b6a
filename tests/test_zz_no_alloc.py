"""The backward entry point that allocates nothing (``cp_partial_attn_bwd_noalloc``).

Some callers cannot allocate device memory: a runtime that forbids cudaMalloc once it has
started, code running inside a memory pool it does not own, or a hook that is handed only its
inputs and outputs.  For them the library keeps the backward's per-row workspace in a fixed
array of its own.  These tests check, through the C ABI, that this entry point gives the same
gradients as the ordinary two-call path (``cp_attn_bwd_prep`` into a caller-allocated workspace,
then ``cp_partial_attn_bwd``), on several calls in a row with different shapes, so that what one
call leaves in the shared array cannot leak into the next; that on one case its gradients match
the CPU oracle's chain rule directly; that once the first call has placed the array, further calls
leave the device's free memory unchanged; and that sizes above the array's limit are refused
with a clear message.

The file is named so that pytest collects it after every other test file.
"""

import ctypes

import numpy as np
import pytest
import torch

import helpers
import oracle
from helpers import TOL_GRAD_BF16, TOL_GRAD_F32, compare_grad

helpers.ensure_built()

import context_blockwise_attention_gb300 as cpa  # noqa: E402
from context_blockwise_attention_gb300 import PosMap, api  # noqa: E402
from context_blockwise_attention_gb300 import workloads as wl  # noqa: E402


def _desc(sq, hq, aux=None):
    d = api._AttnBwdDesc()
    p = 0x1000
    d.q = d.k = d.v = d.d_o = p
    d.in_dtype = api.CP_BF16
    d.aux = aux
    d.dq = d.dk = d.dv = p
    d.sq, d.skv, d.hq, d.hkv, d.d = sq, 128, hq, 1, 128
    d.causal = 1
    d.q_pos = api._PosMap(0, 1)
    d.kv_pos = api._PosMap(0, 1)
    return d


def test_noalloc_rejects_on_host():
    """Refusals that happen before any device work (no GPU needed)."""
    lib = cpa.load_library()
    p = ctypes.c_void_p(0x1000)
    # one row more than the largest shard that fits: 2 * 64 * round_up(32769, 128) floats
    big = _desc(32769, 64)
    assert lib.cp_partial_attn_bwd_noalloc(ctypes.byref(big), p, api.CP_BF16, p, None) == api.CP_ERR_INVALID_ARG
    msg = lib.cp_last_error().decode()
    assert "limit" in msg and str(cpa.NOALLOC_AUX_MAX_FLOATS) in msg
    assert cpa.bwd_aux_floats(32768, 64) == cpa.NOALLOC_AUX_MAX_FLOATS
    with_aux = _desc(16, 2, aux=0x2000)
    assert lib.cp_partial_attn_bwd_noalloc(ctypes.byref(with_aux), p, api.CP_BF16, p, None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_partial_attn_bwd_noalloc(None, p, api.CP_BF16, p, None) == api.CP_ERR_INVALID_ARG


# (dtype, sq, skv, hq, hkv, d, causal, q_pos, kv_pos): shapes differ from call to call
_CASES = [
    (torch.bfloat16, 300, 400, 4, 2, 128, True, PosMap(200, 1), PosMap(0, 1)),
    (torch.bfloat16, 130, 257, 8, 8, 64, True, PosMap(1, 2), PosMap(0, 1)),
    (torch.float32, 77, 190, 2, 1, 64, False, PosMap(0, 1), PosMap(0, 1)),
]


def _inputs(case, seed, dev):
    dtype, sq, skv, hq, hkv, d, causal, qm, km = case
    q = wl.normal((sq, hq, d), dtype, seed, device=dev)
    k = wl.normal((skv, hkv, d), dtype, seed + 1, device=dev)
    v = wl.normal((skv, hkv, d), dtype, seed + 2, device=dev)
    d_o = wl.normal((sq, hq, d), dtype, seed + 3, device=dev)
    # the chunk is the shard's only one, so this partial is the final (O, LSE)
    o, lse = cpa.partial_attn(q, k, v, qm, km, causal=causal)
    return q, k, v, d_o, o, lse


@pytest.mark.gpu
def test_noalloc_matches_two_call_backward():
    dev = torch.device("cuda", 0)
    for i, case in enumerate(_CASES):
        dtype, sq, skv, hq, hkv, d, causal, qm, km = case
        q, k, v, d_o, o, lse = _inputs(case, 100 + 10 * i, dev)
        ref = [torch.zeros(t.shape, dtype=torch.float32, device=dev) for t in (q, k, v)]
        aux = cpa.attn_bwd_prep(o, d_o, lse)  # caller-allocated workspace
        cpa.partial_attn_bwd(q, k, v, d_o, aux, qm, km, *ref, causal=causal)
        got = [torch.zeros(t.shape, dtype=torch.float32, device=dev) for t in (q, k, v)]
        cpa.partial_attn_bwd_noalloc(q, k, v, d_o, o, lse, qm, km, *got, causal=causal)
        torch.cuda.synchronize()
        tol = TOL_GRAD_BF16 if dtype == torch.bfloat16 else TOL_GRAD_F32
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            compare_grad(g.cpu().numpy(), r.cpu().numpy(), tol, f"no-alloc {name} call {i} {case[:7]}")


@pytest.mark.gpu
def test_noalloc_matches_oracle():
    # bf16 GQA 8/2, D=128, a causal chunk whose keys straddle the query shard's positions; the
    # rows' final O and LSE come from the oracle (fp32) and feed both sides, so the comparison
    # isolates the backward
    dev = torch.device("cuda", 0)
    sq, skv, hq, hkv, d = 200, 300, 8, 2, 128
    qm, km = PosMap(150, 1), PosMap(0, 1)
    q = wl.normal((sq, hq, d), torch.bfloat16, 501, device=dev)
    k = wl.normal((skv, hkv, d), torch.bfloat16, 502, device=dev)
    v = wl.normal((skv, hkv, d), torch.bfloat16, 503, device=dev)
    d_o = wl.normal((sq, hq, d), torch.bfloat16, 504, device=dev)
    qpos = qm.base + np.arange(sq)
    kpos = km.base + np.arange(skv)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), qpos, kpos, causal=True)
    o32 = torch.from_numpy(o_ref).float().to(dev)
    l32 = torch.from_numpy(l_ref).float().to(dev)
    got = [torch.zeros(t.shape, dtype=torch.float32, device=dev) for t in (q, k, v)]
    cpa.partial_attn_bwd_noalloc(q, k, v, d_o, o32, l32, qm, km, *got, causal=True)
    torch.cuda.synchronize()
    ref = oracle.chunk_backward(q.cpu(), k.cpu(), v.cpu(), d_o.cpu(), o32.cpu(), l32.cpu(), qpos, kpos,
                                causal=True)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        compare_grad(g.cpu().numpy(), r, TOL_GRAD_BF16, f"no-alloc {name} vs oracle")


@pytest.mark.gpu
def test_noalloc_leaves_free_memory_unchanged():
    # the first call on the device places the array (lazy module loading); after it, calls must
    # not change the device's free memory (the library has its own CUDA runtime, so torch's
    # allocator counters would not see an allocation: read the device's own figure)
    dev = torch.device("cuda", 0)
    case = _CASES[0]
    q, k, v, d_o, o, lse = _inputs(case, 700, dev)
    qm, km = case[7], case[8]
    grads = [torch.zeros(t.shape, dtype=torch.float32, device=dev) for t in (q, k, v)]
    cpa.partial_attn_bwd_noalloc(q, k, v, d_o, o, lse, qm, km, *grads, causal=True)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    for _ in range(4):
        cpa.partial_attn_bwd_noalloc(q, k, v, d_o, o, lse, qm, km, *grads, causal=True)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


@pytest.mark.gpu
def test_noalloc_rejects_oversize_on_gpu():
    dev = torch.device("cuda", 0)
    sq, hq, d = 32769, 64, 64
    q = torch.zeros((sq, hq, d), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((128, 8, d), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((sq, hq), dtype=torch.float32, device=dev)
    dq = torch.zeros(q.shape, dtype=torch.float32, device=dev)
    dk = torch.zeros(k.shape, dtype=torch.float32, device=dev)
    with pytest.raises(cpa.CpError, match="limit"):
        cpa.partial_attn_bwd_noalloc(q, k, k, q, q, lse, PosMap(0, 1), PosMap(0, 1), dq, dk, dk.clone())


def test_noalloc_binding_rejects_bad_tensors():
    """The Python binding checks devices and shapes before calling the library (no GPU needed)."""
    q = torch.zeros((4, 2, 64), dtype=torch.bfloat16)
    k = torch.zeros((4, 1, 64), dtype=torch.bfloat16)
    lse = torch.zeros((4, 2))
    g = torch.zeros((4, 2, 64))
    gk = torch.zeros((4, 1, 64))
    with pytest.raises(cpa.CpError):  # host tensors
        cpa.partial_attn_bwd_noalloc(q, k, k, q, q, lse, PosMap(0, 1), PosMap(0, 1), g, gk, gk.clone())
