"""Stream-pipelined chunk arrival (the FCP article, section 4.3) against the oracle.

The KV chunks of one query rank arrive by copies on a second stream, from pinned host memory or
from another device buffer; each partial waits on its own chunk's CUDA event, either with a
receive buffer per chunk or with two receive buffers reused in turn (the copy of chunk i waits
for the partial of chunk i-2).  After the merge, O and LSE of sampled query rows must match the
oracle's unsharded attention over every key -- the schedule may change when data lands, never
what is computed.  Chunk sizes span the page's 4K-8K range (8192 needs workload 3's shards).
"""

import numpy as np
import pytest
import torch

import helpers
import oracle
from helpers import TOL_BF16_LSE, TOL_BF16_O, compare_partial

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    helpers.ensure_built()

import bench  # noqa: E402
from context_blockwise_attention_gb300 import workloads as wl  # noqa: E402

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None

def _reference(ps, rows):
    """Oracle O and LSE of the sampled rows of the step's query shard over every key of the
    workload, from the very tensors the step holds (its Q from the device, K and V from the host
    copies the chunks arrive from)."""
    w = ps.w
    pos = [oracle.shard_positions(w.seq_len, w.cp, r, w.layout) for r in range(w.cp)]
    k = torch.cat(ps.host_k)
    v = torch.cat(ps.host_v)
    q = ps.q.cpu()[torch.from_numpy(rows)]
    return oracle.attention(q, k, v, pos[ps.qr][rows], np.concatenate(pos), causal=w.causal)


@pytest.mark.parametrize("cfg,chunk_tokens,source", [
    (2, 1024, "pinned_host"), (2, 4096, "device"), (3, 2048, "device"), (3, 8192, "pinned_host")])
def test_pipelined_schedules_match_oracle(cfg, chunk_tokens, source):
    w = wl.WORKLOADS[cfg]
    ps = bench.PipelinedStep(cfg, DEV, chunk_tokens, source)
    assert ps.n == w.cp * (w.local_len // chunk_tokens)
    rows = wl.sample_rows(w.local_len, 256, seed=chunk_tokens + cfg,
                          must=[0, 127, 128, w.local_len - 1])
    o_ref, l_ref = _reference(ps, rows)
    idx = torch.from_numpy(rows).to(DEV)
    for name in ("serial", "overlapped", "double_buffered"):
        # poison every partial and the merged output so rows a schedule skipped cannot pass
        for c in ps.chunks:
            for t in (c["o"], c["l"], c["dk"], c["dv"]):
                t.fill_(float("nan"))
        for dk, dv in ps.ring:
            dk.fill_(float("nan"))
            dv.fill_(float("nan"))
        ps.out.fill_(float("nan"))
        ps.lse.fill_(float("nan"))
        getattr(ps, name)()
        torch.cuda.synchronize()
        compare_partial(ps.out[idx].float().cpu().numpy(), ps.lse[idx].cpu().numpy(), o_ref, l_ref,
                        TOL_BF16_O, TOL_BF16_LSE, f"cfg{cfg} {source} {chunk_tokens}-token chunks, {name}")
