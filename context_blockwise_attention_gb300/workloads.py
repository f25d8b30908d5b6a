"""Seeded synthetic inputs for the five benchmark workloads.

This module draws random numbers and nothing else: no positions, masks, scores or merges.  The
library's tests feed the same tensors to the CUDA path and to the CPU oracle, so neither side
gets its inputs from the other.

Workloads (shapes follow the pages' examples; there is no dataset or trained model):

  1  fp32, non-causal MHA, H=2, D=64, S=512, CP=4 contiguous; every rank's 128 queries against
     the 4 KV chunks in a seeded random order, then merge.
  2  bf16, causal GQA 32 Q / 8 KV heads, D=128, S=32768, CP=8 strided; rank 7's 4096 queries
     against the 8 KV shards (one chunk each) in a seeded random order.
  3  bf16, causal MHA 32 heads, D=128, S=65536, CP=8, contiguous and strided layouts; all 8
     ranks against all 8 chunks, then 8 merges.
  4  bf16, causal GQA 64 / 8, D=64, S=131072, Ulysses cp=4: seq->head reshard of Q and fused
     K|V, full-sequence attention per head-rank (16 Q / 2 KV heads), head->seq reshard of O.
  5  bf16, causal GQA 64 / 8, D=64, S=262144, CP=8 strided; rank 7's 32768 queries against 64
     KV chunks of 4096 tokens (each rank's shard cut into 8) in a seeded random order; K has
     1% of its entries multiplied by 8.

Values are iid N(0,1) * value_scale drawn with ``torch.Generator`` (seed derived from the
workload seed, the tensor name and the rank), then rounded once to the input dtype.
"""

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    dtype: str          # "f32" or "bf16"
    causal: bool
    hq: int
    hkv: int
    d: int
    seq_len: int
    cp: int
    layout: str         # "contiguous" or "strided"
    chunks_per_shard: int = 1
    value_scale: float = 1.0
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    query_rank: int = -1  # -1: all ranks

    @property
    def local_len(self) -> int:
        return self.seq_len // self.cp

    @property
    def chunk_len(self) -> int:
        return self.local_len // self.chunks_per_shard

    @property
    def n_chunks(self) -> int:
        return self.cp * self.chunks_per_shard

    @property
    def input_seed(self) -> int:
        return 1000 + self.index

    @property
    def order_seed(self) -> int:
        return 2000 + self.index

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    1: Workload(1, "fp32 MHA H=2 D=64 S=512 CP=4 contiguous, non-causal", "f32", False,
                2, 2, 64, 512, 4, "contiguous"),
    2: Workload(2, "bf16 causal GQA 32/8 D=128 S=32768 CP=8 strided, rank 7 x 8 chunks", "bf16",
                True, 32, 8, 128, 32768, 8, "strided", value_scale=0.5, query_rank=7),
    3: Workload(3, "bf16 causal MHA 32 D=128 S=65536 CP=8, all ranks", "bf16", True,
                32, 32, 128, 65536, 8, "strided", value_scale=0.5),
    4: Workload(4, "bf16 causal GQA 64/8 D=64 S=131072 Ulysses cp=4", "bf16", True,
                64, 8, 64, 131072, 4, "contiguous", value_scale=0.5),
    5: Workload(5, "bf16 causal GQA 64/8 D=64 S=262144 CP=8 strided, rank 7 x 64 chunks, "
                   "K outliers", "bf16", True, 64, 8, 64, 262144, 8, "strided",
                chunks_per_shard=8, value_scale=1.0, outlier_frac=0.01, outlier_mult=8.0,
                query_rank=7),
}

_TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "o": 4}


def _sub_seed(seed: int, tensor: str, rank: int) -> int:
    return seed * 100003 + _TENSOR_IDS[tensor] * 1009 + rank


def normal(shape, dtype, seed, scale=1.0, device="cpu"):
    """iid N(0,1)*scale from a seeded generator, rounded once to ``dtype``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


def outlier_normal(shape, dtype, seed, frac, mult, device="cpu"):
    """iid N(0,1) where a seeded Bernoulli(frac) subset of entries is multiplied by ``mult``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    u = torch.rand(tuple(shape), generator=g, device=device, dtype=torch.float32)
    x = torch.where(u < frac, x * mult, x)
    return x.to(dtype)


def shard_tensor(w: Workload, tensor: str, rank: int, device="cpu", tokens=None, heads=None):
    """The ``tensor`` ('q', 'k' or 'v') shard of CP rank ``rank``: [S/cp, H, D] in w's dtype."""
    tokens = w.local_len if tokens is None else tokens
    if heads is None:
        heads = w.hq if tensor == "q" else w.hkv
    seed = _sub_seed(w.input_seed, tensor, rank)
    shape = (tokens, heads, w.d)
    if tensor == "k" and w.outlier_frac > 0:
        return outlier_normal(shape, w.torch_dtype, seed, w.outlier_frac, w.outlier_mult, device)
    return normal(shape, w.torch_dtype, seed, w.value_scale, device)


def arrival_order(n: int, seed: int) -> np.ndarray:
    """A seeded random permutation of 0..n-1 (the order in which KV chunks arrive)."""
    return np.random.default_rng(seed).permutation(n)


def ring_order(cp: int, rank: int) -> np.ndarray:
    """Chunk held by ``rank`` at each of the cp steps of a fixed ring: (rank - t) mod cp."""
    return np.array([(rank - t) % cp for t in range(cp)], dtype=np.int64)


def sample_rows(n_rows: int, count: int, seed: int, must=()) -> np.ndarray:
    """Seeded sorted sample of ``count`` distinct rows plus every row listed in ``must``."""
    must = sorted({int(r) for r in must if 0 <= int(r) < n_rows})
    rest = max(0, min(count, n_rows) - len(must))
    pool = np.setdiff1d(np.arange(n_rows), np.asarray(must, dtype=np.int64))
    rng = np.random.default_rng(seed)
    pick = rng.choice(pool, size=min(rest, len(pool)), replace=False) if rest else []
    return np.unique(np.concatenate([np.asarray(must, dtype=np.int64),
                                     np.asarray(pick, dtype=np.int64)]))
