// Ulysses sequence <-> head reshard as one local, bit-exact permutation per tensor.
//
// "Halo context parallelism (CP + Ulysses attention)", section "Ulysses attention: three
// all-to-alls for one exact computation": each of the cp ranks holds S/cp tokens of all heads;
// after the exchange rank r holds all S tokens of heads [r*H/cp, (r+1)*H/cp).  A token lands
// at row = its global position.
//   seq -> head: Y_r[pos_s(i), j, :] = X_s[i, r*H/cp + j, :]
//   head -> seq: X_s[i, r*H/cp + j, :] = Y_r[pos_s(i), j, :]
//
// Bandwidth-bound: each 16-byte vector is read once and written once.  The walk is linear over
// the sequence-sharded side (X), so one side is fully sequential; on the head-sharded side
// each (token, rank) segment of (H/cp)*d elements is contiguous.  Shard layouts: contiguous,
// strided, or two blocks per rank (blocks r and 2cp-1-r of S/(2cp) tokens).
#include "internal.h"

namespace cpattn {

constexpr int kMaxReshardTensors = 4;
constexpr int kMaxReshardRanks = 64;

struct ReshardParams {
  const uint4* in[kMaxReshardTensors * kMaxReshardRanks];
  uint4* out[kMaxReshardTensors * kMaxReshardRanks];
  int64_t row_vecs[kMaxReshardTensors];  // H_t * d * esize / 16  (one token of X)
  int64_t seg_vecs[kMaxReshardTensors];  // row_vecs / cp         (one rank's head block)
  int64_t local;                         // S / cp
  // Shard s's positions: local token i < seg0 is at s * pos_base_step + pos_stride * i; the
  // rest (two-block layout only) at (2cp - 1 - s) * seg0 + (i - seg0).
  int64_t seg0;                          // contiguous / strided: local;  two-block: local / 2
  int64_t pos_base_step;                 // contiguous: local; strided: 1; two-block: local / 2
  int64_t pos_stride;                    // contiguous: 1;     strided: cp; two-block: 1
  int32_t cp;
  int32_t dir;
};

__global__ void __launch_bounds__(256) reshard_kernel(const __grid_constant__ ReshardParams p) {
  const int ts = blockIdx.y;  // tensor * cp + source shard
  const int t = ts / p.cp;
  const int s = ts % p.cp;
  const int64_t row_vecs = p.row_vecs[t];
  const int64_t seg_vecs = p.seg_vecs[t];
  const int64_t total = p.local * row_vecs;
  const int64_t pos_base = static_cast<int64_t>(s) * p.pos_base_step;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += step) {
    const int64_t i = g / row_vecs;        // local token of shard s
    const int64_t rem = g - i * row_vecs;
    const int64_t r = rem / seg_vecs;      // head-rank
    const int64_t v = rem - r * seg_vecs;  // vector inside the head block
    const int64_t pos = i < p.seg0 ? pos_base + p.pos_stride * i
                                   : (2 * p.cp - 1 - s) * p.seg0 + (i - p.seg0);
    const int64_t y_off = pos * seg_vecs + v;
    if (p.dir == 0) {
      const uint4 x = __ldcs(p.in[ts] + g);
      __stcs(p.out[t * p.cp + r] + y_off, x);
    } else {
      const uint4 x = __ldcs(p.in[t * p.cp + r] + y_off);
      __stcs(p.out[ts] + g, x);
    }
  }
}

cp_status launch_reshard(const ReshardArgs& a, int num_sms, cudaStream_t s) {
  ReshardParams p;
  const int n = a.n_tensors * a.cp;
  for (int k = 0; k < kMaxReshardTensors * kMaxReshardRanks; ++k) {
    p.in[k] = k < n ? static_cast<const uint4*>(a.in[k]) : nullptr;
    p.out[k] = k < n ? static_cast<uint4*>(a.out[k]) : nullptr;
  }
  for (int t = 0; t < kMaxReshardTensors; ++t) {
    if (t < a.n_tensors) {
      p.row_vecs[t] = int64_t(a.heads[t]) * a.d * a.esize / 16;
      p.seg_vecs[t] = p.row_vecs[t] / a.cp;
    } else {
      p.row_vecs[t] = p.seg_vecs[t] = 1;
    }
  }
  p.local = a.seq_len / a.cp;
  p.seg0 = p.local;
  if (a.layout == CP_LAYOUT_CONTIGUOUS) {
    p.pos_base_step = p.local;
    p.pos_stride = 1;
  } else if (a.layout == CP_LAYOUT_STRIDED) {
    p.pos_base_step = 1;
    p.pos_stride = a.cp;
  } else {  // two blocks: r and 2cp - 1 - r
    p.seg0 = p.local / 2;
    p.pos_base_step = p.seg0;
    p.pos_stride = 1;
  }
  p.cp = a.cp;
  p.dir = a.dir;
  const int threads = 256;
  // enough resident threads to cover every SM several times over, split across the
  // (tensor, shard) planes in blockIdx.y
  int64_t per_plane = (static_cast<int64_t>(num_sms) * 8 + n - 1) / n;
  int64_t max_vecs = 0;
  for (int t = 0; t < a.n_tensors; ++t)
    if (p.local * p.row_vecs[t] > max_vecs) max_vecs = p.local * p.row_vecs[t];
  int64_t need = (max_vecs + threads - 1) / threads;
  if (per_plane > need) per_plane = need;
  if (per_plane < 1) per_plane = 1;
  dim3 grid(static_cast<unsigned>(per_plane), static_cast<unsigned>(n));
  reshard_kernel<<<grid, threads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "reshard_kernel launch");
}

}  // namespace cpattn
