// Order-independent merge of (O, LSE) partials into exact softmax attention.
//
// "PCP and DCP sequence parallelism guide", section 2.3 (numerical stability) and section 4.2
// (global_softmax): the global maximum first, then exponentials against it and their global
// sum, then normalisation.  With partials (O_i, LSE_i) of the same query row:
//     M = max_i LSE_i,  w_i = exp(LSE_i - M),  O = sum_i w_i O_i / sum_i w_i,
//     LSE = M + ln(sum_i w_i).
//
// Bandwidth-bound.  One (row, head) item is handled by a group of 8 lanes; each lane owns d/32
// 16-byte vectors of the d-vector.  The group reads the n LSE values cooperatively, reduces max
// and sum with warp shuffles, then streams the O rows of the partials whose weight is non-zero
// (rows with LSE = -inf are never read), several partials' loads in flight at once.
#include <math.h>

#include <cuda_bf16.h>

#include "internal.h"

namespace cpattn {

struct MergeParams {
  const float* o[CP_MAX_PARTIALS];
  const float* lse[CP_MAX_PARTIALS];
  int32_t n;
  int32_t h;
  int64_t items;  // sq * h
  void* out;
  float* lse_out;
  int32_t out_bf16;
};

// Eight lanes own one (row, head) item for every D: each lane streams D/32 16-byte vectors of a
// partial's O row (interleaved so that the eight lanes cover 128 contiguous bytes per vector
// index), four items per warp.
// MAXC = number of 8-partial chunks the kernel is instantiated for (n <= 8 * MAXC).
template <int D, int MAXC>
struct MergeShape {
  static constexpr int kLanes = 8;
  static constexpr int kVpl = D / 4 / kLanes;  // float4 vectors per lane
  static constexpr int kItemsPerWarp = 32 / kLanes;
  static constexpr int kMaxChunks = MAXC;
  static constexpr int kUnroll = kVpl >= 4 ? 2 : (kVpl == 2 ? 4 : 8);  // partials in flight
};

__device__ __forceinline__ float4 ld_stream(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}

template <int D, int MAXC>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ MergeParams p) {
  using S = MergeShape<D, MAXC>;
  const int lane = threadIdx.x & 31;
  const int sub = lane % S::kLanes;
  const int group_base = lane - sub;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int nchunks = (p.n + S::kLanes - 1) / S::kLanes;

  for (int64_t base = warp_global * S::kItemsPerWarp; base < p.items;
       base += warps * S::kItemsPerWarp) {
    const int64_t item = base + lane / S::kLanes;
    const bool valid = item < p.items;

    // 1. LSE values (lane `sub` holds partials sub, sub+8, ...) and the global maximum
    float lv[S::kMaxChunks];
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < S::kMaxChunks; ++c) {
      const int i = c * S::kLanes + sub;
      lv[c] = -INFINITY;
      if (c < nchunks && i < p.n && valid) lv[c] = __ldcs(p.lse[i] + item);
      m = fmaxf(m, lv[c]);
    }
#pragma unroll
    for (int off = S::kLanes / 2; off > 0; off >>= 1)
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float m_ref = (m == -INFINITY) ? 0.0f : m;

    // 2. weights against the global maximum and their sum
    float w[S::kMaxChunks];
    float z = 0.0f;
#pragma unroll
    for (int c = 0; c < S::kMaxChunks; ++c) {
      w[c] = expf(lv[c] - m_ref);  // exp(-inf) = 0
      z += w[c];
    }
#pragma unroll
    for (int off = S::kLanes / 2; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);

    // 3. weighted sum of the O rows with non-zero weight; kUnroll partials' loads in flight
    float4 acc[S::kVpl];
#pragma unroll
    for (int v = 0; v < S::kVpl; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t row_off = item * D + sub * 4;
#pragma unroll
    for (int c = 0; c < S::kMaxChunks; ++c) {
      if (c >= nchunks) break;
      // partials of this chunk that some item of the warp needs (warp-uniform bit set); the
      // items of a warp are neighbouring heads of one row, so they usually agree
      const unsigned bal = __ballot_sync(0xffffffffu, w[c] > 0.0f);
      unsigned need = (bal | (bal >> 8) | (bal >> 16) | (bal >> 24)) & 0xFFu;
      while (need != 0u) {
        int idx[S::kUnroll];
#pragma unroll
        for (int u = 0; u < S::kUnroll; ++u) {
          idx[u] = need != 0u ? __ffs(need) - 1 : -1;
          need &= need - 1u;
        }
        float wi[S::kUnroll];
        float4 x[S::kUnroll][S::kVpl];
#pragma unroll
        for (int u = 0; u < S::kUnroll; ++u) {
          wi[u] = idx[u] >= 0 ? __shfl_sync(0xffffffffu, w[c], group_base + idx[u]) : 0.0f;
          const bool use = wi[u] > 0.0f && valid;
          const float* src = p.o[c * S::kLanes + (idx[u] >= 0 ? idx[u] : 0)] + row_off;
#pragma unroll
          for (int v = 0; v < S::kVpl; ++v)
            x[u][v] = use ? ld_stream(src + v * (S::kLanes * 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < S::kUnroll; ++u)
#pragma unroll
          for (int v = 0; v < S::kVpl; ++v) {
            acc[v].x = fmaf(wi[u], x[u][v].x, acc[v].x);
            acc[v].y = fmaf(wi[u], x[u][v].y, acc[v].y);
            acc[v].z = fmaf(wi[u], x[u][v].z, acc[v].z);
            acc[v].w = fmaf(wi[u], x[u][v].w, acc[v].w);
          }
      }
    }
    if (!valid) continue;  // no shuffles below
    const float inv = z > 0.0f ? 1.0f / z : 0.0f;
#pragma unroll
    for (int v = 0; v < S::kVpl; ++v) {
      const int64_t e = row_off + v * (S::kLanes * 4);
      const float4 r = make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv);
      if (p.out_bf16) {
        __nv_bfloat162 a = __floats2bfloat162_rn(r.x, r.y);
        __nv_bfloat162 b = __floats2bfloat162_rn(r.z, r.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&a);
        pk.y = *reinterpret_cast<uint32_t*>(&b);
        __stcs(reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + e), pk);
      } else {
        __stcs(reinterpret_cast<float4*>(static_cast<float*>(p.out) + e), r);
      }
    }
    if (p.lse_out != nullptr && sub == 0)
      p.lse_out[item] = (z > 0.0f) ? m_ref + logf(z) : -INFINITY;
  }
}

cp_status launch_merge(const MergeArgs& a, int num_sms, cudaStream_t s) {
  MergeParams p;
  for (int i = 0; i < a.n; ++i) {
    p.o[i] = a.o_parts[i];
    p.lse[i] = a.lse_parts[i];
  }
  for (int i = a.n; i < CP_MAX_PARTIALS; ++i) {
    p.o[i] = nullptr;
    p.lse[i] = nullptr;
  }
  p.n = a.n;
  p.h = a.h;
  p.items = a.sq * a.h;
  p.out = a.o_out;
  p.lse_out = a.lse_out;
  p.out_bf16 = a.out_bf16;
  const int threads = 256;
  // 8 resident blocks of 256 threads per SM; grid-stride over items
  const int64_t items_per_block = static_cast<int64_t>(threads / 32) * 4;
  int64_t blocks = (p.items + items_per_block - 1) / items_per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const int maxc = a.n <= 8 ? 1 : a.n <= 16 ? 2 : a.n <= 32 ? 4 : a.n <= 64 ? 8 : 16;
  const unsigned nb = static_cast<unsigned>(blocks);
#define CP_MERGE_CASE(DD)                                              \
  case DD:                                                             \
    switch (maxc) {                                                    \
      case 1: merge_kernel<DD, 1><<<nb, threads, 0, s>>>(p); break;   \
      case 2: merge_kernel<DD, 2><<<nb, threads, 0, s>>>(p); break;   \
      case 4: merge_kernel<DD, 4><<<nb, threads, 0, s>>>(p); break;   \
      case 8: merge_kernel<DD, 8><<<nb, threads, 0, s>>>(p); break;   \
      default: merge_kernel<DD, 16><<<nb, threads, 0, s>>>(p); break; \
    }                                                                  \
    break;
  switch (a.d) {
    CP_MERGE_CASE(32)
    CP_MERGE_CASE(64)
    CP_MERGE_CASE(128)
    CP_MERGE_CASE(256)
    default: set_error("merge: unsupported d %d", a.d); return CP_ERR_INVALID_ARG;
  }
#undef CP_MERGE_CASE
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "merge_kernel launch");
}

}  // namespace cpattn
