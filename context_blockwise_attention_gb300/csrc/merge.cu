// Order-independent merge of (O, LSE) partials into exact softmax attention.
//
// "PCP and DCP sequence parallelism guide", section 2.3 (numerical stability) and section 4.2
// (global_softmax): the global maximum first, then exponentials against it and their global
// sum, then normalisation.  With partials (O_i, LSE_i) of the same query row:
//     M = max_i LSE_i,  w_i = exp(LSE_i - M),  O = sum_i w_i O_i / sum_i w_i,
//     LSE = M + ln(sum_i w_i).
//
// Bandwidth-bound.  One (row, head) item is handled by a group of LANES = d/4 (capped at 32)
// lanes; each lane owns 16-byte vectors of the d-vector.  The group reads the n LSE values
// cooperatively, reduces max and sum with warp shuffles, then streams the O rows of the
// partials whose weight is non-zero (rows with LSE = -inf are never read).
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

template <int D>
struct MergeShape {
  static constexpr int kVecs = D / 4;                      // float4 vectors per row
  static constexpr int kLanes = kVecs < 32 ? kVecs : 32;   // lanes per item
  static constexpr int kVpl = kVecs / kLanes;              // vectors per lane
  static constexpr int kItemsPerWarp = 32 / kLanes;
  static constexpr int kMaxChunks = (CP_MAX_PARTIALS + kLanes - 1) / kLanes;
};

__device__ __forceinline__ float4 ld_stream(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ MergeParams p) {
  using S = MergeShape<D>;
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

    // 1. LSE values and the global maximum
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

    // 3. weighted sum of the O rows with non-zero weight
    float4 acc[S::kVpl];
#pragma unroll
    for (int v = 0; v < S::kVpl; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t row_off = item * D;
#pragma unroll
    for (int c = 0; c < S::kMaxChunks; ++c) {
      if (c >= nchunks) break;
#pragma unroll 4
      for (int t = 0; t < S::kLanes; ++t) {
        const int i = c * S::kLanes + t;
        const float wi = __shfl_sync(0xffffffffu, w[c], group_base + t);
        if (i < p.n && wi > 0.0f && valid) {
          const float* src = p.o[i] + row_off;
#pragma unroll
          for (int v = 0; v < S::kVpl; ++v) {
            const float4 x = ld_stream(src + (v * S::kLanes + sub) * 4);
            acc[v].x = fmaf(wi, x.x, acc[v].x);
            acc[v].y = fmaf(wi, x.y, acc[v].y);
            acc[v].z = fmaf(wi, x.z, acc[v].z);
            acc[v].w = fmaf(wi, x.w, acc[v].w);
          }
        }
      }
    }
    if (!valid) continue;  // no shuffles below
    const float inv = z > 0.0f ? 1.0f / z : 0.0f;
#pragma unroll
    for (int v = 0; v < S::kVpl; ++v) {
      const int64_t e = row_off + static_cast<int64_t>(v * S::kLanes + sub) * 4;
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
  const int64_t items_per_block =
      static_cast<int64_t>(threads / 32) * (32 / (a.d / 4 < 32 ? a.d / 4 : 32));
  int64_t blocks = (p.items + items_per_block - 1) / items_per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  switch (a.d) {
    case 32: merge_kernel<32><<<(unsigned)blocks, threads, 0, s>>>(p); break;
    case 64: merge_kernel<64><<<(unsigned)blocks, threads, 0, s>>>(p); break;
    case 128: merge_kernel<128><<<(unsigned)blocks, threads, 0, s>>>(p); break;
    case 256: merge_kernel<256><<<(unsigned)blocks, threads, 0, s>>>(p); break;
    default: set_error("merge: unsupported d %d", a.d); return CP_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "merge_kernel launch");
}

}  // namespace cpattn
