// Per-row quantities of the backward pass, once per query shard.
//
// The softmax Jacobian needs, for every query row i and head h, D_ih = sum over ALL of the row's
// keys of P_ij dP_ij, which equals dO_ih . O_ih for the row's final output O ("PCP and DCP
// sequence parallelism guide", section 2.3: the gradients are those of the globally normalised
// softmax, whichever rank holds a key).  With the final LSE this is all a per-chunk backward
// needs to know about the other chunks.
//
//   aux[0][h][i] = -LSE_ih * log2(e)     (-inf when LSE_ih = -inf)
//   aux[1][h][i] = -D_ih
//   rows [sq, round_up(sq, 128)): -inf and 0, so 128-row tiles past the end contribute nothing.
//
// Head-major and padded, so a 128-row tile of one head is one contiguous 512-byte run (a single
// bulk copy in the tensor-core backward).  Eight lanes own one (row, head): D/8 elements each,
// 16-byte loads, a 3-step shuffle reduction.  HBM-bound: reads O and dO once.
#include <math.h>

#include <cuda_bf16.h>

#include "internal.h"

namespace cpattn {

namespace {

template <bool BF16>
__device__ __forceinline__ void load8(const void* base, int64_t elem, float (&x)[8]) {
  if (BF16) {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + elem);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
    const float4 a = p[0], b = p[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

template <int D, bool O_BF16, bool DO_BF16>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const void* __restrict__ o, const void* __restrict__ d_o,
                                                       const float* __restrict__ lse, int64_t sq,
                                                       int64_t sq_pad, int32_t hq, float* __restrict__ aux) {
  constexpr int kPer = D / 8;  // elements per lane
  const int sub = threadIdx.x & 7;
  const int64_t items = sq_pad * hq;
  // a warp owns 4 consecutive items per step; the loop condition is the same for all its lanes
  // (the shuffles below need the whole warp)
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t step = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5) * 4;
  for (int64_t first = warp_id * 4; first < items; first += step) {
    const int64_t it = first + ((threadIdx.x & 31) >> 3);
    const bool valid = it < items;
    const int64_t row = valid ? it / hq : sq;
    const int h = valid ? static_cast<int>(it - row * hq) : 0;
    float acc = 0.0f;
    if (row < sq) {
      const int64_t base = (row * hq + h) * D + sub * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 8) {
        float a[8], b[8];
        load8<O_BF16>(o, base + e, a);
        load8<DO_BF16>(d_o, base + e, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = fmaf(a[i], b[i], acc);
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (sub == 0 && valid) {
      float nl = -INFINITY, nd = 0.0f;
      if (row < sq) {
        const float l = lse[row * hq + h];
        nl = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
        nd = -acc;
      }
      aux[static_cast<int64_t>(h) * sq_pad + row] = nl;
      aux[(static_cast<int64_t>(hq) + h) * sq_pad + row] = nd;
    }
  }
}

template <int D>
cp_status launch_prep_d(const void* o, bool o_bf16, const void* d_o, bool do_bf16, const float* lse, int64_t sq,
                        int64_t sq_pad, int32_t hq, float* aux, int num_sms, cudaStream_t s) {
  const int64_t items = sq_pad * hq;
  int64_t blocks = (items + 31) / 32;  // 8 warps x 4 items per block and step
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const unsigned g = static_cast<unsigned>(blocks);
  if (o_bf16 && do_bf16)
    bwd_prep_kernel<D, true, true><<<g, 256, 0, s>>>(o, d_o, lse, sq, sq_pad, hq, aux);
  else if (o_bf16)
    bwd_prep_kernel<D, true, false><<<g, 256, 0, s>>>(o, d_o, lse, sq, sq_pad, hq, aux);
  else if (do_bf16)
    bwd_prep_kernel<D, false, true><<<g, 256, 0, s>>>(o, d_o, lse, sq, sq_pad, hq, aux);
  else
    bwd_prep_kernel<D, false, false><<<g, 256, 0, s>>>(o, d_o, lse, sq, sq_pad, hq, aux);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "bwd_prep_kernel launch");
}

}  // namespace

cp_status launch_bwd_prep(const void* o, bool o_bf16, const void* d_o, bool do_bf16, const float* lse,
                          int64_t sq, int32_t hq, int32_t d, float* aux, int num_sms, cudaStream_t s) {
  const int64_t sq_pad = (sq + 127) / 128 * 128;
  if (sq_pad == 0) return CP_OK;
  if (d == 64) return launch_prep_d<64>(o, o_bf16, d_o, do_bf16, lse, sq, sq_pad, hq, aux, num_sms, s);
  return launch_prep_d<128>(o, o_bf16, d_o, do_bf16, lse, sq, sq_pad, hq, aux, num_sms, s);
}

}  // namespace cpattn
