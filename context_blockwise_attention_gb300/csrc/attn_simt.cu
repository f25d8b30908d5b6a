// Partial attention for fp32 inputs on CUDA cores (FFMA), fp32 accumulation.
//
// "FCP: from a fixed ring to a free topology", section 3.3: for each block of keys, scores
// q . k^T / sqrt(head_dim), the block's row maximum, a new running maximum, rescaling of the
// accumulator and running sum by exp(old_max - new_max), then accumulation of exp(scores -
// new_max) @ V and its row sum; the output is acc / running_sum.  Here the blocks are 32-key
// tiles of one or more chunks (in arrival order, the running state carried across chunks), and
// the result is emitted as the normalised partial (O, LSE).
//
// A query row is owned by a quad of 4 lanes; lane t of the quad holds 16-byte vectors
// t, t+4, t+8, ... of q and of the accumulator, and the dot product is completed with two
// __shfl_xor_sync steps.  Causal visibility: key j is visible iff kv_pos(j) <= q_pos(i).
#include <math.h>

#include <cuda_bf16.h>

#include "internal.h"

namespace cpattn {

struct SimtParams {
  const float* q;
  void* o;
  float* lse;
  int64_t sq;
  int32_t hq, hkv, group;
  int32_t causal, o_bf16, descending;
  float scale;
  int64_t q_base, q_stride;
  int32_t n_chunks;
  // KV chunks in arrival order: the running (m, l, acc) is carried from one to the next
  const float* k[CP_MAX_CHUNKS];
  const float* v[CP_MAX_CHUNKS];
  int64_t skv[CP_MAX_CHUNKS];
  int64_t k_base[CP_MAX_CHUNKS];
  int64_t k_stride[CP_MAX_CHUNKS];
};

constexpr int kSimtRows = 32;   // query rows per block
constexpr int kSimtKeys = 32;   // keys per tile

template <int D>
__global__ void __launch_bounds__(128) attn_simt_kernel(const __grid_constant__ SimtParams p) {
  constexpr int kV = D / 16;  // float4 vectors per lane (D/4 vectors over 4 lanes)
  __shared__ float4 ks[kSimtKeys][D / 4];
  __shared__ float4 vs[kSimtKeys][D / 4];

  const int tid = threadIdx.x;
  const int quad_lane = tid & 3;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kSimtRows + (tid >> 2);
  const int h = blockIdx.y;
  const int g = h / p.group;
  const bool row_ok = row < p.sq;

  float4 q[kV], acc[kV];
#pragma unroll
  for (int c = 0; c < kV; ++c) {
    acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    q[c] = row_ok ? reinterpret_cast<const float4*>(p.q + (row * p.hq + h) * D)[quad_lane + 4 * c]
                  : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY, l = 0.0f;
  const int64_t qp = p.q_base + p.q_stride * row;

  for (int ch = 0; ch < p.n_chunks; ++ch) {
    const float* __restrict__ kc = p.k[ch];
    const float* __restrict__ vc = p.v[ch];
    const int64_t skv = p.skv[ch];
    // number of keys of this chunk the row may see: keys with kv_pos(j) <= q_pos(row)
    int64_t lim = skv;
    if (p.causal) {
      lim = qp < p.k_base[ch] ? 0 : (qp - p.k_base[ch]) / p.k_stride[ch] + 1;
      if (lim > skv) lim = skv;
    }
    const int64_t ntiles = (skv + kSimtKeys - 1) / kSimtKeys;
    for (int64_t it = 0; it < ntiles; ++it) {
      const int64_t tile = p.descending ? ntiles - 1 - it : it;
      const int64_t k0 = tile * kSimtKeys;
      __syncthreads();
      for (int e = tid; e < kSimtKeys * (D / 4); e += blockDim.x) {
        const int j = e / (D / 4), c = e % (D / 4);
        const int64_t key = k0 + j;
        float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
        if (key < skv) {
          kv = reinterpret_cast<const float4*>(kc + (key * p.hkv + g) * D)[c];
          vv = reinterpret_cast<const float4*>(vc + (key * p.hkv + g) * D)[c];
        }
        ks[j][c] = kv;
        vs[j][c] = vv;
      }
      __syncthreads();

      float s[kSimtKeys];
      float tmax = -INFINITY;
  #pragma unroll
      for (int j = 0; j < kSimtKeys; ++j) {
        float part = 0.0f;
  #pragma unroll
        for (int c = 0; c < kV; ++c) {
          const float4 kk = ks[j][quad_lane + 4 * c];
          part = fmaf(q[c].x, kk.x, part);
          part = fmaf(q[c].y, kk.y, part);
          part = fmaf(q[c].z, kk.z, part);
          part = fmaf(q[c].w, kk.w, part);
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        const bool vis = (k0 + j) < lim;
        s[j] = vis ? part * p.scale : -INFINITY;
        tmax = fmaxf(tmax, s[j]);
      }
      const float m_new = fmaxf(m, tmax);
      if (m_new == -INFINITY) continue;  // nothing visible yet for this row
      const float corr = expf(m - m_new);  // m = -inf -> 0
      l *= corr;
  #pragma unroll
      for (int c = 0; c < kV; ++c) {
        acc[c].x *= corr;
        acc[c].y *= corr;
        acc[c].z *= corr;
        acc[c].w *= corr;
      }
  #pragma unroll
      for (int j = 0; j < kSimtKeys; ++j) {
        const float pj = expf(s[j] - m_new);
        l += pj;
  #pragma unroll
        for (int c = 0; c < kV; ++c) {
          const float4 vv = vs[j][quad_lane + 4 * c];
          acc[c].x = fmaf(pj, vv.x, acc[c].x);
          acc[c].y = fmaf(pj, vv.y, acc[c].y);
          acc[c].z = fmaf(pj, vv.z, acc[c].z);
          acc[c].w = fmaf(pj, vv.w, acc[c].w);
        }
      }
      m = m_new;
    }
  }

  if (!row_ok) return;
  const bool has = (m != -INFINITY) && l > 0.0f;
  const float inv = has ? 1.0f / l : 0.0f;
  const int64_t obase = (row * p.hq + h) * D;
#pragma unroll
  for (int c = 0; c < kV; ++c) {
    const int col = (quad_lane + 4 * c) * 4;
    const float4 r = make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv);
    if (p.o_bf16) {
      __nv_bfloat162 a = __floats2bfloat162_rn(r.x, r.y);
      __nv_bfloat162 b = __floats2bfloat162_rn(r.z, r.w);
      __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.o) + obase + col);
      dst[0] = a;
      dst[1] = b;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(p.o) + obase + col) = r;
    }
  }
  if (quad_lane == 0) p.lse[row * p.hq + h] = has ? m + logf(l) : -INFINITY;
}

cp_status launch_partial_attn_simt(const cp_attn_desc& d, const cp_kv_chunk* chunks, int n, float scale,
                                   cudaStream_t s) {
  SimtParams p;
  p.q = static_cast<const float*>(d.q);
  p.o = d.o;
  p.lse = d.lse;
  p.sq = d.sq;
  p.hq = d.hq;
  p.hkv = d.hkv;
  p.group = d.hq / d.hkv;
  p.causal = d.causal;
  p.o_bf16 = d.o_dtype == CP_BF16;
  p.descending = (d.flags & CP_FLAG_KV_DESCENDING) ? 1 : 0;
  p.scale = scale;
  p.q_base = d.q_pos.base;
  p.q_stride = d.q_pos.stride;
  p.n_chunks = n;
  for (int i = 0; i < CP_MAX_CHUNKS; ++i) {
    const bool live = i < n;
    p.k[i] = live ? static_cast<const float*>(chunks[i].k) : nullptr;
    p.v[i] = live ? static_cast<const float*>(chunks[i].v) : nullptr;
    p.skv[i] = live ? chunks[i].skv : 0;
    p.k_base[i] = live ? chunks[i].kv_pos.base : 0;
    p.k_stride[i] = live ? chunks[i].kv_pos.stride : 1;
  }
  dim3 grid(static_cast<unsigned>((d.sq + kSimtRows - 1) / kSimtRows), static_cast<unsigned>(d.hq));
  if (d.d == 64)
    attn_simt_kernel<64><<<grid, 128, 0, s>>>(p);
  else
    attn_simt_kernel<128><<<grid, 128, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "attn_simt_kernel launch");
}

}  // namespace cpattn
