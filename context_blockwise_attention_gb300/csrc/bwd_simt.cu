// Backward of one (query shard, KV chunk) partial for fp32 inputs, on CUDA cores (FFMA).
//
// The gradients of the attention definition (chain rule; "PCP and DCP sequence parallelism
// guide", section 2.3 places them: split like the sequence, reduce-scattered across ranks):
//   P_ij = 2^(scale*log2(e) * q_i.k_j + aux0_i)        aux0 = -LSE*log2(e)  (prep kernel)
//   dS_ij = P_ij (dO_i.v_j + aux1_i)                   aux1 = -dO_i.O_i
//   dV_j += sum_i P_ij dO_i,  dK_j += scale sum_i dS_ij q_i,  dQ_i += scale sum_j dS_ij k_j
// Two kernels, each the exclusive owner of what it writes (so the += needs no atomics and the
// summation order is fixed):
//   * dkdv: a block owns 32 keys of one KV head and walks every query row of the group's heads
//     that can see them;
//   * dq:   a block owns 32 query rows of one head and walks every KV tile they can see.
// As in the forward fp32 kernel, a quad of 4 lanes owns one row: lane t holds 16-byte vectors
// t, t+4, ... and dot products finish with two __shfl_xor_sync steps.
#include <math.h>

#include "internal.h"

namespace cpattn {

namespace {

constexpr int kBRows = 32;  // rows (keys or queries) owned by a block
constexpr int kBTile = 32;  // rows of the streamed operand per shared-memory tile

struct BwdSimtParams {
  const float* q;
  const float* k;
  const float* v;
  const float* d_o;
  const float* aux;  // [2][hq][sq_pad]
  float* dq;
  float* dk;
  float* dv;
  int64_t sq, skv, sq_pad;
  int32_t hq, hkv, group, causal;
  float scale, sl2;  // scale, scale * log2(e)
  int64_t q_base, q_stride, k_base, k_stride;
};

template <int D>
__device__ __forceinline__ float quad_dot(const float4 (&a)[D / 16], const float4* b, int ql) {
  float part = 0.0f;
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    const float4 x = b[ql + 4 * c];
    part = fmaf(a[c].x, x.x, part);
    part = fmaf(a[c].y, x.y, part);
    part = fmaf(a[c].z, x.z, part);
    part = fmaf(a[c].w, x.w, part);
  }
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  return part;
}

template <int D>
__global__ void __launch_bounds__(128) bwd_simt_dkdv_kernel(const __grid_constant__ BwdSimtParams p) {
  constexpr int kV = D / 16;
  __shared__ float4 qs[kBTile][D / 4];
  __shared__ float4 dos[kBTile][D / 4];
  __shared__ float nl[kBTile], nd[kBTile];
  const int tid = threadIdx.x;
  const int ql = tid & 3;
  const int64_t key = static_cast<int64_t>(blockIdx.x) * kBRows + (tid >> 2);
  const int g = blockIdx.y;
  const bool key_ok = key < p.skv;
  const int64_t kpos = p.k_base + p.k_stride * key;

  float4 kr[kV], vr[kV], dk[kV], dv[kV];
#pragma unroll
  for (int c = 0; c < kV; ++c) {
    const int64_t off = (key * p.hkv + g) * D;
    kr[c] = key_ok ? reinterpret_cast<const float4*>(p.k + off)[ql + 4 * c] : make_float4(0.f, 0.f, 0.f, 0.f);
    vr[c] = key_ok ? reinterpret_cast<const float4*>(p.v + off)[ql + 4 * c] : make_float4(0.f, 0.f, 0.f, 0.f);
    dk[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    dv[c] = dk[c];
  }
  // first query row that can see the block's first key (positions grow with the index)
  int64_t row0 = 0;
  if (p.causal) {
    const int64_t kp0 = p.k_base + p.k_stride * (static_cast<int64_t>(blockIdx.x) * kBRows);
    if (kp0 > p.q_base) row0 = (kp0 - p.q_base + p.q_stride - 1) / p.q_stride;
  }
  row0 = row0 / kBTile * kBTile;

  for (int hh = 0; hh < p.group; ++hh) {
    const int h = g * p.group + hh;
    const float* nl_h = p.aux + static_cast<int64_t>(h) * p.sq_pad;
    const float* nd_h = p.aux + (static_cast<int64_t>(p.hq) + h) * p.sq_pad;
    for (int64_t r0 = row0; r0 < p.sq; r0 += kBTile) {
      __syncthreads();
      for (int e = tid; e < kBTile * (D / 4); e += blockDim.x) {
        const int i = e / (D / 4), c = e % (D / 4);
        const int64_t row = r0 + i;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (row < p.sq) {
          a = reinterpret_cast<const float4*>(p.q + (row * p.hq + h) * D)[c];
          b = reinterpret_cast<const float4*>(p.d_o + (row * p.hq + h) * D)[c];
        }
        qs[i][c] = a;
        dos[i][c] = b;
      }
      if (tid < kBTile) {
        // padded rows carry -inf / 0 already (prep kernel); r0 + tid < sq_pad always holds
        nl[tid] = nl_h[r0 + tid];
        nd[tid] = nd_h[r0 + tid];
      }
      __syncthreads();
      for (int i = 0; i < kBTile; ++i) {
        const float s = quad_dot<D>(kr, qs[i], ql);
        const float dp = quad_dot<D>(vr, dos[i], ql);
        const int64_t row = r0 + i;
        const bool vis = key_ok && row < p.sq && (!p.causal || kpos <= p.q_base + p.q_stride * row);
        const float pr = vis ? exp2f(fmaf(s, p.sl2, nl[i])) : 0.0f;
        const float ds = pr * (dp + nd[i]);
#pragma unroll
        for (int c = 0; c < kV; ++c) {
          const float4 x = qs[i][ql + 4 * c];
          const float4 y = dos[i][ql + 4 * c];
          dv[c].x = fmaf(pr, y.x, dv[c].x);
          dv[c].y = fmaf(pr, y.y, dv[c].y);
          dv[c].z = fmaf(pr, y.z, dv[c].z);
          dv[c].w = fmaf(pr, y.w, dv[c].w);
          dk[c].x = fmaf(ds, x.x, dk[c].x);
          dk[c].y = fmaf(ds, x.y, dk[c].y);
          dk[c].z = fmaf(ds, x.z, dk[c].z);
          dk[c].w = fmaf(ds, x.w, dk[c].w);
        }
      }
    }
  }
  if (!key_ok) return;
  const int64_t off = (key * p.hkv + g) * D;
#pragma unroll
  for (int c = 0; c < kV; ++c) {
    float4* pk = reinterpret_cast<float4*>(p.dk + off) + ql + 4 * c;
    float4* pv = reinterpret_cast<float4*>(p.dv + off) + ql + 4 * c;
    float4 a = *pk, b = *pv;
    a.x = fmaf(p.scale, dk[c].x, a.x);
    a.y = fmaf(p.scale, dk[c].y, a.y);
    a.z = fmaf(p.scale, dk[c].z, a.z);
    a.w = fmaf(p.scale, dk[c].w, a.w);
    b.x += dv[c].x;
    b.y += dv[c].y;
    b.z += dv[c].z;
    b.w += dv[c].w;
    *pk = a;
    *pv = b;
  }
}

template <int D>
__global__ void __launch_bounds__(128) bwd_simt_dq_kernel(const __grid_constant__ BwdSimtParams p) {
  constexpr int kV = D / 16;
  __shared__ float4 ks[kBTile][D / 4];
  __shared__ float4 vs[kBTile][D / 4];
  const int tid = threadIdx.x;
  const int ql = tid & 3;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kBRows + (tid >> 2);
  const int h = blockIdx.y;
  const int g = h / p.group;
  const bool row_ok = row < p.sq;
  const int64_t qpos = p.q_base + p.q_stride * row;

  float4 qr[kV], dor[kV], dq[kV];
#pragma unroll
  for (int c = 0; c < kV; ++c) {
    const int64_t off = (row * p.hq + h) * D;
    qr[c] = row_ok ? reinterpret_cast<const float4*>(p.q + off)[ql + 4 * c] : make_float4(0.f, 0.f, 0.f, 0.f);
    dor[c] = row_ok ? reinterpret_cast<const float4*>(p.d_o + off)[ql + 4 * c] : make_float4(0.f, 0.f, 0.f, 0.f);
    dq[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float nlr = row_ok ? p.aux[static_cast<int64_t>(h) * p.sq_pad + row] : -INFINITY;
  const float ndr = row_ok ? p.aux[(static_cast<int64_t>(p.hq) + h) * p.sq_pad + row] : 0.0f;
  // keys any row of the block can see: those up to the block's last row
  int64_t nk = p.skv;
  if (p.causal) {
    int64_t last = static_cast<int64_t>(blockIdx.x) * kBRows + kBRows - 1;
    if (last > p.sq - 1) last = p.sq - 1;
    const int64_t lp = p.q_base + p.q_stride * last;
    nk = lp < p.k_base ? 0 : (lp - p.k_base) / p.k_stride + 1;
    if (nk > p.skv) nk = p.skv;
  }
  for (int64_t j0 = 0; j0 < nk; j0 += kBTile) {
    __syncthreads();
    for (int e = tid; e < kBTile * (D / 4); e += blockDim.x) {
      const int j = e / (D / 4), c = e % (D / 4);
      const int64_t key = j0 + j;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      if (key < p.skv) {
        a = reinterpret_cast<const float4*>(p.k + (key * p.hkv + g) * D)[c];
        b = reinterpret_cast<const float4*>(p.v + (key * p.hkv + g) * D)[c];
      }
      ks[j][c] = a;
      vs[j][c] = b;
    }
    __syncthreads();
    for (int j = 0; j < kBTile; ++j) {
      const float s = quad_dot<D>(qr, ks[j], ql);
      const float dp = quad_dot<D>(dor, vs[j], ql);
      const int64_t key = j0 + j;
      const bool vis = row_ok && key < p.skv && (!p.causal || p.k_base + p.k_stride * key <= qpos);
      const float pr = vis ? exp2f(fmaf(s, p.sl2, nlr)) : 0.0f;
      const float ds = pr * (dp + ndr);
#pragma unroll
      for (int c = 0; c < kV; ++c) {
        const float4 x = ks[j][ql + 4 * c];
        dq[c].x = fmaf(ds, x.x, dq[c].x);
        dq[c].y = fmaf(ds, x.y, dq[c].y);
        dq[c].z = fmaf(ds, x.z, dq[c].z);
        dq[c].w = fmaf(ds, x.w, dq[c].w);
      }
    }
  }
  if (!row_ok) return;
  const int64_t off = (row * p.hq + h) * D;
#pragma unroll
  for (int c = 0; c < kV; ++c) {
    float4* pq = reinterpret_cast<float4*>(p.dq + off) + ql + 4 * c;
    float4 a = *pq;
    a.x = fmaf(p.scale, dq[c].x, a.x);
    a.y = fmaf(p.scale, dq[c].y, a.y);
    a.z = fmaf(p.scale, dq[c].z, a.z);
    a.w = fmaf(p.scale, dq[c].w, a.w);
    *pq = a;
  }
}

}  // namespace

cp_status launch_partial_attn_bwd_simt(const cp_attn_bwd_desc& d, float scale, cudaStream_t s) {
  BwdSimtParams p;
  p.q = static_cast<const float*>(d.q);
  p.k = static_cast<const float*>(d.k);
  p.v = static_cast<const float*>(d.v);
  p.d_o = static_cast<const float*>(d.d_o);
  p.aux = d.aux;
  p.dq = d.dq;
  p.dk = d.dk;
  p.dv = d.dv;
  p.sq = d.sq;
  p.skv = d.skv;
  p.sq_pad = (d.sq + 127) / 128 * 128;
  p.hq = d.hq;
  p.hkv = d.hkv;
  p.group = d.hq / d.hkv;
  p.causal = d.causal;
  p.scale = scale;
  p.sl2 = scale * 1.4426950408889634f;
  p.q_base = d.q_pos.base;
  p.q_stride = d.q_pos.stride;
  p.k_base = d.kv_pos.base;
  p.k_stride = d.kv_pos.stride;
  const dim3 g1(static_cast<unsigned>((d.skv + kBRows - 1) / kBRows), static_cast<unsigned>(d.hkv));
  const dim3 g2(static_cast<unsigned>((d.sq + kBRows - 1) / kBRows), static_cast<unsigned>(d.hq));
  if (d.d == 64) {
    bwd_simt_dkdv_kernel<64><<<g1, 128, 0, s>>>(p);
    bwd_simt_dq_kernel<64><<<g2, 128, 0, s>>>(p);
  } else {
    bwd_simt_dkdv_kernel<128><<<g1, 128, 0, s>>>(p);
    bwd_simt_dq_kernel<128><<<g2, 128, 0, s>>>(p);
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "bwd_simt kernels launch");
}

}  // namespace cpattn
