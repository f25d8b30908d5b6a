// Fill a rank's global token positions: pos(i) = base + stride * i.
// "PCP and DCP sequence parallelism guide", section 3.5 (contiguous split, positions stay
// global); "Zig-Zag Ring Attention" article, section 4.2 (strided assignment).
#include "internal.h"

namespace cpattn {

__global__ void fill_positions_kernel(int32_t* __restrict__ out, int64_t n, int64_t base,
                                      int64_t stride) {
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += step)
    out[i] = static_cast<int32_t>(base + stride * i);
}

cp_status launch_fill_positions(int32_t* out, int64_t n, int64_t base, int64_t stride,
                                cudaStream_t s) {
  if (n == 0) return CP_OK;
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  fill_positions_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(out, n, base, stride);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "fill_positions_kernel launch");
}

}  // namespace cpattn
