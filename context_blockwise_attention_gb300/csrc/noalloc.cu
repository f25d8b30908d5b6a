// Backward of one (query shard, KV chunk) pair for callers that cannot allocate device memory.
//
// The ordinary backward needs a per-row workspace (aux: -LSE*log2(e) and -dO.O for every row and
// head) that the caller allocates and passes in.  Some callers have no way to do that: code that
// runs inside a memory pool it does not own, a runtime that forbids cudaMalloc after start-up, or
// a framework hook that only hands out its inputs and outputs.  This entry point keeps that
// workspace in a fixed array in the library's own device memory instead, so the call itself
// allocates nothing.  It runs the existing prep and backward launches on that array.
//
// The array is a module-scope __device__ variable: every device that loads the library holds
// CP_NOALLOC_AUX_MAX_FLOATS floats (16 MiB) until the process exits.  Host code cannot use the
// array's name as a device address (on the host it names a stand-in object), so the device
// address is looked up with cudaGetSymbolAddress on the first call made with that device
// current, and cached per device together with the identity of the CUDA context it belongs to.
// With CUDA's lazy module loading that first lookup is also where the array is placed in device
// memory, so the first call per device should be made at start-up.  If the context is destroyed
// and recreated (cudaDeviceReset), the array moves: the next call sees a different context and
// looks the address up again (placing the array again).

#include <mutex>

#include "internal.h"

// The shared workspace.  Every call overwrites all of the part it uses (prep writes every row,
// padding rows included, before the backward reads any), so nothing has to start at zero.
static __device__ __align__(256) float g_noalloc_aux[CP_NOALLOC_AUX_MAX_FLOATS];

namespace {

constexpr int kMaxDev = 64;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(ptr);
  return nullptr;
}

// Unique id of the calling thread's current context, or 0 if there is none (or it cannot be
// read, in which case every call looks the address up again).
unsigned long long current_ctx_id() {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

std::mutex g_mu;
float* g_aux_addr[kMaxDev];              // device address of g_noalloc_aux, per device
unsigned long long g_aux_ctx[kMaxDev];  // id of the context that address belongs to (0: none)

}  // namespace

using namespace cpattn;

CP_API cp_status cp_partial_attn_bwd_noalloc(const cp_attn_bwd_desc* desc, const void* o, int32_t o_dtype,
                                             const float* lse, cudaStream_t stream) {
  clear_error();
  if (desc == nullptr) {
    set_error("cp_partial_attn_bwd_noalloc: desc is NULL");
    return CP_ERR_INVALID_ARG;
  }
  if (desc->aux != nullptr) {
    set_error("cp_partial_attn_bwd_noalloc: desc->aux must be NULL (the workspace is the library's own)");
    return CP_ERR_INVALID_ARG;
  }
  if (desc->sq < 0 || desc->hq <= 0) {
    set_error("cp_partial_attn_bwd_noalloc: sq must be >= 0 and hq > 0");
    return CP_ERR_INVALID_ARG;
  }
  const int64_t need = CP_BWD_AUX_FLOATS(desc->sq, desc->hq);
  if (need > CP_NOALLOC_AUX_MAX_FLOATS) {
    set_error(
        "cp_partial_attn_bwd_noalloc: sq=%lld, hq=%d needs a %lld-float workspace, above the fixed "
        "limit of %lld floats (2 * hq * round_up(sq, 128) must not exceed it); use "
        "cp_attn_bwd_prep + cp_partial_attn_bwd with a caller-allocated workspace",
        static_cast<long long>(desc->sq), desc->hq, static_cast<long long>(need),
        static_cast<long long>(CP_NOALLOC_AUX_MAX_FLOATS));
    return CP_ERR_INVALID_ARG;
  }
  int dev = 0;
  cp_status st = require_sm103(&dev, nullptr);
  if (st != CP_OK) return st;
  if (dev >= kMaxDev) {
    set_error("cp_partial_attn_bwd_noalloc: device ordinal %d out of range", dev);
    return CP_ERR_UNSUPPORTED;
  }
  float* aux = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const unsigned long long ctx = current_ctx_id();
    if (g_aux_addr[dev] == nullptr || ctx == 0 || ctx != g_aux_ctx[dev]) {
      // first call on this device (which is current), or its context changed since: the
      // array's device address in the current context
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_aux);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_noalloc_aux)");
      g_aux_addr[dev] = static_cast<float*>(p);
      g_aux_ctx[dev] = current_ctx_id();  // the lookup made the primary context current
    }
    aux = g_aux_addr[dev];
  }
  st = cp_attn_bwd_prep(o, o_dtype, desc->d_o, desc->in_dtype, lse, desc->sq, desc->hq, desc->d, aux, stream);
  if (st != CP_OK) return st;
  cp_attn_bwd_desc d = *desc;
  d.aux = aux;
  return cp_partial_attn_bwd(&d, stream);
}
