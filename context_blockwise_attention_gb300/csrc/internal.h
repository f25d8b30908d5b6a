// Internal declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cpattn.h"

#define CP_API extern "C" __attribute__((visibility("default")))

namespace cpattn {

// Records a printf-style message for cp_last_error() on the calling thread.
void set_error(const char* fmt, ...);
void clear_error();

// Checks that the current device is an sm_103 part; caches per device.
cp_status require_sm103(int* device_out, int* num_sms_out);

// Maps a CUDA error to CP_ERR_CUDA with a message naming `what`.
cp_status cuda_fail(cudaError_t e, const char* what);

// 2-D tensor map over a token-major tensor viewed as [tokens, row_elems] (bf16 or fp32): box =
// 128 bytes of columns x box_rows rows, 128-byte swizzle, zero fill out of bounds.  False if the
// driver entry point is unavailable or the encoding is rejected.
bool encode_map_2d(CUtensorMap* m, const void* base, int64_t tokens, int64_t row_elems, bool fp32,
                   int box_rows);

// ---- launchers (arguments already validated by the C entry points) ----
cp_status launch_fill_positions(int32_t* out, int64_t n, int64_t base, int64_t stride,
                                cudaStream_t s);

// Partial attention of desc's query shard against chunks[0..n) (n >= 1, chunks with skv > 0
// only), consumed in order with the running state carried across chunks.
cp_status launch_partial_attn_simt(const cp_attn_desc& d, const cp_kv_chunk* chunks, int n, float scale,
                                   cudaStream_t s);
cp_status launch_partial_attn_tc(const cp_attn_desc& d, const cp_kv_chunk* chunks, int n, float scale,
                                 int64_t timeout_ns, int num_sms, cudaStream_t s);
// O = 0, LSE = -inf for every row of desc's query shard (no visible key at all).
cp_status launch_fill_empty(const cp_attn_desc& d, cudaStream_t s);

// Backward pass (arguments validated by the entry points).
cp_status launch_bwd_prep(const void* o, bool o_bf16, const void* d_o, bool do_bf16, const float* lse,
                          int64_t sq, int32_t hq, int32_t d, float* aux, int num_sms, cudaStream_t s);
// One chunk (desc's k, v, dk, dv, skv, kv_pos), fp32 inputs.
cp_status launch_partial_attn_bwd_simt(const cp_attn_bwd_desc& d, float scale, cudaStream_t s);
// chunks[0..n), each with skv > 0; bf16 inputs.
cp_status launch_partial_attn_bwd_tc(const cp_attn_bwd_desc& d, const cp_kv_bwd_chunk* chunks, int n, float scale,
                                     int64_t timeout_ns, int num_sms, cudaStream_t s);

struct MergeArgs {
  int32_t n;
  const float* const* o_parts;
  const float* const* lse_parts;
  int64_t sq;
  int32_t h, d;
  void* o_out;
  int32_t out_bf16;
  float* lse_out;
};
cp_status launch_merge(const MergeArgs& a, int num_sms, cudaStream_t s);

struct ReshardArgs {
  int32_t dir, cp, n_tensors;
  int64_t seq_len;
  const int32_t* heads;
  int32_t d, esize;
  int32_t layout;
  const void* const* in;
  void* const* out;
};
cp_status launch_reshard(const ReshardArgs& a, int num_sms, cudaStream_t s);

}  // namespace cpattn
