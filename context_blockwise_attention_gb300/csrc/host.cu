// C entry points of libcpattn.so: argument validation (host only, before any launch), device
// check, dispatch to the kernels' launchers, and the per-thread error message.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "internal.h"

namespace cpattn {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}
void clear_error() { g_err[0] = '\0'; }

cp_status cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
  return CP_ERR_CUDA;
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int g_dev_state[kMaxDevices];  // 0 unknown, 1 ok, 2 unsupported
int g_dev_sms[kMaxDevices];
int g_dev_cc[kMaxDevices];
}  // namespace

cp_status require_sm103(int* device_out, int* num_sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal %d out of range", dev);
    return CP_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_state[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(major)");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    g_dev_cc[dev] = major * 10 + minor;
    g_dev_sms[dev] = sms;
    g_dev_state[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  if (g_dev_state[dev] != 1) {
    set_error("device %d has compute capability %d.%d; this library is built for sm_103a (GB300)",
              dev, g_dev_cc[dev] / 10, g_dev_cc[dev] % 10);
    return CP_ERR_UNSUPPORTED;
  }
  if (device_out) *device_out = dev;
  if (num_sms_out) *num_sms_out = g_dev_sms[dev];
  return CP_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int64_t dtype_size(int32_t t) { return t == CP_F32 ? 4 : (t == CP_BF16 ? 2 : 0); }

}  // namespace cpattn

using namespace cpattn;

#define CP_INVALID(...)          \
  do {                           \
    cpattn::set_error(__VA_ARGS__); \
    return CP_ERR_INVALID_ARG;   \
  } while (0)

CP_API int32_t cp_version(void) { return CP_ABI_VERSION; }

CP_API const char* cp_last_error(void) { return cpattn::g_err; }

// Work-balanced split: the smallest b with b (b + 1) cp >= r S (S + 1), i.e. the first b whose
// causal pair count W(b) = b (b + 1) / 2 reaches r / cp of the whole sequence's (b_0 = 0,
// b_cp = S).  128-bit integers: r S (S + 1) exceeds 64 bits for long sequences.
static int64_t balanced_bound(int64_t seq_len, int32_t cp, int32_t r) {
  if (r <= 0) return 0;
  if (r >= cp) return seq_len;
  typedef unsigned __int128 u128;
  const u128 need = static_cast<u128>(r) * static_cast<u128>(seq_len) * static_cast<u128>(seq_len + 1);
  // start from the floating-point root, then step to the exact smallest b
  int64_t b = static_cast<int64_t>(sqrtl(static_cast<long double>(need) / cp));
  auto reach = [&](int64_t x) { return static_cast<u128>(x) * static_cast<u128>(x + 1) * static_cast<u128>(cp) >= need; };
  while (b > 0 && reach(b - 1)) --b;
  while (!reach(b)) ++b;
  return b;
}

// The affine segments of rank `rank`'s shard under layout `kind`, in local order.
static cp_status shard_segments(const char* who, int64_t seq_len, int32_t cp, int32_t rank,
                                int32_t kind, cp_posmap* maps, int64_t* lens, int32_t* n) {
  if (seq_len <= 0) CP_INVALID("%s: seq_len must be positive (got %lld)", who, (long long)seq_len);
  if (cp <= 0) CP_INVALID("%s: cp must be positive (got %d)", who, cp);
  if (rank < 0 || rank >= cp) CP_INVALID("%s: rank %d not in [0, %d)", who, rank, cp);
  if (kind == CP_LAYOUT_BALANCED) {
    if (seq_len > (int64_t(1) << 40)) CP_INVALID("%s: seq_len too large for the balanced split", who);
    const int64_t lo = balanced_bound(seq_len, cp, rank);
    const int64_t hi = balanced_bound(seq_len, cp, rank + 1);
    // every rank must hold tokens: the bounds must increase strictly
    for (int32_t r = 0; r < cp; ++r)
      if (balanced_bound(seq_len, cp, r) >= balanced_bound(seq_len, cp, r + 1))
        CP_INVALID("%s: the balanced split of %lld tokens leaves rank %d of %d without tokens", who,
                   (long long)seq_len, r, cp);
    maps[0] = cp_posmap{lo, 1};
    lens[0] = hi - lo;
    *n = 1;
    return CP_OK;
  }
  if (seq_len % cp != 0)
    CP_INVALID("%s: seq_len %lld is not a multiple of cp %d", who, (long long)seq_len, cp);
  const int64_t local = seq_len / cp;
  if (kind == CP_LAYOUT_CONTIGUOUS) {
    maps[0] = cp_posmap{static_cast<int64_t>(rank) * local, 1};
    lens[0] = local;
    *n = 1;
  } else if (kind == CP_LAYOUT_STRIDED) {
    maps[0] = cp_posmap{rank, cp};
    lens[0] = local;
    *n = 1;
  } else if (kind == CP_LAYOUT_TWO_BLOCK) {
    if (seq_len % (2 * static_cast<int64_t>(cp)) != 0)
      CP_INVALID("%s: the two-block split needs seq_len %lld to be a multiple of 2*cp = %d", who,
                 (long long)seq_len, 2 * cp);
    const int64_t b = local / 2;
    maps[0] = cp_posmap{static_cast<int64_t>(rank) * b, 1};
    maps[1] = cp_posmap{static_cast<int64_t>(2 * cp - 1 - rank) * b, 1};
    lens[0] = lens[1] = b;
    *n = 2;
  } else {
    CP_INVALID("%s: unknown layout kind %d", who, kind);
  }
  return CP_OK;
}

static cp_status fill_segments(const char* who, int64_t seq_len, const cp_posmap* maps,
                               const int64_t* lens, int32_t n, int32_t* dev_positions_out,
                               cudaStream_t stream) {
  if (dev_positions_out == nullptr) return CP_OK;
  if (seq_len > INT32_MAX) CP_INVALID("%s: int32 positions need seq_len <= INT32_MAX", who);
  cp_status st = require_sm103(nullptr, nullptr);
  if (st != CP_OK) return st;
  int64_t off = 0;
  for (int32_t i = 0; i < n; ++i) {
    st = launch_fill_positions(dev_positions_out + off, lens[i], maps[i].base, maps[i].stride, stream);
    if (st != CP_OK) return st;
    off += lens[i];
  }
  return CP_OK;
}

CP_API cp_status cp_shard_layout(int64_t seq_len, int32_t cp, int32_t rank, int32_t kind,
                                 cp_posmap* map_out, int32_t* dev_positions_out,
                                 cudaStream_t stream) {
  clear_error();
  if (map_out == nullptr) CP_INVALID("cp_shard_layout: map_out is NULL");
  cp_posmap maps[CP_MAX_SEGMENTS];
  int64_t lens[CP_MAX_SEGMENTS];
  int32_t n = 0;
  cp_status st = shard_segments("cp_shard_layout", seq_len, cp, rank, kind, maps, lens, &n);
  if (st != CP_OK) return st;
  if (n != 1 || lens[0] * cp != seq_len)
    CP_INVALID("cp_shard_layout: layout %d is not one map of seq_len/cp tokens; use cp_shard_segments", kind);
  st = fill_segments("cp_shard_layout", seq_len, maps, lens, n, dev_positions_out, stream);
  if (st != CP_OK) return st;
  *map_out = maps[0];
  return CP_OK;
}

CP_API cp_status cp_shard_segments(int64_t seq_len, int32_t cp, int32_t rank, int32_t kind,
                                   cp_posmap* maps_out, int64_t* lens_out, int32_t* n_segments_out,
                                   int32_t* dev_positions_out, cudaStream_t stream) {
  clear_error();
  if (maps_out == nullptr || lens_out == nullptr || n_segments_out == nullptr)
    CP_INVALID("cp_shard_segments: maps_out, lens_out and n_segments_out must not be NULL");
  cp_posmap maps[CP_MAX_SEGMENTS];
  int64_t lens[CP_MAX_SEGMENTS];
  int32_t n = 0;
  cp_status st = shard_segments("cp_shard_segments", seq_len, cp, rank, kind, maps, lens, &n);
  if (st != CP_OK) return st;
  st = fill_segments("cp_shard_segments", seq_len, maps, lens, n, dev_positions_out, stream);
  if (st != CP_OK) return st;
  for (int32_t i = 0; i < n; ++i) {
    maps_out[i] = maps[i];
    lens_out[i] = lens[i];
  }
  *n_segments_out = n;
  return CP_OK;
}

// Checks every descriptor field except k, v, skv and kv_pos.
static cp_status validate_desc(const cp_attn_desc& d) {
  if (d.in_dtype != CP_F32 && d.in_dtype != CP_BF16)
    CP_INVALID("partial attention: in_dtype %d is not CP_F32 or CP_BF16", d.in_dtype);
  if (d.o_dtype != CP_F32 && d.o_dtype != CP_BF16)
    CP_INVALID("partial attention: o_dtype %d is not CP_F32 or CP_BF16", d.o_dtype);
  if (d.sq < 0) CP_INVALID("partial attention: negative query count");
  if (d.sq > (int64_t(1) << 31) - 256) CP_INVALID("partial attention: token counts must stay below 2^31");
  if (d.hq <= 0 || d.hkv <= 0) CP_INVALID("partial attention: head counts must be positive");
  if (d.hq % d.hkv != 0) CP_INVALID("partial attention: hq %d is not a multiple of hkv %d", d.hq, d.hkv);
  if (d.d != 64 && d.d != 128) CP_INVALID("partial attention: head_dim %d not in {64, 128}", d.d);
  if (d.causal != 0 && d.causal != 1) CP_INVALID("partial attention: causal must be 0 or 1");
  if (d.q_pos.stride < 1) CP_INVALID("partial attention: position strides must be >= 1");
  if (d.q_pos.base < 0) CP_INVALID("partial attention: positions must be >= 0");
  if (double(d.q_pos.base) + double(d.q_pos.stride) * double(d.sq) > 2.0e9)
    CP_INVALID("partial attention: global positions exceed 2e9");
  if (!(d.scale >= 0.0f) || isinf(d.scale)) CP_INVALID("partial attention: scale must be finite and >= 0");
  if (d.flags & ~(CP_FLAG_KV_DESCENDING | CP_FLAG_TEST_STALL))
    CP_INVALID("partial attention: unknown flag bits 0x%x", d.flags);
  if (d.wait_timeout_ms < 0) CP_INVALID("partial attention: wait_timeout_ms must be >= 0");
  if (d.sq > 0) {
    if (d.q == nullptr || d.o == nullptr || d.lse == nullptr)
      CP_INVALID("partial attention: q, o and lse must not be NULL");
    if (!aligned16(d.q) || !aligned16(d.o) || (reinterpret_cast<uintptr_t>(d.lse) & 3u))
      CP_INVALID("partial attention: q and o must be 16-byte aligned, lse 4-byte aligned");
    if (d.in_dtype == CP_BF16 && (int64_t(d.hq) * d.d * 2) % 16 != 0)
      CP_INVALID("partial attention: row strides must be multiples of 16 bytes");
  }
  return CP_OK;
}

static cp_status validate_chunk(const cp_attn_desc& d, const cp_kv_chunk& c, int idx) {
  if (c.skv < 0) CP_INVALID("partial attention: chunk %d has a negative token count", idx);
  if (c.skv > (int64_t(1) << 31) - 256) CP_INVALID("partial attention: chunk %d token count must stay below 2^31", idx);
  if (c.kv_pos.stride < 1) CP_INVALID("partial attention: chunk %d position stride must be >= 1", idx);
  if (c.kv_pos.base < 0) CP_INVALID("partial attention: chunk %d positions must be >= 0", idx);
  if (double(c.kv_pos.base) + double(c.kv_pos.stride) * double(c.skv) > 2.0e9)
    CP_INVALID("partial attention: chunk %d global positions exceed 2e9", idx);
  if (c.skv > 0 && d.sq > 0) {
    if (c.k == nullptr || c.v == nullptr) CP_INVALID("partial attention: chunk %d k and v must not be NULL", idx);
    if (!aligned16(c.k) || !aligned16(c.v)) CP_INVALID("partial attention: chunk %d k and v must be 16-byte aligned", idx);
    if (d.in_dtype == CP_BF16 && (int64_t(d.hkv) * d.d * 2) % 16 != 0)
      CP_INVALID("partial attention: row strides must be multiples of 16 bytes");
  }
  return CP_OK;
}

// Launches the partial over the chunks that hold keys (chunks without keys contribute nothing).
static cp_status run_partial(const cp_attn_desc& d, const cp_kv_chunk* chunks, int n, cudaStream_t stream) {
  if (d.sq == 0) return CP_OK;
  int dev = 0, sms = 0;
  cp_status st = require_sm103(&dev, &sms);
  if (st != CP_OK) return st;
  cp_kv_chunk live[CP_MAX_CHUNKS];
  int m = 0;
  for (int i = 0; i < n; ++i)
    if (chunks[i].skv > 0) live[m++] = chunks[i];
  if (m == 0) return launch_fill_empty(d, stream);
  const float scale = d.scale > 0.0f ? d.scale : 1.0f / sqrtf(static_cast<float>(d.d));
  const int64_t timeout_ns =
      static_cast<int64_t>(d.wait_timeout_ms > 0 ? d.wait_timeout_ms : 2000) * 1000000LL;
  if (d.in_dtype == CP_F32) return launch_partial_attn_simt(d, live, m, scale, stream);
  return launch_partial_attn_tc(d, live, m, scale, timeout_ns, sms, stream);
}

CP_API cp_status cp_partial_attn(const cp_attn_desc* desc, cudaStream_t stream) {
  clear_error();
  if (desc == nullptr) CP_INVALID("cp_partial_attn: desc is NULL");
  cp_status st = validate_desc(*desc);
  if (st != CP_OK) return st;
  cp_kv_chunk c;
  c.k = desc->k;
  c.v = desc->v;
  c.skv = desc->skv;
  c.kv_pos = desc->kv_pos;
  if ((st = validate_chunk(*desc, c, 0)) != CP_OK) return st;
  return run_partial(*desc, &c, 1, stream);
}

CP_API cp_status cp_partial_attn_chunks(const cp_attn_desc* desc, int32_t n_chunks, const cp_kv_chunk* chunks,
                                        cudaStream_t stream) {
  clear_error();
  if (desc == nullptr) CP_INVALID("cp_partial_attn_chunks: desc is NULL");
  if (n_chunks < 1 || n_chunks > CP_MAX_CHUNKS)
    CP_INVALID("cp_partial_attn_chunks: n_chunks=%d not in [1, %d]", n_chunks, CP_MAX_CHUNKS);
  if (chunks == nullptr) CP_INVALID("cp_partial_attn_chunks: chunks is NULL");
  cp_status st = validate_desc(*desc);
  if (st != CP_OK) return st;
  for (int i = 0; i < n_chunks; ++i)
    if ((st = validate_chunk(*desc, chunks[i], i)) != CP_OK) return st;
  return run_partial(*desc, chunks, n_chunks, stream);
}

CP_API cp_status cp_attn_bwd_prep(const void* o, int32_t o_dtype, const void* d_o, int32_t do_dtype,
                                  const float* lse, int64_t sq, int32_t hq, int32_t d, float* aux,
                                  cudaStream_t stream) {
  clear_error();
  if (o_dtype != CP_F32 && o_dtype != CP_BF16) CP_INVALID("cp_attn_bwd_prep: bad o_dtype %d", o_dtype);
  if (do_dtype != CP_F32 && do_dtype != CP_BF16) CP_INVALID("cp_attn_bwd_prep: bad do_dtype %d", do_dtype);
  if (sq < 0 || sq > (int64_t(1) << 31) - 256) CP_INVALID("cp_attn_bwd_prep: sq out of range");
  if (hq <= 0) CP_INVALID("cp_attn_bwd_prep: hq must be positive");
  if (d != 64 && d != 128) CP_INVALID("cp_attn_bwd_prep: head_dim %d not in {64, 128}", d);
  if (sq == 0) return CP_OK;
  if (o == nullptr || d_o == nullptr || lse == nullptr || aux == nullptr)
    CP_INVALID("cp_attn_bwd_prep: o, d_o, lse and aux must not be NULL");
  if (!aligned16(o) || !aligned16(d_o) || !aligned16(aux) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    CP_INVALID("cp_attn_bwd_prep: o, d_o and aux must be 16-byte aligned, lse 4-byte aligned");
  int sms = 0;
  cp_status st = require_sm103(nullptr, &sms);
  if (st != CP_OK) return st;
  return launch_bwd_prep(o, o_dtype == CP_BF16, d_o, do_dtype == CP_BF16, lse, sq, hq, d, aux, sms, stream);
}

// Checks every backward descriptor field except k, v, dk, dv, skv and kv_pos.
static cp_status validate_bwd_desc(const cp_attn_bwd_desc& d) {
  if (d.in_dtype != CP_F32 && d.in_dtype != CP_BF16)
    CP_INVALID("partial attention backward: in_dtype %d is not CP_F32 or CP_BF16", d.in_dtype);
  if (d.sq < 0) CP_INVALID("partial attention backward: negative token count");
  if (d.sq > (int64_t(1) << 31) - 256) CP_INVALID("partial attention backward: token counts must stay below 2^31");
  if (d.hq <= 0 || d.hkv <= 0) CP_INVALID("partial attention backward: head counts must be positive");
  if (d.hq % d.hkv != 0) CP_INVALID("partial attention backward: hq %d is not a multiple of hkv %d", d.hq, d.hkv);
  if (d.d != 64 && d.d != 128) CP_INVALID("partial attention backward: head_dim %d not in {64, 128}", d.d);
  if (d.causal != 0 && d.causal != 1) CP_INVALID("partial attention backward: causal must be 0 or 1");
  if (d.q_pos.stride < 1) CP_INVALID("partial attention backward: position strides must be >= 1");
  if (d.q_pos.base < 0) CP_INVALID("partial attention backward: positions must be >= 0");
  if (double(d.q_pos.base) + double(d.q_pos.stride) * double(d.sq) > 2.0e9)
    CP_INVALID("partial attention backward: global positions exceed 2e9");
  if (!(d.scale >= 0.0f) || isinf(d.scale)) CP_INVALID("partial attention backward: scale must be finite and >= 0");
  if (d.flags & ~CP_FLAG_TEST_STALL) CP_INVALID("partial attention backward: unknown flag bits 0x%x", d.flags);
  if ((d.flags & CP_FLAG_TEST_STALL) && d.in_dtype != CP_BF16)
    CP_INVALID("partial attention backward: CP_FLAG_TEST_STALL applies to the bf16 (tensor-core) path only");
  if (d.wait_timeout_ms < 0) CP_INVALID("partial attention backward: wait_timeout_ms must be >= 0");
  if (d.sq > 0) {
    if (d.q == nullptr || d.d_o == nullptr || d.aux == nullptr || d.dq == nullptr)
      CP_INVALID("partial attention backward: q, d_o, aux and dq must not be NULL");
    if (!aligned16(d.q) || !aligned16(d.d_o) || !aligned16(d.aux) || !aligned16(d.dq))
      CP_INVALID("partial attention backward: every buffer must be 16-byte aligned");
  }
  return CP_OK;
}

static cp_status validate_bwd_chunk(const cp_attn_bwd_desc& d, const cp_kv_bwd_chunk& c, int idx) {
  if (c.skv < 0) CP_INVALID("partial attention backward: chunk %d has a negative token count", idx);
  if (c.skv > (int64_t(1) << 31) - 256) CP_INVALID("partial attention backward: chunk %d token count must stay below 2^31", idx);
  if (c.kv_pos.stride < 1) CP_INVALID("partial attention backward: chunk %d position stride must be >= 1", idx);
  if (c.kv_pos.base < 0) CP_INVALID("partial attention backward: chunk %d positions must be >= 0", idx);
  if (double(c.kv_pos.base) + double(c.kv_pos.stride) * double(c.skv) > 2.0e9)
    CP_INVALID("partial attention backward: chunk %d global positions exceed 2e9", idx);
  if (c.skv > 0 && d.sq > 0) {
    if (c.k == nullptr || c.v == nullptr || c.dk == nullptr || c.dv == nullptr)
      CP_INVALID("partial attention backward: chunk %d k, v, dk and dv must not be NULL", idx);
    if (!aligned16(c.k) || !aligned16(c.v) || !aligned16(c.dk) || !aligned16(c.dv))
      CP_INVALID("partial attention backward: chunk %d buffers must be 16-byte aligned", idx);
  }
  return CP_OK;
}

static cp_status run_partial_bwd(const cp_attn_bwd_desc& d, const cp_kv_bwd_chunk* chunks, int n,
                                 cudaStream_t stream) {
  if (d.sq == 0) return CP_OK;  // nothing to add
  cp_kv_bwd_chunk live[CP_MAX_CHUNKS];
  int m = 0;
  for (int i = 0; i < n; ++i)
    if (chunks[i].skv > 0) live[m++] = chunks[i];
  if (m == 0) return CP_OK;
  int dev = 0, sms = 0;
  cp_status st = require_sm103(&dev, &sms);
  if (st != CP_OK) return st;
  const float scale = d.scale > 0.0f ? d.scale : 1.0f / sqrtf(static_cast<float>(d.d));
  const int64_t timeout_ns =
      static_cast<int64_t>(d.wait_timeout_ms > 0 ? d.wait_timeout_ms : 2000) * 1000000LL;
  if (d.in_dtype == CP_BF16) return launch_partial_attn_bwd_tc(d, live, m, scale, timeout_ns, sms, stream);
  for (int i = 0; i < m; ++i) {  // fp32: one exclusive-owner pass per chunk
    cp_attn_bwd_desc one = d;
    one.k = live[i].k;
    one.v = live[i].v;
    one.dk = live[i].dk;
    one.dv = live[i].dv;
    one.skv = live[i].skv;
    one.kv_pos = live[i].kv_pos;
    if ((st = launch_partial_attn_bwd_simt(one, scale, stream)) != CP_OK) return st;
  }
  return CP_OK;
}

CP_API cp_status cp_partial_attn_bwd(const cp_attn_bwd_desc* desc, cudaStream_t stream) {
  clear_error();
  if (desc == nullptr) CP_INVALID("cp_partial_attn_bwd: desc is NULL");
  cp_status st = validate_bwd_desc(*desc);
  if (st != CP_OK) return st;
  cp_kv_bwd_chunk c;
  c.k = desc->k;
  c.v = desc->v;
  c.dk = desc->dk;
  c.dv = desc->dv;
  c.skv = desc->skv;
  c.kv_pos = desc->kv_pos;
  if ((st = validate_bwd_chunk(*desc, c, 0)) != CP_OK) return st;
  return run_partial_bwd(*desc, &c, 1, stream);
}

CP_API cp_status cp_partial_attn_bwd_chunks(const cp_attn_bwd_desc* desc, int32_t n_chunks,
                                            const cp_kv_bwd_chunk* chunks, cudaStream_t stream) {
  clear_error();
  if (desc == nullptr) CP_INVALID("cp_partial_attn_bwd_chunks: desc is NULL");
  if (n_chunks < 1 || n_chunks > CP_MAX_CHUNKS)
    CP_INVALID("cp_partial_attn_bwd_chunks: n_chunks=%d not in [1, %d]", n_chunks, CP_MAX_CHUNKS);
  if (chunks == nullptr) CP_INVALID("cp_partial_attn_bwd_chunks: chunks is NULL");
  cp_status st = validate_bwd_desc(*desc);
  if (st != CP_OK) return st;
  for (int i = 0; i < n_chunks; ++i)
    if ((st = validate_bwd_chunk(*desc, chunks[i], i)) != CP_OK) return st;
  return run_partial_bwd(*desc, chunks, n_chunks, stream);
}

CP_API cp_status cp_merge_partials(int32_t n, const float* const* o_parts,
                                   const float* const* lse_parts, int64_t sq, int32_t h, int32_t d,
                                   void* o_out, int32_t out_dtype, float* lse_out,
                                   cudaStream_t stream) {
  clear_error();
  if (n < 1 || n > CP_MAX_PARTIALS) CP_INVALID("cp_merge_partials: n=%d not in [1, %d]", n, CP_MAX_PARTIALS);
  if (o_parts == nullptr || lse_parts == nullptr) CP_INVALID("cp_merge_partials: pointer arrays are NULL");
  if (sq < 0) CP_INVALID("cp_merge_partials: negative row count");
  if (h <= 0) CP_INVALID("cp_merge_partials: h must be positive");
  if (d != 32 && d != 64 && d != 128 && d != 256) CP_INVALID("cp_merge_partials: d=%d not in {32, 64, 128, 256}", d);
  if (out_dtype != CP_F32 && out_dtype != CP_BF16) CP_INVALID("cp_merge_partials: bad out_dtype %d", out_dtype);
  if (sq == 0) return CP_OK;
  if (o_out == nullptr || !aligned16(o_out)) CP_INVALID("cp_merge_partials: o_out NULL or not 16-byte aligned");
  if (lse_out != nullptr && (reinterpret_cast<uintptr_t>(lse_out) & 3u)) CP_INVALID("cp_merge_partials: lse_out misaligned");
  for (int i = 0; i < n; ++i) {
    if (o_parts[i] == nullptr || lse_parts[i] == nullptr) CP_INVALID("cp_merge_partials: partial %d is NULL", i);
    if (!aligned16(o_parts[i])) CP_INVALID("cp_merge_partials: partial %d O not 16-byte aligned", i);
    if (reinterpret_cast<uintptr_t>(lse_parts[i]) & 3u) CP_INVALID("cp_merge_partials: partial %d LSE misaligned", i);
  }
  int sms = 0;
  cp_status st = require_sm103(nullptr, &sms);
  if (st != CP_OK) return st;
  MergeArgs a{n, o_parts, lse_parts, sq, h, d, o_out, out_dtype == CP_BF16 ? 1 : 0, lse_out};
  return launch_merge(a, sms, stream);
}

CP_API cp_status cp_ulysses_reshard(int32_t dir, int32_t cp, int64_t seq_len, int32_t n_tensors,
                                    const int32_t* heads, int32_t d, int32_t dtype, int32_t layout,
                                    const void* const* in, void* const* out, cudaStream_t stream) {
  clear_error();
  if (dir != 0 && dir != 1) CP_INVALID("cp_ulysses_reshard: dir must be 0 (seq->head) or 1 (head->seq)");
  if (cp < 1) CP_INVALID("cp_ulysses_reshard: cp must be >= 1");
  if (seq_len <= 0 || seq_len % cp != 0) CP_INVALID("cp_ulysses_reshard: seq_len %lld not a positive multiple of cp %d", (long long)seq_len, cp);
  if (n_tensors < 1 || n_tensors > 4) CP_INVALID("cp_ulysses_reshard: n_tensors must be in [1, 4]");
  if (heads == nullptr || in == nullptr || out == nullptr) CP_INVALID("cp_ulysses_reshard: NULL array argument");
  if (d <= 0) CP_INVALID("cp_ulysses_reshard: d must be positive");
  const int64_t es = dtype_size(dtype);
  if (es == 0) CP_INVALID("cp_ulysses_reshard: bad dtype %d", dtype);
  if (layout != CP_LAYOUT_CONTIGUOUS && layout != CP_LAYOUT_STRIDED && layout != CP_LAYOUT_TWO_BLOCK)
    CP_INVALID("cp_ulysses_reshard: bad layout %d", layout);
  if (layout == CP_LAYOUT_TWO_BLOCK && seq_len % (2 * static_cast<int64_t>(cp)) != 0)
    CP_INVALID("cp_ulysses_reshard: the two-block split needs seq_len to be a multiple of 2*cp");
  if (cp > 64) CP_INVALID("cp_ulysses_reshard: cp must be <= 64");
  for (int t = 0; t < n_tensors; ++t) {
    if (heads[t] <= 0 || heads[t] % cp != 0) CP_INVALID("cp_ulysses_reshard: heads[%d]=%d not a positive multiple of cp %d", t, heads[t], cp);
    if ((int64_t(heads[t] / cp) * d * es) % 16 != 0) CP_INVALID("cp_ulysses_reshard: per-rank head block of tensor %d is not a multiple of 16 bytes", t);
    for (int r = 0; r < cp; ++r) {
      const void* pi = in[t * cp + r];
      const void* po = out[t * cp + r];
      if (pi == nullptr || po == nullptr) CP_INVALID("cp_ulysses_reshard: NULL buffer (tensor %d, rank %d)", t, r);
      if (!aligned16(pi) || !aligned16(po)) CP_INVALID("cp_ulysses_reshard: buffer not 16-byte aligned (tensor %d, rank %d)", t, r);
    }
  }
  int sms = 0;
  cp_status st = require_sm103(nullptr, &sms);
  if (st != CP_OK) return st;
  ReshardArgs a{dir, cp, n_tensors, seq_len, heads, d, static_cast<int32_t>(es), layout, in, out};
  return launch_reshard(a, sms, stream);
}
