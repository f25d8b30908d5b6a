// Backward of one (query shard, KV chunk) partial for bf16 inputs on the tcgen05 tensor cores.
//
// What it computes: the chain rule of the partial attention ("PCP and DCP sequence parallelism
// guide", section 2.3: in training the split sequence's gradients are reduce-scattered across
// ranks; this is one rank's share for one chunk).  Per head, against the rows' final LSE and
// D = dO . O (prep kernel):
//   S^T  = K Q^T                 P^T  = 2^(scale*log2(e) S^T - LSE*log2(e))   (keys x queries)
//   dP^T = V dO^T                dS^T = P^T o (dP^T - D)
//   dV  += P^T dO                dK  += scale dS^T Q                dQ += scale dS K
//
// How (GB300 design):
//   * Persistent, one CTA per SM.  A unit is one 128-key KV tile of one Q head; it walks every
//     128-row query tile that can see the KV tile (causal: tiles whose last row's position is at
//     least the tile's first key position).  Units are dealt round by round in snake order, in
//     one of two orders (decode_bunit): earliest keys first across the call's chunks for small
//     launches, or chunk by chunk in blocks of 16 KV tiles of one head for large ones, which keeps
//     the dQ tiles a head's units reduce into resident in L2.
//   * warp 0: TMA producer (K, V once per unit; Q, dO tiles and the rows' -LSE*log2(e), -D runs
//     per query tile).  warp 1: allocates tensor memory, issues tcgen05.mma (whole warp waits,
//     one elected lane issues).  warps 4-7: gradient warpgroup, one thread per key row -- turns
//     S^T into P^T and dP^T into dS^T.  warps 8-11: reduction warpgroup -- adds dQ (per query
//     tile; all of a tile's dQ is read from tensor memory before the first reduction) and dK, dV
//     (per unit) into global memory with TMA bulk reductions (fp32 add), so concurrent CTAs and
//     GQA heads accumulate without a separate pass.
//   * Tensor memory: S^T (128 fp32 columns, P^T bf16 written over its first 64), dP^T (128,
//     dS^T bf16 over its first 64), dV and dK accumulators (D each), dQ (D; for D = 128 it
//     reuses the dP^T columns once the dK product has consumed dS^T).
//   * Issue order per query tile g: dP^T(g), dV(g), then S^T(g+1) of the same unit -- so the
//     gradient warps start P^T(g+1) as soon as dS^T(g) is done, while dK(g) and dQ(g) run --
//     then dK(g), dQ(g).  Q tiles (with the rows' aux runs) have two stages, dO a ring of one
//     (D = 128) or two (D = 64) stages.
//   * The five products: S^T and dP^T are K-major x K-major from shared memory; dV and dK take
//     P^T / dS^T straight from tensor memory with dO / Q as MN-major B operands; dQ takes dS from
//     shared memory as an MN-major A operand (the gradient warps write it there in the 128-byte
//     swizzled layout a TMA load would produce) and K as MN-major B.
//   * Every mbarrier wait is bounded by %globaltimer; see sync.cuh.
#include <math.h>
#include <string.h>

#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "sync.cuh"

namespace cpattn {

namespace {

constexpr int kRows = 128;     // query rows per tile
constexpr int kKeys = 128;     // keys per KV tile
constexpr int kThreads = 384;  // 12 warps
constexpr int kBwdMaxChunksPerLaunch = 32;  // chunk table size limit (kernel parameter space)
constexpr int kJtBlock = 16;  // KV tiles of one head dealt together (blocked unit order)
constexpr int kBlockedMinUnitsPerSm = 16;  // launches with fewer units keep the KV-tile-major order

enum BwdSite : int {
  kSKvFull = 1,
  kSKvEmpty = 2,
  kSQFull = 3,
  kSQEmpty = 4,
  kSSFull = 5,
  kSPReady = 6,
  kSDpFull = 7,
  kSDsReady = 8,
  kSDqFull = 9,
  kSDqFree = 10,
  kSAccFull = 11,
  kSAccEmpty = 12,
  kSDoFull = 13,
  kSDoEmpty = 14,
  kSTest = 15,
};

struct BwdParams {
  int32_t* status;
  const float* aux;  // [2][hq][sq_pad]: -LSE*log2(e), -D
  int64_t sq, sq_pad;
  int32_t hq, hkv, group, causal;
  int32_t n_qt;        // query tiles
  int32_t max_kt;      // KV tiles of the longest chunk
  int32_t kt_blocks;   // blocks of kJtBlock KV tiles covering it
  int32_t blocked;     // unit order: 0 KV-tile-major, 1 blocked (see decode_bunit)
  int64_t n_units;     // (blocked ? kt_blocks * kJtBlock : max_kt) * n_chunks * hq
  float scale, sl2;    // scale, scale * log2(e)
  int64_t q_base, q_stride;
  int64_t timeout_ns;
  int32_t test_stall;  // test only: block 0's MMA warp first waits on a barrier nothing completes
};

// The KV chunks of one launch: TMA maps of K, V ([skv, hkv*d] bf16) and of their gradients dK,
// dV ([skv, hkv*d] fp32, reduction targets), token counts and affine global positions.  Chunks
// are independent here (each adds its own share); one launch just saves launches and lets the
// units of all chunks share one schedule.
template <int MAXC>
struct BwdChunks {
  CUtensorMap k[MAXC];
  CUtensorMap v[MAXC];
  CUtensorMap dk[MAXC];
  CUtensorMap dv[MAXC];
  int64_t skv[MAXC];
  int64_t base[MAXC];
  int64_t stride[MAXC];
  int32_t n;
};

template <int D>
struct BLayout {
  static constexpr int kChunkBytes = 128 * 128;     // 128 rows x 128 bytes
  static constexpr int kTileBytes = kRows * D * 2;  // bf16 [128, D]
  static constexpr int kChunks = D / 64;
  static constexpr int kQStages = 2;                // Q tile + the rows' aux runs
  static constexpr int kDoStages = (D == 64) ? 2 : 1;
  static constexpr int kStageBufs = (D == 64) ? 4 : 2;  // reduction staging boxes per warp
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;
  static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;
  static constexpr int kOffDS = kOffDO + kDoStages * kTileBytes;  // dS, 128 keys x 128 queries bf16
  static constexpr int kOffAux = kOffDS + 2 * kChunkBytes;        // per Q stage: 128 + 128 floats
  static constexpr int kOffStage = kOffAux + kQStages * 1024;     // 4 warps x kStageBufs x 4 KB
  static constexpr int kDataBytes = kOffStage + 4 * kStageBufs * 4096;  // from a 1024-byte boundary
  // kv_full, kv_empty, q_full[Q], q_empty[Q], do_full[DO], do_empty[DO], s_full, p_ready, dp_full,
  // ds_ready, dq_full, dq_free, acc_full, acc_empty, drain, never; then the control words
  static constexpr int kNumBars = 2 + 2 * kQStages + 2 * kDoStages + 10;
  static constexpr int kOffCtl = kNumBars * 8;
  static constexpr int kCtlBytes = 256;  // barriers + control words, placed in the alignment gap
  // The data region starts at the first 1024-byte boundary of the dynamic window; the barriers
  // sit in the gap before it when that gap holds them, else right after the data: either way the
  // whole layout fits in kDataBytes + 1024 bytes whatever the window's alignment.
  static constexpr int kSmemLaunch = kDataBytes + 1024;
  // tensor memory columns; dQ: own columns at D=64, the dP^T columns at D=128 (free once the
  // dK product has consumed dS^T, and read out before the next dP^T)
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr uint32_t kColDQ = (D == 64) ? 384 : 128;
};
static_assert(BLayout<128>::kOffCtl + 16 <= BLayout<128>::kCtlBytes, "barrier area");
static_assert(BLayout<128>::kSmemLaunch <= 232448, "shared memory budget (D=128)");
static_assert(BLayout<64>::kSmemLaunch <= 232448, "shared memory budget (D=64)");
static_assert(BLayout<64>::kColDQ + 64 <= 512 && BLayout<128>::kColDK + 128 <= 512, "tensor memory budget");

// Register split (setmaxnreg), 12 warps x 168 at launch.  D = 128: 4 warps x 120 (TMA / MMA) +
// 4 x 232 (gradient) + 4 x 152 (reduction: all four dQ boxes of a tile fit in registers, so the
// dQ tensor-memory columns, which the next dP^T reuses, are released before any reduction is
// issued).  D = 64: 4 x 128 + 4 x 248 + 4 x 128 (two dQ boxes; the gradient warps keep more).
template <int D>
struct BRegs {
  static constexpr uint32_t kControl = (D == 128) ? 120 : 128;
  static constexpr uint32_t kGrad = (D == 128) ? 232 : 248;
  static constexpr uint32_t kRed = (D == 128) ? 152 : 128;
  static_assert(4 * kControl + 4 * kGrad + 4 * kRed == 12 * 168, "register split must match launch");
};

struct Bars {
  uint32_t kv_full, kv_empty, q_full, q_empty, do_full, do_empty;  // q_*, do_*: stage 0, +8 per stage
  uint32_t s_full, p_ready, dp_full, ds_ready, dq_full, dq_free, acc_full, acc_empty, drain, never;
};

struct BUnit {
  int c;      // chunk
  int jt, h, g;
  int t0;     // first query tile that sees the KV tile
  int nit;    // query tiles to visit (0: nothing to do)
};

// Two unit orders.  KV-tile-major: (KV tile, chunk, head), earliest keys first across every
// chunk -- unit lengths fall monotonically, which balances the snake deal best when a launch has
// few rounds.  Blocked: (chunk, block of kJtBlock KV tiles, head, KV tile in the block) --
// concurrent CTAs hold about 152 / kJtBlock heads with kJtBlock neighbouring KV tiles each, whose
// walks start about a query tile apart and advance together, so each dQ tile they reduce into
// and each Q and dO tile they read is touched by all of them within a short window while it is
// in L2; in the KV-tile-major order those touches are spread over the whole launch and, once
// the shard's fp32 dQ outgrows L2, most dQ reductions go to DRAM.  Blocks go earliest keys first,
// so a launch still ends on a chunk's shortest units.  Tiles past a chunk's end are empty units.
template <int MAXC>
__device__ __forceinline__ BUnit decode_bunit(const BwdParams& p, const BwdChunks<MAXC>& ch, int64_t u) {
  BUnit w;
  if (p.blocked) {
    const int64_t per_block = static_cast<int64_t>(kJtBlock) * p.hq;
    const int64_t per_chunk = static_cast<int64_t>(p.kt_blocks) * per_block;
    w.c = static_cast<int>(u / per_chunk);
    int64_t rem = u - static_cast<int64_t>(w.c) * per_chunk;
    const int jb = static_cast<int>(rem / per_block);
    rem -= static_cast<int64_t>(jb) * per_block;
    w.h = static_cast<int>(rem / kJtBlock);
    w.jt = jb * kJtBlock + static_cast<int>(rem - static_cast<int64_t>(w.h) * kJtBlock);
  } else {
    const int64_t per_tile = static_cast<int64_t>(ch.n) * p.hq;
    w.jt = static_cast<int>(u / per_tile);
    const int64_t rem = u - static_cast<int64_t>(w.jt) * per_tile;
    w.c = static_cast<int>(rem / p.hq);
    w.h = static_cast<int>(rem - static_cast<int64_t>(w.c) * p.hq);
  }
  w.g = w.h / p.group;
  w.t0 = 0;
  if (static_cast<int64_t>(w.jt) * kKeys >= ch.skv[w.c]) {
    w.t0 = p.n_qt;
  } else if (p.causal) {
    const int64_t kp0 = ch.base[w.c] + ch.stride[w.c] * static_cast<int64_t>(w.jt) * kKeys;
    int64_t rmin = 0;  // first query row whose position reaches the tile's first key
    if (kp0 > p.q_base) rmin = (kp0 - p.q_base + p.q_stride - 1) / p.q_stride;
    w.t0 = rmin >= p.sq ? p.n_qt : static_cast<int>(rmin / kRows);
  }
  w.nit = p.n_qt - w.t0;
  return w;
}

// One warp's bulk reduction: 32 fp32 columns of its 32 rows, times `mul`, staged in one of its
// BUFS 4 KB swizzled boxes and added into `tm` at (x, y).  Rows past `rows` are clipped by the
// tensor map; a box that starts past them is skipped.  Returns the updated reduction count.
template <int BUFS>
__device__ __forceinline__ uint32_t reduce_box(uint32_t stage0, int lane, uint32_t nred, const uint32_t (&v)[32],
                                               float mul, const CUtensorMap* tm, int32_t x, int32_t y, int64_t rows) {
  if (y >= rows) return nred;
  const uint32_t sb = stage0 + (nred % BUFS) * 4096u;
  // the reduction that used this buffer last has finished reading it
  if (lane == 0) ptx::bulk_wait_read<BUFS - 1>();
  __syncwarp();
  const uint32_t row = sb + static_cast<uint32_t>(lane) * 128u;
  const uint32_t sw = static_cast<uint32_t>(lane & 7);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    ptx::sts128(row + ((static_cast<uint32_t>(q) ^ sw) << 4), __float_as_uint(__uint_as_float(v[4 * q]) * mul),
                __float_as_uint(__uint_as_float(v[4 * q + 1]) * mul), __float_as_uint(__uint_as_float(v[4 * q + 2]) * mul),
                __float_as_uint(__uint_as_float(v[4 * q + 3]) * mul));
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ptx::tma_reduce_add_2d(tm, sb, x, y);
    ptx::bulk_commit();
  }
  return nred + 1;
}

template <int D, int MAXC>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_tc_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dq,
                       const __grid_constant__ BwdChunks<MAXC> ch) {
  using L = BLayout<D>;
  using namespace sync;
  // bounded waits probe the phase with test_wait first at D = 64 (measured faster there)
  constexpr bool kProbe = (D == 64);
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* ctl_area = (smem - smem_raw >= L::kCtlBytes) ? smem_raw : smem + L::kDataBytes;
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t cbase = ptx::smem_u32(ctl_area);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t cta = blockIdx.x;
  const int64_t grid = gridDim.x;

  Bars b;
  b.kv_full = cbase;
  b.kv_empty = b.kv_full + 8;
  b.q_full = b.kv_empty + 8;
  b.q_empty = b.q_full + 8 * L::kQStages;
  b.do_full = b.q_empty + 8 * L::kQStages;
  b.do_empty = b.do_full + 8 * L::kDoStages;
  b.s_full = b.do_empty + 8 * L::kDoStages;
  b.p_ready = b.s_full + 8;
  b.dp_full = b.p_ready + 8;
  b.ds_ready = b.dp_full + 8;
  b.dq_full = b.ds_ready + 8;
  b.dq_free = b.dq_full + 8;
  b.acc_full = b.dq_free + 8;
  b.acc_empty = b.acc_full + 8;
  b.drain = b.acc_empty + 8;
  b.never = b.drain + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl_area + L::kOffCtl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl_area + L::kOffCtl + 4);
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    ptx::mbar_init(b.kv_full, 1);
    ptx::mbar_init(b.kv_empty, 1);
    for (int s = 0; s < L::kQStages; ++s) {
      ptx::mbar_init(b.q_full + 8 * s, 1);
      ptx::mbar_init(b.q_empty + 8 * s, 1);
    }
    for (int s = 0; s < L::kDoStages; ++s) {
      ptx::mbar_init(b.do_full + 8 * s, 1);
      ptx::mbar_init(b.do_empty + 8 * s, 1);
    }
    ptx::mbar_init(b.s_full, 1);
    ptx::mbar_init(b.p_ready, 4);
    ptx::mbar_init(b.dp_full, 1);
    ptx::mbar_init(b.ds_ready, 4);
    ptx::mbar_init(b.dq_full, 1);
    ptx::mbar_init(b.dq_free, 4);
    ptx::mbar_init(b.acc_full, 1);
    ptx::mbar_init(b.acc_empty, 4);
    ptx::mbar_init(b.drain, 1);
    ptx::mbar_init(b.never, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint32_t sK = sbase + L::kOffK;
  const uint32_t sV = sbase + L::kOffV;
  const uint32_t sQ = sbase + L::kOffQ;
  const uint32_t sDO = sbase + L::kOffDO;
  const uint32_t sDS = sbase + L::kOffDS;
  const uint32_t sAux = sbase + L::kOffAux;

  if (warp < 4) {
    ptx::regs_dec<BRegs<D>::kControl>();
    if (warp == 0) {
      // ============================================================== TMA producer
      const bool leader = ptx::elect_one();
      if (leader) {
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_do);
        for (int c = 0; c < ch.n; ++c) {
          ptx::tma_prefetch_desc(&ch.k[c]);
          ptx::tma_prefetch_desc(&ch.v[c]);
        }
      }
      int64_t gi = 0, ku = 0;  // query tiles and units with work issued so far
      int64_t ql = 0, dl = 0;  // Q and dO loads issued
      bool ok = true;
      for (int64_t k = 0; ok; ++k) {
        const int64_t u = unit_of(k, cta, grid);
        if (u >= p.n_units) break;
        const BUnit w = decode_bunit(p, ch, u);
        if (w.nit <= 0) continue;
        if (ku > 0 && !(ok = wait_warp<kProbe>(b.kv_empty, static_cast<uint32_t>((ku - 1) & 1), ctl, kSKvEmpty))) break;
        if (leader) {
          ptx::mbar_arrive_expect_tx(b.kv_full, 2 * L::kTileBytes);
          for (int cc = 0; cc < L::kChunks; ++cc) {
            ptx::tma_load_2d(sK + cc * L::kChunkBytes, &ch.k[w.c], w.g * D + cc * 64, w.jt * kKeys, b.kv_full);
            ptx::tma_load_2d(sV + cc * L::kChunkBytes, &ch.v[w.c], w.g * D + cc * 64, w.jt * kKeys, b.kv_full);
          }
        }
        __syncwarp();
        for (int it = 0; it < w.nit; ++it, ++gi) {
          const int t = w.t0 + it;
          const int st = static_cast<int>(gi % L::kQStages);
          const uint32_t ph = static_cast<uint32_t>((gi / L::kQStages) & 1);
          if (!(ok = wait_warp<kProbe>(b.q_empty + 8 * st, ph ^ 1, ctl, kSQEmpty))) break;
          if (leader) {
            const uint32_t full = b.q_full + 8 * st;
            ptx::mbar_arrive_expect_tx(full, L::kTileBytes + 1024);
            for (int cc = 0; cc < L::kChunks; ++cc)
              ptx::tma_load_2d(sQ + st * L::kTileBytes + cc * L::kChunkBytes, &tm_q, w.h * D + cc * 64,
                               t * kRows, full);
            const float* a0 = p.aux + static_cast<int64_t>(w.h) * p.sq_pad + static_cast<int64_t>(t) * kRows;
            const float* a1 = p.aux + (static_cast<int64_t>(p.hq) + w.h) * p.sq_pad + static_cast<int64_t>(t) * kRows;
            ptx::bulk_load(sAux + st * 1024, a0, 512, full);
            ptx::bulk_load(sAux + st * 1024 + 512, a1, 512, full);
          }
          __syncwarp();
          ql = gi + 1;
          const int sd = static_cast<int>(gi % L::kDoStages);
          const uint32_t phd = static_cast<uint32_t>((gi / L::kDoStages) & 1);
          if (!(ok = wait_warp<kProbe>(b.do_empty + 8 * sd, phd ^ 1, ctl, kSDoEmpty))) break;
          if (leader) {
            const uint32_t full = b.do_full + 8 * sd;
            ptx::mbar_arrive_expect_tx(full, L::kTileBytes);
            for (int cc = 0; cc < L::kChunks; ++cc)
              ptx::tma_load_2d(sDO + sd * L::kTileBytes + cc * L::kChunkBytes, &tm_do, w.h * D + cc * 64,
                               t * kRows, full);
          }
          __syncwarp();
          dl = gi + 1;
        }
        ++ku;
      }
      if (*abort_flag && leader) {
        // loads in flight must land before the CTA's shared memory goes away
        if (ku > 0) wait_drain(b.kv_full, static_cast<uint32_t>((ku - 1) & 1), p.timeout_ns);
        // the last load issued into every stage: load n went to stage n % S, phase (n / S) & 1
        for (int s = 0; s < L::kQStages; ++s) {
          const int64_t last = (ql - 1 - s >= 0) ? ql - 1 - ((ql - 1 - s) % L::kQStages) : -1;
          if (last >= 0)
            wait_drain(b.q_full + 8 * s, static_cast<uint32_t>((last / L::kQStages) & 1), p.timeout_ns);
        }
        for (int s = 0; s < L::kDoStages; ++s) {
          const int64_t last = (dl - 1 - s >= 0) ? dl - 1 - ((dl - 1 - s) % L::kDoStages) : -1;
          if (last >= 0)
            wait_drain(b.do_full + 8 * s, static_cast<uint32_t>((last / L::kDoStages) & 1), p.timeout_ns);
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ============================================================== MMA issuer
      const bool leader = ptx::elect_one();
      // How the MMAs are issued (measured per head dim, same-box A/B): at D = 128 a group of MMAs
      // is issued inside one branch the elected lane takes; at D = 64 the converged warp runs the
      // issue code and each MMA is guarded by its own elected-lane test (2.5 % faster there, 6 %
      // slower at D = 128).
      constexpr bool kGroupIssue = (D == 128);
      const bool issuer = kGroupIssue ? leader : true;
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kKeys, kRows, 0, 0);  // S^T, dP^T
      constexpr uint32_t kIdescG = ptx::idesc_bf16_f32(kKeys, D, 0, 1);      // dV, dK (A in TMEM)
      constexpr uint32_t kIdescQ = ptx::idesc_bf16_f32(kRows, D, 1, 1);      // dQ (A = dS, MN-major)
      const uint64_t dK_k = ptx::smem_desc_sw128(sK, 16, 1024);
      const uint64_t dV_k = ptx::smem_desc_sw128(sV, 16, 1024);
      const uint64_t dQ_k = ptx::smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dDO_k = ptx::smem_desc_sw128(sDO, 16, 1024);
      const uint64_t dQ_mn = ptx::smem_desc_sw128(sQ, L::kChunkBytes, 1024);
      const uint64_t dDO_mn = ptx::smem_desc_sw128(sDO, L::kChunkBytes, 1024);
      const uint64_t dK_mn = ptx::smem_desc_sw128(sK, L::kChunkBytes, 1024);
      const uint64_t dDS_mn = ptx::smem_desc_sw128(sDS, L::kChunkBytes, 1024);
      constexpr uint64_t kTileUnits = L::kTileBytes >> 4;

      // M=128, N=128, K=D; both operands K-major (rows x D, 64-column swizzled boxes)
      auto issue_kk = [&](uint32_t d_tmem, uint64_t a0, uint64_t b0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4);
          if (kGroupIssue || leader) ptx::mma_ss(d_tmem, a0 + off, b0 + off, kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      // M=128 keys, N=D, K=128 queries: A (bf16 packed, 8 columns per 16 queries) in tensor memory
      auto issue_ts = [&](uint32_t d_tmem, uint32_t a_tmem, uint64_t b_mn, bool acc) {
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk)
          if (kGroupIssue || leader)
            ptx::mma_ts(d_tmem, a_tmem + kk * 8, b_mn + static_cast<uint64_t>(kk * 128), kIdescG,
                        (acc || kk > 0) ? 1u : 0u);
      };
      // M=128 queries, N=D, K=128 keys: dS (MN-major) x K (MN-major)
      auto issue_dq = [&](uint32_t d_tmem) {
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          if (kGroupIssue || leader)
            ptx::mma_ss(d_tmem, dDS_mn + static_cast<uint64_t>(kk * 128), dK_mn + static_cast<uint64_t>(kk * 128),
                        kIdescQ, kk > 0 ? 1u : 0u);
      };

      // Per query tile gi of a unit: [S^T(gi) if first of the unit] dP^T(gi), dV(gi), S^T(gi+1) of
      // the same unit (overlaps the gradient warps' dS(gi)), dK(gi), dQ(gi).
      auto issue_s = [&](int64_t g) -> bool {
        const int sq = static_cast<int>(g % L::kQStages);
        if (!wait_warp<kProbe>(b.q_full + 8 * sq, static_cast<uint32_t>((g / L::kQStages) & 1), ctl, kSQFull)) return false;
        ptx::tc_fence_after();
        if (issuer) issue_kk(tmem + L::kColS, dK_k, dQ_k + sq * kTileUnits);
        if (leader) ptx::mma_commit(b.s_full);
        __syncwarp();
        return true;
      };
      int64_t gi = 0, ku = 0;
      bool ok = true;
      if (p.test_stall && blockIdx.x == 0) ok = wait_warp<kProbe>(b.never, 0, ctl, kSTest);
      for (int64_t k = 0; ok; ++k) {
        const int64_t u = unit_of(k, cta, grid);
        if (u >= p.n_units) break;
        const BUnit w = decode_bunit(p, ch, u);
        if (w.nit <= 0) continue;
        if (!(ok = wait_warp<kProbe>(b.kv_full, static_cast<uint32_t>(ku & 1), ctl, kSKvFull))) break;
        if (!(ok = issue_s(gi))) break;
        for (int it = 0; it < w.nit; ++it, ++gi) {
          const bool first = (it == 0);
          const int st = static_cast<int>(gi % L::kQStages);
          const int sd = static_cast<int>(gi % L::kDoStages);
          const uint32_t phd = static_cast<uint32_t>((gi / L::kDoStages) & 1);
          const uint32_t prev = static_cast<uint32_t>((gi - 1) & 1);
          const uint32_t cur = static_cast<uint32_t>(gi & 1);
          if (!(ok = wait_warp<kProbe>(b.do_full + 8 * sd, phd, ctl, kSDoFull))) break;
          // D = 128: the previous dQ sits in the dP^T columns until the reduction warps read it
          if (D == 128 && gi > 0 && !(ok = wait_warp<kProbe>(b.dq_free, prev, ctl, kSDqFree))) break;
          ptx::tc_fence_after();
          if (issuer) issue_kk(tmem + L::kColDP, dV_k, dDO_k + sd * kTileUnits);
          if (leader) ptx::mma_commit(b.dp_full);
          __syncwarp();
          if (!(ok = wait_warp<kProbe>(b.p_ready, cur, ctl, kSPReady))) break;
          // the unit's first dV overwrites the accumulators: the previous unit's must be read out
          if (first && ku > 0 && !(ok = wait_warp<kProbe>(b.acc_empty, static_cast<uint32_t>((ku - 1) & 1), ctl, kSAccEmpty)))
            break;
          ptx::tc_fence_after();
          if (issuer) issue_ts(tmem + L::kColDV, tmem + L::kColS, dDO_mn + sd * kTileUnits, !first);
          if (leader) ptx::mma_commit(b.do_empty + 8 * sd);
          __syncwarp();
          // the next S^T may overwrite P^T: the dV product just issued reads it first (issue order)
          if (it + 1 < w.nit && !(ok = issue_s(gi + 1))) break;
          if (!(ok = wait_warp<kProbe>(b.ds_ready, cur, ctl, kSDsReady))) break;
          ptx::tc_fence_after();
          if (issuer) issue_ts(tmem + L::kColDK, tmem + L::kColDP, dQ_mn + st * kTileUnits, !first);
          __syncwarp();
          if (D == 64 && gi > 0 && !(ok = wait_warp<kProbe>(b.dq_free, prev, ctl, kSDqFree))) break;
          ptx::tc_fence_after();
          if (issuer) issue_dq(tmem + L::kColDQ);
          if (leader) {
            ptx::mma_commit(b.dq_full);
            ptx::mma_commit(b.q_empty + 8 * st);
            if (it == w.nit - 1) {
              ptx::mma_commit(b.acc_full);
              ptx::mma_commit(b.kv_empty);
            }
          }
          __syncwarp();
        }
        ++ku;
      }
      if (!ok) {
        if (leader) {
          ptx::mma_commit(b.drain);
          wait_drain(b.drain, 0, p.timeout_ns);
        }
        __syncwarp();
      }
    }
  } else if (warp < 8) {
    ptx::regs_inc<BRegs<D>::kGrad>();
    // ================================================================ gradient warpgroup
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key row inside the KV tile
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + L::kColS + lane_bits;
    const uint32_t tDP = tmem + L::kColDP + lane_bits;
    const uint64_t sl2x2 = ptx::f2_pack(p.sl2, p.sl2);
    const uint32_t ds_row = sDS + static_cast<uint32_t>(r) * 128u;
    const uint32_t sw = static_cast<uint32_t>(r & 7);
    int64_t gi = 0;
    bool ok = true;
    for (int64_t k = 0; ok; ++k) {
      const int64_t u = unit_of(k, cta, grid);
      if (u >= p.n_units) break;
      const BUnit w = decode_bunit(p, ch, u);
      if (w.nit <= 0) continue;
      const int64_t key = static_cast<int64_t>(w.jt) * kKeys + r;
      const int64_t kpos = ch.base[w.c] + ch.stride[w.c] * key;
      const int64_t skv = ch.skv[w.c];
      int64_t rmin_k = 0;  // first query row that sees this key
      if (p.causal && kpos > p.q_base) rmin_k = (kpos - p.q_base + p.q_stride - 1) / p.q_stride;
      // rows past the chunk's end (zero-filled K, V) get P = 0 too: against a very negative LSE
      // their exponent could overflow, and 0 * inf would reach dQ
      if (key >= skv) rmin_k = INT64_MAX / 2;
      for (int it = 0; it < w.nit; ++it, ++gi) {
        const int t = w.t0 + it;
        const int st = static_cast<int>(gi % L::kQStages);
        const uint32_t cur = static_cast<uint32_t>(gi & 1);
        int cmin = 0;  // query columns below cmin do not see this key
        if (p.causal || key >= skv) {
          const int64_t c = rmin_k - static_cast<int64_t>(t) * kRows;
          cmin = c <= 0 ? 0 : (c >= kRows ? kRows : static_cast<int>(c));
        }
        const uint32_t a_nl = sAux + st * 1024;  // -LSE*log2(e) of the tile's 128 rows
        const uint32_t a_nd = a_nl + 512;        // -D
        // the per-row runs were copied by the bulk engine: observe their barrier directly
        if (!(ok = wait_warp<kProbe>(b.q_full + 8 * st, static_cast<uint32_t>((gi / L::kQStages) & 1), ctl, kSQFull))) break;
        if (!(ok = wait_warp<kProbe>(b.s_full, cur, ctl, kSSFull))) break;
        ptx::tc_fence_after();
        // all 128 columns of S^T in one go (one wait), then P in place
        uint32_t pf[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + c * 32, pf[c]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 nl = ptx::lds128(a_nl + (c * 32 + e4 * 4) * 4);
            const uint64_t x01 = ptx::f2_fma(
                ptx::f2_pack(__uint_as_float(pf[c][4 * e4]), __uint_as_float(pf[c][4 * e4 + 1])), sl2x2,
                ptx::f2_pack(nl.x, nl.y));
            const uint64_t x23 = ptx::f2_fma(
                ptx::f2_pack(__uint_as_float(pf[c][4 * e4 + 2]), __uint_as_float(pf[c][4 * e4 + 3])), sl2x2,
                ptx::f2_pack(nl.z, nl.w));
            float x0, x1, x2, x3;
            ptx::f2_unpack(x01, x0, x1);
            ptx::f2_unpack(x23, x2, x3);
            pf[c][4 * e4] = __float_as_uint(ptx::ex2(x0));
            pf[c][4 * e4 + 1] = __float_as_uint(ptx::ex2(x1));
            pf[c][4 * e4 + 2] = __float_as_uint(ptx::ex2(x2));
            pf[c][4 * e4 + 3] = __float_as_uint(ptx::ex2(x3));
          }
          if (cmin > c * 32) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e < cmin) pf[c][e] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = ptx::pack_bf16x2(__uint_as_float(pf[c][2 * e]), __uint_as_float(pf[c][2 * e + 1]));
          ptx::tmem_st16(tS + c * 16, pk);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b.p_ready);

        if (!(ok = wait_warp<kProbe>(b.dp_full, cur, ctl, kSDpFull))) break;
        // the dS buffer in shared memory is free once the previous dQ product has read it
        if (gi > 0 && !(ok = wait_warp<kProbe>(b.dq_full, static_cast<uint32_t>((gi - 1) & 1), ctl, kSDqFull))) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t dr[32];
          ptx::tmem_ld32(tDP + c * 32, dr);
          ptx::tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const int col = c * 32 + e4 * 4;
            const float4 nd = ptx::lds128(a_nd + col * 4);
            const uint64_t t01 = ptx::f2_add(ptx::f2_pack(__uint_as_float(dr[4 * e4]), __uint_as_float(dr[4 * e4 + 1])),
                                             ptx::f2_pack(nd.x, nd.y));
            const uint64_t t23 = ptx::f2_add(
                ptx::f2_pack(__uint_as_float(dr[4 * e4 + 2]), __uint_as_float(dr[4 * e4 + 3])), ptx::f2_pack(nd.z, nd.w));
            const uint64_t d01 = ptx::f2_mul(
                ptx::f2_pack(__uint_as_float(pf[c][4 * e4]), __uint_as_float(pf[c][4 * e4 + 1])), t01);
            const uint64_t d23 = ptx::f2_mul(
                ptx::f2_pack(__uint_as_float(pf[c][4 * e4 + 2]), __uint_as_float(pf[c][4 * e4 + 3])), t23);
            float s0, s1, s2, s3;
            ptx::f2_unpack(d01, s0, s1);
            ptx::f2_unpack(d23, s2, s3);
            pk[2 * e4] = ptx::pack_bf16x2(s0, s1);
            pk[2 * e4 + 1] = ptx::pack_bf16x2(s2, s3);
          }
          ptx::tmem_st16(tDP + c * 16, pk);
          // dS row r, queries c*32 .. c*32+31: four 16-byte chunks of the 64-query box c/2
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t q8 = static_cast<uint32_t>((c & 1) * 4 + i);
            ptx::sts128(ds_row + static_cast<uint32_t>(c >> 1) * L::kChunkBytes + ((q8 ^ sw) << 4), pk[4 * i],
                        pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        ptx::tmem_wait_st();
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b.ds_ready);
      }
    }
  } else {
    ptx::regs_dec<BRegs<D>::kRed>();  // below the launch allocation: give registers back
    // ================================================================ reduction warpgroup
    const int wq = warp & 3;
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t stage0 = sbase + L::kOffStage + static_cast<uint32_t>(wq * L::kStageBufs) * 4096u;
    int64_t gi = 0, ku = 0;
    uint32_t nred = 0;  // bulk reductions issued by this warp (staging double buffer)
    bool ok = true;

    for (int64_t k = 0; ok; ++k) {
      const int64_t u = unit_of(k, cta, grid);
      if (u >= p.n_units) break;
      const BUnit w = decode_bunit(p, ch, u);
      if (w.nit <= 0) continue;
      for (int it = 0; it < w.nit; ++it, ++gi) {
        const int t = w.t0 + it;
        if (!(ok = wait_warp<kProbe>(b.dq_full, static_cast<uint32_t>(gi & 1), ctl, kSDqFull))) break;
        ptx::tc_fence_after();
        // all of dQ into registers first, so the tensor memory goes back to the MMA warp (which
        // at D = 128 puts the next dP^T there) before any reduction is issued
        uint32_t v[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(tmem + L::kColDQ + lane_bits + c * 32, v[c]);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b.dq_free);
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          nred = reduce_box<L::kStageBufs>(stage0, lane, nred, v[c], p.scale, &tm_dq, w.h * D + c * 32, t * kRows + wq * 32,
                                           p.sq);
      }
      if (!ok) break;
      // end of the unit: dK (scaled) and dV
      if (!(ok = wait_warp<kProbe>(b.acc_full, static_cast<uint32_t>(ku & 1), ctl, kSAccFull))) break;
      ptx::tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        ptx::tmem_ld32(tmem + L::kColDK + lane_bits + c * 32, v);
        ptx::tmem_wait_ld();
        nred = reduce_box<L::kStageBufs>(stage0, lane, nred, v, p.scale, &ch.dk[w.c], w.g * D + c * 32, w.jt * kKeys + wq * 32,
                                         ch.skv[w.c]);
      }
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        ptx::tmem_ld32(tmem + L::kColDV + lane_bits + c * 32, v);
        ptx::tmem_wait_ld();
        nred = reduce_box<L::kStageBufs>(stage0, lane, nred, v, 1.0f, &ch.dv[w.c], w.g * D + c * 32, w.jt * kKeys + wq * 32,
                                         ch.skv[w.c]);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(b.acc_empty);
      ++ku;
    }
    if (lane == 0) ptx::bulk_wait_all();  // every reduction has completed
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int D, int MAXC>
cp_status launch_bwd_dc(const BwdParams& p0, const cp_attn_bwd_desc& d, const cp_kv_bwd_chunk* chunks, int n,
                        int num_sms, cudaStream_t s) {
  BwdChunks<MAXC> ch;
  memset(&ch, 0, sizeof(ch));
  ch.n = n;
  BwdParams p = p0;
  const int64_t ke = int64_t(d.hkv) * D;
  int64_t max_kt = 0;
  for (int c = 0; c < n; ++c) {
    const cp_kv_bwd_chunk& k = chunks[c];
    if (!encode_map_2d(&ch.k[c], k.k, k.skv, ke, false, 128) || !encode_map_2d(&ch.v[c], k.v, k.skv, ke, false, 128) ||
        !encode_map_2d(&ch.dk[c], k.dk, k.skv, ke, true, 32) || !encode_map_2d(&ch.dv[c], k.dv, k.skv, ke, true, 32)) {
      set_error("cuTensorMapEncodeTiled failed for chunk %d (or the driver entry point is unavailable)", c);
      return CP_ERR_CUDA;
    }
    ch.skv[c] = k.skv;
    ch.base[c] = k.kv_pos.base;
    ch.stride[c] = k.kv_pos.stride;
    const int64_t kt = (k.skv + kKeys - 1) / kKeys;
    if (kt > max_kt) max_kt = kt;
  }
  p.max_kt = static_cast<int32_t>(max_kt);
  p.kt_blocks = static_cast<int32_t>((max_kt + kJtBlock - 1) / kJtBlock);
  p.blocked = (max_kt * n * d.hq >= static_cast<int64_t>(kBlockedMinUnitsPerSm) * num_sms) ? 1 : 0;
  p.n_units = (p.blocked ? static_cast<int64_t>(p.kt_blocks) * kJtBlock : max_kt) * n * d.hq;
  CUtensorMap mq, mdo, mdq;
  const int64_t qe = int64_t(d.hq) * D;
  if (!encode_map_2d(&mq, d.q, d.sq, qe, false, 128) || !encode_map_2d(&mdo, d.d_o, d.sq, qe, false, 128) ||
      !encode_map_2d(&mdq, d.dq, d.sq, qe, true, 32)) {
    set_error("cuTensorMapEncodeTiled failed (or the driver entry point is unavailable)");
    return CP_ERR_CUDA;
  }
  const int64_t grid = p.n_units < num_sms ? p.n_units : num_sms;
  constexpr int smem = BLayout<D>::kSmemLaunch;
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_tc_kernel<D, MAXC>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attn_bwd_tc_kernel)");
  attn_bwd_tc_kernel<D, MAXC><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(p, mq, mdo, mdq, ch);
  e = cudaGetLastError();
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "attn_bwd_tc_kernel launch");
}

template <int D>
cp_status launch_bwd_d(const BwdParams& p, const cp_attn_bwd_desc& d, const cp_kv_bwd_chunk* chunks, int n,
                       int num_sms, cudaStream_t s) {
  // the chunk table travels in the kernel parameters: size it to the call; longer lists go in
  // batches (the chunks are independent)
  for (int at = 0; at < n;) {
    const int m = (n - at) < kBwdMaxChunksPerLaunch ? (n - at) : kBwdMaxChunksPerLaunch;
    cp_status st;
    if (m == 1)
      st = launch_bwd_dc<D, 1>(p, d, chunks + at, m, num_sms, s);
    else if (m <= 8)
      st = launch_bwd_dc<D, 8>(p, d, chunks + at, m, num_sms, s);
    else
      st = launch_bwd_dc<D, kBwdMaxChunksPerLaunch>(p, d, chunks + at, m, num_sms, s);
    if (st != CP_OK) return st;
    at += m;
  }
  return CP_OK;
}

}  // namespace

cp_status launch_partial_attn_bwd_tc(const cp_attn_bwd_desc& d, const cp_kv_bwd_chunk* chunks, int n, float scale,
                                     int64_t timeout_ns, int num_sms, cudaStream_t s) {
  BwdParams p;
  p.status = d.status;
  p.aux = d.aux;
  p.sq = d.sq;
  p.sq_pad = (d.sq + 127) / 128 * 128;
  p.hq = d.hq;
  p.hkv = d.hkv;
  p.group = d.hq / d.hkv;
  p.causal = d.causal;
  p.n_qt = static_cast<int32_t>((d.sq + kRows - 1) / kRows);
  p.max_kt = 0;
  p.kt_blocks = 0;
  p.blocked = 0;
  p.n_units = 0;
  p.scale = scale;
  p.sl2 = scale * 1.4426950408889634f;
  p.q_base = d.q_pos.base;
  p.q_stride = d.q_pos.stride;
  p.timeout_ns = timeout_ns;
  p.test_stall = (d.flags & CP_FLAG_TEST_STALL) ? 1 : 0;
  if (d.d == 64) return launch_bwd_d<64>(p, d, chunks, n, num_sms, s);
  return launch_bwd_d<128>(p, d, chunks, n, num_sms, s);
}

}  // namespace cpattn
