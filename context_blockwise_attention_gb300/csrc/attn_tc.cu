// Partial attention for bf16 inputs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// What it computes ("FCP: from a fixed ring to a free topology", section 3.3): for a query
// block, visit KV blocks in any order; per block form scores q . k^T / sqrt(head_dim), update
// the running maximum, rescale the accumulator and running sum by exp(old - new), add
// exp(scores - new_max) @ V and its row sum; output = acc / running_sum.  The kernel emits the
// normalised partial O and LSE = ln(sum exp(scores)) of one KV chunk; partials from different
// chunks are combined by the merge kernel.
//
// How (GB300 design, not the pages'):
//   * Persistent: one CTA per SM walks a list of units -- a pair of 128-row Q tiles (A, B) of
//     one head -- in longest-first order, snaking across CTAs round by round (causal units
//     shrink towards the start of the shard); Q heads of one KV group are adjacent so their
//     K/V tiles are shared through L2.  KV tiles are 128 keys.
//   * warp 0: TMA producer.  K and V tiles stream through rings of shared-memory stages
//     (128-byte swizzle) straight across unit boundaries; a unit's Q is loaded as soon as the
//     previous unit's last QK has completed.  warp 1: allocates tensor memory and issues
//     tcgen05.mma (whole warp waits, one elected lane issues).  warps 4-7 / 8-11: softmax
//     warpgroups for Q tiles A / B, one thread per row.
//   * Tensor memory (512 columns): S_A, S_B (128 fp32 columns each), O_A, O_B (D columns).
//     P (bf16) is written over the first 64 columns of its S tile and fed to the PV product
//     from tensor memory.
//   * Tensor-pipe order per KV step j: QK_A(j), PV_B(j-1), QK_B(j), PV_A(j); each softmax
//     warpgroup has two MMA slots to turn its S tile into P, and releases P in two halves so the
//     PV product starts on keys 0..63 while 64..127 are still being exponentiated.
//   * Online softmax in base 2 with a lazy rescale: O and l are rescaled only when a row's
//     maximum grows by more than 2^8; otherwise exponentials use the stale maximum.  The final
//     O / l and LSE use that same reference, so the result is exact.
//   * Causal visibility is by global position: key j is visible to query i iff
//     kv_pos(j) <= q_pos(i).  KV tiles entirely in the future of a unit's last row are never
//     loaded or multiplied; only tiles that straddle the boundary (or the ragged end of the
//     chunk) are masked element by element.
//   * Epilogue: after a unit's last PV the softmax warpgroup copies O into registers, releases
//     its tensor memory (the next unit's PV may start) and streams O / l through a 16 KB
//     swizzled staging box per warpgroup with TMA bulk stores (rows past sq are clipped).
//   * Every mbarrier wait is bounded by %globaltimer; on expiry the kernel records
//     CP_ERR_TIMEOUT in the caller's status word, every role leaves its loops, outstanding TMA
//     loads, MMAs and bulk stores are drained and tensor memory is freed before the CTA exits.
#include <math.h>
#include <string.h>

#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "sync.cuh"

namespace cpattn {

namespace {

using sync::Ctl;
using sync::unit_of;
using sync::wait_drain;
using sync::wait_warp;

constexpr int kRows = 128;     // rows per Q tile
constexpr int kKeys = 128;     // keys per KV tile
constexpr int kThreads = 384;  // 12 warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum WaitSite : int {
  kSiteQ = 1,
  kSiteKFull = 2,
  kSiteKEmpty = 3,
  kSiteVFull = 4,
  kSiteVEmpty = 5,
  kSiteSFull = 6,
  kSitePFull = 7,
  kSiteOFinal = 8,
  kSiteTest = 9,
  kSiteQEmpty = 10,
  kSiteOEmpty = 11,
};

struct TcParams {
  void* o;
  float* lse;
  int32_t* status;
  int64_t sq;
  int32_t hq, hkv, group;
  int32_t n_pairs;
  int64_t n_units;  // n_pairs * hq
  int32_t causal, o_bf16, descending, test_stall;
  float scale_log2;
  int64_t q_base, q_stride;
  int64_t timeout_ns;
};

// The KV chunks of one launch, in arrival order: TMA maps of K and V ([skv, hkv*d] bf16) and
// the affine global positions.  A unit's KV tiles are the visible tiles of chunk 0, then of
// chunk 1, ...; the online-softmax state runs across all of them.
template <int MAXC>
struct ChunkTable {
  CUtensorMap k[MAXC];
  CUtensorMap v[MAXC];
  int64_t skv[MAXC];
  int64_t base[MAXC];
  int64_t stride[MAXC];
  int32_t n;
};

template <int D>
struct Layout {
  static constexpr int kChunks = D / 64;             // 128-byte column chunks of a tile
  static constexpr int kChunkBytes = 128 * 128;      // 128 rows x 128 bytes
  static constexpr int kTileBytes = kRows * D * 2;   // bf16 tile
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  // 16 KB staging boxes per warpgroup: two at D = 64 (shared memory has room; an fp32 O tile is
  // two boxes, so neither waits for the other's bulk store), one at D = 128
  static constexpr int kStageBufs = (D == 64) ? 2 : 1;
  static constexpr int kOffStage = kOffV + kStages * kTileBytes;
  static constexpr int kOffBar = kOffStage + 2 * kStageBufs * kChunkBytes;
  // barriers: q_full, q_empty, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2],
  //           p_half[2], p_full[2], o_final[2], o_empty[2], never, drain
  static constexpr int kNumBars = 2 + 4 * kStages + 10 + 2;
  static constexpr int kOffCtl = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffCtl + 16;
  static constexpr int kSmemLaunch = kBytes + 1024;  // slack for 1024-byte alignment
  static constexpr int kBoxesF32 = D / 32;           // 32 fp32 columns per 128-byte box
  static constexpr int kBoxesBf16 = D / 64;          // 64 bf16 columns per box
};
static_assert(Layout<128>::kSmemLaunch <= 232448, "shared memory budget (D=128)");
static_assert(Layout<64>::kSmemLaunch <= 232448, "shared memory budget (D=64)");

// Register split (setmaxnreg): the TMA/MMA warpgroup gives registers to the two softmax
// warpgroups.  4 warps x 120 + 8 warps x 192 = 12 warps x 168, the launch's allocation (measured
// best of the splits without spills: the chunk loops of the TMA/MMA warps need > 104).
#ifndef CP_REGS_CONTROL
#define CP_REGS_CONTROL 120
#define CP_REGS_SOFTMAX 192
#endif
constexpr uint32_t kRegsControl = CP_REGS_CONTROL;
constexpr uint32_t kRegsSoftmax = CP_REGS_SOFTMAX;
static_assert(4 * kRegsControl + 8 * kRegsSoftmax == 12 * 168, "register split must match launch");

struct Bars {
  uint32_t q_full, q_empty;
  uint32_t k_full, k_empty, v_full, v_empty;  // stage 0; +8 per stage
  uint32_t s_full, p_half, p_full, o_final, o_empty;  // tile A; +8 for tile B
  uint32_t never, drain;
};

// Keys of chunk c that query `row` may see: all of them when not causal, else the keys j with
// base + stride * j <= q_pos(row) (positions grow with the index, so they are a prefix).
template <int MAXC>
__device__ __forceinline__ int64_t visible_keys(const TcParams& p, const ChunkTable<MAXC>& ch, int c,
                                                int64_t row) {
  const int64_t skv = ch.skv[c];
  if (!p.causal) return skv;
  const int64_t qp = p.q_base + p.q_stride * row;
  if (qp < ch.base[c]) return 0;
  const int64_t n = (qp - ch.base[c]) / ch.stride[c] + 1;
  return n < skv ? n : skv;
}

struct Unit {
  int64_t row0;   // first query row of tile A
  int64_t last;   // last query row of the unit that exists
  int h, kvh;
  int n_tiles;    // KV tiles over all chunks
};

// KV tiles of chunk c the unit has to visit: those holding a key visible to its last row.
template <int MAXC>
__device__ __forceinline__ int chunk_tiles(const TcParams& p, const ChunkTable<MAXC>& ch, int c,
                                           const Unit& w) {
  return static_cast<int>((visible_keys(p, ch, c, w.last) + kKeys - 1) / kKeys);
}

// Units are numbered longest first: pairs in decreasing order when causal, heads innermost.
template <int MAXC>
__device__ __forceinline__ Unit decode_unit(const TcParams& p, const ChunkTable<MAXC>& ch, int64_t u) {
  Unit w;
  const int64_t pair = p.causal ? (p.n_pairs - 1 - u / p.hq) : (u / p.hq);
  w.h = static_cast<int>(u % p.hq);
  w.kvh = w.h / p.group;
  w.row0 = pair * (2 * kRows);
  w.last = w.row0 + 2 * kRows - 1;
  if (w.last > p.sq - 1) w.last = p.sq - 1;
  w.n_tiles = 0;
  for (int c = 0; c < ch.n; ++c) w.n_tiles += chunk_tiles(p, ch, c, w);
  return w;
}

// Issue of MMAs, commits and TMA copies by the control warps: at D = 128 the converged warp issues
// under a lane predicate (the MMA issue rate bounds that head dim; measured +10 %), at D = 64 the
// elected lane alone (measured 2-4 % faster there).
template <bool kPred>
struct Issue {
  uint32_t lead;
  __device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) const {
    if (kPred) ptx::mma_ss_p(d, a, b, idesc, acc, lead);
    else if (lead) ptx::mma_ss(d, a, b, idesc, acc);
  }
  __device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) const {
    if (kPred) ptx::mma_ts_p(d, a, b, idesc, acc, lead);
    else if (lead) ptx::mma_ts(d, a, b, idesc, acc);
  }
  __device__ __forceinline__ void commit(uint32_t bar) const {
    if (kPred) ptx::mma_commit_p(bar, lead);
    else if (lead) ptx::mma_commit(bar);
  }
  __device__ __forceinline__ void expect_tx(uint32_t bar, uint32_t bytes) const {
    if (kPred) ptx::mbar_arrive_expect_tx_p(bar, bytes, lead);
    else if (lead) ptx::mbar_arrive_expect_tx(bar, bytes);
  }
  __device__ __forceinline__ void load(uint32_t dst, const void* tmap, int32_t x, int32_t y, uint32_t bar) const {
    if (kPred) ptx::tma_load_2d_p(dst, tmap, x, y, bar, lead);
    else if (lead) ptx::tma_load_2d(dst, tmap, x, y, bar);
  }
};

// exp2 of 32 scaled scores (x = s * sl2 - m) packed to 16 bf16 pairs; adds the fp32 values to
// the two packed partial sums.  (Evaluating part of the exponentials with a polynomial on the FMA
// pipe was measured slower on GB300 for both head dims: the softmax is bound by instruction issue
// and latency, not by the MUFU unit.)
__device__ __forceinline__ void exp_pack32(const uint32_t (&s)[32], uint64_t sl2x2, uint64_t negm2,
                                           uint32_t (&pk)[16], uint64_t& sum_a, uint64_t& sum_b) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint64_t x2 = ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])),
                                    sl2x2, negm2);
    float x0, x1;
    ptx::f2_unpack(x2, x0, x1);
    const float p0 = ptx::ex2(x0);
    const float p1 = ptx::ex2(x1);
    pk[e] = ptx::pack_bf16x2(p0, p1);
    if (e & 1)
      sum_b = ptx::f2_add(sum_b, ptx::f2_pack(p0, p1));
    else
      sum_a = ptx::f2_add(sum_a, ptx::f2_pack(p0, p1));
  }
}

template <int D, int MAXC>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ ChunkTable<MAXC> ch) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t cta = blockIdx.x;
  const int64_t grid = gridDim.x;

  Bars b;
  b.q_full = sbase + L::kOffBar;
  b.q_empty = b.q_full + 8;
  b.k_full = b.q_empty + 8;
  b.k_empty = b.k_full + 8 * L::kStages;
  b.v_full = b.k_empty + 8 * L::kStages;
  b.v_empty = b.v_full + 8 * L::kStages;
  b.s_full = b.v_empty + 8 * L::kStages;
  b.p_half = b.s_full + 16;
  b.p_full = b.p_half + 16;
  b.o_final = b.p_full + 16;
  b.o_empty = b.o_final + 16;
  b.never = b.o_empty + 16;
  b.drain = b.never + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffCtl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffCtl + 4);
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    ptx::mbar_init(b.q_full, 1);
    ptx::mbar_init(b.q_empty, 1);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(b.k_full + 8 * s, 1);
      ptx::mbar_init(b.k_empty + 8 * s, 1);
      ptx::mbar_init(b.v_full + 8 * s, 1);
      ptx::mbar_init(b.v_empty + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(b.s_full + 8 * t, 1);
      ptx::mbar_init(b.p_half + 8 * t, 4);
      ptx::mbar_init(b.p_full + 8 * t, 4);
      ptx::mbar_init(b.o_final + 8 * t, 1);
      ptx::mbar_init(b.o_empty + 8 * t, 4);
    }
    ptx::mbar_init(b.never, 1);
    ptx::mbar_init(b.drain, 1);
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

  const uint32_t sQ = sbase + L::kOffQ;
  const uint32_t sK = sbase + L::kOffK;
  const uint32_t sV = sbase + L::kOffV;

  if (warp < 4) {
    ptx::regs_dec<kRegsControl>();
    if (warp == 0) {
      // ============================================================== TMA producer
      const bool leader = ptx::elect_one();
      const Issue<D == 128> is{leader ? 1u : 0u};
      if (leader) {
        ptx::tma_prefetch_desc(&tm_q);
        for (int c = 0; c < ch.n; ++c) {
          ptx::tma_prefetch_desc(&ch.k[c]);
          ptx::tma_prefetch_desc(&ch.v[c]);
        }
      }
      int64_t g = 0;        // global KV-tile counter (ring stage / phase)
      int64_t kq = 0;       // units with work seen so far (Q buffer phase)
      int64_t kl = 0, vl = 0, ql = 0;  // K, V, Q loads issued
      bool ok = true;
      for (int64_t k = 0; ok; ++k) {
        const int64_t u = unit_of(k, cta, grid);
        if (u >= p.n_units) break;
        const Unit w = decode_unit(p, ch, u);
        if (w.n_tiles == 0) continue;
        int j = 0;  // tile index within the unit, over all chunks
        for (int c = 0; ok && c < ch.n; ++c) {
          const int nt = chunk_tiles(p, ch, c, w);
          for (int ti = 0; ok && ti < nt; ++ti, ++j) {
            const int t = p.descending ? nt - 1 - ti : ti;
            const int64_t gj = g + j;
            const int st = static_cast<int>(gj % L::kStages);
            const uint32_t ph = static_cast<uint32_t>((gj / L::kStages) & 1);
            if (!(ok = wait_warp(b.k_empty + 8 * st, ph ^ 1, ctl, kSiteKEmpty))) break;
            is.expect_tx(b.k_full + 8 * st, L::kTileBytes);
#pragma unroll
            for (int cc = 0; cc < L::kChunks; ++cc)
              is.load(sK + st * L::kTileBytes + cc * L::kChunkBytes, &ch.k[c], w.kvh * D + cc * 64, t * kKeys,
                      b.k_full + 8 * st);
          __syncwarp();
          kl = gj + 1;
          if (j == 0) {
            // the Q buffer is free once every QK of the previous unit has completed
            if (kq > 0 && !(ok = wait_warp(b.q_empty, static_cast<uint32_t>((kq - 1) & 1), ctl, kSiteQEmpty)))
              break;
            is.expect_tx(b.q_full, 2 * L::kTileBytes);
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
              for (int cc = 0; cc < L::kChunks; ++cc)
                is.load(sQ + x * L::kTileBytes + cc * L::kChunkBytes, &tm_q, w.h * D + cc * 64,
                        static_cast<int32_t>(w.row0 + x * kRows), b.q_full);
            __syncwarp();
            ql = kq + 1;
          }
          if (!(ok = wait_warp(b.v_empty + 8 * st, ph ^ 1, ctl, kSiteVEmpty))) break;
          is.expect_tx(b.v_full + 8 * st, L::kTileBytes);
#pragma unroll
          for (int cc = 0; cc < L::kChunks; ++cc)
            is.load(sV + st * L::kTileBytes + cc * L::kChunkBytes, &ch.v[c], w.kvh * D + cc * 64, t * kKeys,
                    b.v_full + 8 * st);
          __syncwarp();
          vl = gj + 1;
          }
        }
        g += w.n_tiles;
        kq += 1;
      }
      if (*abort_flag && leader) {
        // copies in flight must land before the CTA's shared memory goes away: wait (bounded)
        // for the last load issued into every stage, and for the last Q load
        if (ql > 0) wait_drain(b.q_full, static_cast<uint32_t>((ql - 1) & 1), p.timeout_ns);
        for (int s = 0; s < L::kStages; ++s) {
          const int64_t lk = (kl - 1 - s >= 0) ? kl - 1 - ((kl - 1 - s) % L::kStages) : -1;
          if (lk >= 0) wait_drain(b.k_full + 8 * s, static_cast<uint32_t>((lk / L::kStages) & 1), p.timeout_ns);
          const int64_t lv = (vl - 1 - s >= 0) ? vl - 1 - ((vl - 1 - s) % L::kStages) : -1;
          if (lv >= 0) wait_drain(b.v_full + 8 * s, static_cast<uint32_t>((lv / L::kStages) & 1), p.timeout_ns);
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ============================================================== MMA issuer
      // The whole warp runs the loop and waits; one elected lane issues each tcgen05 instruction.
      const bool leader = ptx::elect_one();
      const Issue<D == 128> is{leader ? 1u : 0u};
      constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kRows, kKeys, 0, 0);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kRows, D, 0, 1);
      // descriptor bases (start address field counts 16-byte units)
      const uint64_t dQ0 = ptx::smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = ptx::smem_desc_sw128(sK, 16, 1024);
      const uint64_t dV0 = ptx::smem_desc_sw128(sV, L::kChunkBytes, 1024);
      constexpr uint64_t kTileUnits = L::kTileBytes >> 4;
      bool ok = true;
      if (p.test_stall && blockIdx.x == 0) ok = wait_warp(b.never, 0, ctl, kSiteTest);

      auto issue_qk = [&](int x, int st) {
        const uint64_t qd = dQ0 + x * kTileUnits;
        const uint64_t kd = dK0 + st * kTileUnits;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4);
          is.mma_ss(tmem + x * 128u, qd + off, kd + off, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int x, int st, int half, bool acc) {
        const uint64_t vd = dV0 + st * kTileUnits;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int kk = half * 4 + q;
          is.mma_ts(tmem + 256u + x * 128u, tmem + x * 128u + kk * 8, vd + static_cast<uint64_t>(kk * 128),
                    kIdescPV, (acc || kk > 0) ? 1u : 0u);
        }
      };
      // PV for Q tile x with the V tile of global step gg (stage st): first half as soon as P's
      // first 64 keys are in tensor memory.  `first` = first PV of the unit (overwrites O), which
      // waits until the previous unit's epilogue has copied O out (o_empty).
      auto pv_tile = [&](int x, int st, int64_t gg, bool first, int64_t kq) -> bool {
        if (first && kq > 0 &&
            !wait_warp(b.o_empty + 8 * x, static_cast<uint32_t>((kq - 1) & 1), ctl, kSiteOEmpty))
          return false;
        if (!wait_warp(b.p_half + 8 * x, static_cast<uint32_t>(gg & 1), ctl, kSitePFull)) return false;
        ptx::tc_fence_after();
        issue_pv(x, st, 0, !first);
        __syncwarp();
        if (!wait_warp(b.p_full + 8 * x, static_cast<uint32_t>(gg & 1), ctl, kSitePFull)) return false;
        ptx::tc_fence_after();
        issue_pv(x, st, 1, true);
        __syncwarp();
        return true;
      };

      int64_t g = 0, kq = 0;
      for (int64_t k = 0; ok; ++k) {
        const int64_t u = unit_of(k, cta, grid);
        if (u >= p.n_units) break;
        const Unit w = decode_unit(p, ch, u);
        if (w.n_tiles == 0) continue;
        if (!(ok = wait_warp(b.q_full, static_cast<uint32_t>(kq & 1), ctl, kSiteQ))) break;
        const int n = w.n_tiles;
        for (int j = 0; j < n; ++j) {
          const int64_t gj = g + j;
          const int st = static_cast<int>(gj % L::kStages);
          const uint32_t ph = static_cast<uint32_t>((gj / L::kStages) & 1);
          if (!(ok = wait_warp(b.k_full + 8 * st, ph, ctl, kSiteKFull))) break;
          ptx::tc_fence_after();
          issue_qk(0, st);
          is.commit(b.s_full);
          __syncwarp();
          if (j > 0) {
            const int pst = static_cast<int>((gj - 1) % L::kStages);
            if (!(ok = pv_tile(1, pst, gj - 1, j - 1 == 0, kq))) break;
            is.commit(b.v_empty + 8 * pst);
            __syncwarp();
          }
          issue_qk(1, st);
          is.commit(b.s_full + 8);
          is.commit(b.k_empty + 8 * st);
          if (j == n - 1) is.commit(b.q_empty);  // every QK of this unit issued
          __syncwarp();
          if (!(ok = wait_warp(b.v_full + 8 * st, ph, ctl, kSiteVFull))) break;
          if (!(ok = pv_tile(0, st, gj, j == 0, kq))) break;
          if (j == n - 1) {
            is.commit(b.o_final);
            __syncwarp();
          }
        }
        if (!ok) break;
        {
          const int64_t gl = g + n - 1;
          const int st = static_cast<int>(gl % L::kStages);
          if (!(ok = pv_tile(1, st, gl, n == 1, kq))) break;
          is.commit(b.v_empty + 8 * st);
          is.commit(b.o_final + 8);
          __syncwarp();
        }
        g += n;
        kq += 1;
      }
      if (!ok) {
        // every MMA issued so far must complete before tensor memory is released
        if (leader) {
          ptx::mma_commit(b.drain);
          wait_drain(b.drain, 0, p.timeout_ns);
        }
        __syncwarp();
      }
    }
  } else {
    ptx::regs_inc<kRegsSoftmax>();
    // ================================================================ softmax warpgroups
    const int x = (warp - 4) >> 2;           // 0: tile A, 1: tile B
    const int wq = warp & 3;                 // lane quarter of tensor memory
    const int r = wq * 32 + lane;            // row inside the tile
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + x * 128u + lane_bits;
    const uint32_t tO = tmem + 256u + x * 128u + lane_bits;
    const uint32_t stage0 = sbase + L::kOffStage + static_cast<uint32_t>(x * L::kStageBufs) * L::kChunkBytes;
    const uint32_t sw = static_cast<uint32_t>(r & 7);
    const bool store_leader = (wq == 0 && lane == 0);
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
    bool ok = true;
    bool staged = false;  // a bulk store from the staging box may still be reading it
    uint32_t nbox = 0;    // staging boxes written so far (every thread of the warpgroup counts)
    int64_t g = 0, kq = 0;

    for (int64_t k = 0;; ++k) {
      const int64_t u = unit_of(k, cta, grid);
      if (u >= p.n_units) break;
      const Unit w = decode_unit(p, ch, u);
      const int64_t tile_row0 = w.row0 + x * kRows;
      const int64_t grow = tile_row0 + r;
      float m_ref = -INFINITY;  // running maximum (log2 units of scaled scores)
      float l = 0.0f;           // running sum of 2^(x - m_ref)

      int j = 0;  // tile index within the unit, over all chunks
      for (int ci = 0; ok && ci < ch.n; ++ci) {
        const int nt = chunk_tiles(p, ch, ci, w);
        // keys of this chunk visible to my row, and the leading tiles every row of my tile sees
        // completely (keys visible to the tile's first row, whole tiles only): no mask there
        const int lim = static_cast<int>(visible_keys(p, ch, ci, grow));
        const int nomask = static_cast<int>(visible_keys(p, ch, ci, tile_row0) / kKeys);
        for (int ti = 0; ti < nt; ++ti, ++j) {
          const int t = p.descending ? nt - 1 - ti : ti;
          const int64_t gj = g + j;
          if (!(ok = wait_warp(b.s_full + 8 * x, static_cast<uint32_t>(gj & 1), ctl, kSiteSFull))) break;
          ptx::tc_fence_after();
          uint32_t sr[4][32];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) ptx::tmem_ld32(tS + cc * 32, sr[cc]);
          ptx::tmem_wait_ld();

          if (t >= nomask) {
            const int lim_local = lim - t * kKeys;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (c * 32 + e >= lim_local) sr[c][e] = __float_as_uint(-INFINITY);
          }
          // row maximum: eight independent 3-input max chains, then a small tree
          float am[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) am[q] = fmaxf(__uint_as_float(sr[0][2 * q]), __uint_as_float(sr[0][2 * q + 1]));
#pragma unroll
          for (int i = 16; i < 128; i += 16)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              am[q] = ptx::max3(am[q], __uint_as_float(sr[i >> 5][(i + 2 * q) & 31]),
                                __uint_as_float(sr[i >> 5][(i + 2 * q + 1) & 31]));
          const float mx = ptx::max3(ptx::max3(am[0], am[1], am[2]), ptx::max3(am[3], am[4], am[5]),
                                     fmaxf(am[6], am[7]));
          const float m_tile = mx * sl2;  // -inf stays -inf
          bool rescale = false;
          float factor = 1.0f;
          if (m_ref == -INFINITY) {
            m_ref = m_tile;  // first visible keys: O and l are still zero
          } else if (m_tile > m_ref + kRescaleThreshold) {
            rescale = true;
            factor = ptx::ex2(m_ref - m_tile);
            m_ref = m_tile;
            l *= factor;
          }
          if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              ptx::tmem_ld32(tO + c * 32, o);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
              ptx::tmem_st32(tO + c * 32, o);
            }
          }
          const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;
          const uint64_t negm2 = ptx::f2_pack(-m_use, -m_use);
          uint64_t sum_a = ptx::f2_pack(0.0f, 0.0f), sum_b = sum_a;
          // keys 0..63: P released early so the PV product can start on them
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
            exp_pack32(sr[c], sl2x2, negm2, pk, sum_a, sum_b);
            ptx::tmem_st16(tS + c * 16, pk);
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(b.p_half + 8 * x);
          // keys 64..127
#pragma unroll
          for (int c = 2; c < 4; ++c) {
            uint32_t pk[16];
            exp_pack32(sr[c], sl2x2, negm2, pk, sum_a, sum_b);
            ptx::tmem_st16(tS + c * 16, pk);
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(b.p_full + 8 * x);
          float s0, s1, s2, s3;
          ptx::f2_unpack(sum_a, s0, s1);
          ptx::f2_unpack(sum_b, s2, s3);
          l += (s0 + s1) + (s2 + s3);
        }
      }

      // -------------------------------------------------------------- epilogue of the unit
      if (ok && w.n_tiles > 0)
        ok = wait_warp(b.o_final + 8 * x, static_cast<uint32_t>(kq & 1), ctl, kSiteOFinal);
      // every warp of the warpgroup arrives here exactly once per unit; the staging barriers
      // below are entered only if all four warps finished the unit and saw its final O
      if (!(ok = ptx::named_bar_and(1 + x, 128, ok))) break;
      // O into registers, then tensor memory goes back to the MMA warp for the next unit
      uint32_t o[D / 32][32];
      if (w.n_tiles > 0) {
        ptx::tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(tO + c * 32, o[c]);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b.o_empty + 8 * x);
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) o[c][e] = 0u;
      }
      const bool has = (m_ref != -INFINITY) && (l > 0.0f);
      const float inv = has ? 1.0f / l : 0.0f;
      const int boxes = p.o_bf16 ? L::kBoxesBf16 : L::kBoxesF32;
      for (int c = 0; c < boxes; ++c) {
        // boxes rotate through the staging buffers across units (one bulk group per box), so the
        // box is reusable once the bulk store kStageBufs boxes back has finished reading it
        const uint32_t stage = stage0 + (nbox % L::kStageBufs) * L::kChunkBytes;
        const uint32_t row_addr = stage + static_cast<uint32_t>(r) * 128u;
        ++nbox;
        if (staged && store_leader) {
          if (L::kStageBufs == 2)
            ptx::bulk_wait_read<1>();
          else
            ptx::bulk_wait_read_all();
        }
        ptx::named_bar_sync(1 + x, 128);
        if (p.o_bf16) {
          // box = 64 bf16 columns = O chunks 2c, 2c+1; 16-byte chunk q holds columns 8q..8q+7
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t* src = &o[0][0] + (2 * c) * 32 + 8 * q;
            const uint32_t a = row_addr + ((static_cast<uint32_t>(q) ^ sw) << 4);
            const uint32_t w0 = ptx::pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv);
            const uint32_t w1 = ptx::pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
            const uint32_t w2 = ptx::pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv);
            const uint32_t w3 = ptx::pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                         : "memory");
          }
        } else {
          // box = 32 fp32 columns = O chunk c; 16-byte chunk q holds columns 4q..4q+3
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t* src = &o[0][0] + c * 32 + 4 * q;
            const uint32_t a = row_addr + ((static_cast<uint32_t>(q) ^ sw) << 4);
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                         "f"(__uint_as_float(src[0]) * inv), "f"(__uint_as_float(src[1]) * inv),
                         "f"(__uint_as_float(src[2]) * inv), "f"(__uint_as_float(src[3]) * inv)
                         : "memory");
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::named_bar_sync(1 + x, 128);
        if (store_leader) {
          const int box_cols = p.o_bf16 ? 64 : 32;
          ptx::tma_store_2d(&tm_o, stage, w.h * D + c * box_cols, static_cast<int32_t>(tile_row0));
          ptx::bulk_commit();
        }
        staged = true;
      }
      if (grow < p.sq)
        p.lse[grow * p.hq + w.h] = has ? (m_ref * 0.69314718055994531f + logf(l)) : -INFINITY;
      g += w.n_tiles;
      if (w.n_tiles > 0) kq += 1;
    }
    if (store_leader) ptx::bulk_wait_all();  // the last bulk stores must complete
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// O = 0, LSE = -inf for every row (no chunk holds a key).
__global__ void fill_empty_kernel(void* o, int o_bf16, float* lse, int64_t rows, int64_t row_elems) {
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t n = rows * row_elems;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += step) {
    if (o_bf16)
      static_cast<__nv_bfloat16*>(o)[i] = __float2bfloat16(0.0f);
    else
      static_cast<float*>(o)[i] = 0.0f;
    if (i < rows) lse[i] = -INFINITY;
  }
}

// 2-D map over a token-major tensor viewed as [tokens, heads*d]; box = 128 bytes of columns x
// 128 rows with 128-byte swizzle (bf16 operands: the canonical K-major / MN-major UMMA layout;
// the output: the staging layout of the epilogue).
bool make_map(CUtensorMap* m, const void* base, int64_t tokens, int64_t row_elems, bool fp32 = false) {
  return encode_map_2d(m, base, tokens, row_elems, fp32, 128);
}

template <int D, int MAXC>
cp_status launch_tc(const TcParams& p, const CUtensorMap& mq, const CUtensorMap& mo, const cp_attn_desc& d,
                    const cp_kv_chunk* chunks, int n, int64_t grid, cudaStream_t s) {
  ChunkTable<MAXC> ch;
  memset(&ch, 0, sizeof(ch));
  ch.n = n;
  for (int c = 0; c < n; ++c) {
    if (!make_map(&ch.k[c], chunks[c].k, chunks[c].skv, int64_t(d.hkv) * d.d) ||
        !make_map(&ch.v[c], chunks[c].v, chunks[c].skv, int64_t(d.hkv) * d.d)) {
      set_error("cuTensorMapEncodeTiled failed for chunk %d (or the driver entry point is unavailable)", c);
      return CP_ERR_CUDA;
    }
    ch.skv[c] = chunks[c].skv;
    ch.base[c] = chunks[c].kv_pos.base;
    ch.stride[c] = chunks[c].kv_pos.stride;
  }
  constexpr int smem = Layout<D>::kSmemLaunch;
  cudaError_t e =
      cudaFuncSetAttribute(attn_tc_kernel<D, MAXC>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attn_tc_kernel)");
  attn_tc_kernel<D, MAXC><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(p, mq, mo, ch);
  e = cudaGetLastError();
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "attn_tc_kernel launch");
}

template <int D>
cp_status launch_tc_chunks(const TcParams& p, const CUtensorMap& mq, const CUtensorMap& mo, const cp_attn_desc& d,
                           const cp_kv_chunk* chunks, int n, int64_t grid, cudaStream_t s) {
  // the chunk table travels in the kernel parameters: size it to the call
  if (n <= 1) return launch_tc<D, 1>(p, mq, mo, d, chunks, n, grid, s);
  if (n <= 8) return launch_tc<D, 8>(p, mq, mo, d, chunks, n, grid, s);
  return launch_tc<D, CP_MAX_CHUNKS>(p, mq, mo, d, chunks, n, grid, s);
}

}  // namespace

cp_status launch_fill_empty(const cp_attn_desc& d, cudaStream_t s) {
  const int64_t n = d.sq * d.hq * d.d;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  fill_empty_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(d.o, d.o_dtype == CP_BF16, d.lse, d.sq * d.hq,
                                                                   d.d);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "fill_empty_kernel launch");
}

cp_status launch_partial_attn_tc(const cp_attn_desc& d, const cp_kv_chunk* chunks, int n, float scale,
                                 int64_t timeout_ns, int num_sms, cudaStream_t s) {
  TcParams p;
  p.o = d.o;
  p.lse = d.lse;
  p.status = d.status;
  p.sq = d.sq;
  p.hq = d.hq;
  p.hkv = d.hkv;
  p.group = d.hq / d.hkv;
  p.n_pairs = static_cast<int32_t>((d.sq + 2 * kRows - 1) / (2 * kRows));
  p.causal = d.causal;
  p.o_bf16 = d.o_dtype == CP_BF16;
  p.descending = (d.flags & CP_FLAG_KV_DESCENDING) ? 1 : 0;
  p.test_stall = (d.flags & CP_FLAG_TEST_STALL) ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q_base = d.q_pos.base;
  p.q_stride = d.q_pos.stride;
  p.timeout_ns = timeout_ns;
  CUtensorMap mq, mo;
  if (!make_map(&mq, d.q, d.sq, int64_t(d.hq) * d.d) ||
      !make_map(&mo, d.o, d.sq, int64_t(d.hq) * d.d, d.o_dtype == CP_F32)) {
    set_error("cuTensorMapEncodeTiled failed (or the driver entry point is unavailable)");
    return CP_ERR_CUDA;
  }
  p.n_units = static_cast<int64_t>(p.n_pairs) * d.hq;
  // persistent: one CTA per SM (shared memory use keeps it at one), never more CTAs than units
  const int64_t grid = p.n_units < num_sms ? p.n_units : num_sms;
  if (d.d == 64) return launch_tc_chunks<64>(p, mq, mo, d, chunks, n, grid, s);
  return launch_tc_chunks<128>(p, mq, mo, d, chunks, n, grid, s);
}

}  // namespace cpattn
