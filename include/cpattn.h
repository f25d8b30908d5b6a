/*
 * cpattn.h -- C ABI of the per-rank context-parallel (CP) attention library (libcpattn.so).
 *
 * One CP rank's attention work on one GPU: which global token positions a rank holds, blockwise
 * attention of the rank's query shard against one KV chunk at a time (chunks may arrive in any
 * order) producing an (O, LSE) partial, the order-independent merge of partials into exact
 * softmax attention, and the Ulysses sequence <-> head reshard.  CP ranks are logical shards;
 * nothing here communicates between processes or GPUs.
 *
 * Sources (pages cited by title and section):
 *   [FCP]     "FCP: from a fixed ring to a free topology" (lqnn.cn/news/264049)
 *   [PCP/DCP] "PCP and DCP sequence parallelism guide" (hmyw.cn/news/122838)
 *   [ZigZag]  "Zig-Zag Ring Attention" article (intelliparadigm.com, article 2133809)
 *   [Halo]    "Halo context parallelism (CP + Ulysses attention)" (sheratonhq.com/news/191935)
 *
 * Conventions shared by every call:
 *   - Tensors are token-major, batch 1: [tokens, heads, head_dim], contiguous, head_dim fastest.
 *   - Global positions are affine per shard: pos(i) = base + stride * i, stride >= 1.
 *   - All device pointers are caller-owned device memory; the library allocates no device memory
 *     and keeps no state between calls (one exception: the fixed workspace array behind
 *     cp_partial_attn_bwd_noalloc).  Host pointer arrays are read during the call only.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream).  Argument checks run on
 *     the host before anything is launched; a rejected call launches nothing.
 *   - On a non-OK status, cp_last_error() returns a message for the calling thread.
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CP_ABI_VERSION 4
/* Largest number of partials one cp_merge_partials call accepts. */
#define CP_MAX_PARTIALS 128

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = 1, /* rejected on the host; nothing launched                     */
  CP_ERR_UNSUPPORTED = 2, /* device is not sm_103 (GB300) or the shape is not supported  */
  CP_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed               */
  CP_ERR_TIMEOUT = 4      /* a bounded in-kernel wait expired (reported via *status)     */
} cp_status;

typedef enum {
  CP_LAYOUT_CONTIGUOUS = 0, /* one block of seq_len/cp tokens per rank                       */
  CP_LAYOUT_STRIDED = 1,    /* every cp-th token ("zig-zag" on the pages)                    */
  CP_LAYOUT_TWO_BLOCK = 2,  /* blocks r and 2cp-1-r of seq_len/(2cp) tokens (two segments)   */
  CP_LAYOUT_BALANCED = 3    /* contiguous blocks of equal causal work (unequal token counts) */
} cp_layout;

/* Most affine segments a shard layout has (cp_shard_segments). */
#define CP_MAX_SEGMENTS 2
typedef enum { CP_F32 = 0, CP_BF16 = 1 } cp_dtype;

/* Global position of local token i: base + stride * i. */
typedef struct {
  int64_t base;
  int64_t stride;
} cp_posmap;

/*
 * cp_shard_layout -- which global tokens rank `rank` of `cp` holds.
 *   [PCP/DCP] section 3.5 (split_sequence_for_cp): contiguous block starting at rank*seq_len/cp,
 *             seq_len must divide by cp; positions stay global.
 *   [ZigZag]  section 4.2: strided assignment, rank r holds r, r+cp, r+2cp, ...
 * Arguments:
 *   seq_len, cp, rank   sequence length (> 0), CP size (> 0), rank in [0, cp).
 *   kind                CP_LAYOUT_CONTIGUOUS (base = rank*seq_len/cp, stride 1) or
 *                       CP_LAYOUT_STRIDED    (base = rank,             stride cp).
 *   map_out             host pointer, required: receives the affine map.
 *   dev_positions_out   device int32 [seq_len/cp] or NULL; filled with pos(i) on `stream`
 *                       (requires seq_len <= INT32_MAX).
 * Errors: CP_ERR_INVALID_ARG when seq_len % cp != 0, rank out of range, map_out NULL, or an
 *         unknown kind.  CP_ERR_CUDA if the fill kernel fails to launch.
 */
cp_status cp_shard_layout(int64_t seq_len, int32_t cp, int32_t rank, int32_t kind,
                          cp_posmap* map_out, int32_t* dev_positions_out, cudaStream_t stream);

/*
 * cp_shard_segments -- the same question for any layout, answered as a list of affine segments
 * in local order (local tokens [0, lens[0]) follow maps[0], the next lens[1] follow maps[1]).
 *   CP_LAYOUT_CONTIGUOUS, CP_LAYOUT_STRIDED: one segment, the cp_shard_layout map.
 *   CP_LAYOUT_TWO_BLOCK: [ZigZag] sections 4.2 / 5.2 give the aim of the zig-zag split (every
 *     rank gets early and late tokens, so causal work is even); this is its block-granular form,
 *     which the pages do not print: 2*cp blocks of b = seq_len/(2cp) tokens, rank r holds block r
 *     then block 2cp-1-r -- maps {r*b, 1} and {(2cp-1-r)*b, 1}, b tokens each.  Every rank then
 *     sees exactly b*b*(2cp-1) + b*(b+1) causal pairs.  Needs seq_len % (2*cp) == 0.
 *   CP_LAYOUT_BALANCED: [PCP/DCP] section 2.3 (load balancing): an even split by tokens leaves
 *     causal work uneven; DCP splits by the work instead.  Reading taken: contiguous blocks of
 *     equal causal work at token granularity -- with W(b) = b(b+1)/2, rank r holds [b_r, b_r+1)
 *     where b_r is the smallest b with W(b) >= r*W(seq_len)/cp (b_0 = 0, b_cp = seq_len).  One
 *     segment per rank, lengths differ between ranks; seq_len need not divide by cp, but every
 *     rank must get at least one token.
 * Arguments:
 *   seq_len, cp, rank, kind   as cp_shard_layout.
 *   maps_out, lens_out        host arrays [CP_MAX_SEGMENTS], required; entries past the count
 *                             are left untouched.
 *   n_segments_out            host pointer, required: 1 or 2.
 *   dev_positions_out         device int32 [sum of lens] (seq_len/cp except for the balanced
 *                             split) or NULL: every local token's position, written on `stream`
 *                             (requires seq_len <= INT32_MAX).
 * Errors: CP_ERR_INVALID_ARG as cp_shard_layout (and seq_len % (2cp) != 0 for the two-block
 *         split, a rank left without tokens for the balanced one); CP_ERR_CUDA if the fill
 *         kernel fails to launch.
 * cp_shard_layout rejects CP_LAYOUT_TWO_BLOCK and CP_LAYOUT_BALANCED (not one map of
 * seq_len/cp tokens).  cp_ulysses_reshard needs equal shards and rejects CP_LAYOUT_BALANCED.
 */
cp_status cp_shard_segments(int64_t seq_len, int32_t cp, int32_t rank, int32_t kind,
                            cp_posmap* maps_out, int64_t* lens_out, int32_t* n_segments_out,
                            int32_t* dev_positions_out, cudaStream_t stream);

/* Flags for cp_attn_desc.flags. */
#define CP_FLAG_KV_DESCENDING 0x1 /* visit the chunk's KV tiles last-to-first (same result)   */
#define CP_FLAG_TEST_STALL 0x100  /* test only: block 0 waits on a barrier nobody arrives on; */
                                  /* its bounded wait expires, *status gets CP_ERR_TIMEOUT.   */

/*
 * Partial attention of one query shard against one KV chunk.
 *   [FCP] section 3.3: scores = q . k^T / sqrt(head_dim); running max and running sum with
 *   online-softmax rescaling over KV blocks; output = acc / running_sum.  The result does not
 *   depend on the order in which chunks (or the tiles inside a chunk) are visited.
 * Output is the normalised partial: O = softmax-weighted sum of the chunk's visible V rows and
 * LSE = natural-log sum of exp(scores) over those keys.  A query row with no visible key in the
 * chunk gets O = 0 and LSE = -inf.
 * Fields:
 *   q         device [sq, hq, d]  (in_dtype)
 *   k, v      device [skv, hkv, d] (in_dtype)
 *   in_dtype  CP_F32 (fp32 CUDA-core path) or CP_BF16 (tensor-core path, fp32 accumulation)
 *   o         device [sq, hq, d]  (o_dtype: CP_F32, or CP_BF16 when this partial is final)
 *   lse       device fp32 [sq, hq]
 *   sq, skv   token counts (>= 0); hq, hkv head counts, hq % hkv == 0; Q head h reads KV head
 *             h / (hq/hkv) ([Halo] native GQA, contiguous groups).  d in {64, 128}.
 *   causal    1: key visible iff kv_pos(j) <= q_pos(i) (global positions, self included)
 *   scale     softmax scale; 0 means 1/sqrt(d)
 *   q_pos, kv_pos  affine position maps of the query shard and of the chunk
 *   status    device int32 or NULL: set to CP_ERR_TIMEOUT | (site << 8) if a bounded wait
 *             inside the kernel expires (the kernel then returns early; outputs undefined).
 *             The caller zeroes it; read it after synchronising.
 *   flags     CP_FLAG_* bits
 *   wait_timeout_ms  limit of each in-kernel wait; 0 means 2000 ms
 * Positions: base >= 0, stride >= 1, and every global position of the shard and of the chunk
 * below 2e9 (a checked limit that keeps positions within the int32 position arrays of the layout
 * calls; far beyond any sequence length).
 * Errors: CP_ERR_INVALID_ARG (null pointers, d not 64/128, hq % hkv, stride < 1, negative base,
 * positions at or above 2e9, bad dtype, pointers not 16-byte aligned), CP_ERR_UNSUPPORTED
 * (device not sm_103), CP_ERR_CUDA.
 */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  int32_t in_dtype;
  int32_t o_dtype;
  void* o;
  float* lse;
  int64_t sq;
  int64_t skv;
  int32_t hq;
  int32_t hkv;
  int32_t d;
  int32_t causal;
  float scale;
  int32_t flags;
  cp_posmap q_pos;
  cp_posmap kv_pos;
  int32_t* status;
  int32_t wait_timeout_ms;
  int32_t reserved;
} cp_attn_desc;

cp_status cp_partial_attn(const cp_attn_desc* desc, cudaStream_t stream);

/* Largest number of KV chunks one cp_partial_attn_chunks call accepts. */
#define CP_MAX_CHUNKS 64

/* One KV chunk for cp_partial_attn_chunks: device [skv, hkv, d] K and V (in_dtype of the
 * descriptor) and the global positions of its tokens. */
typedef struct {
  const void* k;
  const void* v;
  int64_t skv;
  cp_posmap kv_pos;
} cp_kv_chunk;

/*
 * Attention of one query shard against a list of KV chunks, consumed in the given (arrival)
 * order inside one launch, with the running maximum, running sum and accumulator carried from
 * chunk to chunk.
 *   [FCP] section 3.3: each arriving KV block updates the running max and running sum of every
 *   local query block; the result equals attention over the union of the blocks whatever their
 *   order.  Equivalent to one cp_partial_attn per chunk followed by cp_merge_partials, without
 *   writing or re-reading the per-chunk partials.
 * desc supplies q, o, lse, sq, hq, hkv, d, causal, scale, q_pos, in_dtype, o_dtype, flags,
 * status and wait_timeout_ms exactly as for cp_partial_attn; its k, v, skv and kv_pos are
 * ignored.  o/lse receive the (O, LSE) over the union of the chunks' keys (O = 0, LSE = -inf for
 * rows that see no key).
 * Arguments:
 *   n_chunks   1 <= n_chunks <= CP_MAX_CHUNKS
 *   chunks     host array [n_chunks], read during the call
 * Errors: as cp_partial_attn, plus CP_ERR_INVALID_ARG for a bad chunk (null pointer with
 * skv > 0, misaligned pointer, stride < 1, negative base or skv).
 */
cp_status cp_partial_attn_chunks(const cp_attn_desc* desc, int32_t n_chunks, const cp_kv_chunk* chunks,
                                 cudaStream_t stream);

/*
 * Merge n partials of the same query rows into exact attention.
 *   [PCP/DCP] sections 2.3 and 4.2 (global_softmax): global max first, then exponentials
 *   against it and their global sum, then normalise.  In (O, LSE) form:
 *     M = max_i LSE_i;  w_i = exp(LSE_i - M);  O = sum_i w_i O_i / sum_i w_i;
 *     LSE = M + ln sum_i w_i.
 *   A partial with LSE_i = -inf contributes nothing and its O_i row is not read; if all are
 *   -inf the result is O = 0, LSE = -inf.  The result does not depend on the order of parts.
 * Arguments:
 *   n          1 <= n <= CP_MAX_PARTIALS
 *   o_parts    host array of n device pointers, each fp32 [sq, h, d]
 *   lse_parts  host array of n device pointers, each fp32 [sq, h]
 *   sq, h, d   rows, heads, head_dim (d in {32, 64, 128, 256})
 *   o_out      device [sq, h, d] in out_dtype (CP_F32 or CP_BF16, round-to-nearest-even)
 *   lse_out    device fp32 [sq, h], or NULL to skip
 * Errors: CP_ERR_INVALID_ARG (n out of range, null or unaligned pointers, bad sizes),
 *         CP_ERR_CUDA.
 */
cp_status cp_merge_partials(int32_t n, const float* const* o_parts, const float* const* lse_parts,
                            int64_t sq, int32_t h, int32_t d, void* o_out, int32_t out_dtype,
                            float* lse_out, cudaStream_t stream);

/*
 * Ulysses reshard between sequence-sharded and head-sharded layouts, as a local permutation.
 *   [Halo] "Ulysses attention": each rank holds S/cp tokens of all heads; the exchange gives
 *   rank r all S tokens of heads [r*H/cp, (r+1)*H/cp); Q once, fused K|V once, O back.
 *     dir 0 (seq -> head): out[t*cp + r][pos_s(i), j, :] = in[t*cp + s][i, r*H_t/cp + j, :]
 *     dir 1 (head -> seq): out[t*cp + s][i, r*H_t/cp + j, :] = in[t*cp + r][pos_s(i), j, :]
 *   where pos_s is shard s's layout (cp_shard_layout) and t indexes the tensors of one call.
 * Arguments:
 *   dir        0 or 1
 *   cp         number of ranks, 1 <= cp <= 64; seq_len % cp == 0
 *   n_tensors  1..4 tensors moved in one launch (e.g. 2 for fused K|V)
 *   heads      host array [n_tensors]: full head count H_t of each tensor; H_t % cp == 0
 *   d          head_dim; (H_t/cp) * d * sizeof(dtype) must be a multiple of 16 bytes
 *   dtype      CP_F32 or CP_BF16
 *   layout     cp_layout of the sequence shards (CP_LAYOUT_TWO_BLOCK needs seq_len % (2cp) == 0)
 *   in, out    host arrays [n_tensors*cp] of device pointers (16-byte aligned), shapes above
 * Bit-exact copy.  Errors: CP_ERR_INVALID_ARG, CP_ERR_CUDA.
 */
cp_status cp_ulysses_reshard(int32_t dir, int32_t cp, int64_t seq_len, int32_t n_tensors,
                             const int32_t* heads, int32_t d, int32_t dtype, int32_t layout,
                             const void* const* in, void* const* out, cudaStream_t stream);

/*
 * ---------------------------------------------------------------- backward pass
 * [PCP/DCP] section 2.3 (gradient handling): in training the gradients of the split sequence
 * are split the same way and reduce-scattered across ranks; [Halo] (Ulysses): the backward pass
 * runs the same exchanges in reverse.  What is differentiated is the partial attention above.
 * For one (query shard, KV chunk) pair and one head, with the rows' FINAL (merged over every
 * chunk) output O and LSE:
 *     P_ij   = exp(scale * q_i . k_j - LSE_i)   visible pairs only; 0 when LSE_i = -inf
 *     D_i    = dO_i . O_i                        (cp_attn_bwd_prep)
 *     dV_j  += sum_i P_ij dO_i
 *     dS_ij  = P_ij (dO_i . v_j - D_i)
 *     dQ_i  += scale * sum_j dS_ij k_j
 *     dK_j  += scale * sum_i dS_ij q_i
 * A KV head's dK, dV sum over the Q heads of its group.  Summing dQ over a shard's chunks, and
 * a chunk's dK, dV over every query shard that saw it (the pages' reduce-scatter, here a plain
 * accumulation into the chunk owner's buffers), gives the gradients of unsharded attention.
 */

/* Floats of the per-row workspace cp_attn_bwd_prep writes for a query shard of sq rows, hq heads:
 * [2][hq][sq rounded up to 128]. */
#define CP_BWD_AUX_FLOATS(sq, hq) (2 * (int64_t)(hq) * ((((int64_t)(sq)) + 127) / 128 * 128))

/*
 * cp_attn_bwd_prep -- per query row and head, once per shard before its backward calls:
 *   aux[0][h][i] = -LSE_ih * log2(e)  (-inf where LSE_ih = -inf: the row has no P)
 *   aux[1][h][i] = -D_ih = -(dO_ih . O_ih)
 * and -inf / 0 in the padding rows [sq, round_up(sq, 128)).
 * Arguments:
 *   o        device [sq, hq, d] final output of the shard (o_dtype CP_F32 or CP_BF16)
 *   d_o      device [sq, hq, d] gradient of the loss w.r.t. that output (do_dtype CP_F32/CP_BF16)
 *   lse      device fp32 [sq, hq] final LSE (natural log)
 *   sq >= 0, hq >= 1, d in {64, 128}
 *   aux      device fp32 [CP_BWD_AUX_FLOATS(sq, hq)], 16-byte aligned (caller-owned)
 * Errors: CP_ERR_INVALID_ARG (null or misaligned pointers, bad sizes or dtypes),
 *         CP_ERR_UNSUPPORTED, CP_ERR_CUDA.
 */
cp_status cp_attn_bwd_prep(const void* o, int32_t o_dtype, const void* d_o, int32_t do_dtype,
                           const float* lse, int64_t sq, int32_t hq, int32_t d, float* aux,
                           cudaStream_t stream);

/*
 * Backward of one (query shard, KV chunk) partial: ACCUMULATES (+=) the pair's share into
 * dq [sq, hq, d], dk and dv [skv, hkv, d] (fp32, caller-owned, zeroed by the caller before the
 * first call).  Fields as cp_attn_desc where the names match; also:
 *   d_o       device [sq, hq, d], in_dtype (bf16: tensor-core path; fp32: CUDA-core path)
 *   aux       the shard's cp_attn_bwd_prep output
 *   dq, dk, dv  device fp32, 16-byte aligned
 *   status, wait_timeout_ms  as cp_attn_desc (bounded in-kernel waits of the tensor-core path)
 *   flags     0, or CP_FLAG_TEST_STALL (bf16 only; same meaning as for cp_attn_desc)
 * Within one call dq, dk, dv are updated with atomic reductions (bf16 path) or by exclusive
 * owners (fp32 path); calls on one stream follow stream order.  The summation order of dq and
 * of a GQA group's dk, dv is not fixed on the bf16 path.
 * Positions as cp_partial_attn (every global position below 2e9).
 * Errors: CP_ERR_INVALID_ARG, CP_ERR_UNSUPPORTED, CP_ERR_CUDA.
 */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  const void* d_o;
  int32_t in_dtype;
  int32_t flags;
  const float* aux;
  float* dq;
  float* dk;
  float* dv;
  int64_t sq;
  int64_t skv;
  int32_t hq;
  int32_t hkv;
  int32_t d;
  int32_t causal;
  float scale;
  int32_t wait_timeout_ms;
  cp_posmap q_pos;
  cp_posmap kv_pos;
  int32_t* status;
} cp_attn_bwd_desc;

cp_status cp_partial_attn_bwd(const cp_attn_bwd_desc* desc, cudaStream_t stream);

/* One KV chunk for cp_partial_attn_bwd_chunks: device K, V [skv, hkv, d] (in_dtype), the chunk's
 * gradient buffers dK, dV [skv, hkv, d] (fp32, accumulated), and its global positions. */
typedef struct {
  const void* k;
  const void* v;
  float* dk;
  float* dv;
  int64_t skv;
  cp_posmap kv_pos;
} cp_kv_bwd_chunk;

/*
 * The backward of one query shard against a list of KV chunks in one call (f1's counterpart):
 * the same as one cp_partial_attn_bwd per chunk (desc's k, v, dk, dv, skv and kv_pos are
 * ignored), with the chunks' work dealt out in one persistent launch per 32 chunks.  The order of
 * the chunks does not matter (each adds its own share).  n_chunks in [1, CP_MAX_CHUNKS].
 * Errors: as cp_partial_attn_bwd, per chunk.
 */
cp_status cp_partial_attn_bwd_chunks(const cp_attn_bwd_desc* desc, int32_t n_chunks,
                                     const cp_kv_bwd_chunk* chunks, cudaStream_t stream);

/* Largest workspace (floats) cp_partial_attn_bwd_noalloc can use: CP_BWD_AUX_FLOATS(sq, hq) must
 * not exceed it (16 MiB; e.g. 32768 rows x 64 heads, or 131072 rows x 16 heads). */
#define CP_NOALLOC_AUX_MAX_FLOATS ((int64_t)4194304)

/*
 * cp_partial_attn_bwd_noalloc -- cp_attn_bwd_prep followed by cp_partial_attn_bwd for one
 * (query shard, KV chunk) pair, with the per-row workspace held in the library's own device
 * memory, so that the call allocates nothing.  The pages have no counterpart: this exists for
 * callers that cannot allocate device memory themselves (a runtime that forbids cudaMalloc after
 * start-up, code that runs inside a memory pool it does not own, a hook that is handed only its
 * inputs and outputs).
 * Arguments:
 *   desc      as cp_partial_attn_bwd, except that desc->aux must be NULL; d_o is read with
 *             desc->in_dtype by both steps
 *   o, o_dtype, lse  as cp_attn_bwd_prep: the shard's final output and LSE
 * dq, dk, dv are ACCUMULATED exactly as by cp_partial_attn_bwd (the caller zeroes them before the
 * first call); nothing else needs to start at zero.
 * The workspace is one fixed array of CP_NOALLOC_AUX_MAX_FLOATS floats per device, held by every
 * device that loads the library until the process exits.  The first call on a device (with that
 * device current) looks up the array's device address; under CUDA's lazy module loading that
 * lookup is also where the 16 MiB are placed in device memory, so it can fail with
 * CP_ERR_CUDA (out of memory) inside a pool that owns all device memory: make that first call at
 * start-up, before such a pool takes the memory and before any stream capture.  The address is
 * cached per device with the identity of its CUDA context; after a cudaDeviceReset the next call
 * looks it up again (and the array is placed again).  Every call shares the array and leaves its contents behind: calls that may overlap on
 * the GPU (different streams, or different host threads, without ordering between them) race on
 * it and give wrong gradients.  Calls on one stream are ordered and safe.
 * No cudaMalloc, cudaFree or other allocating call is made.
 * Errors: CP_ERR_INVALID_ARG (desc NULL, desc->aux not NULL, CP_BWD_AUX_FLOATS(sq, hq) above
 * CP_NOALLOC_AUX_MAX_FLOATS, and everything cp_attn_bwd_prep and cp_partial_attn_bwd reject),
 * CP_ERR_UNSUPPORTED, CP_ERR_CUDA.
 */
cp_status cp_partial_attn_bwd_noalloc(const cp_attn_bwd_desc* desc, const void* o, int32_t o_dtype,
                                      const float* lse, cudaStream_t stream);

/* Message for the calling thread's last non-OK status ("" if none).  Valid until the next call. */
const char* cp_last_error(void);

/* CP_ABI_VERSION of the loaded library. */
int32_t cp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */
