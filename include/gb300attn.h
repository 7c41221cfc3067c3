/*
 * gb300attn — exact packed-THD attention hot path for one GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only.  Unless stated otherwise every
 * pointer is a DEVICE pointer owned by the caller; the library allocates no
 * device memory and keeps no state between calls.  Every call validates its
 * arguments on the host first and returns ATTN_ERR_INVALID_ARG /
 * ATTN_ERR_UNSUPPORTED without launching anything; otherwise it enqueues its
 * kernels asynchronously on `stream` and returns ATTN_OK (or ATTN_ERR_CUDA if
 * a launch failed).  Nothing synchronises implicitly except
 * attn_read_device_status.
 *
 * Notation (pages: "Context parallelism and ring attention", sections "The
 * attention problem", "Online softmax", "Causal attention", "Load balance";
 * "JAX: Context-Parallel Attention with TransformerEngine", sections 1
 * "Packed THD inputs", 3 "Fused attention call", 4 "Striped load balancing
 * and sharding"; "Implementation:NVIDIA TransformerEngine JAX Cpp
 * Attention", "I/O Contract"):
 *
 *   q            bf16 [b, s_q, h_q, d]   contiguous ("THD" separate-QKV layout)
 *   k, v         bf16 [b, s_kv, h_kv, d] contiguous
 *   segment ids  int32 [b, s]   0 = padding slot, >0 = segment id
 *   segment pos  int32 [b, s]   position of the token inside its segment
 *   visible(i,j) <=> ids_q[i] == ids_kv[j] != 0 and pos_kv[j] <= pos_q[i]
 *                    and (window_left < 0 or pos_q[i] - pos_kv[j] <= window_left)
 *   out          O = softmax(scale * Q K^T + M) V   per head, M = 0 / -inf
 *   lse          fp32 [b, h_q, s_q], natural log of the softmax denominator
 *                including the scale; rows with no visible key: O = 0, lse = -inf
 *   GQA          query head h reads kv head h / (h_q / h_kv)
 */
#ifndef GB300ATTN_H
#define GB300ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GB300ATTN_API __attribute__((visibility("default")))
#else
#define GB300ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* == cudaStream_t; NULL = legacy default stream */

enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or flag; nothing launched */
  ATTN_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. d not in {64,128,256}) */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed */
  ATTN_ERR_TIMEOUT = 4      /* a device-side bounded wait gave up (see attn_read_device_status) */
};

enum { ATTN_REORDER_DUAL_CHUNK = 0, ATTN_REORDER_STRIPED = 1 };

/* Forward attention parameters.
 * Page: "Context parallelism and ring attention", section "The attention
 * problem" (O = softmax(QK^T/sqrt(H) + M) V); TE tutorial section 3 (packed
 * THD, PADDING_CAUSAL mask, window (left, 0), scaling_factor); TE Cpp
 * Attention page, "I/O Contract" (outputs: output, softmax_aux).
 *
 *  q, k, v        bf16, layouts above; 16-byte aligned base pointers.
 *  q_segment_ids, q_segment_pos    int32 [b, s_q]
 *  kv_segment_ids, kv_segment_pos  int32 [b, s_kv]  (may alias the q ones)
 *  b, s_q, s_kv, h_q, h_kv, d      sizes; h_q % h_kv == 0; d in {64, 128, 256}
 *                                  (forward and backward); d is the head
 *                                  dim of q and k, and of v unless d_v says
 *                                  otherwise;
 *                                  s_q, s_kv >= 1 (ragged lengths allowed)
 *  window_left    -1 = unlimited, else >= 0 (inclusive, W+1 keys incl. self)
 *  window_right   must be 0 (causal)
 *  scale          softmax scale, usually 1/sqrt(d)
 *  out            bf16 [b, s_q, h_q, d_v], or fp32 when out_fp32 != 0
 *  lse            fp32 [b, h_q, s_q]
 *  workspace      device scratch of at least attn_fwd_workspace_bytes() bytes,
 *                 256-byte aligned; contents need no initialisation and are
 *                 overwritten (the tile plan and the device status word).
 *  merge_into_out 0: out / lse receive this call's result.
 *                 1: out (fp32; out_fp32 must be 1) and lse hold a finished
 *                 partial (O_acc, LSE_acc) of the same query rows over other
 *                 key blocks; the kernel's epilogue folds this call's result
 *                 (O_blk, LSE_blk) into it with exactly the merge of
 *                 attn_merge_partial below ("Context parallelism and ring
 *                 attention", section "Online softmax"), so a ring step needs
 *                 no separate merge pass over HBM.  lse is updated; out is
 *                 updated unless out_final is given.  A row whose LSE_acc is
 *                 -inf takes the block as is (its out value is ignored).
 *  out_final      NULL, or (merge_into_out only) bf16 [b, s_q, h_q, d_v]: the
 *                 merged O goes there, rounded to bf16 (RNE), instead of into
 *                 out (the last ring step).  Must not overlap out.
 *  kv_token_stride  elements between consecutive tokens of k and of v (and of
 *                 dk / dv in the backward); 0 = h_kv * d (contiguous).  The
 *                 packed K/V layout of the TE tutorial (section 1, THD_T2HD:
 *                 kv [b, s_kv, 2, h_kv, d]) is k = kv, v = kv + h_kv * d,
 *                 kv_token_stride = 2 * h_kv * d.  Must be >= h_kv * d and a
 *                 multiple of 8; batch rows are s_kv * kv_token_stride apart.
 *                 Must be 0 when d_v differs from d.
 *  d_v            head dim of v and out; 0 = d.  Other than d, only d = 192
 *                 with d_v = 128 (the MLA shape the TE tutorial's closing
 *                 section points to), forward and backward: v is then bf16
 *                 [b, s_kv, h_kv, 128], contiguous.
 */
typedef struct attn_fwd_params {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* q_segment_ids;
  const int32_t* q_segment_pos;
  const int32_t* kv_segment_ids;
  const int32_t* kv_segment_pos;
  int64_t b, s_q, s_kv, h_q, h_kv, d;
  int32_t window_left;
  int32_t window_right;
  float scale;
  int32_t out_fp32;
  void* out;
  float* lse;
  void* workspace;
  size_t workspace_bytes;
  int32_t merge_into_out;
  void* out_final;
  int64_t kv_token_stride;
  int64_t d_v;
} attn_fwd_params;

/* Backward parameters: gradient of sum(out * dout) with respect to q, k, v
 * (TE tutorial section 5 differentiates jnp.vdot(out, dout)).  The forward
 * fields mean the same as in attn_fwd_params (out_fp32 must be 0), plus:
 *  out      bf16 [b, s_q, h_q, d]  forward output (as written by attn_fwd)
 *  lse      fp32 [b, h_q, s_q]     forward LSE (as written by attn_fwd)
 *  dout     bf16 [b, s_q, h_q, d]
 *  (merge_into_out must be 0 and out_final NULL in the embedded fwd fields)
 *  dq       bf16 [b, s_q, h_q, d]     (written)
 *  dk       bf16 [b, s_kv, h_kv, d]   (written; summed over the GQA group),
 *  dv       bf16 [b, s_kv, h_kv, d_v] tokens fwd.kv_token_stride elements apart
 *           like k and v
 *  workspace  >= attn_bwd_workspace_bytes() bytes, 256-byte aligned; holds
 *             D = rowsum(dO * O), the tile plan and (fused path) the fp32 dQ
 *             accumulator.
 *  accumulate_fp32  0: dq/dk/dv are bf16 and are overwritten.
 *                   1: dq/dk/dv are fp32 and this call's gradients are ADDED to
 *                   their contents (ring context parallelism sums per-block
 *                   contributions; "Context parallelism and ring attention",
 *                   section "Ring attention").  out / lse must then be the final
 *                   forward output and LSE of the query rows (D and P use them).
 *  deterministic    0: at d = 64 / 128 one fused kernel computes dQ, dK and dV and
 *                   sums dQ over key tiles with fp32 reduce-adds into a global
 *                   accumulator, in an order the hardware schedules (the last
 *                   bits of dq may differ from run to run).
 *                   1: a dK / dV kernel and a dQ kernel; dQ of each query tile is
 *                   summed in a fixed order on chip and written once, so every
 *                   output is bit-identical from run to run (slower at d <= 128).
 *                   d = 256 and (192, 128) always take this pair.
 *  kernel_events    optional timing hook: two events (cudaEvent_t cast to
 *                   void*) that the caller created, or both NULL.  attn_bwd then
 *                   records kernel_events[0] on the stream just before its main
 *                   kernel (the fused kernel, or the dK / dV kernel of the pair)
 *                   and kernel_events[1] just after it (after the dQ kernel of
 *                   the pair), so that their elapsed time is the main kernels'
 *                   alone, without the tile plan, the D pre-pass and the dQ
 *                   finalise.  Setting only one of them is ATTN_ERR_INVALID_ARG.
 *  delta            optional output (NULL: none): fp32 [b, h_q, s_q], 4-byte
 *                   aligned, D = rowsum(dO * O) of every query row and head,
 *                   as the backward uses it (its workspace copy otherwise).
 *                   Rows of a 128-row query tile that sees no key at all
 *                   (padding, where attn_fwd leaves O = 0) get 0 without O and
 *                   dO being read.  Its sum is vdot(out, dout), the loss whose
 *                   gradient this call computes (TE tutorial section 5
 *                   differentiates that vdot).  Must not overlap the other
 *                   buffers.
 */
typedef struct attn_bwd_params {
  attn_fwd_params fwd;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  int32_t accumulate_fp32;
  int32_t deterministic;
  void* kernel_events[2];
  float* delta;
} attn_bwd_params;

/* Scratch sizes (bytes) for the given problem; 0 on invalid sizes. */
GB300ATTN_API size_t attn_fwd_workspace_bytes(const attn_fwd_params* p);
GB300ATTN_API size_t attn_bwd_workspace_bytes(const attn_bwd_params* p);

/* Forward attention (tile plan + fused tcgen05 kernel).  See attn_fwd_params. */
GB300ATTN_API int attn_fwd(const attn_fwd_params* p, attn_stream_t stream);

/* Backward attention: D = rowsum(dO*O), then either the fused dQ/dK/dV kernel
 * and the dQ finalise (d = 64 / 128, deterministic = 0), or the dK / dV kernel
 * and the dQ kernel (deterministic = 1, and always at d = 256 and d = 192 with
 * d_v = 128, where a 128-key tile's dK and dV would not fit the fused
 * kernel's 512 TMEM columns).  scale must be at least 1e-30
 * (ATTN_ERR_UNSUPPORTED otherwise): the kernels subtract (LSE - ln scale) /
 * scale from S on the tensor core, which must stay within the fp32 range. */
GB300ATTN_API int attn_bwd(const attn_bwd_params* p, attn_stream_t stream);

/* Online-softmax merge of a partial result into an accumulator, per row-head.
 * Page: "Context parallelism and ring attention", section "Online softmax"
 * (m' = max(m, m_b); z' = e^(m-m') z + e^(m_b-m') z_b; u' likewise; output
 * u'/z'), applied to finished partials (O, LSE) == (u/z, m + ln z):
 *   M = max(l_acc, l_blk); if M == -inf the row stays (0, -inf); else
 *   l' = M + ln(e^(l_acc-M) + e^(l_blk-M)),
 *   O' = e^(l_acc-l') O_acc + e^(l_blk-l') O_blk.
 *  out_acc   fp32 [b, s, h, d]  accumulator (read; written unless out_final)
 *  lse_acc   fp32 [b, h, s]     accumulator LSE (read and written)
 *  out_blk   [b, s, h, d], fp32 or bf16 (blk_is_bf16 != 0)
 *  lse_blk   fp32 [b, h, s]
 *  out_final NULL, or bf16 [b, s, h, d]: then O' goes there (as bf16, RNE)
 *            instead of into out_acc.
 * A row whose accumulator LSE is -inf takes the block as is (its out_acc
 * value is ignored, so the accumulator needs no initialisation).  Pointers
 * 16-byte aligned; d % 8 == 0.
 */
GB300ATTN_API int attn_merge_partial(float* out_acc, float* lse_acc, const void* out_blk,
                       const float* lse_blk, int blk_is_bf16, void* out_final,
                       int64_t b, int64_t s, int64_t h, int64_t d, attn_stream_t stream);

/* Causal load-balancing reorder along the sequence axis of a tensor viewed as
 * [outer, s, inner_bytes] (q/k/v/out: inner = h*d*2; ids/pos: outer = b,
 * inner = 4; lse [b, h, s]: outer = b*h, inner = 4).
 * Page: "Context parallelism and ring attention", section "Load balance"
 * (pair early and late pieces on each device); TE tutorial section 4.
 *  strategy DUAL_CHUNK: 2R chunks of s/(2R); shard r = [chunk r, chunk 2R-1-r],
 *           shards in order r = 0..R-1.  Needs s % (2R) == 0.
 *  strategy STRIPED: stripes of stripe_size tokens; stripe t -> shard t mod R,
 *           kept in order.  Needs s % (R*stripe_size) == 0.
 *  out[o, i, :] = in[o, src(i), :].  in != out (no in-place).
 */
GB300ATTN_API int reorder_causal_lb(const void* in, void* out, int64_t outer, int64_t s, int64_t inner_bytes,
                      int strategy, int cp_size, int stripe_size, attn_stream_t stream);

/* Inverse of reorder_causal_lb with the same arguments: out[o, src(i), :] = in[o, i, :]. */
GB300ATTN_API int inverse_reorder_causal_lb(const void* in, void* out, int64_t outer, int64_t s,
                              int64_t inner_bytes, int strategy, int cp_size, int stripe_size,
                              attn_stream_t stream);

/* Segment descriptors (ids, pos) from per-row sequence lengths.
 * TE tutorial section 1 ("Packed THD inputs": a SequenceDescriptor of segment
 * ids counted from 1, positions from each segment's first token, padding id
 * 0); TE Cpp attention page, "I/O Contract" (seqlen_q / seqlen_kv inputs).
 * Covers BSHD batches (nseg = 1 per row), packed variable-length rows
 * (offsets NULL: segments back to back) and padded slots (explicit offsets).
 *  seqlens  int32 [b, nseg] segment lengths (negative counts as 0)
 *  offsets  NULL, or int32 [b, nseg] segment starts, non-decreasing per row;
 *           NULL = each segment starts where the previous one ends (row 0 at 0)
 *  ids, pos int32 [b, s] (written): token t belongs to the last segment j of
 *           its row with start_j <= t; pos = t - start_j and id = j + 1 while
 *           pos < seqlen_j, else id = 0 (padding); tokens before every start
 *           get id 0, pos = t.  Segments past s are cut at s.
 *  1 <= nseg <= 8192; s >= 1; pointers 4-byte aligned; ids / pos must not
 *  overlap the inputs.
 */
GB300ATTN_API int attn_segments_from_seqlens(const int32_t* seqlens, const int32_t* offsets,
                                             int64_t b, int64_t nseg, int64_t s, int32_t* ids,
                                             int32_t* pos, attn_stream_t stream);

/* Debug hook: the per-tile work classification the forward pass uses.
 * Page: "Context parallelism and ring attention", section "Causal attention"
 * (skip future blocks, process fully valid blocks, mask overlapping ones).
 *  classes  uint8 [b, ceil(s_q/128), ceil(s_kv/128)]: 0 SKIP, 1 PARTIAL, 2 FULL
 *  ranges   int32 [b, ceil(s_q/128), 2]: first / last non-SKIP kv tile (0, -1 if none)
 * Uses p->workspace like attn_fwd.
 */
GB300ATTN_API int attn_tile_plan(const attn_fwd_params* p, uint8_t* classes, int32_t* ranges,
                   attn_stream_t stream);

/* Debug hook: the order in which the kernels take their work units.  Each
 * side's order is one of two, chosen per call from the plan's weights (a
 * unit's weight: its non-SKIP tiles of the other side):
 *  - index order, descending on the query side and ascending on the key
 *    side (heavy first within each causal segment; neighbouring tiles run
 *    together and share their inputs through L2), taken when the heaviest
 *    unit's CTA is at most 1/20 of an SM's share of the launch:
 *    w_max * SMs * 20 <= (sum of w) * (CTAs per unit);
 *  - otherwise heaviest first over all units, equal weights in index order
 *    (a stable sort).
 *  q_order   int32 [b * ceil(s_q/128)]:  (b, query tile) indices b * nq + tile,
 *            as the forward takes them (CTAs per unit: h_kv * ceil(g / 2),
 *            g = h_q / h_kv, or h_q when d_v = 256)
 *  kv_order  int32 [b * ceil(s_kv/128)]: (b, key tile) indices b * nk + tile,
 *            as the fused backward takes them (CTAs per unit: h_kv)
 * (The dQ kernel of the deterministic backward decides with h_q CTAs per
 * unit, its dK / dV kernel with h_kv, or 2 * h_kv at d = 256.)
 * Uses p->workspace like attn_fwd.  Not part of any computation's result:
 * the order only decides which CTAs run first. */
GB300ATTN_API int attn_tile_order(const attn_fwd_params* p, int32_t* q_order, int32_t* kv_order,
                                  attn_stream_t stream);

/* Test hook for the device-side timeout path: runs attn_fwd with every key /
 * value tile load withheld, so the bounded waits of the launch run out (about
 * one second) instead of completing.  The kernel then stops early, leaves its
 * outputs undefined and records ATTN_ERR_TIMEOUT in the status word, which
 * attn_read_device_status reports; the CUDA context stays usable.  Returns
 * the launch status like attn_fwd.  Not for production use. */
GB300ATTN_API int attn_fwd_test_timeout(const attn_fwd_params* p, attn_stream_t stream);

/* Synchronises `stream`, then returns the device status word kept at the start
 * of `workspace` by the last attn_fwd / attn_bwd that used it: ATTN_OK, or
 * ATTN_ERR_TIMEOUT if a bounded device-side wait gave up (the kernel then
 * stopped early and its outputs are undefined). */
GB300ATTN_API int attn_read_device_status(const void* workspace, attn_stream_t stream);

/* attn_fwd without a caller-provided workspace, for callers that cannot
 * allocate device memory (for example code inside a host framework that owns
 * all device memory through its own pool, or a latency-critical path that
 * cannot afford an allocation's implicit synchronisation).  The pages have no
 * counterpart to this entry point.
 *  - Same parameters and results as attn_fwd; p->workspace and
 *    p->workspace_bytes are ignored.  The caller still provides q, k, v, the
 *    descriptors, out and lse.
 *  - The scratch (tile plan + status word) is a fixed 4 MiB array in the
 *    library's device memory, held on every GPU that loads the library until
 *    the process exits.  Problems whose attn_fwd_workspace_bytes() exceeds
 *    4 MiB are rejected with ATTN_ERR_UNSUPPORTED (about b * ceil(s_q/128) *
 *    ceil(s_kv/128) <= 3.5M tiles, e.g. b=2 with s=160k).
 *  - No cudaMalloc / cudaFree or other allocating call is made.  Every call
 *    looks up the array's device address (cudaGetSymbolAddress, with the
 *    caller's device current); the first call on a device also loads the
 *    library's module there, so make that first call before any stream
 *    capture.
 *  - All calls share the one array and it keeps the last call's contents (the
 *    status word is cleared at the start of every call): calls that overlap on
 *    the GPU (different streams, or different host threads) race on it.
 *  - A device-side timeout (see ATTN_ERR_TIMEOUT) is recorded in that array's
 *    status word, not returned: read it with attn_fwd_noalloc_status.
 */
GB300ATTN_API int attn_fwd_noalloc(const attn_fwd_params* p, attn_stream_t stream);

/* Synchronises `stream`, then returns the status word of attn_fwd_noalloc's
 * scratch on the current device (the counterpart of attn_read_device_status
 * for that entry point): ATTN_OK, or ATTN_ERR_TIMEOUT if a bounded wait of
 * the last attn_fwd_noalloc on this device gave up, its outputs then being
 * undefined.  ATTN_ERR_CUDA if the stream or the copy fails.  The pages have
 * no counterpart to this call either. */
GB300ATTN_API int attn_fwd_noalloc_status(attn_stream_t stream);

/* Static description of a status code. */
GB300ATTN_API const char* attn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GB300ATTN_H */
