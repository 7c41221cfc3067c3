// Shared host-side declarations of the gb300attn library (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "gb300attn.h"

namespace gb300 {

constexpr int kMaxDevices = 64;

// Checks a kernel's register count and raises its dynamic shared memory
// limit, once per device.  Idempotent and safe to call from several host
// threads: a flag is only set after both succeeded, and a repeated call is
// harmless.
inline cudaError_t ensure_smem_limit(const void* kernel, int bytes, int launch_regs,
                                     std::atomic<int>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  // The kernels split the block's registers between warpgroups with
  // setmaxnreg, which assumes the block was launched with exactly
  // `launch_regs` per thread; refuse to launch a build that differs.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != launch_regs) return cudaErrorInvalidKernelImage;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) done[dev].store(1, std::memory_order_release);
  return e;
}

constexpr int kTile = 128;  // query / key tile edge used by the plan and the kernels
constexpr int kFwdKeyTile = 64;  // keys per tile inside the forward kernel (half a plan tile)

constexpr int kSortChunk = 1024;  // rows per CTA of the heavy-first sort

// Per-128-token tile summary of a segment descriptor (32 bytes).
struct TileSummary {
  int any_valid;  // some token has id != 0
  int has_pad;    // some slot is padding or past the end of the sequence
  int id_min;     // min / max nonzero id (valid only if any_valid)
  int id_max;
  int pos_min;    // min / max position over valid tokens
  int pos_max;
  int reserved0;
  int reserved1;
};

enum : uint8_t { kSkip = 0, kPartial = 1, kFull = 2 };

// Byte offsets of the tile plan inside a workspace.
struct PlanLayout {
  size_t status;      // int: device status word
  size_t q_sum;       // TileSummary [b, nq]
  size_t kv_sum;      // TileSummary [b, nk]
  size_t q_range;     // int2 [b, nq]  first/last non-SKIP kv tile
  size_t kv_range;    // int2 [b, nk]  first/last non-SKIP q tile
  size_t q_weight;    // int  [b, nq]  number of non-SKIP kv tiles
  size_t kv_weight;   // int  [b, nk]  number of non-SKIP q tiles
  size_t q_order;     // int  [b, nq]  (b, q tile) work order
  size_t kv_order;    // int  [b, nk]  (b, kv tile) work order
  size_t classes;     // uint8 [b, nq, nk]
  size_t sort_hist;   // int [chunks, buckets]  heavy-first sort: per-chunk weight counts
  size_t sort_rank;   // int [max(b*nq, b*nk)]   rank among equal weights in the chunk
  size_t sort_start;  // int [buckets + 1]       first position of each weight; the order chosen
  int64_t sort_buckets;  // max(nq, nk) + 1: weights are tile counts of the other side
  size_t end;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline PlanLayout plan_layout(int64_t b, int64_t nq, int64_t nk, size_t base = 0) {
  PlanLayout L;
  size_t o = base;
  L.status = o;    o = align_up(o + 256, 256);
  L.q_sum = o;     o = align_up(o + (size_t)(b * nq) * sizeof(TileSummary), 256);
  L.kv_sum = o;    o = align_up(o + (size_t)(b * nk) * sizeof(TileSummary), 256);
  L.q_range = o;   o = align_up(o + (size_t)(b * nq) * 8, 256);
  L.kv_range = o;  o = align_up(o + (size_t)(b * nk) * 8, 256);
  L.q_weight = o;  o = align_up(o + (size_t)(b * nq) * 4, 256);
  L.kv_weight = o; o = align_up(o + (size_t)(b * nk) * 4, 256);
  L.q_order = o;   o = align_up(o + (size_t)(b * nq) * 4, 256);
  L.kv_order = o;  o = align_up(o + (size_t)(b * nk) * 4, 256);
  L.classes = o;   o = align_up(o + (size_t)(b * nq * nk), 256);
  const int64_t nmax = b * (nq > nk ? nq : nk);
  L.sort_buckets = (nq > nk ? nq : nk) + 1;
  const int64_t chunks = (nmax + kSortChunk - 1) / kSortChunk;
  L.sort_hist = o;  o = align_up(o + (size_t)(chunks * L.sort_buckets) * 4, 256);
  L.sort_rank = o;  o = align_up(o + (size_t)nmax * 4, 256);
  L.sort_start = o; o = align_up(o + (size_t)(L.sort_buckets + 1) * 4, 256);
  L.end = o;
  return L;
}

struct PlanPtrs {
  int* status;
  TileSummary* q_sum;
  TileSummary* kv_sum;
  int2* q_range;
  int2* kv_range;
  int* q_weight;
  int* kv_weight;
  int* q_order;
  int* kv_order;
  uint8_t* classes;
  int* sort_hist;
  int* sort_rank;
  int* sort_start;
  int64_t sort_buckets;
};

inline PlanPtrs plan_ptrs(void* ws, const PlanLayout& L) {
  char* c = static_cast<char*>(ws);
  return PlanPtrs{reinterpret_cast<int*>(c + L.status),
                  reinterpret_cast<TileSummary*>(c + L.q_sum),
                  reinterpret_cast<TileSummary*>(c + L.kv_sum),
                  reinterpret_cast<int2*>(c + L.q_range),
                  reinterpret_cast<int2*>(c + L.kv_range),
                  reinterpret_cast<int*>(c + L.q_weight),
                  reinterpret_cast<int*>(c + L.kv_weight),
                  reinterpret_cast<int*>(c + L.q_order),
                  reinterpret_cast<int*>(c + L.kv_order),
                  reinterpret_cast<uint8_t*>(c + L.classes),
                  reinterpret_cast<int*>(c + L.sort_hist),
                  reinterpret_cast<int*>(c + L.sort_rank),
                  reinterpret_cast<int*>(c + L.sort_start),
                  L.sort_buckets};
}

// ---- kernels_misc.cu
// q_ctas / kv_ctas: CTAs the kernel that takes the query / key side's work
// order launches per unit (the order is chosen from it; kernels_misc.cu).
cudaError_t launch_tile_plan(const attn_fwd_params& p, const PlanPtrs& pp, int64_t nq, int64_t nk,
                             bool need_kv_side, int64_t q_ctas, int64_t kv_ctas, cudaStream_t st);
cudaError_t launch_permute(const void* in, void* out, int64_t outer, int64_t s, int64_t inner_bytes,
                           int strategy, int cp, int stripe, bool inverse, cudaStream_t st);
cudaError_t launch_merge(float* out_acc, float* lse_acc, const void* out_blk, const float* lse_blk,
                         int blk_bf16, void* out_final, int64_t b, int64_t s, int64_t h, int64_t d,
                         cudaStream_t st);
// D = rowsum(dout * out) per row-head; also zeroes zero_acc (fp32, out's
// layout) when it is not null.  Query tiles of plan weight 0 (q_weight
// [b, ceil(s/128)]) get D = 0 and keep their accumulator rows untouched.
cudaError_t launch_bwd_preprocess(const void* out, const void* dout, float* D, float* zero_acc,
                                  const int* q_weight, int64_t b, int64_t s, int64_t h, int64_t d,
                                  cudaStream_t st);
// dq (bf16, [b, s, h, d]) from the fp32 accumulator; zeros for query tiles of
// plan weight 0, whose accumulator rows are not read.
cudaError_t launch_dq_finalize(const float* acc, void* dq, const int* q_weight, int64_t b,
                               int64_t s, int64_t h, int64_t d, cudaStream_t st);
constexpr int kSegMax = 8192;  // segments per row accepted by launch_segments
cudaError_t launch_segments(const int* seqlens, const int* offsets, int64_t b, int64_t nseg,
                            int64_t s, int* ids, int* pos, cudaStream_t st);

// ---- attn_fwd.cu
struct FwdLaunch {
  const attn_fwd_params* p;
  PlanPtrs plan;
  int64_t nq, nk;
  CUtensorMap tm_q, tm_k, tm_v;
  bool withhold_kv = false;  // debug hook (attn_fwd_test_timeout)
};
cudaError_t launch_attn_fwd(const FwdLaunch& L, cudaStream_t st);
// forward CTAs per (b, query tile): one per kv head and slot group of its query heads
int64_t fwd_ctas_per_tile(const attn_fwd_params& p);

// ---- attn_bwd.cu
struct BwdLaunch {
  const attn_bwd_params* p;
  PlanPtrs plan;
  int64_t nq, nk;
  float* D;       // [b, hq, s_q]
  float* dq_acc;  // [b, s_q, hq, d]
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  CUtensorMap tm_dq;  // fp32 dQ accumulator, 32 d x 128 rows boxes, 128B swizzle
};
cudaError_t launch_attn_bwd(const BwdLaunch& L, cudaStream_t st);

// ---- attn_bwd_split.cu
// Backward as a dK / dV kernel plus a dQ kernel (no fp32 dQ accumulator).
struct SplitLaunch {
  const attn_bwd_params* p;
  PlanPtrs plan;
  int64_t nq, nk;
  float* D;                      // [b, hq, s_q]
  CUtensorMap tm_q, tm_do;       // 128-row boxes (dQ kernel)
  CUtensorMap tm_q_a, tm_do_a;   // split_bwd_query_rows()-row boxes (dK / dV kernel)
  CUtensorMap tm_k, tm_v;        // 128-row boxes (dK / dV kernel)
  CUtensorMap tm_kb, tm_vb;      // split_bwd_key_rows()-row boxes (dQ kernel)
};
int split_bwd_query_rows(int64_t d, int64_t dv);
int split_bwd_key_rows(int64_t d, int64_t dv);
// dK / dV kernel CTAs per (b, key tile) and kv head: column slices of dK / dV
int split_bwd_col_slices(int64_t d, int64_t dv);
cudaError_t launch_attn_bwd_split(const SplitLaunch& L, cudaStream_t st);

// ---- attn_api.cu
bool encode_qkv_map(CUtensorMap* m, const void* base, int64_t b, int64_t s, int64_t h, int64_t d,
                    int64_t token_stride, int box_rows = kTile);
bool encode_acc_map(CUtensorMap* m, const float* base, int64_t b, int64_t s, int64_t h, int64_t d);

}  // namespace gb300
