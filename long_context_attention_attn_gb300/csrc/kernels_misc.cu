// HBM-bound and integer kernels of the hot path: tile plan, causal
// load-balancing permutation, online-softmax merge, backward pre/post passes.
#include <cuda_bf16.h>

#include <climits>

#include "internal.h"
#include "merge_math.cuh"

namespace gb300 {

// ============================================================== tile plan
// Page: "Context parallelism and ring attention", section "Causal attention":
// skip key blocks entirely in the future, process fully valid blocks without
// a mask, mask the overlapping ones.  Generalised to segments, padding and a
// left window through per-tile summaries of the segment descriptors.

// Summary of tile t of batch row bi (one warp; every lane returns it).
__device__ __forceinline__ TileSummary warp_tile_summary(const int* __restrict__ ids,
                                                         const int* __restrict__ pos, int64_t s,
                                                         int64_t bi, int64_t t, int lane) {
  int any_valid = 0, has_pad = 0;
  int id_min = INT_MAX, id_max = INT_MIN, pmin = INT_MAX, pmax = INT_MIN;
#pragma unroll
  for (int k = 0; k < kTile / 32; ++k) {
    const int64_t tok = t * kTile + k * 32 + lane;
    if (tok < s) {
      const int id = ids[bi * s + tok];
      if (id != 0) {
        const int ps = pos[bi * s + tok];
        any_valid = 1;
        id_min = min(id_min, id);
        id_max = max(id_max, id);
        pmin = min(pmin, ps);
        pmax = max(pmax, ps);
      } else {
        has_pad = 1;
      }
    } else {
      has_pad = 1;
    }
  }
  any_valid = __reduce_or_sync(0xffffffffu, any_valid);
  has_pad = __reduce_or_sync(0xffffffffu, has_pad);
  id_min = __reduce_min_sync(0xffffffffu, id_min);
  id_max = __reduce_max_sync(0xffffffffu, id_max);
  pmin = __reduce_min_sync(0xffffffffu, pmin);
  pmax = __reduce_max_sync(0xffffffffu, pmax);
  TileSummary r;
  r.any_valid = any_valid;
  r.has_pad = has_pad;
  r.id_min = any_valid ? id_min : 0;
  r.id_max = any_valid ? id_max : 0;
  r.pos_min = any_valid ? pmin : 0;
  r.pos_max = any_valid ? pmax : 0;
  r.reserved0 = r.reserved1 = 0;
  return r;
}

__global__ void tile_summary_kernel(const int* __restrict__ ids, const int* __restrict__ pos,
                                    int64_t b, int64_t s, int64_t ntile,
                                    TileSummary* __restrict__ out) {
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= b * ntile) return;
  const TileSummary r = warp_tile_summary(ids, pos, s, w / ntile, w % ntile, lane);
  if (lane == 0) out[w] = r;
}

__device__ __forceinline__ uint8_t classify(const TileSummary& q, const TileSummary& k, int window) {
  if (!q.any_valid || !k.any_valid) return kSkip;
  if (q.id_max < k.id_min || k.id_max < q.id_min) return kSkip;
  if (k.pos_min > q.pos_max) return kSkip;  // every key after every query
  if (window >= 0 && (int64_t)k.pos_max < (int64_t)q.pos_min - window) return kSkip;
  const bool one_id = !q.has_pad && !k.has_pad && q.id_min == q.id_max && k.id_min == k.id_max &&
                      q.id_min == k.id_min;
  if (one_id && k.pos_max <= q.pos_min &&
      (window < 0 || (int64_t)q.pos_max - k.pos_min <= window))
    return kFull;
  return kPartial;
}

// One CTA per (q tile, b): the class of every kv tile and the q-side range.
__global__ void tile_class_kernel(const TileSummary* __restrict__ qs,
                                  const TileSummary* __restrict__ ks, int64_t nq, int64_t nk,
                                  int window, uint8_t* __restrict__ cls, int2* __restrict__ qrange,
                                  int* __restrict__ qweight) {
  const int64_t a = blockIdx.x, bi = blockIdx.y;
  __shared__ int s_first, s_last, s_count;
  if (threadIdx.x == 0) {
    s_first = INT_MAX;
    s_last = -1;
    s_count = 0;
  }
  __syncthreads();
  const TileSummary q = qs[bi * nq + a];
  int first = INT_MAX, last = -1, count = 0;
  for (int64_t c = threadIdx.x; c < nk; c += blockDim.x) {
    const uint8_t k = classify(q, ks[bi * nk + c], window);
    cls[(bi * nq + a) * nk + c] = k;
    if (k != kSkip) {
      first = min(first, (int)c);
      last = max(last, (int)c);
      ++count;
    }
  }
  atomicMin(&s_first, first);
  atomicMax(&s_last, last);
  atomicAdd(&s_count, count);
  __syncthreads();
  if (threadIdx.x == 0) {
    qrange[bi * nq + a] = s_last < 0 ? make_int2(0, -1) : make_int2(s_first, s_last);
    qweight[bi * nq + a] = s_count;
  }
}

// The range of q tiles that see each kv tile (backward side).  A CTA takes 32
// neighbouring kv tiles of one batch row (lane = kv tile, so a warp reads 32
// consecutive class bytes of a row: one sector), its 32 warps split the rows,
// and each warp keeps eight independent loads in flight.
__global__ void __launch_bounds__(1024)
    kv_range_kernel(const uint8_t* __restrict__ cls, int64_t nq, int64_t nk,
                    int2* __restrict__ krange, int* __restrict__ kweight) {
  __shared__ int s_first[32][33], s_last[32][33], s_count[32][33];
  const int64_t bi = blockIdx.y;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 32 + lane;
  int first = INT_MAX, last = -1, count = 0;
  if (c < nk) {
    const uint8_t* col = cls + bi * nq * nk + c;
    for (int64_t a0 = (int64_t)wid * 8; a0 < nq; a0 += 32 * 8) {
      uint8_t v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = (a0 + u < nq) ? col[(a0 + u) * nk] : (uint8_t)kSkip;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (v[u] != kSkip) {
          first = min(first, (int)(a0 + u));
          last = max(last, (int)(a0 + u));
          ++count;
        }
      }
    }
  }
  s_first[wid][lane] = first;
  s_last[wid][lane] = last;
  s_count[wid][lane] = count;
  __syncthreads();
  if (wid == 0 && c < nk) {
    for (int w = 1; w < 32; ++w) {
      first = min(first, s_first[w][lane]);
      last = max(last, s_last[w][lane]);
      count += s_count[w][lane];
    }
    krange[bi * nk + c] = last < 0 ? make_int2(0, -1) : make_int2(first, last);
    kweight[bi * nk + c] = count;
  }
}

// SM count of the current device (cached per device; safe across host threads).
static int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  int n = cached ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (cached) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Work order of the units (rows) of one side: the CTAs of a launch take them
// in this order.  Two orders, chosen per call on the device:
// * index order (key side: ascending; query side: descending).  Under the
//   causal mask a segment's key tiles get lighter and its query tiles heavier
//   with the tile index, so both are heavy first within every segment, and
//   neighbouring tiles run at the same time, sharing their K / V, Q / dO and
//   fp32 dQ tiles through L2;
// * heavy first over all units (a stable counting sort by weight): the last
//   units to start are the lightest, which bounds the tail of the launch, but
//   CTAs running at the same time come from different segments.
// The largest unit bounds what the index order can lose at the tail: when one
// CTA of it is under 1/kTailShare of an SM's share of the launch (weight_max *
// SMs * kTailShare <= sum of weights * CTAs per unit) the index order is
// taken.  On GB300 at b 2 s 65536 Hq 128 Hkv 8 d 128 window 8192 (ratio 3.7 %
// for the fused backward, 0.5 % for the forward) it halved the kernels' DRAM
// traffic at the same speed; on the same packing at s 16384 Hq 32 window 1024
// (11.9 %) heavy first ran the backward 13 % faster.
//
// The sort places row i at
//   (rows with a larger weight) + (rows of its weight in earlier chunks)
//   + (rows of its weight earlier in its own chunk of kSortChunk rows).
// order_chunk_kernel: per chunk, the weight counts (a [chunks, buckets]
// table in global memory) and each row's rank within the chunk among the
// rows of its weight (a bitonic sort of (weight, index) pairs in shared
// memory, then the distance to the first pair of the same weight).
// order_colscan_kernel / order_bucketscan_kernel: the table's prefix down the
// chunks of each weight, and the first position of each weight (a suffix sum
// over the weights); the bucket scan also takes the choice of order and
// stores it after the weights' positions.
// order_scatter_kernel: order[position] = row.
constexpr int kTailShare = 20;

__device__ __forceinline__ int clamp_weight(int w, int buckets) {
  return w < 0 ? 0 : (w >= buckets ? buckets - 1 : w);
}

__global__ void __launch_bounds__(kSortChunk)
    order_chunk_kernel(const int* __restrict__ weight, int n, int buckets, int* __restrict__ hist,
                       int* __restrict__ rank) {
  __shared__ uint64_t keys[kSortChunk];
  __shared__ int warp_max[kSortChunk / 32];
  const int t = threadIdx.x;
  const int64_t i = (int64_t)blockIdx.x * kSortChunk + t;
  uint64_t key = ~0ull;  // rows past n sort last
  if (i < n) {
    const int w = clamp_weight(weight[i], buckets);
    atomicAdd(&hist[(int64_t)blockIdx.x * buckets + w], 1);
    key = ((uint64_t)w << 32) | (uint32_t)t;
  }
  keys[t] = key;
  __syncthreads();
  for (int k = 2; k <= kSortChunk; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int p = t ^ j;
      if (p > t) {
        const uint64_t x = keys[t], y = keys[p];
        if ((x > y) == ((t & k) == 0)) {
          keys[t] = y;
          keys[p] = x;
        }
      }
      __syncthreads();
    }
  }
  // position of the first pair with this weight: inclusive max-scan of the
  // group starts over the sorted positions
  const uint64_t kt = keys[t];
  int first = (t == 0 || (keys[t - 1] >> 32) != (kt >> 32)) ? t : 0;
  const int lane = t & 31, wid = t >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, first, o);
    if (lane >= o) first = max(first, v);
  }
  if (lane == 31) warp_max[wid] = first;
  __syncthreads();
  if (wid == 0) {
    int v = warp_max[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v = max(v, u);
    }
    warp_max[lane] = v;
  }
  __syncthreads();
  if (wid > 0) first = max(first, warp_max[wid - 1]);
  if (kt != ~0ull) rank[(int64_t)blockIdx.x * kSortChunk + (uint32_t)kt] = t - first;
}

// Exclusive prefix of each weight's counts down the chunks (one thread per
// weight, the chunk counts loaded eight at a time); the totals go to `total`.
__global__ void __launch_bounds__(256)
    order_colscan_kernel(int* __restrict__ hist, int chunks, int buckets, int* __restrict__ total) {
  const int w = blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= buckets) return;
  int run = 0;
  for (int c0 = 0; c0 < chunks; c0 += 8) {
    int v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = (c0 + u < chunks) ? hist[(int64_t)(c0 + u) * buckets + w] : 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (c0 + u < chunks) hist[(int64_t)(c0 + u) * buckets + w] = run;
      run += v[u];
    }
  }
  total[w] = run;
}

// start[w] = number of rows whose weight is larger than w: one CTA; thread t
// takes a run of consecutive weights from the largest down, sums it, and a
// block-wide exclusive scan of the run sums gives each run's base.  The same
// pass sums weight * count and finds the largest weight present, and thread 0
// stores start[buckets] = 1 (heavy first) or 0 (index order).
__global__ void __launch_bounds__(1024)
    order_bucketscan_kernel(int* __restrict__ start, int buckets, int64_t ctas_per_unit, int sms) {
  __shared__ int warp_sum[32];
  __shared__ long long warp_work[32];
  __shared__ int warp_wmax[32];
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int per = (buckets + blockDim.x - 1) / blockDim.x;
  const int p0 = t * per;  // positions p0.. of the list of weights from the largest down
  int sum = 0;
  long long work = 0;
  int wmax = 0;
  for (int k0 = 0; k0 < per; k0 += 8) {
    int v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int w = buckets - 1 - (p0 + k0 + u);
      v[u] = (k0 + u < per && w >= 0) ? start[w] : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int w = buckets - 1 - (p0 + k0 + u);
      sum += v[u];
      work += (long long)v[u] * w;
      if (v[u] > 0) wmax = max(wmax, w);
    }
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  long long wk = work;
  int wm = wmax;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    wk += __shfl_xor_sync(0xffffffffu, wk, o);
    wm = max(wm, __shfl_xor_sync(0xffffffffu, wm, o));
  }
  if (lane == 31) warp_sum[wid] = incl;
  if (lane == 0) {
    warp_work[wid] = wk;
    warp_wmax[wid] = wm;
  }
  __syncthreads();
  if (wid == 0) {
    int x = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += u;
    }
    warp_sum[lane] = x;
    long long tw = lane < (int)(blockDim.x >> 5) ? warp_work[lane] : 0;
    int tm = lane < (int)(blockDim.x >> 5) ? warp_wmax[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tw += __shfl_xor_sync(0xffffffffu, tw, o);
      tm = max(tm, __shfl_xor_sync(0xffffffffu, tm, o));
    }
    if (lane == 0)
      start[buckets] = (long long)tm * sms * kTailShare > tw * ctas_per_unit ? 1 : 0;
  }
  __syncthreads();
  int run = (wid > 0 ? warp_sum[wid - 1] : 0) + incl - sum;
  for (int k = 0; k < per; ++k) {
    const int w = buckets - 1 - (p0 + k);
    if (w < 0) break;
    const int v = start[w];
    start[w] = run;
    run += v;
  }
}

// order[position] = row: the sorted position (heavy first), or the row's own
// index (reversed on the query side) when the bucket scan chose index order.
__global__ void order_scatter_kernel(const int* __restrict__ weight, int n, int buckets,
                                     const int* __restrict__ hist, const int* __restrict__ start,
                                     const int* __restrict__ rank, int reverse,
                                     int* __restrict__ order) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  if (start[buckets] == 0) {
    order[reverse ? n - 1 - i : i] = (int)i;
    return;
  }
  const int w = clamp_weight(weight[i], buckets);
  const int64_t c = i / kSortChunk;
  order[start[w] + hist[c * buckets + w] + rank[i]] = (int)i;
}

// ctas_per_unit: CTAs the consuming kernel launches per unit; reverse: the
// query side (index order descending).
static cudaError_t launch_work_order(const int* weight, int64_t n, int64_t ctas_per_unit,
                                     bool reverse, const PlanPtrs& pp, int* order,
                                     cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t chunks = (n + kSortChunk - 1) / kSortChunk;
  const int buckets = (int)pp.sort_buckets;
  cudaError_t e = cudaMemsetAsync(pp.sort_hist, 0, (size_t)(chunks * buckets) * 4, st);
  if (e != cudaSuccess) return e;
  order_chunk_kernel<<<(unsigned)chunks, kSortChunk, 0, st>>>(weight, (int)n, buckets,
                                                              pp.sort_hist, pp.sort_rank);
  order_colscan_kernel<<<(unsigned)((buckets + 255) / 256), 256, 0, st>>>(pp.sort_hist, (int)chunks,
                                                                         buckets, pp.sort_start);
  order_bucketscan_kernel<<<1, 1024, 0, st>>>(pp.sort_start, buckets,
                                              ctas_per_unit > 0 ? ctas_per_unit : 1, sm_count());
  order_scatter_kernel<<<(unsigned)chunks, kSortChunk, 0, st>>>(
      weight, (int)n, buckets, pp.sort_hist, pp.sort_start, pp.sort_rank, reverse ? 1 : 0, order);
  return cudaGetLastError();
}

// ---- the whole plan in one CTA, for small problems (both sides at most
// kSmallPlanUnits units, at most kSmallPlanPairs class bytes): the same
// summaries, classes, ranges, weights and work orders as the kernels above,
// in one launch instead of up to fifteen (the plan is then most of a small
// call's launches).

constexpr int kSmallPlanUnits = 1024;
// One CTA's serial walk overtakes the parallel kernels' extra launches near
// here: on GB300 the fused plan saved ~20 / 40 µs per forward / backward call
// at 2 x 4096 tokens (2048 class bytes) and cost ~20 µs at 2 x 16384 (32768).
constexpr int64_t kSmallPlanPairs = 4096;

// The work order of one side (n <= 1024 units), block-wide: the choice rule of
// order_bucketscan_kernel from a block reduction, and the heavy-first order
// from one bitonic sort of (heaviest first, index) keys (the single-chunk case
// of the counting sort: same order).  Every thread of the block calls it.
__device__ void small_work_order(const int* __restrict__ weight, int n, int64_t ctas_per_unit,
                                 int sms, bool reverse, int* __restrict__ order, uint64_t* keys) {
  __shared__ long long r_work[32];
  __shared__ int r_wmax[32];
  __shared__ int s_lpt;
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int w = t < n ? weight[t] : 0;
  long long wk = w;
  int wm = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    wk += __shfl_xor_sync(0xffffffffu, wk, o);
    wm = max(wm, __shfl_xor_sync(0xffffffffu, wm, o));
  }
  if (lane == 0) {
    r_work[wid] = wk;
    r_wmax[wid] = wm;
  }
  __syncthreads();
  if (wid == 0) {
    long long tw = r_work[lane];
    int tm = r_wmax[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tw += __shfl_xor_sync(0xffffffffu, tw, o);
      tm = max(tm, __shfl_xor_sync(0xffffffffu, tm, o));
    }
    if (lane == 0)
      s_lpt = (long long)tm * sms * kTailShare > tw * (ctas_per_unit > 0 ? ctas_per_unit : 1);
  }
  __syncthreads();
  if (!s_lpt) {  // uniform over the block
    if (t < n) order[reverse ? n - 1 - t : t] = t;
    return;
  }
  keys[t] = t < n ? ((uint64_t)(uint32_t)(INT_MAX - w) << 32) | (uint32_t)t : ~0ull;
  __syncthreads();
  for (int k = 2; k <= kSmallPlanUnits; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int q = t ^ j;
      if (q > t) {
        const uint64_t x = keys[t], y = keys[q];
        if ((x > y) == ((t & k) == 0)) {
          keys[t] = y;
          keys[q] = x;
        }
      }
      __syncthreads();
    }
  }
  if (t < n) order[t] = (int)(uint32_t)keys[t];
}

struct SmallPlanArgs {
  const int* q_ids;
  const int* q_pos;
  const int* kv_ids;
  const int* kv_pos;
  int64_t b, s_q, s_kv, nq, nk, q_ctas, kv_ctas;
  int window, need_kv, sms;
};

__global__ void __launch_bounds__(kSmallPlanUnits)
    small_plan_kernel(const SmallPlanArgs a, const PlanPtrs pp) {
  __shared__ uint64_t keys[kSmallPlanUnits];
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  constexpr int kWarps = kSmallPlanUnits / 32;
  const int64_t nqt = a.b * a.nq, nkt = a.b * a.nk;
  // summaries: one warp per tile, query tiles then key tiles
  for (int64_t u = wid; u < nqt + nkt; u += kWarps) {
    const bool qside = u < nqt;
    const int64_t v = qside ? u : u - nqt, nt = qside ? a.nq : a.nk;
    const TileSummary r = qside ? warp_tile_summary(a.q_ids, a.q_pos, a.s_q, v / nt, v % nt, lane)
                                : warp_tile_summary(a.kv_ids, a.kv_pos, a.s_kv, v / nt, v % nt, lane);
    if (lane == 0) (qside ? pp.q_sum : pp.kv_sum)[v] = r;
  }
  __syncthreads();
  // classes, and each query tile's range and weight: one warp per query tile
  for (int64_t r = wid; r < nqt; r += kWarps) {
    const int64_t bi = r / a.nq;
    const TileSummary qsum = pp.q_sum[r];
    int first = INT_MAX, last = -1, count = 0;
    for (int64_t c = lane; c < a.nk; c += 32) {
      const uint8_t k = classify(qsum, pp.kv_sum[bi * a.nk + c], a.window);
      pp.classes[r * a.nk + c] = k;
      if (k != kSkip) {
        first = min(first, (int)c);
        last = max(last, (int)c);
        ++count;
      }
    }
    first = __reduce_min_sync(0xffffffffu, first);
    last = __reduce_max_sync(0xffffffffu, last);
    count = __reduce_add_sync(0xffffffffu, count);
    if (lane == 0) {
      pp.q_range[r] = last < 0 ? make_int2(0, -1) : make_int2(first, last);
      pp.q_weight[r] = count;
    }
  }
  __syncthreads();
  // each key tile's range and weight: one warp per key tile
  if (a.need_kv) {
    for (int64_t kc = wid; kc < nkt; kc += kWarps) {
      const int64_t bi = kc / a.nk, c = kc % a.nk;
      int first = INT_MAX, last = -1, count = 0;
      for (int64_t r = lane; r < a.nq; r += 32) {
        if (pp.classes[(bi * a.nq + r) * a.nk + c] != kSkip) {
          first = min(first, (int)r);
          last = max(last, (int)r);
          ++count;
        }
      }
      first = __reduce_min_sync(0xffffffffu, first);
      last = __reduce_max_sync(0xffffffffu, last);
      count = __reduce_add_sync(0xffffffffu, count);
      if (lane == 0) {
        pp.kv_range[kc] = last < 0 ? make_int2(0, -1) : make_int2(first, last);
        pp.kv_weight[kc] = count;
      }
    }
  }
  __syncthreads();
  small_work_order(pp.q_weight, (int)nqt, a.q_ctas, a.sms, true, pp.q_order, keys);
  if (a.need_kv) {
    __syncthreads();
    small_work_order(pp.kv_weight, (int)nkt, a.kv_ctas, a.sms, false, pp.kv_order, keys);
  }
}

cudaError_t launch_tile_plan(const attn_fwd_params& p, const PlanPtrs& pp, int64_t nq, int64_t nk,
                             bool need_kv_side, int64_t q_ctas, int64_t kv_ctas, cudaStream_t st) {
  if (p.b * nq <= kSmallPlanUnits && p.b * nk <= kSmallPlanUnits &&
      p.b * nq * nk <= kSmallPlanPairs) {
    SmallPlanArgs a;
    a.q_ids = p.q_segment_ids;
    a.q_pos = p.q_segment_pos;
    a.kv_ids = p.kv_segment_ids;
    a.kv_pos = p.kv_segment_pos;
    a.b = p.b;
    a.s_q = p.s_q;
    a.s_kv = p.s_kv;
    a.nq = nq;
    a.nk = nk;
    a.q_ctas = q_ctas;
    a.kv_ctas = kv_ctas;
    a.window = (int)p.window_left;
    a.need_kv = need_kv_side ? 1 : 0;
    a.sms = sm_count();
    small_plan_kernel<<<1, kSmallPlanUnits, 0, st>>>(a, pp);
    return cudaGetLastError();
  }
  const int wpb = 8;
  tile_summary_kernel<<<(unsigned)((p.b * nq + wpb - 1) / wpb), wpb * 32, 0, st>>>(
      p.q_segment_ids, p.q_segment_pos, p.b, p.s_q, nq, pp.q_sum);
  tile_summary_kernel<<<(unsigned)((p.b * nk + wpb - 1) / wpb), wpb * 32, 0, st>>>(
      p.kv_segment_ids, p.kv_segment_pos, p.b, p.s_kv, nk, pp.kv_sum);
  tile_class_kernel<<<dim3((unsigned)nq, (unsigned)p.b), 256, 0, st>>>(
      pp.q_sum, pp.kv_sum, nq, nk, p.window_left, pp.classes, pp.q_range, pp.q_weight);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    e = launch_work_order(pp.q_weight, p.b * nq, q_ctas, true, pp, pp.q_order, st);
  if (e == cudaSuccess && need_kv_side) {
    kv_range_kernel<<<dim3((unsigned)((nk + 31) / 32), (unsigned)p.b), 1024, 0, st>>>(
        pp.classes, nq, nk, pp.kv_range, pp.kv_weight);
    e = launch_work_order(pp.kv_weight, p.b * nk, kv_ctas, false, pp, pp.kv_order, st);
  }
  return e;
}

// ============================================================== permutation
// Page: "Context parallelism and ring attention", section "Load balance"
// (dual chunk: shard r holds chunks r and 2R-1-r of 2R); TE tutorial section 4
// (striped: stripe t goes to shard t mod R).  src(i) is the input row of
// output row i.
__device__ __forceinline__ int64_t perm_src(int64_t i, int64_t s, int strategy, int R, int stripe) {
  if (strategy == ATTN_REORDER_DUAL_CHUNK) {
    const int64_t c = s / (2 * R);
    const int64_t r = i / (2 * c), w = i - r * 2 * c;
    return w < c ? r * c + w : (2 * R - 1 - r) * c + (w - c);
  }
  const int64_t n = s / R;
  const int64_t r = i / n, t = i - r * n;
  return ((t / stripe) * R + r) * stripe + (t % stripe);
}

// One warp per row; 16-byte vectors along the row.
constexpr int kPermVecs = 16;  // 16-byte vectors in flight per lane
__global__ void permute_vec16_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                     int64_t rows, int64_t s, int64_t vpr, int strategy, int R,
                                     int stripe, int inverse) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; row < rows;
       row += nwarps) {
    const int64_t o = row / s, i = row - o * s;
    const int64_t j = perm_src(i, s, strategy, R, stripe);
    const int64_t src = o * s + (inverse ? i : j);
    const int64_t dst = o * s + (inverse ? j : i);
    const uint4* a = in + src * vpr;
    uint4* bptr = out + dst * vpr;
    // 16 loads in flight per lane (8 KB per warp) before the stores
    for (int64_t w = lane; w < vpr; w += 32 * kPermVecs) {
      uint4 x[kPermVecs];
#pragma unroll
      for (int u = 0; u < kPermVecs; ++u)
        if (w + 32 * u < vpr) x[u] = a[w + 32 * u];
#pragma unroll
      for (int u = 0; u < kPermVecs; ++u)
        if (w + 32 * u < vpr) bptr[w + 32 * u] = x[u];
    }
  }
}

// One thread per element of `esize` bytes (4 or 1).
template <typename T>
__global__ void permute_elem_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t rows,
                                    int64_t s, int64_t epr, int strategy, int R, int stripe,
                                    int inverse) {
  const int64_t total = rows * epr;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = e / epr, k = e - row * epr;
    const int64_t o = row / s, i = row - o * s;
    const int64_t j = perm_src(i, s, strategy, R, stripe);
    const int64_t src = o * s + (inverse ? i : j);
    const int64_t dst = o * s + (inverse ? j : i);
    out[dst * epr + k] = in[src * epr + k];
  }
}

cudaError_t launch_permute(const void* in, void* out, int64_t outer, int64_t s, int64_t inner_bytes,
                           int strategy, int cp, int stripe, bool inverse, cudaStream_t st) {
  const int64_t rows = outer * s;
  const int sms = sm_count();
  const bool aligned16 = (reinterpret_cast<uintptr_t>(in) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(out) % 16 == 0);
  if (inner_bytes % 16 == 0 && aligned16) {
    const int64_t need = (rows + 7) / 8;
    const unsigned grid = (unsigned)std::min<int64_t>(need, (int64_t)sms * 16);
    permute_vec16_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(in),
                                               static_cast<uint4*>(out), rows, s, inner_bytes / 16,
                                               strategy, cp, stripe, inverse ? 1 : 0);
  } else if (inner_bytes % 4 == 0 && reinterpret_cast<uintptr_t>(in) % 4 == 0 &&
             reinterpret_cast<uintptr_t>(out) % 4 == 0) {
    const int64_t total = rows * (inner_bytes / 4);
    const unsigned grid = (unsigned)std::min<int64_t>((total + 255) / 256, (int64_t)sms * 16);
    permute_elem_kernel<uint32_t><<<grid, 256, 0, st>>>(
        static_cast<const uint32_t*>(in), static_cast<uint32_t*>(out), rows, s, inner_bytes / 4,
        strategy, cp, stripe, inverse ? 1 : 0);
  } else {
    const int64_t total = rows * inner_bytes;
    const unsigned grid = (unsigned)std::min<int64_t>((total + 255) / 256, (int64_t)sms * 16);
    permute_elem_kernel<uint8_t><<<grid, 256, 0, st>>>(
        static_cast<const uint8_t*>(in), static_cast<uint8_t*>(out), rows, s, inner_bytes,
        strategy, cp, stripe, inverse ? 1 : 0);
  }
  return cudaGetLastError();
}

// ============================================================== merge
// Page: "Context parallelism and ring attention", section "Online softmax".
// A finished partial (O, LSE) is the running triple (m = LSE, z = 1, u = O);
// the page's update then gives, with M = max(l_a, l_b):
//   z' = e^(l_a - M) + e^(l_b - M),  LSE' = M + ln z',
//   O' = (e^(l_a - M) O_a + e^(l_b - M) O_b) / z'.
// A warp merges 8 consecutive tokens of one (batch, head): lane j < 8 reads
// and writes the LSE pair of token j (one 32-byte sector per group), and the
// 8 rows' accumulator / block vectors (d = 128: one float4 per lane per row)
// are all loaded before the arithmetic, so their latencies overlap.  Warps
// with consecutive indices take consecutive heads, i.e. adjacent rows of the
// [b, s, h, d] tensors.  A row whose weight is 0 ignores its (possibly
// uninitialised) values through a select.
constexpr int kMergeRows = 8;

template <bool BLK_BF16>
__device__ __forceinline__ float4 load_blk4(const void* out_blk, int64_t idx4) {
  if (BLK_BF16) {
    const uint2 raw = reinterpret_cast<const uint2*>(out_blk)[idx4];
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    return make_float4(f0.x, f0.y, f1.x, f1.y);
  }
  return reinterpret_cast<const float4*>(out_blk)[idx4];
}


template <bool FINAL>
__device__ __forceinline__ void store_merged(float* out_acc, __nv_bfloat16* out_final, int64_t idx4,
                                             const float4& o) {
  if (FINAL) {
    const __nv_bfloat162 q0 = __floats2bfloat162_rn(o.x, o.y);
    const __nv_bfloat162 q1 = __floats2bfloat162_rn(o.z, o.w);
    uint2 raw;
    raw.x = *reinterpret_cast<const uint32_t*>(&q0);
    raw.y = *reinterpret_cast<const uint32_t*>(&q1);
    reinterpret_cast<uint2*>(out_final)[idx4] = raw;
  } else {
    reinterpret_cast<float4*>(out_acc)[idx4] = o;
  }
}

template <bool BLK_BF16, bool FINAL>
__global__ void merge_kernel(float* __restrict__ out_acc, float* __restrict__ lse_acc,
                             const void* __restrict__ out_blk, const float* __restrict__ lse_blk,
                             __nv_bfloat16* __restrict__ out_final, int64_t b, int64_t s,
                             int64_t h, int64_t d) {
  const int lane = threadIdx.x & 31;
  const int64_t ngroups = (s + kMergeRows - 1) / kMergeRows;
  const int64_t nwork = b * ngroups * h;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t v4 = d / 4;
  for (int64_t wi = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; wi < nwork;
       wi += nwarps) {
    const int64_t hh = wi % h;
    const int64_t tg = (wi / h) % ngroups;
    const int64_t bi = wi / (h * ngroups);
    const int64_t t0 = tg * kMergeRows;
    const int nrows = (s - t0 < kMergeRows) ? (int)(s - t0) : kMergeRows;
    // LSE pair of token t0 + lane (lanes < nrows)
    const int64_t lbase = (bi * h + hh) * s + t0;
    float la = -INFINITY, lb = -INFINITY;
    if (lane < nrows) {
      la = lse_acc[lbase + lane];
      lb = lse_blk[lbase + lane];
    }
    // row r of token t: (bi * s + t) * h + hh; one float4 per lane when d <= 128
    float4 av[kMergeRows], xv[kMergeRows];
    if (v4 <= 32) {
#pragma unroll
      for (int j = 0; j < kMergeRows; ++j) {
        av[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        xv[j] = av[j];
        if (j < nrows && lane < v4) {
          const int64_t r = (bi * s + t0 + j) * h + hh;
          av[j] = reinterpret_cast<const float4*>(out_acc)[r * v4 + lane];
          xv[j] = load_blk4<BLK_BF16>(out_blk, r * v4 + lane);
        }
      }
    }
    float ca, cb, lnew;
    merge_coeffs(la, lb, ca, cb, lnew);
#pragma unroll
    for (int j = 0; j < kMergeRows; ++j) {
      const float caj = __shfl_sync(0xffffffffu, ca, j);
      const float cbj = __shfl_sync(0xffffffffu, cb, j);
      if (j >= nrows) continue;
      const int64_t r = (bi * s + t0 + j) * h + hh;
      if (v4 <= 32) {
        if (lane < v4) store_merged<FINAL>(out_acc, out_final, r * v4 + lane, merge4(caj, cbj, av[j], xv[j]));
      } else {
        for (int64_t w = lane; w < v4; w += 32) {
          const float4 a = reinterpret_cast<const float4*>(out_acc)[r * v4 + w];
          const float4 x = load_blk4<BLK_BF16>(out_blk, r * v4 + w);
          store_merged<FINAL>(out_acc, out_final, r * v4 + w, merge4(caj, cbj, a, x));
        }
      }
    }
    if (lane < nrows) lse_acc[lbase + lane] = lnew;
  }
}

cudaError_t launch_merge(float* out_acc, float* lse_acc, const void* out_blk, const float* lse_blk,
                         int blk_bf16, void* out_final, int64_t b, int64_t s, int64_t h, int64_t d,
                         cudaStream_t st) {
  const int64_t work = b * ((s + kMergeRows - 1) / kMergeRows) * h;  // warp-sized items
  const unsigned grid = (unsigned)std::min<int64_t>((work + 7) / 8, (int64_t)sm_count() * 4);
  __nv_bfloat16* fin = static_cast<__nv_bfloat16*>(out_final);
  if (blk_bf16) {
    if (fin)
      merge_kernel<true, true><<<grid, 256, 0, st>>>(out_acc, lse_acc, out_blk, lse_blk, fin, b, s, h, d);
    else
      merge_kernel<true, false><<<grid, 256, 0, st>>>(out_acc, lse_acc, out_blk, lse_blk, fin, b, s, h, d);
  } else {
    if (fin)
      merge_kernel<false, true><<<grid, 256, 0, st>>>(out_acc, lse_acc, out_blk, lse_blk, fin, b, s, h, d);
    else
      merge_kernel<false, false><<<grid, 256, 0, st>>>(out_acc, lse_acc, out_blk, lse_blk, fin, b, s, h, d);
  }
  return cudaGetLastError();
}

// ============================================================== backward helpers
// D_i = sum_d dO_i * O_i per (b, head, row): the row term of dS = P * (dP - D).
// Each thread reads 16 bytes (8 bf16) of O and of dO; a row-head of d values
// is handled by d/8 consecutive lanes (16 for d = 128), reduced by shuffles.
// The LSE/D layout is [b, h, s] so each row-head writes one float.  With
// zero_acc the same pass clears the fp32 dQ accumulator (out's layout, 32
// bytes per thread and row), instead of a separate memset over it.
// Work items are (query tile, slice of kPreGroups row groups per warp), so the
// tile's plan weight is read once per item.  Rows of a tile of weight 0 (it
// sees no key tile: padding) take no step of the backward: their D is 0
// (their O is 0) and is written without reading O or dO, and their
// accumulator rows are not cleared (no reduce-add reaches them; the finalise
// writes their zeros).
constexpr int kPreThreads = 256;
constexpr int kPreGroups = 4;  // row groups in flight per warp and item

template <int D>
__global__ void __launch_bounds__(kPreThreads)
    bwd_preprocess_kernel(const uint4* __restrict__ out, const uint4* __restrict__ dout,
                          float* __restrict__ Dv, float4* __restrict__ zero_acc,
                          const int* __restrict__ q_weight, int64_t s, int64_t h, int64_t nq,
                          int64_t nslices, int64_t nitems) {
  constexpr int kLanes = D / 8;  // lanes per row-head
  constexpr int kRowsPerWarp = 32 / kLanes;
  constexpr int kWarps = kPreThreads / 32;
  constexpr int kItemRows = kWarps * kRowsPerWarp * kPreGroups;
  const int lane = threadIdx.x & 31;
  const int sub = lane % kLanes;
  const int wrow = (threadIdx.x / 32) * kRowsPerWarp * kPreGroups + lane / kLanes;
  for (int64_t item = blockIdx.x; item < nitems; item += gridDim.x) {
    const int64_t tile = item / nslices, slice = item % nslices;
    const int64_t bi = tile / nq, t0 = (tile % nq) * kTile;
    const int64_t t1 = t0 + kTile < s ? t0 + kTile : s;
    const int64_t row0 = (bi * s + t0) * h;  // the tile's first row-head
    const int nrows = (int)((t1 - t0) * h);  // row-heads of the tile (<= 128 h)
    const int lo = (int)(slice * kItemRows);
    if (lo >= nrows) continue;
    const bool live = q_weight[tile] != 0;
    uint4 o[kPreGroups], g[kPreGroups];
#pragma unroll
    for (int k = 0; k < kPreGroups; ++k) {
      const int lr = lo + wrow + k * kRowsPerWarp;  // row-head within the tile
      o[k] = make_uint4(0, 0, 0, 0);
      g[k] = o[k];
      if (live && lr < nrows) {
        o[k] = out[(row0 + lr) * kLanes + sub];
        g[k] = dout[(row0 + lr) * kLanes + sub];
      }
    }
    if (zero_acc && live) {
      // the fp32 dQ accumulator has out's layout: clear this thread's 8 values
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < kPreGroups; ++k) {
        const int lr = lo + wrow + k * kRowsPerWarp;
        if (lr < nrows) {
          zero_acc[((row0 + lr) * kLanes + sub) * 2] = z;
          zero_acc[((row0 + lr) * kLanes + sub) * 2 + 1] = z;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kPreGroups; ++k) {
      const uint32_t xs[4] = {o[k].x, o[k].y, o[k].z, o[k].w};
      const uint32_t ys[4] = {g[k].x, g[k].y, g[k].z, g[k].w};
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[u]));
        const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[u]));
        acc += x.x * y.x + x.y * y.y;
      }
#pragma unroll
      for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const int lr = lo + wrow + k * kRowsPerWarp;
      if (sub == 0 && lr < nrows) {
        const int hh = lr % (int)h;
        const int64_t ti = t0 + lr / (int)h;
        Dv[(bi * h + hh) * s + ti] = acc;
      }
    }
  }
}

cudaError_t launch_bwd_preprocess(const void* out, const void* dout, float* D, float* zero_acc,
                                  const int* q_weight, int64_t b, int64_t s, int64_t h, int64_t d,
                                  cudaStream_t st) {
  const int64_t nq = (s + kTile - 1) / kTile;
  const int64_t item_rows = (kPreThreads / 32) * (32 / (d / 8)) * kPreGroups;
  const int64_t nslices = (kTile * h + item_rows - 1) / item_rows;
  const int64_t nitems = b * nq * nslices;
  if (nitems == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<int64_t>(nitems, (int64_t)sm_count() * 16);
  const uint4* o4 = static_cast<const uint4*>(out);
  const uint4* d4 = static_cast<const uint4*>(dout);
  float4* z4 = reinterpret_cast<float4*>(zero_acc);
  if (d == 256)
    bwd_preprocess_kernel<256><<<grid, kPreThreads, 0, st>>>(o4, d4, D, z4, q_weight, s, h, nq,
                                                             nslices, nitems);
  else if (d == 128)
    bwd_preprocess_kernel<128><<<grid, kPreThreads, 0, st>>>(o4, d4, D, z4, q_weight, s, h, nq,
                                                             nslices, nitems);
  else
    bwd_preprocess_kernel<64><<<grid, kPreThreads, 0, st>>>(o4, d4, D, z4, q_weight, s, h, nq,
                                                            nslices, nitems);
  return cudaGetLastError();
}

// dq (bf16) from the fp32 accumulator, both [b, s, h, d].  Work items are
// (query tile, slice of kFinSlice float4 groups) so that a tile's plan weight is
// read once per item; a tile of weight 0 (no key tile reaches it) gets zeros
// without its accumulator rows being read (the pre-pass did not clear them).
constexpr int kFinThreads = 256;
constexpr int64_t kFinSlice = kFinThreads * 8;

__global__ void __launch_bounds__(kFinThreads)
    dq_finalize_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq,
                       const int* __restrict__ q_weight, int64_t s, int64_t nq, int64_t per_tok4,
                       int64_t nslices, int64_t nitems) {
  for (int64_t item = blockIdx.x; item < nitems; item += gridDim.x) {
    const int64_t tile = item / nslices, slice = item % nslices;
    const int64_t bi = tile / nq, t0 = (tile % nq) * kTile;
    const int64_t t1 = t0 + kTile < s ? t0 + kTile : s;
    const int64_t lo = (bi * s + t0) * per_tok4 + slice * kFinSlice;
    const int64_t end = (bi * s + t1) * per_tok4;
    const int64_t hi = lo + kFinSlice < end ? lo + kFinSlice : end;
    const bool live = q_weight[tile] != 0;
#pragma unroll 4
    for (int64_t i = lo + threadIdx.x; i < hi; i += kFinThreads) {
      uint2 o = make_uint2(0u, 0u);
      if (live) {
        const float4 v = acc[i];
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
        const __nv_bfloat162 c = __floats2bfloat162_rn(v.z, v.w);
        o.x = *reinterpret_cast<const uint32_t*>(&a);
        o.y = *reinterpret_cast<const uint32_t*>(&c);
      }
      dq[i] = o;
    }
  }
}

cudaError_t launch_dq_finalize(const float* acc, void* dq, const int* q_weight, int64_t b,
                               int64_t s, int64_t h, int64_t d, cudaStream_t st) {
  const int64_t nq = (s + kTile - 1) / kTile;
  const int64_t per_tok4 = h * d / 4;
  const int64_t nslices = (kTile * per_tok4 + kFinSlice - 1) / kFinSlice;
  const int64_t nitems = b * nq * nslices;
  if (nitems == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<int64_t>(nitems, (int64_t)sm_count() * 16);
  dq_finalize_kernel<<<grid, kFinThreads, 0, st>>>(reinterpret_cast<const float4*>(acc),
                                                   static_cast<uint2*>(dq), q_weight, s, nq,
                                                   per_tok4, nslices, nitems);
  return cudaGetLastError();
}

// ============================================================== descriptors
// Segment ids / positions from per-row lengths and optional start offsets
// (TE tutorial section 1: a packed row's segments are given by ids counted
// from 1 with positions from each segment's start, padding by id 0; the TE
// Cpp attention page's I/O contract takes per-row sequence lengths).  Token t
// of row bi belongs to the last segment j whose start is <= t: pos = t -
// start_j, id = j + 1 inside the segment's length, else 0; a token before
// every start is padding with pos = t.  One CTA takes one row slice: it
// stages the row's starts and lengths in shared memory (running sums of the
// lengths when no offsets are given, saturated at s) and binary-searches
// them per token.
constexpr int kDescTokens = 4096;  // tokens of one row per CTA

__global__ void __launch_bounds__(256) segments_kernel(const int* __restrict__ lens,
                                                       const int* __restrict__ offs, int nseg,
                                                       int64_t s, int* __restrict__ ids,
                                                       int* __restrict__ pos) {
  __shared__ int start[kSegMax];
  __shared__ int len_s[kSegMax];
  const int64_t bi = blockIdx.y;
  const int* lrow = lens + bi * nseg;
  for (int j = threadIdx.x; j < nseg; j += blockDim.x) {
    const int l = lrow[j];
    len_s[j] = l > 0 ? l : 0;
    if (offs) start[j] = offs[bi * nseg + j];
  }
  __syncthreads();
  if (!offs && threadIdx.x < 32) {
    // exclusive running sum of the lengths: lane L scans its own contiguous
    // chunk, the chunk totals are combined with a warp scan.
    const int lane = threadIdx.x;
    const int per = (nseg + 31) / 32;
    const int j0 = lane * per, j1 = min(j0 + per, nseg);
    int64_t sum = 0;
    for (int j = j0; j < j1; ++j) sum += len_s[j];
    int64_t incl = sum;
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int64_t run = incl - sum;
    for (int j = j0; j < j1; ++j) {
      start[j] = (int)(run < s ? run : s);  // saturated: tokens are < s
      run += len_s[j];
    }
  }
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * kDescTokens;
  const int64_t t1 = t0 + kDescTokens < s ? t0 + kDescTokens : s;
  for (int64_t t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
    int lo = 0, hi = nseg;  // first j with start[j] > t
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if ((int64_t)start[mid] <= t) lo = mid + 1;
      else hi = mid;
    }
    const int j = lo - 1;
    int id = 0, p = (int)t;
    if (j >= 0) {
      const int64_t rel = t - start[j];
      p = (int)rel;
      id = rel < len_s[j] ? j + 1 : 0;
    }
    ids[bi * s + t] = id;
    pos[bi * s + t] = p;
  }
}

cudaError_t launch_segments(const int* seqlens, const int* offsets, int64_t b, int64_t nseg,
                            int64_t s, int* ids, int* pos, cudaStream_t st) {
  const dim3 grid((unsigned)((s + kDescTokens - 1) / kDescTokens), (unsigned)b);
  segments_kernel<<<grid, 256, 0, st>>>(seqlens, offsets, (int)nseg, s, ids, pos);
  return cudaGetLastError();
}

}  // namespace gb300
