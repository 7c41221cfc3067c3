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

__global__ void tile_summary_kernel(const int* __restrict__ ids, const int* __restrict__ pos,
                                    int64_t b, int64_t s, int64_t ntile,
                                    TileSummary* __restrict__ out) {
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= b * ntile) return;
  const int64_t bi = w / ntile, t = w % ntile;
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
  if (lane == 0) {
    TileSummary r;
    r.any_valid = any_valid;
    r.has_pad = has_pad;
    r.id_min = any_valid ? id_min : 0;
    r.id_max = any_valid ? id_max : 0;
    r.pos_min = any_valid ? pmin : 0;
    r.pos_max = any_valid ? pmax : 0;
    r.reserved0 = r.reserved1 = 0;
    out[w] = r;
  }
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

// One CTA per (kv tile, b): the range of q tiles that see it (backward side).
__global__ void kv_range_kernel(const uint8_t* __restrict__ cls, int64_t nq, int64_t nk,
                                int2* __restrict__ krange, int* __restrict__ kweight) {
  const int64_t c = blockIdx.x, bi = blockIdx.y;
  __shared__ int s_first, s_last, s_count;
  if (threadIdx.x == 0) {
    s_first = INT_MAX;
    s_last = -1;
    s_count = 0;
  }
  __syncthreads();
  int first = INT_MAX, last = -1, count = 0;
  for (int64_t a = threadIdx.x; a < nq; a += blockDim.x) {
    if (cls[(bi * nq + a) * nk + c] != kSkip) {
      first = min(first, (int)a);
      last = max(last, (int)a);
      ++count;
    }
  }
  atomicMin(&s_first, first);
  atomicMax(&s_last, last);
  atomicAdd(&s_count, count);
  __syncthreads();
  if (threadIdx.x == 0) {
    krange[bi * nk + c] = s_last < 0 ? make_int2(0, -1) : make_int2(s_first, s_last);
    kweight[bi * nk + c] = s_count;
  }
}

// Stable counting sort of n work rows by weight, heaviest first (single CTA):
// rows of equal weight keep their index order, so neighbouring tiles stay
// neighbours in the launch order (their K/V, Q and dQ tiles are then shared
// through L2 by the CTAs running at the same time).  Weights above
// kBuckets - 1 share the top bucket.
constexpr int kBuckets = 2048;
constexpr int kSortChunk = 1024;
__global__ void heavy_first_kernel(const int* __restrict__ weight, int n, int* __restrict__ order) {
  __shared__ int hist[kBuckets];
  __shared__ int start[kBuckets];
  __shared__ int chunk_w[kSortChunk];
  for (int i = threadIdx.x; i < kBuckets; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    atomicAdd(&hist[min(weight[i], kBuckets - 1)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int w = kBuckets - 1; w >= 0; --w) {
      start[w] = acc;
      acc += hist[w];
    }
  }
  __syncthreads();
  for (int c0 = 0; c0 < n; c0 += kSortChunk) {
    const int m = min(kSortChunk, n - c0);
    for (int t = threadIdx.x; t < m; t += blockDim.x)
      chunk_w[t] = min(weight[c0 + t], kBuckets - 1);
    __syncthreads();
    for (int t = threadIdx.x; t < m; t += blockDim.x) {
      const int w = chunk_w[t];
      int before = 0;  // earlier rows of this chunk with the same weight
      for (int j = 0; j < t; ++j) before += (chunk_w[j] == w);
      order[start[w] + before] = c0 + t;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < m; t += blockDim.x) atomicAdd(&start[chunk_w[t]], 1);
    __syncthreads();
  }
}

cudaError_t launch_tile_plan(const attn_fwd_params& p, const PlanPtrs& pp, int64_t nq, int64_t nk,
                             bool need_kv_side, cudaStream_t st) {
  const int wpb = 8;
  tile_summary_kernel<<<(unsigned)((p.b * nq + wpb - 1) / wpb), wpb * 32, 0, st>>>(
      p.q_segment_ids, p.q_segment_pos, p.b, p.s_q, nq, pp.q_sum);
  tile_summary_kernel<<<(unsigned)((p.b * nk + wpb - 1) / wpb), wpb * 32, 0, st>>>(
      p.kv_segment_ids, p.kv_segment_pos, p.b, p.s_kv, nk, pp.kv_sum);
  tile_class_kernel<<<dim3((unsigned)nq, (unsigned)p.b), 256, 0, st>>>(
      pp.q_sum, pp.kv_sum, nq, nk, p.window_left, pp.classes, pp.q_range, pp.q_weight);
  heavy_first_kernel<<<1, 1024, 0, st>>>(pp.q_weight, (int)(p.b * nq), pp.q_order);
  if (need_kv_side) {
    kv_range_kernel<<<dim3((unsigned)nk, (unsigned)p.b), 256, 0, st>>>(pp.classes, nq, nk,
                                                                      pp.kv_range, pp.kv_weight);
    heavy_first_kernel<<<1, 1024, 0, st>>>(pp.kv_weight, (int)(p.b * nk), pp.kv_order);
  }
  return cudaGetLastError();
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
template <int D>
__global__ void bwd_preprocess_kernel(const uint4* __restrict__ out, const uint4* __restrict__ dout,
                                      float* __restrict__ Dv, float4* __restrict__ zero_acc,
                                      int64_t b, int64_t s, int64_t h) {
  constexpr int kLanes = D / 8;            // lanes per row-head
  constexpr int kRowsPerWarp = 32 / kLanes;
  const int lane = threadIdx.x & 31;
  const int sub = lane % kLanes;
  const int64_t nrows = b * s * h;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  for (int64_t r0 = warp0 * kRowsPerWarp; r0 < nrows; r0 += nwarps * kRowsPerWarp * 2) {
    // two independent row groups per iteration keep more bytes in flight
    const int64_t ra = r0 + lane / kLanes;
    const int64_t rb = ra + nwarps * kRowsPerWarp;
    uint4 oa = make_uint4(0, 0, 0, 0), da = oa, ob = oa, db = oa;
    if (ra < nrows) {
      oa = out[ra * kLanes + sub];
      da = dout[ra * kLanes + sub];
    }
    if (rb < nrows) {
      ob = out[rb * kLanes + sub];
      db = dout[rb * kLanes + sub];
    }
    if (zero_acc) {
      // the fp32 dQ accumulator has out's layout: clear this thread's 8 values
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ra < nrows) {
        zero_acc[(ra * kLanes + sub) * 2] = z;
        zero_acc[(ra * kLanes + sub) * 2 + 1] = z;
      }
      if (rb < nrows) {
        zero_acc[(rb * kLanes + sub) * 2] = z;
        zero_acc[(rb * kLanes + sub) * 2 + 1] = z;
      }
    }
    auto dot8 = [](const uint4& x, const uint4& y) {
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
      const uint32_t ys[4] = {y.x, y.y, y.z, y.w};
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[k]));
        const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[k]));
        acc += a.x * c.x + a.y * c.y;
      }
      return acc;
    };
    float sa = dot8(oa, da), sb = dot8(ob, db);
#pragma unroll
    for (int off = kLanes / 2; off > 0; off >>= 1) {
      sa += __shfl_xor_sync(0xffffffffu, sa, off);
      sb += __shfl_xor_sync(0xffffffffu, sb, off);
    }
    if (sub == 0) {
      if (ra < nrows) {
        const int64_t hh = ra % h, ti = (ra / h) % s, bi = ra / (h * s);
        Dv[(bi * h + hh) * s + ti] = sa;
      }
      if (rb < nrows) {
        const int64_t hh = rb % h, ti = (rb / h) % s, bi = rb / (h * s);
        Dv[(bi * h + hh) * s + ti] = sb;
      }
    }
  }
}

cudaError_t launch_bwd_preprocess(const void* out, const void* dout, float* D, float* zero_acc,
                                  int64_t b, int64_t s, int64_t h, int64_t d, cudaStream_t st) {
  const int64_t rows = b * s * h;
  const int rows_per_cta = 8 * (d == 256 ? 1 : d == 128 ? 2 : 4);
  const unsigned grid =
      (unsigned)std::min<int64_t>((rows + rows_per_cta - 1) / rows_per_cta, (int64_t)sm_count() * 16);
  if (d == 256)
    bwd_preprocess_kernel<256><<<grid, 256, 0, st>>>(static_cast<const uint4*>(out),
                                                     static_cast<const uint4*>(dout), D,
                                                     reinterpret_cast<float4*>(zero_acc), b, s, h);
  else if (d == 128)
    bwd_preprocess_kernel<128><<<grid, 256, 0, st>>>(static_cast<const uint4*>(out),
                                                     static_cast<const uint4*>(dout), D,
                                                     reinterpret_cast<float4*>(zero_acc), b, s, h);
  else
    bwd_preprocess_kernel<64><<<grid, 256, 0, st>>>(static_cast<const uint4*>(out),
                                                    static_cast<const uint4*>(dout), D,
                                                    reinterpret_cast<float4*>(zero_acc), b, s, h);
  return cudaGetLastError();
}

__global__ void dq_finalize_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq,
                                   int64_t n4) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = acc[i];
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 c = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&a);
    o.y = *reinterpret_cast<const uint32_t*>(&c);
    dq[i] = o;
  }
}

cudaError_t launch_dq_finalize(const float* acc, void* dq, int64_t n, cudaStream_t st) {
  const int64_t n4 = n / 4;
  const unsigned grid = (unsigned)std::min<int64_t>((n4 + 255) / 256, (int64_t)sm_count() * 16);
  dq_finalize_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const float4*>(acc),
                                           static_cast<uint2*>(dq), n4);
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
