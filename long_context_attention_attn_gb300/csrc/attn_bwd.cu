// Backward attention over packed THD inputs on sm_103a.
//
// Gradient of sum(O * dO) (TE tutorial section 5 differentiates the vdot of
// the output with dout) through O = softmax(scale * Q K^T + M) V ("Context
// parallelism and ring attention", section "The attention problem"):
//   P = exp(scale * S - LSE),  dV = P^T dO,  dP = dO V^T,
//   dS = P * (dP - D) with D = rowsum(dO * O),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
//
// One CTA owns a 128-key tile of one kv head and keeps dK and dV for it in
// TMEM while it walks over every (query tile, query head of the GQA group)
// that can see the tile (a "step").  Per step it recomputes S^T = K Q^T and
// dP^T = V dO^T on tcgen05 (keys on TMEM lanes), forms P^T and dS^T in
// registers (one thread per key row; one extra K = 16 MMA step subtracts the
// per-query LSE / scale from S^T and D from dP^T, so that no per-column vector
// is read from shared memory), writes them back to TMEM as bf16 (the A
// operands of dV += P^T dO and dK += dS^T Q), stages dS in shared memory for
// dQ = dS K, and adds the dQ tile into an fp32 accumulator in global memory
// with TMA tiled reduce-adds staged through the (then free) dS buffer.
//
// Roles (384 threads): warp 0 TMA producer; warp 1 MMA issuer and TMEM owner;
// warp 2 per-step vector loader; warp 3 dQ reduce issuer;
// warps 4-7 and 8-11 the two element-wise warpgroups (query columns 0-63 and
// 64-127 of S^T / dP^T; each also reads back half of the dQ tile).
// TMEM: dV [0,D)  dK [128,128+D)  S^T [256,384)  dP^T [384,512).  Each
// element-wise half w owns the S^T columns of its 64 queries, [256+64w, 320+64w),
// and overwrites them with its bf16 P^T (first 32 columns) and dS^T (last 32),
// so the halves never wait for each other; the dV / dK MMAs take their A
// operand from the two halves in turn.  The dQ tile (one N = d MMA group) lands
// in the dP^T columns [384, 384+D).  So the next step's S^T only waits for dK,
// and only its dP^T waits for the dQ tile to be read out.
// dQ leaves through shared memory: one half through the dS buffer, the other
// through the just-finished Q stage; warp 3 issues the TMA reduce-adds of the
// dS-buffer half first and hands that buffer back to the next step's dS as soon
// as the TMA has read it, then those of the Q-stage half.
// Where an operation needs several events, they complete one mbarrier with
// several expected arrivals (dP^T(t): dO(t) landed and dQ(t-1) read out; the
// element-wise dS phase: dP^T(t) done and the dS buffer's staging read), so
// that the issuing thread waits once: every wait on the MMA thread's and the
// element-wise warps' path costs latency per step.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int BM = 128;  // query rows per step
constexpr int BN = 128;  // key rows per CTA
constexpr int NQ = 2;    // Q tile stages
constexpr int NV = 4;    // per-step vector ring entries
// vector entry: query ids, pos (128 each), then the step's tile class
constexpr int kVecEntry = 2 * 128 + 32;
// Per-step augment tile (no-swizzle K-major, 128 query rows x 16 bf16): row q
// holds -c split into three bf16 (c = (LSE - ln scale) / scale, so that
// 2^(scale log2(e) (S - c)) = scale * P: P and dS carry the factor that dK and
// dQ need, and dV divides it back out) and -D split likewise, then zeros.
// With the constant "ones" tiles E_S (ones in columns 0-2) and E_D (ones in
// columns 3-5) as A, one extra K = 16 MMA step makes the tensor core deliver
// S^T - c and dP^T - D, so no per-column vector is read in the element-wise
// phases.
constexpr int kAugTile = 128 * 16 * 2;
constexpr float kAugNoKeys = 18446744073709551616.0f;  // 2^64: c of a row without keys
constexpr int kThreads = 384;
// Registers per thread at launch (65536 / 384, rounded down to a multiple of 8).
constexpr int kLaunchRegs = 168;
static_assert(128 * kRegsControl + 256 * kRegsCompute <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr float kLog2e = 1.4426950408889634f;

// x as three bf16 (round to nearest even each) whose fp32 sum is x to about
// 24 bits: the high part, then the rounded residuals.
__device__ __forceinline__ void split_bf16x3(float x, uint32_t out[3]) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h);
  const __nv_bfloat16 m = __float2bfloat16_rn(r1);
  const __nv_bfloat16 l = __float2bfloat16_rn(r1 - __bfloat162float(m));
  out[0] = __bfloat16_as_ushort(h);
  out[1] = __bfloat16_as_ushort(m);
  out[2] = __bfloat16_as_ushort(l);
}

struct BwdArgs {
  const int* q_ids;
  const int* q_pos;
  const int* kv_ids;
  const int* kv_pos;
  const float* lse;
  const float* Dv;
  float* dq_acc;
  void* dk;
  void* dv;
  const uint8_t* cls;
  const int2* krange;
  const int* kweight;
  const int* order;
  int* status;
  int b, s_q, s_kv, hq, hkv, g, nq, nk;
  int window;
  int accumulate;  // dk / dv are fp32 accumulators (add), else bf16 (overwrite)
  int64_t kv_stride;  // elements between consecutive tokens of dk / dv
  float scale;
  float scale_log2;
  float c_shift;  // -ln(scale) / scale: added to c so that the exponent gives scale * P
};

template <int D>
struct BLayout {
  static constexpr int kChunk = 128 * 128;  // 128 rows x 128 bytes
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = 128 * D * 2;
  static constexpr int k_off = 0;
  static constexpr int v_off = k_off + kTile;
  static constexpr int q_off = v_off + kTile;          // NQ stages
  static constexpr int do_off = q_off + NQ * kTile;    // 1 stage
  static constexpr int ds_off = do_off + kTile;        // dS: 128 q x 128 keys bf16, MN-major
  static constexpr int e_off = ds_off + 2 * kChunk;    // E_S, E_D ones tiles
  static constexpr int aug_off = e_off + 2 * kAugTile; // NV augment tiles
  static constexpr int vec_off = aug_off + NV * kAugTile;  // NV x kVecEntry words
  static constexpr int bar_off = vec_off + NV * kVecEntry * 4;
  static constexpr int bytes = bar_off + 256;
  static constexpr int alloc = (bytes + 1024) > 150 * 1024 ? (bytes + 1024) : 150 * 1024;
};

struct BBars {
  uint64_t kv_full;
  uint64_t q_full[NQ];
  uint64_t q_empty[NQ];
  uint64_t dp_ready;  // dO(t) landed and dQ(t-1) read out of TMEM: dP^T(t) may go
  uint64_t do_empty;
  uint64_t vec_full[NV];
  uint64_t vec_empty[NV];
  uint64_t s_full, dp_full, p_full, ds_full, dq_full, dk_done;
  uint64_t stg_ready[2];  // dQ staging written: [0] dS buffer half, [1] Q stage half
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BBars) <= 256, "barrier block too large");

// Iterates over the steps (head, query tile) of a CTA: heads outer, query
// tiles inner.  In the plan's index order, CTAs of neighbouring key tiles of
// one kv head run at the same time and walk the same head in step, so a dQ
// tile receives its reduce-adds from them on consecutive steps while it is
// still in L2.
struct StepIter {
  int i, hh, i_first, i_end, g;
  const uint8_t* cls_col;  // cls + b*nq*nk + c, stride nk
  int nk;
  __device__ bool valid() const { return hh < g; }
  __device__ uint8_t kind() const { return cls_col[(size_t)i * nk]; }
  __device__ void skip_to_valid() {
    while (i <= i_end && cls_col[(size_t)i * nk] == kSkip) ++i;
  }
  __device__ void start() {
    i = i_first;
    skip_to_valid();
    if (i > i_end) hh = g;  // no visible query tile at all
  }
  __device__ void next() {
    ++i;
    skip_to_valid();
    if (i > i_end) {
      ++hh;
      i = i_first;
      skip_to_valid();
    }
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
  using L = BLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  BBars* bars = reinterpret_cast<BBars*>(smem + L::bar_off);
  float* vec = reinterpret_cast<float*>(smem + L::vec_off);  // [NV][kVecEntry]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (a.status && *reinterpret_cast<volatile int*>(a.status) != kStatusOk) return;

  // ---- work unit: kv head slowest, then (b, kv tile) in the plan's work order
  const int nunits = a.b * a.nk;
  const int kvh = blockIdx.x / nunits;
  const int rank = blockIdx.x % nunits;
  const int e = a.order[rank];
  const int bi = e / a.nk;
  const int kt = e % a.nk;
  const int2 rng = a.krange[e];
  const int nsteps_total = a.kweight[e] * a.g;  // (non-SKIP query tile, head) steps
  StepIter it0;
  it0.hh = 0;
  it0.i_first = rng.x;
  it0.i_end = rng.y;
  it0.g = a.g;
  it0.cls_col = a.cls + (size_t)bi * a.nq * a.nk + kt;
  it0.nk = a.nk;
  it0.start();

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    mbar_init(&bars->dp_ready, 1 + 256);  // dO(t) (TMA) + the 256 read-outs of dQ(t-1)
    mbar_init(&bars->do_empty, 1);
    for (int i = 0; i < NV; ++i) {
      mbar_init(&bars->vec_full[i], 1);
      mbar_init(&bars->vec_empty[i], 256);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 2);  // dP^T(t) complete, and the dS buffer's staging of step t-1 read
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dk_done, 1);
    mbar_init(&bars->stg_ready[0], 128);
    mbar_init(&bars->stg_ready[1], 128);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 2) {
    // E_S / E_D (ones in columns 0-2 / 3-5 of each key row) and zeroed
    // augment tiles (their second K half stays zero)
    uint4* e = reinterpret_cast<uint4*>(smem + L::e_off);
    constexpr int kE16 = kAugTile / 16;  // 16-byte units per tile
    const uint32_t one = 0x3F80u;        // bf16 1.0
    for (int i = lane; i < 2 * kE16 + NV * kE16; i += 32) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      const bool first_half = ((i % kE16) % 16) < 8;  // K columns 0-7 of its row
      if (i < kE16 && first_half) v = make_uint4(one | (one << 16), one, 0u, 0u);
      if (i >= kE16 && i < 2 * kE16 && first_half) v = make_uint4(0u, one << 16, one | (one << 16), 0u);
      e[i] = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtx ctx{&bars->abort_flag, a.status};
  constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384;
  // P^T / dS^T of half w: columns [kColS + 64w, +32) / [kColS + 64w + 32, +32)
  constexpr uint32_t kColDQ = 384;

  if (warp < 4) {
  regs_dec<kRegsControl>();
  if (warp == 0) {
    // ======================================================== producer
    int last_q[NQ] = {-1, -1};
    int last_do = -1;
    int nsteps = 0;
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * L::kTile);
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_4d(smem_u32(smem + L::k_off + c * L::kChunk), &tm_k, c * 64, kvh, kt * BN, bi,
                    &bars->kv_full);
        tma_load_4d(smem_u32(smem + L::v_off + c * L::kChunk), &tm_v, c * 64, kvh, kt * BN, bi,
                    &bars->kv_full);
      }
    }
    for (StepIter it = it0; it.valid() && ok; it.next(), ++nsteps) {
      const int t = nsteps;
      const int h = kvh * a.g + it.hh;
      const int qt = it.i;
      // Q tile
      if (lane == 0) {
        const int qs = t % NQ, use = t / NQ;
        ok = mbar_wait(&bars->q_empty[qs], (use & 1) ^ 1, ctx);
        if (ok) {
          mbar_arrive_expect_tx(&bars->q_full[qs], L::kTile);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_4d(smem_u32(smem + L::q_off + qs * L::kTile + c * L::kChunk), &tm_q, c * 64, h,
                        qt * BM, bi, &bars->q_full[qs]);
          last_q[qs] = use;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // dO tile
      if (lane == 0) {
        ok = mbar_wait(&bars->do_empty, (t & 1) ^ 1, ctx);
        if (ok) {
          mbar_arrive_expect_tx(&bars->dp_ready, L::kTile);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_4d(smem_u32(smem + L::do_off + c * L::kChunk), &tm_do, c * 64, h, qt * BM, bi,
                        &bars->dp_ready);
          last_do = t;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {
      mbar_wait_drain(&bars->kv_full, 0, a.status);
      for (int i = 0; i < NQ; ++i)
        if (last_q[i] >= 0) mbar_wait_drain(&bars->q_full[i], last_q[i] & 1, a.status);
      if (last_do >= 0) mbar_wait_drain(&bars->dp_ready, last_do & 1, a.status);
    }
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t id_acc = idesc_bf16_f32(128, D, false, true);    // dV, dK (A in TMEM)
      constexpr uint32_t id_dq = idesc_bf16_f32(128, D, true, true);      // dQ
      // split descriptors (low words): K-major for S^T / dP^T, MN-major otherwise
      const uint32_t k_km = sdesc_lo(smem_u32(smem + L::k_off), 16);
      const uint32_t v_km = sdesc_lo(smem_u32(smem + L::v_off), 16);
      const uint32_t q_km = sdesc_lo(smem_u32(smem + L::q_off), 16);
      const uint32_t do_km = sdesc_lo(smem_u32(smem + L::do_off), 16);
      const uint32_t k_mn = sdesc_lo(smem_u32(smem + L::k_off), L::kChunk);
      const uint32_t q_mn = sdesc_lo(smem_u32(smem + L::q_off), L::kChunk);
      const uint32_t do_mn = sdesc_lo(smem_u32(smem + L::do_off), L::kChunk);
      const uint32_t ds_mn = sdesc_lo(smem_u32(smem + L::ds_off), L::kChunk);
      const uint32_t e_s = sdesc_lo_nosw(smem_u32(smem + L::e_off));
      const uint32_t e_d = sdesc_lo_nosw(smem_u32(smem + L::e_off + kAugTile));
      const uint32_t aug0 = sdesc_lo_nosw(smem_u32(smem + L::aug_off));
      const uint32_t t_s = tmem + kColS, t_dp = tmem + kColDP, t_dq = tmem + kColDQ;
      bool ok = mbar_wait(&bars->kv_full, 0, ctx);
      for (int t = 0; t < nsteps_total && ok; ++t) {
        const int qs = t % NQ;
        const uint32_t qstage = (qs * L::kTile) >> 4;
        ok = mbar_wait(&bars->q_full[qs], (t / NQ) & 1, ctx);
        // the step's augment tile (-c, -D)
        if (ok) ok = mbar_wait(&bars->vec_full[t % NV], (t / NV) & 1, ctx);
        // S^T overwrites P^T / dS^T of the previous step: dV and dK must be done
        if (ok && t > 0) ok = mbar_wait(&bars->dk_done, (t - 1) & 1, ctx);
        if (!ok) break;
        tc_fence_after();
        const uint32_t aug = aug0 + (((t % NV) * kAugTile) >> 4);
        // S^T - c = K Q^T + E_S Aug^T  (M = keys, N = queries, K = d, then 16)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * L::kChunk + (kk % 4) * 32) >> 4;
          mma_ss_lo(t_s, k_km + off, q_km + qstage + off, id_kk, kk > 0 ? 1u : 0u);
        }
        mma_ss_nosw(t_s, e_s, aug, id_kk, 1u);
        mma_commit(&bars->s_full);
        // dP^T = V dO^T
        // dO(t) landed and (dP^T overwrites the previous dQ tile) dQ(t-1) read out
        ok = mbar_wait(&bars->dp_ready, t & 1, ctx);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * L::kChunk + (kk % 4) * 32) >> 4;
          mma_ss_lo(t_dp, v_km + off, do_km + off, id_kk, kk > 0 ? 1u : 0u);
        }
        mma_ss_nosw(t_dp, e_d, aug, id_kk, 1u);  // dP^T - D
        mma_commit(&bars->dp_full);
        // dV += P^T dO  (A = P^T in TMEM, B = dO MN-major)
        ok = mbar_wait(&bars->p_full, t & 1, ctx);
        if (!ok) break;
        tc_fence_after();
        const uint32_t acc0 = t > 0 ? 1u : 0u;
        // K-steps 0-3 read half 0's P^T, 4-7 half 1's
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_ts_lo(tmem + kColDV, t_s + (kk / 4) * 64 + (kk % 4) * 8,
                    do_mn + ((kk * 2048) >> 4), id_acc, kk > 0 ? 1u : acc0);
        mma_commit(&bars->do_empty);
        // dQ = dS K  (A = dS in smem MN-major, B = K MN-major), N = d
        ok = mbar_wait(&bars->ds_full, t & 1, ctx);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ss_lo(t_dq, ds_mn + ((kk * 2048) >> 4), k_mn + ((kk * 2048) >> 4), id_dq,
                    kk > 0 ? 1u : 0u);
        mma_commit(&bars->dq_full);
        // dK += dS^T Q  (A = dS^T in TMEM, B = Q MN-major)
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_ts_lo(tmem + kColDK, t_s + (kk / 4) * 64 + 32 + (kk % 4) * 8,
                    q_mn + qstage + ((kk * 2048) >> 4), id_acc, kk > 0 ? 1u : acc0);
        mma_commit(&bars->dk_done);
      }
      mma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, a.status);
    }
  } else if (warp == 3) {
    // ======================================================== dQ reduce issuer
    if (lane == 0) {
      int t = 0;
      bool ok = true;
      mbar_arrive(&bars->dp_full);  // step 0's dS buffer holds no staging
      for (StepIter it = it0; it.valid() && ok; it.next(), ++t) {
        const int h = kvh * a.g + it.hh;
        const int qt = it.i;
        constexpr int kHalfR = D / 2, kRoundsR = kHalfR / 32;
        const uint32_t s0 = smem_u32(smem + L::ds_off);
        const uint32_t s1 = smem_u32(smem + L::q_off + (t % NQ) * L::kTile);
        ok = mbar_wait(&bars->stg_ready[0], t & 1, ctx);
        if (!ok) break;
#pragma unroll
        for (int k = 0; k < kRoundsR; ++k)
          tma_reduce_add_4d(&tm_dq, s0 + k * L::kChunk, 32 * k, h, qt * BM, bi);
        bulk_commit_group();
        // The next step's stg_ready[1] phase must not complete before this wait
        // has seen the current one: it follows the dp_full arrival below.
        ok = mbar_wait(&bars->stg_ready[1], t & 1, ctx);
        if (!ok) break;
#pragma unroll
        for (int k = 0; k < kRoundsR; ++k)
          tma_reduce_add_4d(&tm_dq, s1 + k * L::kChunk, kHalfR + 32 * k, h, qt * BM, bi);
        bulk_commit_group();
        bulk_wait_group_read<1>();
        mbar_arrive(&bars->dp_full);  // dS buffer half read: the next step's dS may go there
        bulk_wait_group_read<0>();
        mbar_arrive(&bars->q_empty[t % NQ]);  // Q stage reusable
      }
      bulk_wait_group0();  // every dQ reduce-add has landed before the CTA exits
    }
  } else if (warp == 2) {
    // ======================================================== vector loader
    // Per step: the augment tile (-LSE / scale and -D, each split into three
    // bf16; a row without keys takes 2^64, so P = 0), read by the S^T and dP^T
    // MMAs, and the query ids / pos and the step's tile class, read by the
    // element-wise warpgroups (off the TMA producer's path).
    int t = 0;
    bool ok = true;
    for (StepIter it = it0; it.valid() && ok; it.next(), ++t) {
      const int h = kvh * a.g + it.hh;
      const int qt = it.i;
      const int en = t % NV, use = t / NV;
      const int64_t lbase = ((int64_t)bi * a.hq + h) * a.s_q;
      const int64_t ibase = (int64_t)bi * a.s_q;
      float vl[BM / 32], vd[BM / 32];
      int vid[BM / 32], vps[BM / 32];
#pragma unroll
      for (int u = 0; u < BM / 32; ++u) {
        const int gq = qt * BM + u * 32 + lane;
        const bool in = gq < a.s_q;
        vl[u] = in ? a.lse[lbase + gq] : -INFINITY;
        vd[u] = in ? a.Dv[lbase + gq] : 0.f;
        vid[u] = in ? a.q_ids[ibase + gq] : 0;
        vps[u] = in ? a.q_pos[ibase + gq] : 0;
      }
      const int kind = it.kind();
      if (lane == 0) ok = mbar_wait(&bars->vec_empty[en], (use & 1) ^ 1, ctx);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      int* vi = reinterpret_cast<int*>(vec + en * kVecEntry);
      uint8_t* aug = smem + L::aug_off + en * kAugTile;
      const float inv_scale = 1.f / a.scale;
#pragma unroll
      for (int u = 0; u < BM / 32; ++u) {
        const int r = u * 32 + lane;
        vi[r] = vid[u];
        vi[BM + r] = vps[u];
        // -c and -D, each as three bf16 whose sum is the fp32 value
        const float c = (vl[u] == -INFINITY) ? kAugNoKeys : vl[u] * inv_scale + a.c_shift;
        uint32_t cs[3], ds[3];
        split_bf16x3(-c, cs);
        split_bf16x3(-vd[u], ds);
        *reinterpret_cast<uint4*>(aug + (r / 8) * 256 + (r % 8) * 16) =
            make_uint4(cs[0] | (cs[1] << 16), cs[2] | (ds[0] << 16), ds[1] | (ds[2] << 16), 0u);
      }
      if (lane == 0) {
        vi[2 * BM] = kind;
      }
      fence_proxy_async_smem();  // the augment tile is read by the MMAs
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->vec_full[en]);
    }
  }
  } else {
  regs_inc<kRegsCompute>();
  {
    // ======================================================== element-wise
    const int w = (warp - 4) / 4;  // query columns [64w, 64w + 64)
    const int wq = warp % 4;
    const int kr = wq * 32 + lane;  // key row (S^T lanes) / query row (dQ lanes)
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int key = kt * BN + kr;
    const bool key_in = key < a.s_kv;
    const int ik = key_in ? a.kv_ids[(int64_t)bi * a.s_kv + key] : 0;
    const int pk = key_in ? a.kv_pos[(int64_t)bi * a.s_kv + key] : 0;
    const float sl2 = a.scale_log2;
    uint8_t* ds_smem = smem + L::ds_off + w * L::kChunk + kr * 128;
    constexpr int kHalf = D / 2;         // dQ columns read back by this half
    constexpr int kRounds = kHalf / 32;  // 32-column staging boxes per half
    int t = 0;
    bool ok = true;
    // step 0's dP^T has no previous dQ tile to wait for
    mbar_arrive(&bars->dp_ready);
    for (; t < nsteps_total; ++t) {
      const int en = t % NV;
      ok = mbar_wait(&bars->vec_full[en], (t / NV) & 1, ctx);
      ok = mbar_wait(&bars->s_full, t & 1, ctx) && ok;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int* ventry = reinterpret_cast<const int*>(vec + en * kVecEntry);
      const bool partial = ventry[2 * BM] == kPartial;
      const int* qid = ventry + 64 * w;
      const int* qpos = ventry + BM + 64 * w;
      uint32_t r[64];
      tmem_ld32(tmem + lane_off + kColS + 64 * w, &r[0]);
      tmem_ld32(tmem + lane_off + kColS + 64 * w + 32, &r[32]);
      tmem_wait_ld();
      // the tensor core already subtracted c: p = 2^(scale log2(e) (S - c)) = scale * P
      float p[64];
#pragma unroll
      for (int u = 0; u < 64; u += 2) {
        float x0, x1;
        mul_f32x2(x0, x1, __uint_as_float(r[u]), __uint_as_float(r[u + 1]), sl2, sl2);
        p[u] = ex2(x0);
        p[u + 1] = ex2(x1);
      }
      if (partial) {
        const int4* id4 = reinterpret_cast<const int4*>(qid);
        const int4* ps4 = reinterpret_cast<const int4*>(qpos);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int4 i4 = id4[c];
          const int4 q4 = ps4[c];
          const int ia[4] = {i4.x, i4.y, i4.z, i4.w};
          const int qa[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            bool vis = (ia[u] == ik) && (ik != 0) && (pk <= qa[u]);
            if (a.window >= 0) vis = vis && (qa[u] - pk <= a.window);
            if (!vis) p[4 * c + u] = 0.f;
          }
        }
      }
      uint32_t pk2[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) pk2[u] = pack_bf16(p[2 * u], p[2 * u + 1]);
      tmem_st32(tmem + lane_off + kColS + 64 * w, pk2);  // own columns: no wait
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
      // dS^T = P^T * (dP^T - D)
      ok = mbar_wait(&bars->dp_full, t & 1, ctx);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_off + kColDP + 64 * w, &r[0]);
      tmem_ld32(tmem + lane_off + kColDP + 64 * w + 32, &r[32]);
      tmem_wait_ld();
      // dP^T - D came from the tensor core
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float d0, d1;
        mul_f32x2(d0, d1, p[2 * c], p[2 * c + 1], __uint_as_float(r[2 * c]),
                  __uint_as_float(r[2 * c + 1]));
        pk2[c] = pack_bf16(d0, d1);
      }
      tmem_st32(tmem + lane_off + kColS + 64 * w + 32, pk2);
      // (The dS buffer doubles as the dQ staging area of the previous step:
      // dp_full also waited until the TMA had read it.)
      // dS (queries x keys) in shared memory, MN-major 128B-swizzled: key row kr
      // holds this half's 64 query values.
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint4 v4 = make_uint4(pk2[4 * u], pk2[4 * u + 1], pk2[4 * u + 2], pk2[4 * u + 3]);
        *reinterpret_cast<uint4*>(ds_smem + ((u ^ (kr & 7)) * 16)) = v4;
      }
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);
      // dQ tile readout: TMEM lanes are query rows here.  Half 1 stages its
      // columns in the Q stage, whose last reader is dK (issued after dQ): it
      // waits for dK alone, whose commit covers dQ too.
      ok = (w == 0) ? mbar_wait(&bars->dq_full, t & 1, ctx) : mbar_wait(&bars->dk_done, t & 1, ctx);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t q[kHalf];
      const uint32_t src = tmem + lane_off + kColDQ + kHalf * w;
#pragma unroll
      for (int c = 0; c < kHalf; c += 32) tmem_ld32(src + c, &q[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->dp_ready);  // for the next step's dP^T
      // dQ (scaled already: dS carries the factor) into the fp32 accumulator.  Half 0 stages its columns in
      // the dS buffer (free: the dQ MMA has read it), half 1 in the Q stage of
      // this step (free once dK, its last reader, is done), as 32-column boxes
      // of 128 rows x 128 B (128B-swizzled); warp 3 issues the reduce-adds.
      {
        uint8_t* stage = (w == 0) ? smem + L::ds_off : smem + L::q_off + (t % NQ) * L::kTile;
#pragma unroll
        for (int k = 0; k < kRounds; ++k) {
          uint8_t* box = stage + k * L::kChunk + kr * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 v4 = make_float4(__uint_as_float(q[32 * k + 4 * u]),
                                          __uint_as_float(q[32 * k + 4 * u + 1]),
                                          __uint_as_float(q[32 * k + 4 * u + 2]),
                                          __uint_as_float(q[32 * k + 4 * u + 3]));
            *reinterpret_cast<float4*>(box + ((u ^ (kr & 7)) * 16)) = v4;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->stg_ready[w]);
      }
      mbar_arrive(&bars->vec_empty[en]);
    }
    // ---- epilogue: dV (half 0) and dK (half 1) rows of this key tile: bf16,
    // or added into fp32 accumulators
    if (ok && t > 0) {
      ok = mbar_wait(&bars->dk_done, (t - 1) & 1, ctx);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    if (ok) {
      // P was formed as scale * P (so dS too): dK and dQ carry their factor
      // already, dV takes it back out
      const float sc = (w == 0) ? 1.f / a.scale : 1.f;
      const int64_t row0 = ((int64_t)bi * a.s_kv + key) * a.kv_stride + (int64_t)kvh * D;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        if (t > 0) {
          tmem_ld32(tmem + lane_off + (w == 0 ? kColDV : kColDK) + c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = 0u;
        }
        if (!key_in) continue;
        if (a.accumulate) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(w == 0 ? a.dv : a.dk) +
                                                  row0 + c);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float4 v = dst[u];
            v.x += __uint_as_float(o[4 * u + 0]) * sc;
            v.y += __uint_as_float(o[4 * u + 1]) * sc;
            v.z += __uint_as_float(o[4 * u + 2]) * sc;
            v.w += __uint_as_float(o[4 * u + 3]) * sc;
            dst[u] = v;
          }
          continue;
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(w == 0 ? a.dv : a.dk) +
                                              row0 + c);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 v;
          v.x = pack_bf16(__uint_as_float(o[8 * u + 0]) * sc, __uint_as_float(o[8 * u + 1]) * sc);
          v.y = pack_bf16(__uint_as_float(o[8 * u + 2]) * sc, __uint_as_float(o[8 * u + 3]) * sc);
          v.z = pack_bf16(__uint_as_float(o[8 * u + 4]) * sc, __uint_as_float(o[8 * u + 5]) * sc);
          v.w = pack_bf16(__uint_as_float(o[8 * u + 6]) * sc, __uint_as_float(o[8 * u + 7]) * sc);
          dst[u] = v;
        }
      }
    }
  }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_attn_bwd(const BwdLaunch& Lc, cudaStream_t st) {
  const attn_bwd_params& p = *Lc.p;
  const attn_fwd_params& f = p.fwd;
  BwdArgs a;
  a.q_ids = f.q_segment_ids;
  a.q_pos = f.q_segment_pos;
  a.kv_ids = f.kv_segment_ids;
  a.kv_pos = f.kv_segment_pos;
  a.lse = f.lse;
  a.Dv = Lc.D;
  a.dq_acc = Lc.dq_acc;
  a.dk = p.dk;
  a.dv = p.dv;
  a.cls = Lc.plan.classes;
  a.krange = Lc.plan.kv_range;
  a.kweight = Lc.plan.kv_weight;
  a.order = Lc.plan.kv_order;
  a.status = Lc.plan.status;
  a.b = (int)f.b;
  a.s_q = (int)f.s_q;
  a.s_kv = (int)f.s_kv;
  a.hq = (int)f.h_q;
  a.hkv = (int)f.h_kv;
  a.g = (int)(f.h_q / f.h_kv);
  a.nq = (int)Lc.nq;
  a.nk = (int)Lc.nk;
  a.window = f.window_left;
  a.accumulate = p.accumulate_fp32 ? 1 : 0;
  a.kv_stride = f.kv_token_stride > 0 ? f.kv_token_stride : f.h_kv * f.d;
  a.scale = f.scale;
  a.scale_log2 = f.scale * kLog2e;
  a.c_shift = -logf(f.scale) / f.scale;
  const int64_t units = f.b * Lc.nk * f.h_kv;
  if (units == 0) return cudaSuccess;
  if (f.d == 128) {
    const int smem = BLayout<128>::alloc;
    static std::atomic<int> smem_set[kMaxDevices];
    cudaError_t e =
        ensure_smem_limit(reinterpret_cast<const void*>(attn_bwd_kernel<128>), smem,
                          kLaunchRegs, smem_set);
    if (e != cudaSuccess) return e;
    attn_bwd_kernel<128><<<(unsigned)units, kThreads, smem, st>>>(Lc.tm_q, Lc.tm_k, Lc.tm_v,
                                                                  Lc.tm_do, Lc.tm_dq, a);
  } else {
    const int smem = BLayout<64>::alloc;
    static std::atomic<int> smem_set[kMaxDevices];
    cudaError_t e =
        ensure_smem_limit(reinterpret_cast<const void*>(attn_bwd_kernel<64>), smem,
                          kLaunchRegs, smem_set);
    if (e != cudaSuccess) return e;
    attn_bwd_kernel<64><<<(unsigned)units, kThreads, smem, st>>>(Lc.tm_q, Lc.tm_k, Lc.tm_v,
                                                                 Lc.tm_do, Lc.tm_dq, a);
  }
  return cudaGetLastError();
}

}  // namespace gb300
