// Backward attention as two kernels, on sm_103a: one for dK / dV, one for dQ.
//
// Gradient of sum(O * dO) (TE tutorial section 5 differentiates the vdot of
// the output with dout) through O = softmax(scale * Q K^T + M) V ("Context
// parallelism and ring attention", section "The attention problem"):
//   P = exp(scale * S - LSE),  dV = P^T dO,  dP = dO V^T,
//   dS = P * (dP - D) with D = rowsum(dO * O),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
//
// attn_bwd_dkdv_kernel: one CTA owns a 128-key tile of one kv head (and, for
// the widest head dims, one column slice of dK / dV) and keeps dK and dV in
// TMEM while it walks every (query head of the GQA group, query rows) step
// that can see the tile.  Per step: S^T = K Q^T and dP^T = V dO^T (keys on
// TMEM lanes; one extra K = 16 MMA step against constant "ones" tiles
// subtracts the per-query c = (LSE - ln scale) / scale and D, so the
// exponent yields scale * P and dS carries the scale dK needs), P^T and dS^T
// in registers, written back to TMEM as bf16 as the A operands of
// dV += P^T dO and dK += dS^T Q.
//
// attn_bwd_dq_tmem_kernel: one CTA owns a 128-row query tile of one query
// head and keeps dQ in TMEM while it walks the key tiles the tile sees, as
// the forward pass does: S = Q K^T and dP = dO V^T (queries on TMEM lanes, so
// LSE and D are per-thread scalars; Q, and dO where it fits, held in TMEM as
// the A operands), scale * dS = scale * P * (dP - D) written back as bf16 over
// the dP columns, the A operand of dQ += dS K.  dQ leaves TMEM once, as bf16
// (or added into an fp32 accumulator), so no partial sum of dQ ever travels
// through global memory.
//
// Both kernels: warp 0 TMA producer, warp 1 MMA issuer and TMEM owner, warp 2
// per-step vector / descriptor loader, warps 4-11 two element-wise
// warpgroups (warp 3 idle).  Every wait is bounded (see ptx.cuh).  Where a
// product needs its operand tile and a TMEM region to be free, both events
// complete the tile's barrier (the region's readers arrive on it as well), so
// the MMA thread waits once per product: each extra wait on its path costs
// latency every step.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;  // 65536 / 384 rounded down to a multiple of 8
static_assert(128 * kRegsControl + 256 * kRegsCompute <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kAugNoKeys = 18446744073709551616.0f;  // 2^64: c of a row without keys
constexpr int NV = 4;    // per-step vector ring entries (dK/dV kernel)
constexpr int NID = 4;   // key descriptor ring entries (dQ kernel)

// x as three bf16 (each rounded to nearest even) whose fp32 sum is x to about
// 24 bits: the high part, then the rounded residuals.
__device__ __forceinline__ void split3(float x, uint32_t out[3]) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h);
  const __nv_bfloat16 m = __float2bfloat16_rn(r1);
  const __nv_bfloat16 l = __float2bfloat16_rn(r1 - __bfloat162float(m));
  out[0] = __bfloat16_as_ushort(h);
  out[1] = __bfloat16_as_ushort(m);
  out[2] = __bfloat16_as_ushort(l);
}

struct SplitArgs {
  const __nv_bfloat16* k;  // read directly when the key / value tile is kept in TMEM
  const __nv_bfloat16* v;
  const int* q_ids;
  const int* q_pos;
  const int* kv_ids;
  const int* kv_pos;
  const float* lse;
  const float* Dv;
  void* dq;
  void* dk;
  void* dv;
  const uint8_t* cls;
  const int2* range;   // kv side (dK/dV kernel) or q side (dQ kernel)
  const int* weight;
  const int* order;
  int* status;
  int b, s_q, s_kv, hq, hkv, g, nq, nk;
  int window;
  int accumulate;    // dq / dk / dv are fp32 accumulators (add), else bf16 (overwrite)
  int64_t k_stride;  // elements between consecutive tokens of dk
  int64_t v_stride;  // ... of dv
  float scale;
  float scale_log2;
  float c_shift;     // -ln(scale) / scale
};

__device__ __forceinline__ bool visible(int iq, int pq, int ik, int pk, int window) {
  bool v = (iq == ik) && (iq != 0) && (pk <= pq);
  if (window >= 0) v = v && (pq - pk <= window);
  return v;
}

// ============================================================== dK / dV
// DK, DV: head dims of q / k and of v; BM: query rows per step (128, or 64
// where the head dims leave no room); NSPLIT: column slices of dK / dV (each
// CTA owns one); NQ / NO: Q / dO shared-memory stages; KT / VT: the key /
// value tile is kept in TMEM (the A operand of S^T = K Q^T / dP^T = V dO^T)
// instead of shared memory, where the TMEM columns allow: at d = 256 the key
// tile (which frees the room for two Q and two dO stages), for MLA the value
// tile (the product then reads only dO from shared memory).
template <int DK, int DV, int BM, int NSPLIT, int NQ, int NO, bool KT = false, bool VT = false>
struct ALayout {
  static constexpr int DKS = DK / NSPLIT;  // dK columns of this CTA
  static constexpr int DVS = DV / NSPLIT;  // dV columns of this CTA
  static constexpr int kKChunk = 128 * 128;  // 128 key rows x 128 B (64 bf16)
  static constexpr int kQChunk = BM * 128;   // BM query rows x 128 B
  static constexpr int kKTile = 128 * DK * 2;
  static constexpr int kVTile = 128 * DV * 2;
  static constexpr int kQTile = BM * DK * 2;
  static constexpr int kOTile = BM * DV * 2;
  static constexpr int kAug = BM * 16 * 2;   // augment tile: BM query rows x 16 bf16
  static constexpr int kE = 128 * 16 * 2;    // "ones" tile: 128 key rows x 16 bf16
  static constexpr int kVec = 2 * BM + 32;   // ids, pos of the step's rows, then the class
  static constexpr int k_off = 0;
  static constexpr int v_off = k_off + (KT ? 0 : kKTile);
  static constexpr int kVTileS = VT ? 0 : kVTile;  // bytes of V in shared memory
  static constexpr int q_off = v_off + kVTileS;
  static constexpr int do_off = q_off + NQ * kQTile;
  static constexpr int e_off = do_off + NO * kOTile;
  static constexpr int aug_off = e_off + 2 * kE;
  static constexpr int vec_off = aug_off + NV * kAug;
  static constexpr int bar_off = vec_off + NV * kVec * 4;
  static constexpr int bytes = bar_off + 256;
  static constexpr int alloc = (bytes + 1024) > 150 * 1024 ? (bytes + 1024) : 150 * 1024;
  // TMEM columns: two BM-wide regions that S^T and dP^T take in turn (step t:
  // S^T in region t & 1, dP^T in the other), then the dV and dK slices
  static constexpr uint32_t kColR = 0, kColDV = 2 * BM, kColDK = 2 * BM + DVS,
                            kColK = 2 * BM + DVS + DKS,                   // the key tile (KT)
                            kColV = 2 * BM + DVS + DKS + (KT ? DK / 2 : 0);  // the value tile (VT)
  static_assert(kColV + (VT ? DV / 2 : 0) <= 512, "TMEM columns");
  static_assert(alloc <= 232448, "shared memory per block");
  static_assert(DKS % 64 == 0 || DKS == 64 || DKS % 32 == 0, "dK slice");
};

struct ABars {
  uint64_t kv_full;
  uint64_t k_full;  // the key / value tiles are in TMEM (KT, VT)
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t do_full[2];
  uint64_t do_empty[2];
  uint64_t vec_full[NV];
  uint64_t vec_empty[NV];
  uint64_t s_full, dp_full, p_full, ds_full, dk_done, drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(ABars) <= 256, "barrier block too large");

// Steps of a dK/dV CTA: heads outer, then the non-SKIP 128-row query tiles,
// then the BM-row parts of each.
template <int BM>
struct AStepIter {
  static constexpr int kSub = 128 / BM;
  int i, sub, hh, i_first, i_end, g;
  const uint8_t* cls_col;  // cls + b*nq*nk + kv tile, stride nk
  int nk;
  __device__ bool valid() const { return hh < g; }
  __device__ uint8_t kind() const { return cls_col[(size_t)i * nk]; }
  __device__ void skip_to_valid() {
    while (i <= i_end && cls_col[(size_t)i * nk] == kSkip) ++i;
  }
  __device__ void start() {
    i = i_first;
    sub = 0;
    skip_to_valid();
    if (i > i_end) hh = g;
  }
  __device__ void next() {
    if (++sub < kSub) return;
    sub = 0;
    ++i;
    skip_to_valid();
    if (i > i_end) {
      ++hh;
      i = i_first;
      skip_to_valid();
    }
  }
  __device__ int row0() const { return i * 128 + sub * BM; }
};

template <int DK, int DV, int BM, int NSPLIT, int NQ, int NO, bool KT, bool VT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do, const SplitArgs a) {
  using L = ALayout<DK, DV, BM, NSPLIT, NQ, NO, KT, VT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  ABars* bars = reinterpret_cast<ABars*>(smem + L::bar_off);
  int* vec = reinterpret_cast<int*>(smem + L::vec_off);  // [NV][kVec]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (a.status && *reinterpret_cast<volatile int*>(a.status) != kStatusOk) return;

  // ---- work unit: kv head slowest, then (b, kv tile) in work order, then slice
  const int nunits = a.b * a.nk;
  const int kvh = blockIdx.x / (nunits * NSPLIT);
  const int rem = blockIdx.x % (nunits * NSPLIT);
  const int ks = rem % NSPLIT;
  const int e = a.order[rem / NSPLIT];
  const int bi = e / a.nk;
  const int kt = e % a.nk;
  const int2 rng = a.range[e];
  const int nsteps_total = a.weight[e] * a.g * AStepIter<BM>::kSub;
  AStepIter<BM> it0;
  it0.hh = 0;
  it0.i_first = rng.x;
  it0.i_end = rng.y;
  it0.g = a.g;
  it0.cls_col = a.cls + (size_t)bi * a.nq * a.nk + kt;
  it0.nk = a.nk;
  it0.start();

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->k_full, 256);  // every element-wise thread stores its part of the key tile
    for (int i = 0; i < 2; ++i) {
      // Q(t) landed (TMA) and dP^T(t-1) read by the 256 element-wise threads
      // (S^T(t) goes into the region dP^T(t-1) leaves)
      mbar_init(&bars->q_full[i], 1 + 256);
      mbar_init(&bars->q_empty[i], 1);
      // dO(t) landed (TMA) and dK(t-1) done (dP^T(t) goes into the region
      // P^T / dS^T(t-1) leave; MMA commit)
      mbar_init(&bars->do_full[i], 1 + 1);
      mbar_init(&bars->do_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&bars->vec_full[i], 1);
      mbar_init(&bars->vec_empty[i], 256);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->dk_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 2) {
    // E_S / E_D (ones in K columns 0-2 / 3-5 of each key row, no-swizzle
    // K-major) and zeroed augment tiles (their K columns 8-15 stay zero)
    uint4* ez = reinterpret_cast<uint4*>(smem + L::e_off);
    constexpr int kE16 = L::kE / 16;
    constexpr int kA16 = L::kAug / 16;
    const uint32_t one = 0x3F80u;  // bf16 1.0
    for (int i = lane; i < 2 * kE16 + NV * kA16; i += 32) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      const bool first_half = ((i % 16) < 8);  // core matrix of K columns 0-7
      if (i < kE16 && first_half) v = make_uint4(one | (one << 16), one, 0u, 0u);
      if (i >= kE16 && i < 2 * kE16 && first_half)
        v = make_uint4(0u, one << 16, one | (one << 16), 0u);
      ez[i] = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtx ctx{&bars->abort_flag, a.status};

  if (warp < 4) {
    regs_dec<kRegsControl>();
    if (warp == 0) {
      // ====================================================== producer
      int last_q[2] = {-1, -1}, last_do[2] = {-1, -1};
      int t = 0;
      bool ok = true;
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        mbar_arrive_expect_tx(&bars->kv_full, (KT ? 0 : L::kKTile) + L::kVTileS);
        if constexpr (!KT) {
          for (int c = 0; c < DK / 64; ++c)
            tma_load_4d(smem_u32(smem + L::k_off + c * L::kKChunk), &tm_k, c * 64, kvh, kt * 128,
                        bi, &bars->kv_full);
        }
        if constexpr (!VT) {
          for (int c = 0; c < DV / 64; ++c)
            tma_load_4d(smem_u32(smem + L::v_off + c * L::kKChunk), &tm_v, c * 64, kvh, kt * 128,
                        bi, &bars->kv_full);
        }
      }
      for (AStepIter<BM> it = it0; it.valid() && ok; it.next(), ++t) {
        const int h = kvh * a.g + it.hh;
        const int r0 = it.row0();
        if (lane == 0) {
          const int qs = t % NQ, use = t / NQ;
          ok = mbar_wait(&bars->q_empty[qs], (use & 1) ^ 1, ctx);
          if (ok) {
            mbar_arrive_expect_tx(&bars->q_full[qs], L::kQTile);
            for (int c = 0; c < DK / 64; ++c)
              tma_load_4d(smem_u32(smem + L::q_off + qs * L::kQTile + c * L::kQChunk), &tm_q,
                          c * 64, h, r0, bi, &bars->q_full[qs]);
            last_q[qs] = use;
          }
          const int os = t % NO, ouse = t / NO;
          if (ok) ok = mbar_wait(&bars->do_empty[os], (ouse & 1) ^ 1, ctx);
          if (ok) {
            mbar_arrive_expect_tx(&bars->do_full[os], L::kOTile);
            for (int c = 0; c < DV / 64; ++c)
              tma_load_4d(smem_u32(smem + L::do_off + os * L::kOTile + c * L::kQChunk), &tm_do,
                          c * 64, h, r0, bi, &bars->do_full[os]);
            last_do[os] = ouse;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (lane == 0) {
        mbar_wait_drain(&bars->kv_full, 0, a.status);
        for (int i = 0; i < NQ; ++i)
          if (last_q[i] >= 0) mbar_wait_drain(&bars->q_full[i], last_q[i] & 1, a.status);
        for (int i = 0; i < NO; ++i)
          if (last_do[i] >= 0) mbar_wait_drain(&bars->do_full[i], last_do[i] & 1, a.status);
      }
    } else if (warp == 1) {
      // ====================================================== MMA issuer
      if (lane == 0) {
        constexpr uint32_t id_st = idesc_bf16_f32(128, BM, false, false);      // S^T, dP^T
        constexpr uint32_t id_dv = idesc_bf16_f32(128, L::DVS, false, true);   // dV (A in TMEM)
        constexpr uint32_t id_dk = idesc_bf16_f32(128, L::DKS, false, true);   // dK (A in TMEM)
        const uint32_t k_km = sdesc_lo(smem_u32(smem + L::k_off), 16);
        const uint32_t v_km = sdesc_lo(smem_u32(smem + L::v_off), 16);
        const uint32_t q_km = sdesc_lo(smem_u32(smem + L::q_off), 16);
        const uint32_t do_km = sdesc_lo(smem_u32(smem + L::do_off), 16);
        // MN-major views of Q / dO (d contiguous): 64-wide d blocks kQChunk apart
        const uint32_t q_mn = sdesc_lo(smem_u32(smem + L::q_off), L::kQChunk);
        const uint32_t do_mn = sdesc_lo(smem_u32(smem + L::do_off), L::kQChunk);
        const uint32_t e_s = sdesc_lo_nosw(smem_u32(smem + L::e_off));
        const uint32_t e_d = sdesc_lo_nosw(smem_u32(smem + L::e_off + L::kE));
        const uint32_t aug0 = sdesc_lo_nosw(smem_u32(smem + L::aug_off));
        // this CTA's slice: d columns [ks * DKS, ...) of dK, [ks * DVS, ...) of dV
        const uint32_t q_slice = (uint32_t)((ks * L::DKS / 64) * L::kQChunk) >> 4;
        const uint32_t do_slice = (uint32_t)((ks * L::DVS / 64) * L::kQChunk) >> 4;
        constexpr int kHB = BM / 2;  // query columns of one element-wise half
        auto region = [&](int r) { return tmem + L::kColR + (uint32_t)((r & 1) * BM); };
        // S^T(t) - c = K Q^T + E_S Aug^T into region t  (M = keys, N = BM queries)
        auto issue_s = [&](int t) -> bool {
          const int qs = t % NQ;
          // the augment tile (usually ready long before), then Q(t) and the region
          bool w_ok = mbar_wait(&bars->vec_full[t % NV], (t / NV) & 1, ctx);
          if (w_ok) w_ok = mbar_wait(&bars->q_full[qs], (t / NQ) & 1, ctx);
          if (!w_ok) return false;
          tc_fence_after();
          const uint32_t qstage = (uint32_t)(qs * L::kQTile) >> 4;
          const uint32_t aug = aug0 + (uint32_t)(((t % NV) * L::kAug) >> 4);
#pragma unroll
          for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t offk = (uint32_t)((kk / 4) * L::kKChunk + (kk % 4) * 32) >> 4;
            const uint32_t offq = (uint32_t)((kk / 4) * L::kQChunk + (kk % 4) * 32) >> 4;
            if constexpr (KT)
              mma_ts_lo(region(t), tmem + L::kColK + kk * 8, q_km + qstage + offq, id_st,
                        kk > 0 ? 1u : 0u);
            else
              mma_ss_lo(region(t), k_km + offk, q_km + qstage + offq, id_st, kk > 0 ? 1u : 0u);
          }
          mma_ss_nosw(region(t), e_s, aug, id_st, 1u);
          mma_commit(&bars->s_full);
          return true;
        };
        // dP^T(t) - D = V dO^T + E_D Aug^T into the other region
        auto issue_dp = [&](int t) -> bool {
          const int os = t % NO;
          if (!mbar_wait(&bars->do_full[os], (t / NO) & 1, ctx)) return false;
          tc_fence_after();
          const uint32_t ostage = (uint32_t)(os * L::kOTile) >> 4;
          const uint32_t aug = aug0 + (uint32_t)(((t % NV) * L::kAug) >> 4);
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk) {
            const uint32_t offv = (uint32_t)((kk / 4) * L::kKChunk + (kk % 4) * 32) >> 4;
            const uint32_t offo = (uint32_t)((kk / 4) * L::kQChunk + (kk % 4) * 32) >> 4;
            if constexpr (VT)
              mma_ts_lo(region(t + 1), tmem + L::kColV + kk * 8, do_km + ostage + offo, id_st,
                        kk > 0 ? 1u : 0u);
            else
              mma_ss_lo(region(t + 1), v_km + offv, do_km + ostage + offo, id_st,
                        kk > 0 ? 1u : 0u);
          }
          mma_ss_nosw(region(t + 1), e_d, aug, id_st, 1u);
          mma_commit(&bars->dp_full);
          return true;
        };
        // Order: S^T(0), dP^T(0); per step t: dV(t) (once P^T(t) is in TMEM),
        // S^T(t+1) (into the region dP^T(t) leaves once the element-wise warps
        // have read it), dK(t) (once dS^T(t) is in TMEM), dP^T(t+1) (into the
        // region P^T / dS^T(t) leave once dV(t) and dK(t) are done).
        bool ok = mbar_wait(&bars->kv_full, 0, ctx);
        if constexpr (KT || VT) {
          if (ok) ok = mbar_wait(&bars->k_full, 0, ctx);
        }
        mbar_arrive(&bars->do_full[0]);  // step 0 has no dK before it
        if (ok && nsteps_total > 0) ok = issue_s(0) && issue_dp(0);
        for (int t = 0; t < nsteps_total && ok; ++t) {
          const int qs = t % NQ, os = t % NO;
          const uint32_t qstage = (uint32_t)(qs * L::kQTile) >> 4;
          const uint32_t ostage = (uint32_t)(os * L::kOTile) >> 4;
          const uint32_t t_s = region(t);
          const uint32_t acc0 = t > 0 ? 1u : 0u;
          // dV += P^T dO  (A = P^T in TMEM: K-step kk reads half kk / (kHB / 16))
          ok = mbar_wait(&bars->p_full, t & 1, ctx);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk) {
            const uint32_t col = (kk / (kHB / 16)) * kHB + (kk % (kHB / 16)) * 8;
            mma_ts_lo(tmem + L::kColDV, t_s + col,
                      do_mn + ostage + do_slice + (uint32_t)((kk * 2048) >> 4), id_dv,
                      kk > 0 ? 1u : acc0);
          }
          mma_commit(&bars->do_empty[os]);
          // With two Q stages S^T(t+1) goes ahead of dK(t); with one, Q(t+1)
          // can only arrive once dK(t) has released the stage.
          if constexpr (NQ > 1) {
            if (t + 1 < nsteps_total) {
              ok = issue_s(t + 1);
              if (!ok) break;
            }
          }
          // dK += dS^T Q  (A = dS^T in TMEM: the second half of each half's columns)
          ok = mbar_wait(&bars->ds_full, t & 1, ctx);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk) {
            const uint32_t col = (kk / (kHB / 16)) * kHB + kHB / 2 + (kk % (kHB / 16)) * 8;
            mma_ts_lo(tmem + L::kColDK, t_s + col,
                      q_mn + qstage + q_slice + (uint32_t)((kk * 2048) >> 4), id_dk,
                      kk > 0 ? 1u : acc0);
          }
          mma_commit(&bars->dk_done);
          mma_commit(&bars->q_empty[qs]);
          if (t + 1 < nsteps_total) mma_commit(&bars->do_full[(t + 1) % NO]);
          if constexpr (NQ == 1) {
            if (t + 1 < nsteps_total) {
              ok = issue_s(t + 1);
              if (!ok) break;
            }
          }
          if (t + 1 < nsteps_total) {
            ok = issue_dp(t + 1);
            if (!ok) break;
          }
        }
        mma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0, a.status);
      }
    } else if (warp == 2) {
      // ====================================================== vector loader
      // Per step: the augment tile (-c and -D per query row, each split into
      // three bf16; a row without keys takes c = 2^64, so P = 0), read by the
      // S^T and dP^T MMAs, and the rows' ids / pos and the tile class, read by
      // the element-wise warps.
      int t = 0;
      bool ok = true;
      const float inv_scale = 1.f / a.scale;
      for (AStepIter<BM> it = it0; it.valid() && ok; it.next(), ++t) {
        const int h = kvh * a.g + it.hh;
        const int r0 = it.row0();
        const int en = t % NV, use = t / NV;
        const int64_t lbase = ((int64_t)bi * a.hq + h) * a.s_q;
        const int64_t ibase = (int64_t)bi * a.s_q;
        float vl[BM / 32], vd[BM / 32];
        int vid[BM / 32], vps[BM / 32];
#pragma unroll
        for (int u = 0; u < BM / 32; ++u) {
          const int gq = r0 + u * 32 + lane;
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
        int* vi = vec + en * L::kVec;
        uint8_t* aug = smem + L::aug_off + en * L::kAug;
#pragma unroll
        for (int u = 0; u < BM / 32; ++u) {
          const int r = u * 32 + lane;
          vi[r] = vid[u];
          vi[BM + r] = vps[u];
          const float c = (vl[u] == -INFINITY) ? kAugNoKeys : vl[u] * inv_scale + a.c_shift;
          uint32_t cs[3], ds[3];
          split3(-c, cs);
          split3(-vd[u], ds);
          *reinterpret_cast<uint4*>(aug + (r / 8) * 256 + (r % 8) * 16) =
              make_uint4(cs[0] | (cs[1] << 16), cs[2] | (ds[0] << 16), ds[1] | (ds[2] << 16), 0u);
        }
        if (lane == 0) vi[2 * BM] = kind;
        fence_proxy_async_smem();  // the augment tile is read by the MMAs
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->vec_full[en]);
      }
    }
  } else {
    regs_inc<kRegsCompute>();
    // ======================================================== element-wise
    constexpr int kHB = BM / 2;  // query columns of this half
    const int w = (warp - 4) / 4;
    const int wq = warp % 4;
    const int kr = wq * 32 + lane;  // key row (TMEM lane)
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int key = kt * 128 + kr;
    const bool key_in = key < a.s_kv;
    const int ik = key_in ? a.kv_ids[(int64_t)bi * a.s_kv + key] : 0;
    const int pk = key_in ? a.kv_pos[(int64_t)bi * a.s_kv + key] : 0;
    const float sl2 = a.scale_log2;
    if constexpr (KT || VT) {
      // this thread's key (KT) and value (VT) rows into TMEM as bf16 pairs
      // (column c holds d elements 2c, 2c + 1): half w stores the d range
      // [w * D / 2, (w + 1) * D / 2) of each
      auto store_row = [&](const __nv_bfloat16* base, int64_t stride, int width, uint32_t col) {
        const uint4* src4 = reinterpret_cast<const uint4*>(
            base + ((int64_t)bi * a.s_kv + key) * stride + (int64_t)kvh * width + w * (width / 2));
        const uint32_t dst = tmem + lane_off + col + w * (width / 4);
#pragma unroll 1
        for (int c = 0; c < width / 4; c += 32) {
          uint32_t v32[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = key_in ? src4[c / 4 + u] : make_uint4(0u, 0u, 0u, 0u);
            v32[4 * u] = x.x;
            v32[4 * u + 1] = x.y;
            v32[4 * u + 2] = x.z;
            v32[4 * u + 3] = x.w;
          }
          tmem_st32(dst + c, v32);
        }
      };
      if constexpr (KT) store_row(a.k, a.k_stride, DK, L::kColK);
      if constexpr (VT) store_row(a.v, a.v_stride, DV, L::kColV);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->k_full);
    }
    int t = 0;
    bool ok = true;
    mbar_arrive(&bars->q_full[0]);  // S^T(0) has no dP^T before it to wait for
    for (; t < nsteps_total; ++t) {
      const int en = t % NV;
      // this half's S^T columns (region t & 1) and dP^T columns (the other region)
      const uint32_t t_sh = tmem + lane_off + L::kColR + (uint32_t)((t & 1) * BM) + kHB * w;
      const uint32_t t_dph = tmem + lane_off + L::kColR + (uint32_t)(((t + 1) & 1) * BM) + kHB * w;
      ok = mbar_wait(&bars->vec_full[en], (t / NV) & 1, ctx);
      ok = mbar_wait(&bars->s_full, t & 1, ctx) && ok;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int* ventry = vec + en * L::kVec;
      const bool partial = ventry[2 * BM] == kPartial;
      uint32_t r[kHB];
#pragma unroll
      for (int c = 0; c < kHB; c += 32) tmem_ld32(t_sh + c, &r[c]);
      tmem_wait_ld();
      // the tensor core already subtracted c: p = 2^(scale log2(e) (S - c)) = scale * P
      float p[kHB];
#pragma unroll
      for (int u = 0; u < kHB; u += 2) {
        float x0, x1;
        mul_f32x2(x0, x1, __uint_as_float(r[u]), __uint_as_float(r[u + 1]), sl2, sl2);
        p[u] = ex2(x0);
        p[u + 1] = ex2(x1);
      }
      if (partial) {
        const int4* id4 = reinterpret_cast<const int4*>(ventry + kHB * w);
        const int4* ps4 = reinterpret_cast<const int4*>(ventry + BM + kHB * w);
#pragma unroll
        for (int c = 0; c < kHB / 4; ++c) {
          const int4 i4 = id4[c];
          const int4 q4 = ps4[c];
          const int ia[4] = {i4.x, i4.y, i4.z, i4.w};
          const int qa[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (!visible(ia[u], qa[u], ik, pk, a.window)) p[4 * c + u] = 0.f;
        }
      }
      uint32_t pk2[kHB / 2];
#pragma unroll
      for (int u = 0; u < kHB / 2; ++u) pk2[u] = pack_bf16(p[2 * u], p[2 * u + 1]);
#pragma unroll
      for (int c = 0; c < kHB / 2; c += 16) tmem_st16(t_sh + c, &pk2[c]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
      // dS^T = P^T * (dP^T - D)  (the tensor core already subtracted D)
      ok = mbar_wait(&bars->dp_full, t & 1, ctx);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kHB; c += 32) tmem_ld32(t_dph + c, &r[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->q_full[(t + 1) % NQ]);  // S^T(t+1) may take the dP^T region
      mbar_arrive(&bars->vec_empty[en]);
#pragma unroll
      for (int c = 0; c < kHB / 2; ++c) {
        float d0, d1;
        mul_f32x2(d0, d1, p[2 * c], p[2 * c + 1], __uint_as_float(r[2 * c]),
                  __uint_as_float(r[2 * c + 1]));
        pk2[c] = pack_bf16(d0, d1);
      }
#pragma unroll
      for (int c = 0; c < kHB / 2; c += 16) tmem_st16(t_sh + kHB / 2 + c, &pk2[c]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);
    }
    // ---- epilogue: this CTA's dV slice (half 0) and dK slice (half 1)
    if (ok && t > 0) {
      ok = mbar_wait(&bars->dk_done, (t - 1) & 1, ctx);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    if (ok) {
      // P was formed as scale * P: dK carries its factor, dV divides it out
      const float sc = (w == 0) ? 1.f / a.scale : 1.f;
      constexpr int kCols0 = L::DVS, kCols1 = L::DKS;
      const int ncols = (w == 0) ? kCols0 : kCols1;
      const int64_t row0 =
          (w == 0) ? ((int64_t)bi * a.s_kv + key) * a.v_stride + (int64_t)kvh * DV + ks * L::DVS
                   : ((int64_t)bi * a.s_kv + key) * a.k_stride + (int64_t)kvh * DK + ks * L::DKS;
      const uint32_t src = tmem + lane_off + (w == 0 ? L::kColDV : L::kColDK);
#pragma unroll 1
      for (int c = 0; c < ncols; c += 32) {
        uint32_t o[32];
        if (t > 0) {
          tmem_ld32(src + c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = 0u;
        }
        if (!key_in) continue;
        if (a.accumulate) {
          float4* dst =
              reinterpret_cast<float4*>(static_cast<float*>(w == 0 ? a.dv : a.dk) + row0 + c);
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
        uint4* dst = reinterpret_cast<uint4*>(
            static_cast<__nv_bfloat16*>(w == 0 ? a.dv : a.dk) + row0 + c);
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

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ============================================================== dQ, TMEM operands
// The dQ computation with the query tile (and, where TMEM has room, the dO
// tile) loaded once into TMEM as the A operands of S = Q K^T (and dP =
// dO V^T), so those products read only K / V from shared memory, and dS
// (bf16) written over the dP columns it was computed from (the A operand of
// dQ += dS K).  One S buffer suffices because S(n+1) may overwrite S(n) as
// soon as the element-wise warps have loaded it, long before dQ(n); dP(n+1)
// waits for dQ(n), which reads dS(n) from the dP columns.  Shared memory
// holds a ring of NKV K / V slots (and the dO tile when it is not in TMEM):
// the K tile of S(n+1) reuses the slot of K(n+1-NKV/2), freed by dQ long
// before, so it is loaded well ahead.
// TMEM: S [0,BN)  dP [BN,2BN)  Q [2BN, 2BN+DK/2)  dO [.., +DV/2) (OT)  dQ [512-DK, 512)
// d <= 128: 128-key tiles, dO in TMEM, six slots; MLA (192 / 128): 64-key
// tiles, dO in TMEM, six slots; d = 256: 64-key tiles, dO in shared memory
// (the Q and dQ columns leave no room), four slots.
template <int DK, int DV, int BN_, int NKV_, bool OT>
struct QTLayout {
  static constexpr int BN = BN_;
  static constexpr int NKV = NKV_;
  static constexpr int kQChunk = 128 * 128;  // 128 query rows x 128 B (the dO tile)
  static_assert(kQChunk == 128 * 128, "dO tile chunk");
  static constexpr int kKVChunk = BN * 128;  // BN key rows x 128 B
  static constexpr int kKSlot = BN * DK * 2;
  static constexpr int kVSlot = BN * DV * 2;
  static constexpr int kSlot = kKSlot > kVSlot ? kKSlot : kVSlot;  // a K or V tile
  static constexpr int kOTile = OT ? 0 : 128 * DV * 2;
  static constexpr int kIdEntry = 2 * BN + 32;
  static constexpr int do_off = 0;
  static constexpr int kv_off = do_off + kOTile;
  static constexpr int id_off = kv_off + NKV * kSlot;
  static constexpr int bar_off = id_off + NID * kIdEntry * 4;
  static constexpr int bytes = bar_off + 512;
  static constexpr int alloc = (bytes + 1024) > 150 * 1024 ? (bytes + 1024) : 150 * 1024;
  static constexpr uint32_t kColS = 0, kColDP = BN, kColQ = 2 * BN, kColO = 2 * BN + DK / 2,
                            kColDQ = 512 - DK;
  static_assert((OT ? kColO + DV / 2 : kColQ + DK / 2) <= kColDQ, "TMEM columns");
  static_assert(NKV >= 4 && NKV <= 8, "K / V slots");
  static_assert(alloc <= 232448, "shared memory per block");
};

struct QTBars {
  uint64_t q_full;
  uint64_t do_full;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t id_full[NID];
  uint64_t id_empty[NID];
  uint64_t s_full, dp_full, ds_full, dq_done, drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(QTBars) <= 512, "barrier block too large");

template <int DK, int DV, int BN_, int NKV_, bool OT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_tmem_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_do, const __nv_bfloat16* q,
                            const __nv_bfloat16* dout, const SplitArgs a) {
  using L = QTLayout<DK, DV, BN_, NKV_, OT>;
  constexpr int BN = L::BN;
  constexpr int NKV = L::NKV;
  constexpr int kSub = 128 / BN;  // key tiles per 128-key plan tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  QTBars* bars = reinterpret_cast<QTBars*>(smem + L::bar_off);
  int* s_ids = reinterpret_cast<int*>(smem + L::id_off);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (a.status && *reinterpret_cast<volatile int*>(a.status) != kStatusOk) return;

  const int rank = blockIdx.x / a.hq;
  const int h = blockIdx.x % a.hq;
  const int kvh = h / a.g;
  const int e = a.order[rank];
  const int bi = e / a.nq;
  const int qt = e % a.nq;
  const int2 rng = a.range[e];
  const int nt = kSub * a.weight[e];  // BN-key tiles of the non-SKIP plan tiles
  const uint8_t* cls_row = a.cls + (size_t)e * a.nk;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 256);  // every element-wise thread stores its row (or arrives)
    mbar_init(&bars->do_full, 1);
    // K tiles take the even slots, V tiles the odd ones (NKV is even).  K(n):
    // landed (TMA) and S(n-1) loaded by the 256 element-wise threads (S(n)
    // overwrites it); V(n): landed and dQ(n-1) done (dP(n) overwrites the dS
    // columns dQ(n-1) reads; MMA commit).
    static_assert(NKV % 2 == 0, "K / V slots alternate");
    for (int i = 0; i < NKV; ++i) {
      mbar_init(&bars->kv_full[i], (i % 2 == 0) ? 1 + 256 : 1 + 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int i = 0; i < NID; ++i) {
      mbar_init(&bars->id_full[i], 1);
      mbar_init(&bars->id_empty[i], 256);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->dq_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtx ctx{&bars->abort_flag, a.status};

  if (warp < 4) {
    regs_dec<kRegsControl>();
    if (warp == 0) {
      // ====================================================== producer (K, V)
      int last_use[NKV];
      for (int i = 0; i < NKV; ++i) last_use[i] = -1;
      bool ok = true;
      if (lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if constexpr (!OT) {
          tma_prefetch_desc(&tm_do);
          mbar_arrive_expect_tx(&bars->do_full, L::kOTile);
          for (int c = 0; c < DV / 64; ++c)
            tma_load_4d(smem_u32(smem + L::do_off + c * L::kQChunk), &tm_do, c * 64, h, qt * 128,
                        bi, &bars->do_full);
        }
      }
      int n = 0;
      for (int j = kSub * rng.x; j < kSub * (rng.y + 1) && ok; ++j) {
        if (cls_row[j / kSub] == kSkip) continue;
#pragma unroll 1
        for (int kv = 0; kv < 2 && ok; ++kv) {
          const int ld = 2 * n + kv, slot = ld % NKV, use = ld / NKV;
          if (lane == 0) {
            ok = mbar_wait(&bars->kv_empty[slot], (use & 1) ^ 1, ctx);
            if (ok) {
              mbar_arrive_expect_tx(&bars->kv_full[slot], kv == 0 ? L::kKSlot : L::kVSlot);
              for (int c = 0; c < (kv == 0 ? DK : DV) / 64; ++c)
                tma_load_4d(smem_u32(smem + L::kv_off + slot * L::kSlot + c * L::kKVChunk),
                            kv == 0 ? &tm_k : &tm_v, c * 64, kvh, j * BN, bi, &bars->kv_full[slot]);
              last_use[slot] = use;
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        ++n;
      }
      if (lane == 0) {
        if constexpr (!OT) mbar_wait_drain(&bars->do_full, 0, a.status);
        for (int i = 0; i < NKV; ++i)
          if (last_use[i] >= 0) mbar_wait_drain(&bars->kv_full[i], last_use[i] & 1, a.status);
      }
    } else if (warp == 1) {
      // ====================================================== MMA issuer
      // S(0), dP(0); then per tile n: S(n+1) once S(n) has been loaded by the
      // element-wise warps, dQ(n) once dS(n) is in TMEM (releases K(n)),
      // dP(n+1) once dQ(n) has read dS(n) from the dP columns (releases V(n+1)).
      if (lane == 0) {
        constexpr uint32_t id_s = idesc_bf16_f32(128, BN, false, false);  // S, dP (A in TMEM)
        constexpr uint32_t id_q = idesc_bf16_f32(128, DK, false, true);   // dQ (A in TMEM)
        const uint32_t kv_km = sdesc_lo(smem_u32(smem + L::kv_off), 16);
        const uint32_t kv_mn = sdesc_lo(smem_u32(smem + L::kv_off), L::kKVChunk);
        const uint32_t do_km = sdesc_lo(smem_u32(smem + L::do_off), 16);
        auto issue_s = [&](int m) -> bool {
          const int slot = (2 * m) % NKV;
          if (!mbar_wait(&bars->kv_full[slot], ((2 * m) / NKV) & 1, ctx)) return false;
          tc_fence_after();
          const uint32_t kb = kv_km + (uint32_t)((slot * L::kSlot) >> 4);
#pragma unroll
          for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t offb = (uint32_t)((kk / 4) * L::kKVChunk + (kk % 4) * 32) >> 4;
            mma_ts_lo(tmem + L::kColS, tmem + L::kColQ + kk * 8, kb + offb, id_s,
                      kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full);
          return true;
        };
        auto issue_dp = [&](int m) -> bool {
          const int slot = (2 * m + 1) % NKV;
          if (!mbar_wait(&bars->kv_full[slot], ((2 * m + 1) / NKV) & 1, ctx)) return false;
          tc_fence_after();
          const uint32_t vb = kv_km + (uint32_t)((slot * L::kSlot) >> 4);
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk) {
            const uint32_t offb = (uint32_t)((kk / 4) * L::kKVChunk + (kk % 4) * 32) >> 4;
            if constexpr (OT) {
              mma_ts_lo(tmem + L::kColDP, tmem + L::kColO + kk * 8, vb + offb, id_s,
                        kk > 0 ? 1u : 0u);
            } else {
              const uint32_t offa = (uint32_t)((kk / 4) * L::kQChunk + (kk % 4) * 32) >> 4;
              mma_ss_lo(tmem + L::kColDP, do_km + offa, vb + offb, id_s, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(&bars->dp_full);
          mma_commit(&bars->kv_empty[slot]);  // V(m) has no other reader
          return true;
        };
        bool ok = mbar_wait(&bars->q_full, 0, ctx);
        if constexpr (!OT) {
          if (ok) ok = mbar_wait(&bars->do_full, 0, ctx);
        }
        mbar_arrive(&bars->kv_full[1]);  // dP(0) has no dQ before it
        if (ok && nt > 0) ok = issue_s(0) && issue_dp(0);
        for (int n = 0; n < nt && ok; ++n) {
          if (n + 1 < nt) {
            ok = issue_s(n + 1);
            if (!ok) break;
          }
          ok = mbar_wait(&bars->ds_full, n & 1, ctx);
          if (!ok) break;
          tc_fence_after();
          const int kslot = (2 * n) % NKV;
          const uint32_t kb = kv_mn + (uint32_t)((kslot * L::kSlot) >> 4);
          // dQ += dS K: K-step kk (16 keys) reads the dS columns of half kk / (BN / 32)
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts_lo(tmem + L::kColDQ,
                      tmem + L::kColDP + (kk / (BN / 32)) * (BN / 2) + (kk % (BN / 32)) * 8,
                      kb + (uint32_t)((kk * 16 * 128) >> 4), id_q, (n > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars->dq_done);
          mma_commit(&bars->kv_empty[kslot]);  // K(n): S(n) and dQ(n) have read it
          if (n + 1 < nt) mma_commit(&bars->kv_full[(2 * n + 3) % NKV]);  // V(n+1)'s barrier
          if (n + 1 < nt) {
            ok = issue_dp(n + 1);
            if (!ok) break;
          }
        }
        mma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0, a.status);
      }
    } else if (warp == 2) {
      // ====================================================== key descriptor loader
      int n = 0;
      bool ok = true;
      for (int j = kSub * rng.x; j < kSub * (rng.y + 1) && ok; ++j) {
        const uint8_t kind = cls_row[j / kSub];
        if (kind == kSkip) continue;
        const int en = n % NID, use = n / NID;
        const int64_t base = (int64_t)bi * a.s_kv;
        int vid[BN / 32], vpos[BN / 32];
#pragma unroll
        for (int u = 0; u < BN / 32; ++u) {
          const int tok = j * BN + u * 32 + lane;
          const bool in = tok < a.s_kv;
          vid[u] = in ? a.kv_ids[base + tok] : 0;
          vpos[u] = in ? a.kv_pos[base + tok] : 0;
        }
        if (lane == 0) ok = mbar_wait(&bars->id_empty[en], (use & 1) ^ 1, ctx);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        int* dst = s_ids + en * L::kIdEntry;
#pragma unroll
        for (int u = 0; u < BN / 32; ++u) {
          dst[u * 32 + lane] = vid[u];
          dst[BN + u * 32 + lane] = vpos[u];
        }
        if (lane == 0) dst[2 * BN] = kind;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->id_full[en]);
        ++n;
      }
    }
  } else {
    regs_inc<kRegsCompute>();
    // ======================================================== element-wise
    constexpr int kHB = BN / 2;  // key columns of this half
    const int w = (warp - 4) / 4;
    const int wq = warp % 4;
    const int row = wq * 32 + lane;  // query row (TMEM lane)
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int grow = qt * 128 + row;
    const bool row_in = grow < a.s_q;
    if (w == 0 || OT) {
      // the query row (half 0) or the dO row (half 1) into TMEM as bf16 pairs:
      // column c holds elements 2c, 2c + 1 (the row's own byte order)
      const int width = (w == 0) ? DK : DV;
      const __nv_bfloat16* src =
          (w == 0 ? q : dout) + (((int64_t)bi * a.s_q + grow) * a.hq + h) * width;
      const uint4* src4 = reinterpret_cast<const uint4*>(src);
      const uint32_t dst = tmem + lane_off + (w == 0 ? L::kColQ : L::kColO);
#pragma unroll 1
      for (int c = 0; c < width / 2; c += 32) {
        uint32_t v32[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = row_in ? src4[c / 4 + u] : make_uint4(0u, 0u, 0u, 0u);
          v32[4 * u] = x.x;
          v32[4 * u + 1] = x.y;
          v32[4 * u + 2] = x.z;
          v32[4 * u + 3] = x.w;
        }
        tmem_st32(dst + c, v32);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->q_full);
    } else {
      mbar_arrive(&bars->q_full);  // the dO tile comes by TMA
    }
    const int iq = row_in ? a.q_ids[(int64_t)bi * a.s_q + grow] : 0;
    const int pq = row_in ? a.q_pos[(int64_t)bi * a.s_q + grow] : 0;
    const int64_t lidx = ((int64_t)bi * a.hq + h) * a.s_q + grow;
    const float lse = row_in ? a.lse[lidx] : -INFINITY;
    const float Dr = row_in ? a.Dv[lidx] : 0.f;
    const float c2 = (lse == -INFINITY) ? INFINITY : (lse + a.c_shift * a.scale) * kLog2e;
    const float sl2 = a.scale_log2;
    const uint32_t t_sh = tmem + lane_off + L::kColS + kHB * w;
    const uint32_t t_dph = tmem + lane_off + L::kColDP + kHB * w;
    int n = 0;
    bool ok = true;
    mbar_arrive(&bars->kv_full[0]);  // S(0) overwrites no earlier S
    for (; n < nt; ++n) {
      const int en = n % NID;
      ok = mbar_wait(&bars->id_full[en], (n / NID) & 1, ctx);
      ok = mbar_wait(&bars->s_full, n & 1, ctx) && ok;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t r[kHB];
#pragma unroll
      for (int c = 0; c < kHB; c += 32) tmem_ld32(t_sh + c, &r[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->kv_full[(2 * n + 2) % NKV]);  // S(n+1) may overwrite the S columns
      float p[kHB];
#pragma unroll
      for (int u = 0; u < kHB; u += 2) {
        float x0, x1;
        fma_f32x2(x0, x1, __uint_as_float(r[u]), __uint_as_float(r[u + 1]), sl2, sl2, -c2, -c2);
        p[u] = ex2(x0);
        p[u + 1] = ex2(x1);
      }
      const int* ent = s_ids + en * L::kIdEntry;
      if (ent[2 * BN] == kPartial) {
        const int4* id4 = reinterpret_cast<const int4*>(ent + kHB * w);
        const int4* ps4 = reinterpret_cast<const int4*>(ent + BN + kHB * w);
#pragma unroll
        for (int c = 0; c < kHB / 4; ++c) {
          const int4 i4 = id4[c];
          const int4 k4 = ps4[c];
          const int ia[4] = {i4.x, i4.y, i4.z, i4.w};
          const int ka[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (!visible(iq, pq, ia[u], ka[u], a.window)) p[4 * c + u] = 0.f;
        }
      }
      mbar_arrive(&bars->id_empty[en]);
      ok = mbar_wait(&bars->dp_full, n & 1, ctx);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kHB; c += 32) tmem_ld32(t_dph + c, &r[c]);
      tmem_wait_ld();
      uint32_t pk2[kHB / 2];
#pragma unroll
      for (int c = 0; c < kHB / 2; ++c) {
        float d0, d1;
        fma_f32x2(d0, d1, p[2 * c], p[2 * c + 1], __uint_as_float(r[2 * c]),
                  __uint_as_float(r[2 * c + 1]), -p[2 * c] * Dr, -p[2 * c + 1] * Dr);
        pk2[c] = pack_bf16(d0, d1);
      }
      // dS over the first half of this half's own dP columns (K-major A operand)
#pragma unroll
      for (int c = 0; c < kHB / 2; c += 16) tmem_st16(t_dph + c, &pk2[c]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);
    }
    if (ok && n > 0) {
      ok = mbar_wait(&bars->dq_done, (n - 1) & 1, ctx);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    if (ok) {
      constexpr int kHalfD = DK / 2;
      const int64_t orow = (((int64_t)bi * a.s_q + grow) * a.hq + h) * DK + kHalfD * w;
      const uint32_t src = tmem + lane_off + L::kColDQ + kHalfD * w;
#pragma unroll 1
      for (int c = 0; c < kHalfD; c += 32) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld32(src + c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = 0u;
        }
        if (!row_in) continue;
        if (a.accumulate) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.dq) + orow + c);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float4 v = dst[u];
            v.x += __uint_as_float(o[4 * u + 0]);
            v.y += __uint_as_float(o[4 * u + 1]);
            v.z += __uint_as_float(o[4 * u + 2]);
            v.w += __uint_as_float(o[4 * u + 3]);
            dst[u] = v;
          }
          continue;
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dq) + orow + c);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 v;
          v.x = pack_bf16(__uint_as_float(o[8 * u + 0]), __uint_as_float(o[8 * u + 1]));
          v.y = pack_bf16(__uint_as_float(o[8 * u + 2]), __uint_as_float(o[8 * u + 3]));
          v.z = pack_bf16(__uint_as_float(o[8 * u + 4]), __uint_as_float(o[8 * u + 5]));
          v.w = pack_bf16(__uint_as_float(o[8 * u + 6]), __uint_as_float(o[8 * u + 7]));
          dst[u] = v;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int DK, int DV, int BN, int NKV, bool OT>
cudaError_t launch_dq_tmem(const SplitArgs& a, const SplitLaunch& Lc, cudaStream_t st) {
  using L = QTLayout<DK, DV, BN, NKV, OT>;
  const int64_t units = (int64_t)a.b * a.nq * a.hq;
  if (units == 0) return cudaSuccess;
  static std::atomic<int> smem_set[kMaxDevices];
  auto kern = attn_bwd_dq_tmem_kernel<DK, DV, BN, NKV, OT>;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), L::alloc, kLaunchRegs,
                                    smem_set);
  if (e != cudaSuccess) return e;
  const attn_fwd_params& f = Lc.p->fwd;
  kern<<<(unsigned)units, kThreads, L::alloc, st>>>(
      Lc.tm_kb, Lc.tm_vb, Lc.tm_do, static_cast<const __nv_bfloat16*>(f.q),
      static_cast<const __nv_bfloat16*>(Lc.p->dout), a);
  return cudaGetLastError();
}

template <int DK, int DV, int BM, int NSPLIT, int NQ, int NO, bool KT = false, bool VT = false>
cudaError_t launch_dkdv(const SplitArgs& a, const SplitLaunch& Lc, cudaStream_t st) {
  using L = ALayout<DK, DV, BM, NSPLIT, NQ, NO, KT, VT>;
  const int64_t units = (int64_t)a.b * a.nk * a.hkv * NSPLIT;
  if (units == 0) return cudaSuccess;
  static std::atomic<int> smem_set[kMaxDevices];
  auto kern = attn_bwd_dkdv_kernel<DK, DV, BM, NSPLIT, NQ, NO, KT, VT>;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), L::alloc, kLaunchRegs,
                                    smem_set);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)units, kThreads, L::alloc, st>>>(Lc.tm_q_a, Lc.tm_k, Lc.tm_v, Lc.tm_do_a, a);
  return cudaGetLastError();
}

}  // namespace

int split_bwd_query_rows(int64_t d, int64_t dv) {
  return (d == 256 || (d == 192 && dv == 128)) ? 64 : 128;
}

int split_bwd_key_rows(int64_t d, int64_t dv) {
  return (d == 256 || (d == 192 && dv == 128)) ? 64 : 128;
}

int split_bwd_col_slices(int64_t d, int64_t dv) { return (d == 256 && dv == 256) ? 2 : 1; }

cudaError_t launch_attn_bwd_split(const SplitLaunch& Lc, cudaStream_t st) {
  const attn_bwd_params& p = *Lc.p;
  const attn_fwd_params& f = p.fwd;
  const int64_t dv = f.d_v > 0 ? f.d_v : f.d;
  SplitArgs a;
  a.k = static_cast<const __nv_bfloat16*>(f.k);
  a.v = static_cast<const __nv_bfloat16*>(f.v);
  a.q_ids = f.q_segment_ids;
  a.q_pos = f.q_segment_pos;
  a.kv_ids = f.kv_segment_ids;
  a.kv_pos = f.kv_segment_pos;
  a.lse = f.lse;
  a.Dv = Lc.D;
  a.dq = p.dq;
  a.dk = p.dk;
  a.dv = p.dv;
  a.cls = Lc.plan.classes;
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
  a.k_stride = f.kv_token_stride > 0 ? f.kv_token_stride : f.h_kv * f.d;
  a.v_stride = f.kv_token_stride > 0 ? f.kv_token_stride : f.h_kv * dv;
  a.scale = f.scale;
  a.scale_log2 = f.scale * kLog2e;
  a.c_shift = -logf(f.scale) / f.scale;
  // dK / dV: kv side of the plan
  SplitArgs ak = a;
  ak.range = Lc.plan.kv_range;
  ak.weight = Lc.plan.kv_weight;
  ak.order = Lc.plan.kv_order;
  cudaError_t e;
  if (f.d == 128 && dv == 128) e = launch_dkdv<128, 128, 128, 1, 2, 2>(ak, Lc, st);
  else if (f.d == 64 && dv == 64) e = launch_dkdv<64, 64, 128, 1, 2, 2>(ak, Lc, st);
  else if (f.d == 192 && dv == 128) e = launch_dkdv<192, 128, 64, 1, 2, 2, false, true>(ak, Lc, st);
  else if (f.d == 256 && dv == 256) e = launch_dkdv<256, 256, 64, 2, 2, 2, true>(ak, Lc, st);
  else return cudaErrorNotSupported;
  if (e != cudaSuccess) return e;
  // dQ: q side of the plan
  SplitArgs aq = a;
  aq.range = Lc.plan.q_range;
  aq.weight = Lc.plan.q_weight;
  aq.order = Lc.plan.q_order;
  if (f.d == 128) return launch_dq_tmem<128, 128, 128, 6, true>(aq, Lc, st);
  if (f.d == 64) return launch_dq_tmem<64, 64, 128, 6, true>(aq, Lc, st);
  if (f.d == 192) return launch_dq_tmem<192, 128, 64, 6, true>(aq, Lc, st);
  return launch_dq_tmem<256, 256, 64, 4, false>(aq, Lc, st);
}

}  // namespace gb300
