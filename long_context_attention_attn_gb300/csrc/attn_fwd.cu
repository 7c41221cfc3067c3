// Forward attention over packed THD inputs on sm_103a.
//
// Page: "Context parallelism and ring attention", sections "The attention
// problem" (O = softmax(QK^T/sqrt(H) + M) V), "Online softmax" (running
// m, z, u with rescaling) and "Causal attention" (skip / full / masked key
// blocks); TE tutorial sections 1 and 3 (segment ids/pos, GQA, causal window).
//
// One CTA computes a 128-row query tile for TWO query heads of one GQA group
// (both read the same kv head, so every K/V tile loaded into shared memory
// feeds both; one head when d_v = 256), walking the keys in 64-key tiles.
// Roles (384 threads):
//   warp 0        TMA producer: Q tiles once, then K and V tiles into two
//                 rings of shared-memory slots, one for K and one for V (at
//                 d_qk 192 / d_v 128 a K tile is 24 KB and a V tile 16 KB, so
//                 separate rings hold a tile more than one ring of 24 KB slots).
//   warps 1, 3    MMA issuers, one thread per head slot: S_h = Q_h K^T and
//                 O_h += P_h V on tcgen05; warp 1 also owns the TMEM allocation.
//   warp 2        descriptor loader: each key tile's ids / pos / class.
//   warps 4-7     softmax for head slot 0 (one thread per query row)
//   warps 8-11    softmax for head slot 1
// TMEM (512 columns x 128 lanes, lane = query row):
//   slot 0 S buffers [0,64) [64,128), slot 1 [128,192) [192,256),
//   O0 [256,256+d_v)  O1 [256+d_v, 256+2d_v)
// (head dims: q / k and v / out both 64, 128 or 256, or 192 / 128; at d_v = 256
// a CTA takes one head slot, whose O fills columns [256, 512), and warps 3 and
// 8-11 stay idle)
// Key tile n's scores go to buffer n & 1 of the slot, so S(n+1) is computed
// while the softmax works on tile n.  P (bf16, 2 per column) overwrites the
// first 32 columns of its S buffer and is the A operand of the P.V MMA
// straight from TMEM.
//
// Softmax runs in the base-2 domain: x = s * scale * log2(e).  The running
// maximum m is only raised (and O rescaled) when a row's new maximum exceeds
// it by more than 8, so exp2(x - m) <= 256; the final u / z is exact for any
// reference m.
#include <cuda_bf16.h>

#include "internal.h"
#include "merge_math.cuh"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int BM = 128;
constexpr int BN = kFwdKeyTile;  // keys per tile (half of the plan's 128-key tile)
// Query heads per CTA and K / V ring slots by head dims (DK of q / k, DV of
// v / out): d <= 128 four K and four V slots; DV = 256 takes one head slot
// (its O accumulator fills TMEM columns [256, 512)) and keeps the query tile
// in TMEM columns [128, 256) (the second slot's S buffers), the A operand of
// S = Q K^T, so shared memory holds three 32 KB K and three 32 KB V slots and
// no Q; DK = 192 (DV = 128): three 24 KB K and three 16 KB V slots next to the
// two 48 KB query tiles.
template <int DK, int DV> constexpr int kSlots = DV <= 128 ? 2 : 1;
template <int DK, int DV> constexpr bool kQInTmem = DK == 256;
template <int DK, int DV> constexpr int kKSlots = DK <= 128 ? 4 : 3;
template <int DK, int DV> constexpr int kVSlots = DK <= 128 ? 4 : 3;
constexpr int kMaxRing = 4;  // slots per ring, at most
constexpr int NID = 4;   // ids/pos ring entries
constexpr int kThreads = 384;
// Registers per thread at launch (65536 / 384, rounded down to a multiple of 8).
constexpr int kLaunchRegs = 168;
static_assert(128 * kRegsControl + 256 * kRegsCompute <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
// ids/pos ring entry: 64 ids, 64 pos, then the tile's class (PARTIAL/FULL)
constexpr int kIdEntry = 2 * BN + 32;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

struct FwdArgs {
  const __nv_bfloat16* q;  // read directly when the query tile is kept in TMEM
  const int* q_ids;
  const int* q_pos;
  const int* kv_ids;
  const int* kv_pos;
  void* out;
  float* lse;
  const uint8_t* cls;
  const int2* qrange;
  const int* qweight;
  const int* order;
  int* status;
  int b, s_q, s_kv, hq, hkv, g, npairs, nq, nk;
  int window;
  int out_fp32;
  int merge;               // fold the result into (out, lse) instead of writing it
  __nv_bfloat16* out_final;  // merge mode: merged O as bf16 here instead of into out
  int withhold_kv;  // debug hook: issue no K/V loads, so every wait runs out
  float scale_log2;
};

template <int DK, int DV>
struct Layout {
  static constexpr int kChunk = BM * 128;             // one 64-wide bf16 chunk of a Q tile
  static constexpr int kChunkKV = BN * 128;           // one 64-wide bf16 chunk of a K / V tile
  static constexpr int kChunksK = DK / 64;            // chunks of a Q or K tile
  static constexpr int kChunksV = DV / 64;            // chunks of a V tile
  static constexpr int kTileBytes = BM * DK * 2;      // a Q tile
  static constexpr int kKBytes = BN * DK * 2;         // a K tile
  static constexpr int kVBytes = BN * DV * 2;         // a V tile
  static constexpr int q_off = 0;                     // kSlots Q tiles (none when in TMEM)
  static constexpr int k_off = q_off + (kQInTmem<DK, DV> ? 0 : kSlots<DK, DV> * kTileBytes);
  static constexpr int v_off = k_off + kKSlots<DK, DV> * kKBytes;  // the V ring
  static constexpr int id_off = v_off + kVSlots<DK, DV> * kVBytes;  // NID x kIdEntry ints
  static constexpr int bar_off = id_off + NID * kIdEntry * 4;
  static constexpr int bytes = bar_off + 512;
  // + slack for 1024-byte alignment; at least 150 KB so that one CTA (which
  // holds all 512 TMEM columns) is resident per SM.
  static constexpr int alloc = (bytes + 1024) > 150 * 1024 ? (bytes + 1024) : 150 * 1024;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kMaxRing];
  uint64_t k_empty[kMaxRing];  // one arrival per softmax warp
  uint64_t v_full[kMaxRing];
  uint64_t v_empty[kMaxRing];
  uint64_t id_full[NID];
  uint64_t id_empty[NID];
  uint64_t s_full[2][2];  // [slot][S buffer]
  uint64_t p_full[2][2];  // [slot][S buffer]
  uint64_t o_done[2][2];  // [slot][S buffer of the P.V's tile]
  uint64_t drain[2];
  uint64_t slot1_go;  // one phase: slot 0's first softmax is done
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block too large");

// First plan tile at or after j in [j, last] whose class is not SKIP (last + 1
// if none): 32 class bytes per warp load.  All 32 lanes must call it.
__device__ __forceinline__ int next_live_tile(const uint8_t* cls_row, int j, int last, int lane) {
  for (; j <= last; j += 32) {
    const uint8_t cl = (j + lane <= last) ? cls_row[j + lane] : (uint8_t)kSkip;
    const uint32_t live = __ballot_sync(0xffffffffu, cl != kSkip);
    if (live != 0u) return j + __ffs(live) - 1;
  }
  return last + 1;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = Layout<DK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::bar_off);
  int* s_ids = reinterpret_cast<int*>(smem + L::id_off);  // [NID][kIdEntry]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  // A CTA of this launch already timed out: the outputs are undefined, stop.
  if (a.status && *reinterpret_cast<volatile int*>(a.status) != kStatusOk) return;

  // ---- work unit: (b, q tile) in the plan's work order, then kv head, then head pair
  const int per_tile = a.hkv * a.npairs;
  const int rank = blockIdx.x / per_tile;
  const int rem = blockIdx.x % per_tile;
  const int kvh = rem / a.npairs;
  const int pair = rem % a.npairs;
  const int e = a.order[rank];
  const int bi = e / a.nq;
  const int qt = e % a.nq;
  const int h0 = kvh * a.g + kSlots<DK, DV> * pair;
  const int nslots = min(kSlots<DK, DV>, a.g - kSlots<DK, DV> * pair);
  constexpr int NKS = kKSlots<DK, DV>;
  constexpr int NVS = kVSlots<DK, DV>;
  static_assert(NKS <= kMaxRing && NVS <= kMaxRing, "ring slots");
  constexpr int NIDD = NID;
  constexpr bool QT = kQInTmem<DK, DV>;
  constexpr uint32_t kColQ = 2 * BN;  // query tile in TMEM (QT only)
  static_assert(!QT || (kSlots<DK, DV> == 1 && kColQ + DK / 2 <= 4 * BN), "TMEM columns");
  static_assert(4 * BN + kSlots<DK, DV> * DV <= 512, "TMEM columns");
  static_assert(Layout<DK, DV>::alloc <= 232448, "shared memory per block");
  const int2 rng = a.qrange[e];
  const int nt = 2 * a.qweight[e];  // 64-key tiles of the non-SKIP 128-key plan tiles
  const uint8_t* cls_row = a.cls + (size_t)e * a.nk;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, QT ? 128 : 1);  // TMA, or the 128 threads storing Q into TMEM
    for (int i = 0; i < NKS; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 4 * nslots);
    }
    for (int i = 0; i < NVS; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 4 * nslots);
    }
    for (int i = 0; i < NIDD; ++i) {
      mbar_init(&bars->id_full[i], 1);
      mbar_init(&bars->id_empty[i], 128 * nslots);
    }
    for (int i = 0; i < 2; ++i) {
      for (int bb = 0; bb < 2; ++bb) {
        mbar_init(&bars->s_full[i][bb], 1);
        mbar_init(&bars->p_full[i][bb], 128);
      }
      mbar_init(&bars->o_done[i][0], 1);
      mbar_init(&bars->o_done[i][1], 1);
    }
    mbar_init(&bars->drain[0], 1);
    mbar_init(&bars->drain[1], 1);
    mbar_init(&bars->slot1_go, 1);
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
    // ======================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      if (!QT) {
        mbar_arrive_expect_tx(&bars->q_full, nslots * L::kTileBytes);
        for (int sl = 0; sl < nslots; ++sl)
          for (int c = 0; c < L::kChunksK; ++c)
            tma_load_4d(smem_u32(smem + L::q_off + sl * L::kTileBytes + c * L::kChunk), &tm_q,
                        c * 64, h0 + sl, qt * BM, bi, &bars->q_full);
      }
    }
    int n = 0;
    int last_k[NKS], last_v[NVS];
    for (int i = 0; i < NKS; ++i) last_k[i] = -1;
    for (int i = 0; i < NVS; ++i) last_v[i] = -1;
    bool ok = true;
    for (int j2 = 2 * rng.x; j2 <= 2 * rng.y + 1 && ok && !a.withhold_kv; ++j2) {
      if (cls_row[j2 >> 1] == kSkip) {
        // jump over the run of SKIP tiles (the loop header then takes j2 to the
        // first half of the next live plan tile)
        j2 = 2 * next_live_tile(cls_row, (j2 >> 1) + 1, rng.y, lane) - 1;
        continue;
      }
      // K tile, then V tile of 64-key tile j2, each into its own ring
      if (lane == 0) {
        const int sk = n % NKS, uk = n / NKS;
        ok = mbar_wait(&bars->k_empty[sk], (uk & 1) ^ 1, ctx);
        if (ok) {
          mbar_arrive_expect_tx(&bars->k_full[sk], L::kKBytes);
          for (int c = 0; c < L::kChunksK; ++c)
            tma_load_4d(smem_u32(smem + L::k_off + sk * L::kKBytes + c * L::kChunkKV), &tm_k,
                        c * 64, kvh, j2 * BN, bi, &bars->k_full[sk]);
          last_k[sk] = uk;
        }
        const int sv = n % NVS, uv = n / NVS;
        if (ok) ok = mbar_wait(&bars->v_empty[sv], (uv & 1) ^ 1, ctx);
        if (ok) {
          mbar_arrive_expect_tx(&bars->v_full[sv], L::kVBytes);
          for (int c = 0; c < L::kChunksV; ++c)
            tma_load_4d(smem_u32(smem + L::v_off + sv * L::kVBytes + c * L::kChunkKV), &tm_v,
                        c * 64, kvh, j2 * BN, bi, &bars->v_full[sv]);
          last_v[sv] = uv;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++n;
    }
    // Drain: every TMA copy this warp issued has landed before the CTA exits
    // (already true on the normal path; bounded after an abort).
    if (lane == 0) {
      if (!QT) mbar_wait_drain(&bars->q_full, 0, a.status);
      for (int i = 0; i < NKS; ++i)
        if (last_k[i] >= 0) mbar_wait_drain(&bars->k_full[i], last_k[i] & 1, a.status);
      for (int i = 0; i < NVS; ++i)
        if (last_v[i] >= 0) mbar_wait_drain(&bars->v_full[i], last_v[i] & 1, a.status);
    }
  } else if (warp == 1 || warp == 3) {
    // ======================================================== MMA issuers
    // One issuing thread per head slot (warp 1: slot 0, warp 3: slot 1).  Each
    // slot has two S buffers in TMEM, so S(n+1) is computed while the softmax
    // works on S(n): the thread issues S(0), S(1), then per tile
    // PV(n) -> [PV(n) done: P(n) consumed, its buffer free] -> S(n+2).
    const int sl = warp == 1 ? 0 : 1;
    if (lane == 0 && sl < nslots) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(BM, DV, false, true);
      // base descriptors: K-major Q / K tiles, MN-major V tiles (128B swizzle)
      const uint32_t da = sdesc_lo(smem_u32(smem + L::q_off + sl * L::kTileBytes), 16);
      const uint32_t k_lo = sdesc_lo(smem_u32(smem + L::k_off), 16);
      const uint32_t v_lo = sdesc_lo(smem_u32(smem + L::v_off), L::kChunkKV);
      const uint32_t d_s0 = tmem + 2 * sl * BN;  // buffer bb at d_s0 + bb * BN
      const uint32_t d_o = tmem + 4 * BN + sl * DV;
      bool ok = mbar_wait(&bars->q_full, 0, ctx);
      // Slot 1 starts once slot 0's first softmax is done, so the two softmax
      // warpgroups do not start in step.
      if (ok && sl == 1 && nt > 0) ok = mbar_wait(&bars->slot1_go, 0, ctx);
      // n = -2, -1 issue S(0), S(1); every later n issues PV(n), then S(n+2)
      for (int n = -2; n < nt && ok; ++n) {
        if (n >= 0) {
          // O_sl += P_sl(n) V(n): needs V(n) and the softmax of tile n
          const int slot_v = n % NVS;
          ok = mbar_wait(&bars->v_full[slot_v], (n / NVS) & 1, ctx);
          if (ok) ok = mbar_wait(&bars->p_full[sl][n & 1], (n >> 1) & 1, ctx);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dv = v_lo + ((slot_v * L::kVBytes) >> 4);
          const uint32_t d_s = d_s0 + (n & 1) * BN;
          const uint32_t acc0 = n > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts_lo(d_o, d_s + kk * 8, dv + ((kk * 16 * 128) >> 4), idesc_o,
                      kk > 0 ? 1u : acc0);
          mma_commit(&bars->o_done[sl][n & 1]);
        }
        const int m2 = n + 2;
        if (m2 < nt) {
          // S_sl(m2) = Q_sl K(m2)^T into buffer m2 & 1: needs K(m2), and PV(n)
          // done (P(n) lives in that buffer)
          const int slot_k = m2 % NKS;
          ok = mbar_wait(&bars->k_full[slot_k], (m2 / NKS) & 1, ctx);
          if (ok && n >= 0) ok = mbar_wait(&bars->o_done[sl][n & 1], (n >> 1) & 1, ctx);
          if (!ok) break;
          tc_fence_after();
          const uint32_t db = k_lo + ((slot_k * L::kKBytes) >> 4);
          const uint32_t d_s = d_s0 + (m2 & 1) * BN;
#pragma unroll
          for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t offa = ((kk / 4) * L::kChunk + (kk % 4) * 32) >> 4;
            const uint32_t offb = ((kk / 4) * L::kChunkKV + (kk % 4) * 32) >> 4;
            if constexpr (QT)
              mma_ts_lo(d_s, tmem + kColQ + kk * 8, db + offb, idesc_s, kk > 0 ? 1u : 0u);
            else
              mma_ss_lo(d_s, da + offa, db + offb, idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[sl][m2 & 1]);
        }
      }
      // Drain: all MMAs issued by this thread complete before TMEM is freed.
      mma_commit(&bars->drain[sl]);
      mbar_wait_drain(&bars->drain[sl], 0, a.status);
    }
  } else if (warp == 2) {
    // ======================================================== descriptor loader
    // ids / pos / class of each non-SKIP key tile into the ring read by the
    // softmax warpgroups (off the TMA producer's path).
    int n = 0;
    bool ok = true;
    for (int j2 = 2 * rng.x; j2 <= 2 * rng.y + 1 && ok; ++j2) {
      const uint8_t kind = cls_row[j2 >> 1];
      if (kind == kSkip) {
        j2 = 2 * next_live_tile(cls_row, (j2 >> 1) + 1, rng.y, lane) - 1;
        continue;
      }
      const int j = j2;  // 64-key tile index
      const int en = n % NIDD, use = n / NIDD;
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
      int* dst = s_ids + en * kIdEntry;
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
  {
    // ======================================================== softmax
    const int sl = (warp - 4) / 4;
    const int wq = warp % 4;  // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    if (sl < nslots) {
      const int h = h0 + sl;
      const int grow = qt * BM + row;
      const bool row_in = grow < a.s_q;
      const int iq = row_in ? a.q_ids[(int64_t)bi * a.s_q + grow] : 0;
      const int pq = row_in ? a.q_pos[(int64_t)bi * a.s_q + grow] : 0;
      const uint32_t t_s0 = tmem + ((uint32_t)(wq * 32) << 16) + 2 * sl * BN;  // + (n & 1) * BN
      const uint32_t t_o = tmem + ((uint32_t)(wq * 32) << 16) + 4 * BN + sl * DV;
      const float sl2 = a.scale_log2;
      if constexpr (QT) {
        // The query row into TMEM as bf16 pairs (column c holds elements 2c,
        // 2c + 1: the row's own byte order), the A operand of S = Q K^T.
        const uint4* src = reinterpret_cast<const uint4*>(
            a.q + (((int64_t)bi * a.s_q + grow) * a.hq + h) * DK);
#pragma unroll 1
        for (int c = 0; c < DK / 2; c += 32) {
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 v = row_in ? src[c / 4 + u] : make_uint4(0u, 0u, 0u, 0u);
            w[4 * u] = v.x;
            w[4 * u + 1] = v.y;
            w[4 * u + 2] = v.z;
            w[4 * u + 3] = v.w;
          }
          tmem_st32(tmem + ((uint32_t)(wq * 32) << 16) + kColQ + c, w);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->q_full);
      }
      float m = -INFINITY;  // running max (base-2 units)
      float l = 0.f;        // running denominator relative to m
      int n = 0;
      bool ok = true;
      for (; n < nt;) {
        const int en = n % NIDD;
        ok = mbar_wait(&bars->id_full[en], (n / NIDD) & 1, ctx);
        ok = mbar_wait(&bars->s_full[sl][n & 1], (n >> 1) & 1, ctx) && ok;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // S_sl(n) is complete, so this slot is done with K(n) and (its S(n) was
        // issued after PV_sl(n-2) completed) with V(n-2): release both slots.
        // (Releasing them with tcgen05.commit from the MMA threads instead, right
        // after the MMAs that read them, made the forward 6-11 % slower.)
        if (lane == 0) {
          mbar_arrive(&bars->k_empty[n % NKS]);
          if (n > 1) mbar_arrive(&bars->v_empty[(n - 2) % NVS]);
        }
        const uint32_t t_s = t_s0 + (n & 1) * BN;
        uint32_t sr[BN];
        tmem_ld32(t_s + 0, &sr[0]);
        tmem_ld32(t_s + 32, &sr[32]);
        tmem_wait_ld();
        const int kind = s_ids[en * kIdEntry + 2 * BN];
        if (kind == kPartial) {
          const int4* ids4 = reinterpret_cast<const int4*>(s_ids + en * kIdEntry);
          const int4* pos4 = reinterpret_cast<const int4*>(s_ids + en * kIdEntry + BN);
#pragma unroll
          for (int c = 0; c < BN / 4; ++c) {
            const int4 ik = ids4[c];
            const int4 pk4 = pos4[c];
            const int ika[4] = {ik.x, ik.y, ik.z, ik.w};
            const int pka[4] = {pk4.x, pk4.y, pk4.z, pk4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              bool vis = (ika[u] == iq) && (iq != 0) && (pka[u] <= pq);
              if (a.window >= 0) vis = vis && (pq - pka[u] <= a.window);
              if (!vis) sr[4 * c + u] = __float_as_uint(-INFINITY);
            }
          }
        }
        mbar_arrive(&bars->id_empty[en]);
        // row max of the raw scores (scale > 0 keeps the order)
        float mx0 = __uint_as_float(sr[0]), mx1 = __uint_as_float(sr[1]);
        float mx2 = __uint_as_float(sr[2]), mx3 = __uint_as_float(sr[3]);
#pragma unroll
        for (int c = 4; c < BN; c += 4) {
          mx0 = fmaxf(mx0, __uint_as_float(sr[c]));
          mx1 = fmaxf(mx1, __uint_as_float(sr[c + 1]));
          mx2 = fmaxf(mx2, __uint_as_float(sr[c + 2]));
          mx3 = fmaxf(mx3, __uint_as_float(sr[c + 3]));
        }
        const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
        const float m_new = fmaxf(m, mt);
        float alpha = 1.f;
        bool rescale = false;
        float m_use = m;
        if (m == -INFINITY) {
          m_use = m_new;  // nothing accumulated yet: O row and l are 0
        } else if (m_new > m + kRescaleThreshold) {
          m_use = m_new;
          alpha = ex2(m - m_new);
          rescale = true;
        }
        const float msub = (m_use == -INFINITY) ? 0.f : m_use;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        // packed bf16 P overwrites the front of the score registers
#pragma unroll
        for (int c = 0; c < BN; c += 4) {
          float p0, p1, p2, p3;
          if constexpr (kSlots<DK, DV> == 2) {
            // two softmax warps per SM sub-partition: issue slots are the limit,
            // so exponent arguments and running sums go two lanes per instruction
            float x0, x1, x2, x3;
            fma_f32x2(x0, x1, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), sl2, sl2,
                      -msub, -msub);
            fma_f32x2(x2, x3, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]), sl2, sl2,
                      -msub, -msub);
            p0 = ex2(x0);
            p1 = ex2(x1);
            p2 = ex2(x2);
            p3 = ex2(x3);
            add_f32x2(s0, s1, s0, s1, p0, p1);
            add_f32x2(s2, s3, s2, s3, p2, p3);
          } else {
            // one softmax warp per sub-partition: latency is the limit
            p0 = ex2(fmaf(__uint_as_float(sr[c]), sl2, -msub));
            p1 = ex2(fmaf(__uint_as_float(sr[c + 1]), sl2, -msub));
            p2 = ex2(fmaf(__uint_as_float(sr[c + 2]), sl2, -msub));
            p3 = ex2(fmaf(__uint_as_float(sr[c + 3]), sl2, -msub));
            s0 += p0;
            s1 += p1;
            s2 += p2;
            s3 += p3;
          }
          sr[c / 2] = pack_bf16(p0, p1);
          sr[c / 2 + 1] = pack_bf16(p2, p3);
        }
        l = l * alpha + ((s0 + s1) + (s2 + s3));
        m = m_use;
        tmem_st32(t_s + 0, &sr[0]);  // P (bf16 pairs) over the first 32 columns
        if (__any_sync(0xffffffffu, rescale) && n > 0) {
          // O += P V of the previous tile must be complete before O is rescaled.
          ok = mbar_wait(&bars->o_done[sl][(n - 1) & 1], ((n - 1) >> 1) & 1, ctx);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DV; c += 32) {
            uint32_t o[32];
            tmem_ld32(t_o + c, o);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
            tmem_st32(t_o + c, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[sl][n & 1]);
        if (n == 0 && sl == 0 && row == 0 && nslots > 1) mbar_arrive(&bars->slot1_go);
        ++n;
      }
      // ---- epilogue: O = u / z, LSE = ln2 * (m + log2 z)
      // The last two P.V groups may both be in flight here (S(n) only waits for
      // P.V(n-2)), which is why each S buffer has its own o_done barrier: the
      // last P.V's phase is then never ahead of or behind the waited one by
      // more than one, and its commit covers every earlier MMA of the slot.
      if (ok && n > 0) {
        ok = mbar_wait(&bars->o_done[sl][(n - 1) & 1], ((n - 1) >> 1) & 1, ctx);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
      }
      if (ok) {
        const bool has = l > 0.f;
        float inv = has ? 1.f / l : 0.f;
        const int64_t orow = ((int64_t)bi * a.s_q + grow) * a.hq + h;
        const int64_t lidx = ((int64_t)bi * a.hq + h) * a.s_q + grow;
        float lse_row = has ? (m + log2f(l)) * kLn2 : -INFINITY;
        // merge mode: out = ca * out + cb * (this block's O), lse = merged
        float ca = 0.f;
        if (a.merge && row_in) {
          float cb;
          merge_coeffs(a.lse[lidx], lse_row, ca, cb, lse_row);
          inv *= cb;
        }
#pragma unroll 1
        for (int c = 0; c < DV; c += 32) {
          uint32_t o[32];
          if (n > 0) {
            tmem_ld32(t_o + c, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = 0u;
          }
          if (!row_in) continue;
          if (a.merge) {
            float* acc = static_cast<float*>(a.out) + orow * DV + c;
            float v[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
              if (ca != 0.f) x = reinterpret_cast<const float4*>(acc)[u];
              v[4 * u] = merge1(ca, 1.f, x.x, __uint_as_float(o[4 * u]) * inv);
              v[4 * u + 1] = merge1(ca, 1.f, x.y, __uint_as_float(o[4 * u + 1]) * inv);
              v[4 * u + 2] = merge1(ca, 1.f, x.z, __uint_as_float(o[4 * u + 2]) * inv);
              v[4 * u + 3] = merge1(ca, 1.f, x.w, __uint_as_float(o[4 * u + 3]) * inv);
            }
            if (a.out_final) {
              uint4* dst = reinterpret_cast<uint4*>(a.out_final + orow * DV + c);
#pragma unroll
              for (int u = 0; u < 4; ++u)
                dst[u] = make_uint4(pack_bf16(v[8 * u], v[8 * u + 1]), pack_bf16(v[8 * u + 2], v[8 * u + 3]),
                                    pack_bf16(v[8 * u + 4], v[8 * u + 5]),
                                    pack_bf16(v[8 * u + 6], v[8 * u + 7]));
            } else {
#pragma unroll
              for (int u = 0; u < 8; ++u)
                reinterpret_cast<float4*>(acc)[u] =
                    make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            }
            continue;
          }
          if (a.out_fp32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow * DV + c);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              dst[u] = make_float4(__uint_as_float(o[4 * u]) * inv, __uint_as_float(o[4 * u + 1]) * inv,
                                   __uint_as_float(o[4 * u + 2]) * inv,
                                   __uint_as_float(o[4 * u + 3]) * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow * DV + c);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint4 w;
              w.x = pack_bf16(__uint_as_float(o[8 * u + 0]) * inv, __uint_as_float(o[8 * u + 1]) * inv);
              w.y = pack_bf16(__uint_as_float(o[8 * u + 2]) * inv, __uint_as_float(o[8 * u + 3]) * inv);
              w.z = pack_bf16(__uint_as_float(o[8 * u + 4]) * inv, __uint_as_float(o[8 * u + 5]) * inv);
              w.w = pack_bf16(__uint_as_float(o[8 * u + 6]) * inv, __uint_as_float(o[8 * u + 7]) * inv);
              dst[u] = w;
            }
          }
        }
        if (row_in) a.lse[lidx] = lse_row;
      }
    }
  }

  // ---- teardown (the producer and MMA threads drained their async work above)
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int DK, int DV>
cudaError_t launch_fwd_d(const FwdArgs& a, const FwdLaunch& Lc, int64_t units, cudaStream_t st) {
  const int smem = Layout<DK, DV>::alloc;
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(attn_fwd_kernel<DK, DV>), smem,
                                    kLaunchRegs, smem_set);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<DK, DV><<<(unsigned)units, kThreads, smem, st>>>(Lc.tm_q, Lc.tm_k, Lc.tm_v, a);
  return cudaGetLastError();
}

}  // namespace

int64_t fwd_ctas_per_tile(const attn_fwd_params& p) {
  const int64_t dv = p.d_v > 0 ? p.d_v : p.d;
  const int64_t slots = dv <= 128 ? 2 : 1;  // query heads per CTA (kSlots)
  const int64_t g = p.h_q / p.h_kv;
  return p.h_kv * ((g + slots - 1) / slots);
}

cudaError_t launch_attn_fwd(const FwdLaunch& Lc, cudaStream_t st) {
  const attn_fwd_params& p = *Lc.p;
  FwdArgs a;
  a.withhold_kv = Lc.withhold_kv ? 1 : 0;
  a.q = static_cast<const __nv_bfloat16*>(p.q);
  a.q_ids = p.q_segment_ids;
  a.q_pos = p.q_segment_pos;
  a.kv_ids = p.kv_segment_ids;
  a.kv_pos = p.kv_segment_pos;
  a.out = p.out;
  a.lse = p.lse;
  a.cls = Lc.plan.classes;
  a.qrange = Lc.plan.q_range;
  a.qweight = Lc.plan.q_weight;
  a.order = Lc.plan.q_order;
  a.status = Lc.plan.status;
  a.b = (int)p.b;
  a.s_q = (int)p.s_q;
  a.s_kv = (int)p.s_kv;
  a.hq = (int)p.h_q;
  a.hkv = (int)p.h_kv;
  a.g = (int)(p.h_q / p.h_kv);
  const int64_t dv = p.d_v > 0 ? p.d_v : p.d;
  a.npairs = (int)(fwd_ctas_per_tile(p) / p.h_kv);
  a.nq = (int)Lc.nq;
  a.nk = (int)Lc.nk;
  a.window = p.window_left;
  a.out_fp32 = p.out_fp32 ? 1 : 0;
  a.merge = p.merge_into_out ? 1 : 0;
  a.out_final = static_cast<__nv_bfloat16*>(p.out_final);
  a.scale_log2 = p.scale * 1.4426950408889634f;
  const int64_t units = p.b * Lc.nq * p.h_kv * a.npairs;
  if (units == 0) return cudaSuccess;
  if (p.d == 128) return launch_fwd_d<128, 128>(a, Lc, units, st);
  if (p.d == 256) return launch_fwd_d<256, 256>(a, Lc, units, st);
  if (p.d == 192 && dv == 128) return launch_fwd_d<192, 128>(a, Lc, units, st);
  return launch_fwd_d<64, 64>(a, Lc, units, st);
}

}  // namespace gb300
