// C ABI of gb300attn: argument validation, tensor-map encoding, launches.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>

#include "internal.h"

using namespace gb300;

namespace {

// cuTensorMapEncodeTiled from the driver, looked up once per process (a
// function-local static: initialised exactly once even when several host
// threads make their first call at the same time).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return nullptr;
  }();
  return fn;
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Head dim of v and out (d_v = 0 means d).
int64_t fwd_dv(const attn_fwd_params* p) { return p->d_v > 0 ? p->d_v : p->d; }

// Shared checks of the forward problem description.
int check_fwd(const attn_fwd_params* p) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (!p->q || !p->k || !p->v || !p->q_segment_ids || !p->q_segment_pos || !p->kv_segment_ids ||
      !p->kv_segment_pos || !p->out || !p->lse)
    return ATTN_ERR_INVALID_ARG;
  if (p->b < 1 || p->s_q < 1 || p->s_kv < 1 || p->h_q < 1 || p->h_kv < 1 || p->d < 1)
    return ATTN_ERR_INVALID_ARG;
  if (p->h_q % p->h_kv) return ATTN_ERR_INVALID_ARG;
  if (p->window_right != 0 || p->window_left < -1) return ATTN_ERR_INVALID_ARG;
  if (!(p->scale > 0.f) || !std::isfinite(p->scale)) return ATTN_ERR_INVALID_ARG;
  if (p->s_q > (1ll << 30) || p->s_kv > (1ll << 30) || p->h_q > 65535 || p->b > 65535)
    return ATTN_ERR_UNSUPPORTED;
  if (p->d_v < 0) return ATTN_ERR_INVALID_ARG;
  const int64_t dv = fwd_dv(p);
  // head dims (q/k, v): (64, 64), (128, 128), (256, 256), (192, 128)
  if (!((dv == p->d && (p->d == 64 || p->d == 128 || p->d == 256)) || (p->d == 192 && dv == 128)))
    return ATTN_ERR_UNSUPPORTED;
  if (dv != p->d && p->kv_token_stride != 0) return ATTN_ERR_INVALID_ARG;
  if (!aligned(p->q, 16) || !aligned(p->k, 16) || !aligned(p->v, 16) || !aligned(p->out, 16) ||
      !aligned(p->lse, 4) || !aligned(p->q_segment_ids, 4) || !aligned(p->q_segment_pos, 4) ||
      !aligned(p->kv_segment_ids, 4) || !aligned(p->kv_segment_pos, 4))
    return ATTN_ERR_INVALID_ARG;
  if (p->kv_token_stride != 0 &&
      (p->kv_token_stride < p->h_kv * p->d || p->kv_token_stride % 8 != 0 ||
       p->kv_token_stride > (1ll << 24)))
    return ATTN_ERR_INVALID_ARG;
  if (p->merge_into_out != 0 && p->merge_into_out != 1) return ATTN_ERR_INVALID_ARG;
  if (p->merge_into_out && !p->out_fp32) return ATTN_ERR_INVALID_ARG;
  if (p->out_final) {
    if (!p->merge_into_out || !aligned(p->out_final, 16)) return ATTN_ERR_INVALID_ARG;
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(p->out);
    const uintptr_t f0 = reinterpret_cast<uintptr_t>(p->out_final);
    const uintptr_t n = (uintptr_t)(p->b * p->s_q * p->h_q * dv);
    if (o0 < f0 + 2 * n && f0 < o0 + 4 * n) return ATTN_ERR_INVALID_ARG;  // overlap
  }
  const int64_t g = p->h_q / p->h_kv;
  const int64_t slots = dv <= 128 ? 2 : 1;  // query heads per forward CTA
  const int64_t units = p->b * cdiv(p->s_q, kTile) * p->h_kv * ((g + slots - 1) / slots);
  if (units > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

PlanLayout fwd_layout(const attn_fwd_params* p) {
  return plan_layout(p->b, cdiv(p->s_q, kTile), cdiv(p->s_kv, kTile));
}

int check_workspace(const attn_fwd_params* p, size_t need) {
  if (!p->workspace || !aligned(p->workspace, 256) || p->workspace_bytes < need)
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

}  // namespace

namespace gb300 {

bool encode_qkv_map(CUtensorMap* m, const void* base, int64_t b, int64_t s, int64_t h, int64_t d,
                    int64_t token_stride, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int64_t ts = token_stride > 0 ? token_stride : h * d;  // elements between tokens
  // dims innermost first: (d, head, token, batch); box = 64 d x 1 head x box_rows tokens.
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)h, (cuuint64_t)s, (cuuint64_t)b};
  cuuint64_t strides[3] = {(cuuint64_t)(d * 2), (cuuint64_t)(ts * 2), (cuuint64_t)(s * ts * 2)};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [b, s, h, d] accumulator viewed as (d, head, token, batch); box =
// 32 d (128 bytes, swizzled) x 1 head x 128 tokens, for tiled reduce-adds.
bool encode_acc_map(CUtensorMap* m, const float* base, int64_t b, int64_t s, int64_t h, int64_t d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)h, (cuuint64_t)s, (cuuint64_t)b};
  cuuint64_t strides[3] = {(cuuint64_t)(d * 4), (cuuint64_t)(h * d * 4), (cuuint64_t)(s * h * d * 4)};
  cuuint32_t box[4] = {32, 1, (cuuint32_t)kTile, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gb300

extern "C" {

size_t attn_fwd_workspace_bytes(const attn_fwd_params* p) {
  if (check_fwd(p) != ATTN_OK) return 0;
  return fwd_layout(p).end;
}

static int fwd_impl(const attn_fwd_params* p, attn_stream_t stream, bool withhold_kv) {
  int rc = check_fwd(p);
  if (rc != ATTN_OK) return rc;
  const PlanLayout L = fwd_layout(p);
  rc = check_workspace(p, L.end);
  if (rc != ATTN_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  FwdLaunch fl;
  fl.p = p;
  fl.plan = plan_ptrs(p->workspace, L);
  fl.nq = cdiv(p->s_q, kTile);
  fl.nk = cdiv(p->s_kv, kTile);
  fl.withhold_kv = withhold_kv;
  if (!encode_qkv_map(&fl.tm_q, p->q, p->b, p->s_q, p->h_q, p->d, 0) ||
      !encode_qkv_map(&fl.tm_k, p->k, p->b, p->s_kv, p->h_kv, p->d, p->kv_token_stride,
                      kFwdKeyTile) ||
      !encode_qkv_map(&fl.tm_v, p->v, p->b, p->s_kv, p->h_kv, fwd_dv(p), p->kv_token_stride,
                      kFwdKeyTile))
    return ATTN_ERR_CUDA;
  cudaError_t e = cudaMemsetAsync(fl.plan.status, 0, sizeof(int), st);
  if (e == cudaSuccess)
    e = launch_tile_plan(*p, fl.plan, fl.nq, fl.nk, false, fwd_ctas_per_tile(*p), 0, st);
  if (e == cudaSuccess) e = launch_attn_fwd(fl, st);
  return cuda_status(e);
}

int attn_fwd(const attn_fwd_params* p, attn_stream_t stream) {
  return fwd_impl(p, stream, false);
}

int attn_fwd_test_timeout(const attn_fwd_params* p, attn_stream_t stream) {
  return fwd_impl(p, stream, true);
}

int attn_tile_plan(const attn_fwd_params* p, uint8_t* classes, int32_t* ranges,
                   attn_stream_t stream) {
  int rc = check_fwd(p);
  if (rc != ATTN_OK) return rc;
  if (!classes || !ranges || !aligned(ranges, 4)) return ATTN_ERR_INVALID_ARG;
  const PlanLayout L = fwd_layout(p);
  rc = check_workspace(p, L.end);
  if (rc != ATTN_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t nq = cdiv(p->s_q, kTile), nk = cdiv(p->s_kv, kTile);
  const PlanPtrs pp = plan_ptrs(p->workspace, L);
  cudaError_t e = launch_tile_plan(*p, pp, nq, nk, false, fwd_ctas_per_tile(*p), 0, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(classes, pp.classes, (size_t)(p->b * nq * nk), cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ranges, pp.q_range, (size_t)(p->b * nq) * 8, cudaMemcpyDeviceToDevice, st);
  return cuda_status(e);
}

// Which backward runs: the fused kernel (dQ summed through an fp32
// accumulator in global memory) or the dK / dV kernel plus the dQ kernel
// (dQ summed on chip in a fixed order: deterministic).  The head dims whose
// dK and dV do not fit the fused kernel's TMEM (256, and 192 / 128) always
// take the pair.
static bool use_split_bwd(const attn_bwd_params* p) {
  const attn_fwd_params* f = &p->fwd;
  const int64_t dv = fwd_dv(f);
  return f->d == 256 || (f->d == 192 && dv == 128) || p->deterministic != 0;
}

int attn_tile_order(const attn_fwd_params* p, int32_t* q_order, int32_t* kv_order,
                    attn_stream_t stream) {
  int rc = check_fwd(p);
  if (rc != ATTN_OK) return rc;
  if (!q_order || !kv_order || !aligned(q_order, 4) || !aligned(kv_order, 4))
    return ATTN_ERR_INVALID_ARG;
  const PlanLayout L = fwd_layout(p);
  rc = check_workspace(p, L.end);
  if (rc != ATTN_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t nq = cdiv(p->s_q, kTile), nk = cdiv(p->s_kv, kTile);
  const PlanPtrs pp = plan_ptrs(p->workspace, L);
  // the orders the forward (query side) and the fused backward (key side) take
  cudaError_t e = launch_tile_plan(*p, pp, nq, nk, true, fwd_ctas_per_tile(*p), p->h_kv, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(q_order, pp.q_order, (size_t)(p->b * nq) * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(kv_order, pp.kv_order, (size_t)(p->b * nk) * 4, cudaMemcpyDeviceToDevice,
                        st);
  return cuda_status(e);
}

size_t attn_bwd_workspace_bytes(const attn_bwd_params* p) {
  if (!p || check_fwd(&p->fwd) != ATTN_OK) return 0;
  const PlanLayout L = fwd_layout(&p->fwd);
  const size_t d_bytes = align_up((size_t)(p->fwd.b * p->fwd.h_q * p->fwd.s_q) * 4, 256);
  if (use_split_bwd(p)) return L.end + d_bytes;
  const size_t dq_bytes = align_up((size_t)(p->fwd.b * p->fwd.s_q * p->fwd.h_q * p->fwd.d) * 4, 256);
  return L.end + d_bytes + dq_bytes;
}

constexpr float kBwdMinScale = 1e-30f;

int attn_bwd(const attn_bwd_params* p, attn_stream_t stream) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  int rc = check_fwd(&p->fwd);
  if (rc != ATTN_OK) return rc;
  if (p->fwd.out_fp32 || p->fwd.merge_into_out || p->fwd.out_final) return ATTN_ERR_INVALID_ARG;
  // The kernel feeds (LSE - ln scale) / scale to the tensor core as bf16
  // parts; below 1e-30 that value could leave the fp32 range.
  if (p->fwd.scale < kBwdMinScale) return ATTN_ERR_UNSUPPORTED;
  if (!p->dout || !p->dq || !p->dk || !p->dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned(p->dout, 16) || !aligned(p->dq, 16) || !aligned(p->dk, 16) || !aligned(p->dv, 16))
    return ATTN_ERR_INVALID_ARG;
  const attn_fwd_params* f = &p->fwd;
  const PlanLayout L = fwd_layout(f);
  const size_t need = attn_bwd_workspace_bytes(p);
  rc = check_workspace(f, need);
  if (rc != ATTN_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t dv = fwd_dv(f);
  if (p->deterministic != 0 && p->deterministic != 1) return ATTN_ERR_INVALID_ARG;
  if ((p->kernel_events[0] == nullptr) != (p->kernel_events[1] == nullptr))
    return ATTN_ERR_INVALID_ARG;
  if (p->delta) {
    // the optional D output: aligned, and clear of every other buffer
    if (!aligned(p->delta, 4)) return ATTN_ERR_INVALID_ARG;
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(p->delta);
    const uintptr_t dn = (uintptr_t)(f->b * f->h_q * f->s_q) * 4;
    const uintptr_t rows = (uintptr_t)(f->b * f->s_q * f->h_q);
    const uintptr_t gsz = p->accumulate_fp32 ? 4 : 2;
    const uintptr_t toks = (uintptr_t)(f->b * f->s_kv);
    const uintptr_t kst = f->kv_token_stride > 0 ? (uintptr_t)f->kv_token_stride
                                                 : (uintptr_t)(f->h_kv * f->d);
    const uintptr_t vst = f->kv_token_stride > 0 ? (uintptr_t)f->kv_token_stride
                                                 : (uintptr_t)(f->h_kv * dv);
    const struct { const void* a; uintptr_t n; } others[] = {
        {f->workspace, (uintptr_t)f->workspace_bytes},
        {f->out, rows * (uintptr_t)dv * 2},
        {p->dout, rows * (uintptr_t)dv * 2},
        {f->lse, dn},
        {p->dq, rows * (uintptr_t)f->d * gsz},
        {p->dk, toks * kst * gsz},
        {p->dv, toks * vst * gsz}};
    for (const auto& o : others) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(o.a);
      if (a0 < d0 + dn && d0 < a0 + o.n) return ATTN_ERR_INVALID_ARG;
    }
  }
  // optional timing hook around the main kernel(s)
  auto mark = [&](int i) -> cudaError_t {
    return p->kernel_events[i]
               ? cudaEventRecord(reinterpret_cast<cudaEvent_t>(p->kernel_events[i]), st)
               : cudaSuccess;
  };
  if (use_split_bwd(p)) {
    SplitLaunch sl;
    sl.p = p;
    sl.plan = plan_ptrs(f->workspace, L);
    sl.nq = cdiv(f->s_q, kTile);
    sl.nk = cdiv(f->s_kv, kTile);
    sl.D = p->delta ? p->delta : reinterpret_cast<float*>(static_cast<char*>(f->workspace) + L.end);
    const int bm = split_bwd_query_rows(f->d, dv), bn = split_bwd_key_rows(f->d, dv);
    if (!encode_qkv_map(&sl.tm_q, f->q, f->b, f->s_q, f->h_q, f->d, 0) ||
        !encode_qkv_map(&sl.tm_do, p->dout, f->b, f->s_q, f->h_q, dv, 0) ||
        !encode_qkv_map(&sl.tm_q_a, f->q, f->b, f->s_q, f->h_q, f->d, 0, bm) ||
        !encode_qkv_map(&sl.tm_do_a, p->dout, f->b, f->s_q, f->h_q, dv, 0, bm) ||
        !encode_qkv_map(&sl.tm_k, f->k, f->b, f->s_kv, f->h_kv, f->d, f->kv_token_stride) ||
        !encode_qkv_map(&sl.tm_v, f->v, f->b, f->s_kv, f->h_kv, dv, f->kv_token_stride) ||
        !encode_qkv_map(&sl.tm_kb, f->k, f->b, f->s_kv, f->h_kv, f->d, f->kv_token_stride, bn) ||
        !encode_qkv_map(&sl.tm_vb, f->v, f->b, f->s_kv, f->h_kv, dv, f->kv_token_stride, bn))
      return ATTN_ERR_CUDA;
    cudaError_t e = cudaMemsetAsync(sl.plan.status, 0, sizeof(int), st);
    // dQ kernel: one CTA per query tile and head; dK / dV kernel: one per key
    // tile, kv head and column slice
    if (e == cudaSuccess)
      e = launch_tile_plan(*f, sl.plan, sl.nq, sl.nk, true, f->h_q,
                           f->h_kv * split_bwd_col_slices(f->d, dv), st);
    if (e == cudaSuccess)
      e = launch_bwd_preprocess(f->out, p->dout, sl.D, nullptr, sl.plan.q_weight, f->b, f->s_q,
                                f->h_q, dv, st);
    if (e == cudaSuccess) e = mark(0);
    if (e == cudaSuccess) e = launch_attn_bwd_split(sl, st);
    if (e == cudaSuccess) e = mark(1);
    if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
    return cuda_status(e);
  }
  if (dv != f->d) return ATTN_ERR_UNSUPPORTED;
  BwdLaunch bl;
  bl.p = p;
  bl.plan = plan_ptrs(f->workspace, L);
  bl.nq = cdiv(f->s_q, kTile);
  bl.nk = cdiv(f->s_kv, kTile);
  char* ws = static_cast<char*>(f->workspace);
  bl.D = p->delta ? p->delta : reinterpret_cast<float*>(ws + L.end);
  const bool acc = p->accumulate_fp32 != 0;
  // accumulate mode: the dQ reduce-adds go straight into the caller's fp32 dq
  bl.dq_acc = acc ? static_cast<float*>(p->dq)
                  : reinterpret_cast<float*>(
                        ws + L.end + align_up((size_t)(f->b * f->h_q * f->s_q) * 4, 256));
  if (!encode_qkv_map(&bl.tm_q, f->q, f->b, f->s_q, f->h_q, f->d, 0) ||
      !encode_qkv_map(&bl.tm_k, f->k, f->b, f->s_kv, f->h_kv, f->d, f->kv_token_stride) ||
      !encode_qkv_map(&bl.tm_v, f->v, f->b, f->s_kv, f->h_kv, f->d, f->kv_token_stride) ||
      !encode_qkv_map(&bl.tm_do, p->dout, f->b, f->s_q, f->h_q, f->d, 0) ||
      !encode_acc_map(&bl.tm_dq, bl.dq_acc, f->b, f->s_q, f->h_q, f->d))
    return ATTN_ERR_CUDA;
  cudaError_t e = cudaMemsetAsync(bl.plan.status, 0, sizeof(int), st);
  if (e == cudaSuccess)
    e = launch_tile_plan(*f, bl.plan, bl.nq, bl.nk, true, f->h_q, f->h_kv, st);
  // the D pre-pass also zeroes the workspace's fp32 dQ accumulator (not the
  // caller's accumulator in accumulate mode)
  if (e == cudaSuccess)
    e = launch_bwd_preprocess(f->out, p->dout, bl.D, acc ? nullptr : bl.dq_acc,
                              bl.plan.q_weight, f->b, f->s_q, f->h_q, f->d, st);
  if (e == cudaSuccess) e = mark(0);
  if (e == cudaSuccess) e = launch_attn_bwd(bl, st);
  if (e == cudaSuccess) e = mark(1);
  if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
  if (e == cudaSuccess && !acc)
    e = launch_dq_finalize(bl.dq_acc, p->dq, bl.plan.q_weight, f->b, f->s_q, f->h_q, f->d, st);
  return cuda_status(e);
}

int attn_segments_from_seqlens(const int32_t* seqlens, const int32_t* offsets, int64_t b,
                               int64_t nseg, int64_t s, int32_t* ids, int32_t* pos,
                               attn_stream_t stream) {
  if (!seqlens || !ids || !pos || b < 1 || nseg < 1 || s < 1) return ATTN_ERR_INVALID_ARG;
  if (!aligned(seqlens, 4) || !aligned(ids, 4) || !aligned(pos, 4) || (offsets && !aligned(offsets, 4)))
    return ATTN_ERR_INVALID_ARG;
  if (nseg > kSegMax || s > (1ll << 30) || b > 65535) return ATTN_ERR_UNSUPPORTED;
  const uintptr_t i0 = reinterpret_cast<uintptr_t>(ids), p0 = reinterpret_cast<uintptr_t>(pos);
  const uintptr_t n = (uintptr_t)(b * s) * 4, m = (uintptr_t)(b * nseg) * 4;
  const uintptr_t l0 = reinterpret_cast<uintptr_t>(seqlens);
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(offsets);
  if (i0 < p0 + n && p0 < i0 + n) return ATTN_ERR_INVALID_ARG;  // ids / pos overlap
  for (uintptr_t out0 : {i0, p0}) {
    if (out0 < l0 + m && l0 < out0 + n) return ATTN_ERR_INVALID_ARG;
    if (offsets && out0 < o0 + m && o0 < out0 + n) return ATTN_ERR_INVALID_ARG;
  }
  return cuda_status(launch_segments(seqlens, offsets, b, nseg, s, ids, pos,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int attn_merge_partial(float* out_acc, float* lse_acc, const void* out_blk, const float* lse_blk,
                       int blk_is_bf16, void* out_final, int64_t b, int64_t s, int64_t h, int64_t d,
                       attn_stream_t stream) {
  if (!out_acc || !lse_acc || !out_blk || !lse_blk) return ATTN_ERR_INVALID_ARG;
  if (b < 1 || s < 1 || h < 1 || d < 8 || d % 8) return ATTN_ERR_INVALID_ARG;
  if (!aligned(out_acc, 16) || !aligned(out_blk, 16) || !aligned(lse_acc, 4) ||
      !aligned(lse_blk, 4) || (out_final && !aligned(out_final, 16)))
    return ATTN_ERR_INVALID_ARG;
  return cuda_status(launch_merge(out_acc, lse_acc, out_blk, lse_blk, blk_is_bf16 ? 1 : 0,
                                  out_final, b, s, h, d, reinterpret_cast<cudaStream_t>(stream)));
}

static int reorder_common(const void* in, void* out, int64_t outer, int64_t s, int64_t inner,
                          int strategy, int cp, int stripe, bool inverse, attn_stream_t stream) {
  if (!in || !out || in == out) return ATTN_ERR_INVALID_ARG;
  if (outer < 1 || s < 1 || inner < 1 || cp < 1) return ATTN_ERR_INVALID_ARG;
  if (strategy == ATTN_REORDER_DUAL_CHUNK) {
    if (s % (2ll * cp)) return ATTN_ERR_INVALID_ARG;
  } else if (strategy == ATTN_REORDER_STRIPED) {
    if (stripe < 1 || s % ((int64_t)cp * stripe)) return ATTN_ERR_INVALID_ARG;
  } else {
    return ATTN_ERR_INVALID_ARG;
  }
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(in), b0 = reinterpret_cast<uintptr_t>(out);
  const uintptr_t n = (uintptr_t)(outer * s * inner);
  if (a0 < b0 + n && b0 < a0 + n) return ATTN_ERR_INVALID_ARG;  // overlapping buffers
  return cuda_status(launch_permute(in, out, outer, s, inner, strategy, cp, stripe, inverse,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int reorder_causal_lb(const void* in, void* out, int64_t outer, int64_t s, int64_t inner_bytes,
                      int strategy, int cp_size, int stripe_size, attn_stream_t stream) {
  return reorder_common(in, out, outer, s, inner_bytes, strategy, cp_size, stripe_size, false,
                        stream);
}

int inverse_reorder_causal_lb(const void* in, void* out, int64_t outer, int64_t s,
                              int64_t inner_bytes, int strategy, int cp_size, int stripe_size,
                              attn_stream_t stream) {
  return reorder_common(in, out, outer, s, inner_bytes, strategy, cp_size, stripe_size, true,
                        stream);
}

int attn_read_device_status(const void* workspace, attn_stream_t stream) {
  if (!workspace || !aligned(workspace, 256)) return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return v;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
