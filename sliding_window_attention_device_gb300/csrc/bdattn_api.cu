// Host side of the bdattn C ABI: argument checks, TMA tensor maps, launches.
// The library allocates no device memory and never synchronises a stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace bd {
cudaError_t launch_seg_build(const int32_t* doc, const Geom& g, int32_t* seg, int32_t* status, cudaStream_t st,
                             int kv_chunk);
cudaError_t launch_merge(const Geom& g, void* out, float* lse, const void* out_c, const float* lse_c,
                         const int32_t* status, cudaStream_t st);
cudaError_t launch_fwd512(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const int32_t* seg,
                          const Geom& g, void* out, float* lse, int32_t* status, bool merge, cudaStream_t st);
cudaError_t launch_fwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const int32_t* seg,
                       const Geom& g, void* out, float* lse, int32_t* status, int merge, cudaStream_t st);
cudaError_t launch_bwd_prep(const Geom& g, const void* dout, const void* out, void* workspace, float* dq_f32,
                            int32_t* status, cudaStream_t st);
cudaError_t launch_bwd_main(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CUtensorMap& mdq, const int32_t* seg, const Geom& g, const float* lse, void* dk,
                            void* dv, int bf16, void* workspace, float* dq_f32, int32_t* status, cudaStream_t st);
cudaError_t launch_bwd_finalize(const Geom& g, void* dq, int bf16, void* workspace, int32_t* status,
                                cudaStream_t st);
size_t bwd_workspace_bytes(const Geom& g);
cudaError_t launch_bwd_delta(const Geom& g, const void* dout, const void* out, void* workspace, int32_t* status,
                             cudaStream_t st);
const float* bwd_delta_ptr(const Geom& g, void* workspace);
cudaError_t launch_bwd_main_nodq(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                                 const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                                 void* dk, void* dv, int bf16, void* workspace, int32_t* status, cudaStream_t st);
cudaError_t launch_bwd_dq(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk,
                          const CUtensorMap& mv, const int32_t* seg, const Geom& g, const float* lse,
                          const float* delta, void* dq, int bf16, int32_t* status, cudaStream_t st);
cudaError_t launch_exchange_plan(const int32_t* doc, int B, int S, int W, int rank, int32_t* plan, int32_t* status,
                                 cudaStream_t st);
cudaError_t launch_needed_gather(const void* x, const int32_t* plan, int B, int C, int L, int vshift, void* send,
                                 int max_rows, int32_t* status, cudaStream_t st);
cudaError_t launch_needed_scatter_add(const void* gsend, const int32_t* plan, int B, int C, int L, int vshift,
                                      int bf16, void* glocal, int max_rows, int32_t* status, cudaStream_t st);
int bwd_q_box_rows(int D);

__global__ void selftest_wait_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nobody arrives on `bar`: the wait must give up after limit_ns
    if (!mbar_wait(&bar, 0, &abort_flag, nullptr, 0, limit_ns)) atomicOr(status, BD_STATUS_TIMEOUT);
  }
}
}  // namespace bd

using namespace bd;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BD_ERR_CUDA;
  int major = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return BD_ERR_CUDA;
  return major == 10 ? BD_OK : BD_ERR_UNSUPPORTED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int to_geom(const bd_geom* in, Geom* g) {
  if (!in) return BD_ERR_ARG;
  if (in->B < 1 || in->Hq < 1 || in->Hkv < 1 || in->Hq % in->Hkv != 0) return BD_ERR_ARG;
  if (in->D != 64 && in->D != 128 && in->D != 256 && in->D != 512) return BD_ERR_ARG;
  if (in->L < 1 || in->S_kv < 1 || in->S_full < 1) return BD_ERR_ARG;
  if (in->row_offset < 0 || static_cast<long long>(in->row_offset) + in->L > in->S_full) return BD_ERR_ARG;
  if (in->kv_offset < 0 || static_cast<long long>(in->kv_offset) + in->S_kv > in->S_full) return BD_ERR_ARG;
  // keep every index the kernels form within 32-bit range
  if (in->S_full > (1 << 28) || static_cast<long long>(in->B) * in->Hq > (1 << 20)) return BD_ERR_ARG;
  if (static_cast<long long>(in->B) * (in->L + 1) * 4 + static_cast<long long>(in->B) * in->S_kv > (1LL << 29))
    return BD_ERR_ARG;
  if (!(in->scale == in->scale)) return BD_ERR_ARG;  // NaN
  if (in->kv_layout != BD_KV_BHSD && in->kv_layout != BD_KV_SBHD) return BD_ERR_ARG;
  if (!(in->dropout_p >= 0.f && in->dropout_p < 1.f)) return BD_ERR_ARG;  // also NaN
  const double t = std::floor(static_cast<double>(in->dropout_p) * 65536.0 + 0.5);
  if (t > 65535.0) return BD_ERR_ARG;
  g->drop_t = static_cast<uint32_t>(t);
  g->drop_scale = static_cast<float>(65536.0 / (65536.0 - t));
  g->seed_lo = in->seed_lo;
  g->seed_hi = in->seed_hi;
  g->B = in->B;
  g->Hq = in->Hq;
  g->Hkv = in->Hkv;
  g->D = in->D;
  g->G = in->Hq / in->Hkv;
  g->S_full = in->S_full;
  g->L = in->L;
  g->row_offset = in->row_offset;
  g->kv_offset = in->kv_offset;
  g->S_kv = in->S_kv;
  g->window = in->window > 0 ? in->window : 0;
  g->scale = in->scale > 0.f ? in->scale : 1.0f / std::sqrt(static_cast<float>(in->D));
  g->kv_tm = in->kv_layout == BD_KV_SBHD;
  seg_layout(g->B, g->L, g->S_kv, g->off, &g->nqt, &g->nkt, &g->nkw);
  return BD_OK;
}

// 3-D bf16 map over [planes][rows][D] with a (64 x box_rows x 1) box, 128B swizzle;
// rows past `rows` read as zero.
int make_map(CUtensorMap* m, const void* ptr, int D, int rows, int planes, int box_rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BD_OK : BD_ERR_CUDA;
}

// K or V: the map above over [B*Hkv][S_kv][D], or, token-major
// ([S_kv][B*Hkv][D]), dims (D, B*Hkv, S_kv) with a (64 x 1 x box_rows) box --
// the same shared-memory tile, loaded at coordinates (d, plane, row) instead
// of (d, row, plane); rows past S_kv read as zero either way.
int make_map_kv(CUtensorMap* m, const void* ptr, const Geom& g, int box_rows) {
  if (!g.kv_tm) return make_map(m, ptr, g.D, g.S_kv, g.B * g.Hkv, box_rows);
  const cuuint64_t planes = static_cast<cuuint64_t>(g.B) * g.Hkv;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.D), planes, static_cast<cuuint64_t>(g.S_kv)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(g.D) * 2, planes * g.D * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BD_OK : BD_ERR_CUDA;
}

// 3-D fp32 map over [planes][rows][D] with a (64 x 64 x 1) box and no swizzle:
// the fp32 dq accumulator, target of the backward's bulk reduce-add.
int make_map_f32(CUtensorMap* m, const void* ptr, int D, int rows, int planes) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(rows) * D * 4};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBwdQ), 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BD_OK : BD_ERR_CUDA;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? BD_OK : BD_ERR_CUDA; }

// Rows of D elements of `dtype` as 16-byte vectors: log2 of the vectors per
// row, or -1 when a row is not a power-of-two number of vectors or an index
// of a [max_rows][B][C] or [B][C][L] array of them would pass 2^31.
int exchange_vshift(int B, int C, int L, int D, int dtype, int max_rows) {
  if (B < 1 || C < 1 || L < 1 || D < 1 || max_rows < 0) return -1;
  if (dtype != BD_DTYPE_F32 && dtype != BD_DTYPE_BF16) return -1;
  const long long bytes = static_cast<long long>(D) * (dtype == BD_DTYPE_F32 ? 4 : 2);
  if (bytes % 16) return -1;
  const long long vpr = bytes / 16;
  if (vpr & (vpr - 1)) return -1;
  int sh = 0;
  while ((1LL << sh) < vpr) ++sh;
  const long long bc = static_cast<long long>(B) * C;
  if (((bc * L) << sh) > 0x7fffffffLL || ((bc * max_rows) << sh) > 0x7fffffffLL) return -1;
  return sh;
}

}  // namespace

extern "C" {

size_t bd_attn_seg_bytes(const bd_geom* gi) {
  Geom g;
  if (to_geom(gi, &g) != BD_OK) return 0;
  return static_cast<size_t>(g.off[BD_SEG_OFF_TOTAL]) * 4;
}

int bd_attn_seg_layout(const bd_geom* gi, int32_t* offsets) {
  Geom g;
  if (!offsets || to_geom(gi, &g) != BD_OK) return BD_ERR_ARG;
  for (int i = 0; i < BD_SEG_NOFF; ++i) offsets[i] = g.off[i];
  offsets[BD_SEG_NOFF] = g.nqt;
  offsets[BD_SEG_NOFF + 1] = g.nkt;
  offsets[BD_SEG_NOFF + 2] = g.nkw;
  return BD_OK;
}

size_t bd_attn_bwd_workspace_bytes(const bd_geom* gi) {
  Geom g;
  if (to_geom(gi, &g) != BD_OK) return 0;
  return bwd_workspace_bytes(g);
}

int bd_attn_seg_build(const int32_t* doc_ids, const bd_geom* gi, void* seg, int32_t* status, bd_stream_t stream) {
  Geom g;
  if (int rc = to_geom(gi, &g)) return rc;
  if (!doc_ids || !seg || !status || !aligned16(seg)) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  return cuda_rc(
      launch_seg_build(doc_ids, g, static_cast<int32_t*>(seg), status, static_cast<cudaStream_t>(stream), 0));
}

int bd_attn_seg_build_chunk(const int32_t* doc_ids, const bd_geom* gi, void* seg, int32_t* status,
                            bd_stream_t stream) {
  Geom g;
  if (int rc = to_geom(gi, &g)) return rc;
  if (!doc_ids || !seg || !status || !aligned16(seg)) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  return cuda_rc(
      launch_seg_build(doc_ids, g, static_cast<int32_t*>(seg), status, static_cast<cudaStream_t>(stream), 1));
}

int bd_attn_merge(void* out, float* lse, const void* out_chunk, const float* lse_chunk, const bd_geom* gi,
                  int32_t* status, bd_stream_t stream) {
  Geom g;
  if (int rc = to_geom(gi, &g)) return rc;
  if (!out || !lse || !out_chunk || !lse_chunk || !status) return BD_ERR_ARG;
  if (!aligned16(out) || !aligned16(out_chunk)) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  return cuda_rc(launch_merge(g, out, lse, out_chunk, lse_chunk, status, static_cast<cudaStream_t>(stream)));
}

size_t bd_attn_plan_bytes(int B, int cp_size, int L) {
  int off[BD_PLAN_NOFF];
  const long long words = plan_layout(B, cp_size, L, off);
  return words < 0 ? 0 : static_cast<size_t>(words) * 4;
}

int bd_attn_plan_layout(int B, int cp_size, int L, int32_t* offsets) {
  int off[BD_PLAN_NOFF];
  if (!offsets || plan_layout(B, cp_size, L, off) < 0) return BD_ERR_ARG;
  for (int i = 0; i < BD_PLAN_NOFF; ++i) offsets[i] = off[i];
  return BD_OK;
}

int bd_attn_exchange_plan(const int32_t* doc_ids, int B, int S_full, int cp_size, int rank, void* plan,
                          int32_t* status, bd_stream_t stream) {
  if (!doc_ids || !plan || !status || !aligned16(plan)) return BD_ERR_ARG;
  if (B < 1 || cp_size < 1 || S_full < 1 || S_full % cp_size || rank < 0 || rank >= cp_size) return BD_ERR_ARG;
  if (B > 65535 || bd_attn_plan_bytes(B, cp_size, S_full / cp_size) == 0) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  return cuda_rc(launch_exchange_plan(doc_ids, B, S_full, cp_size, rank, static_cast<int32_t*>(plan), status,
                                      static_cast<cudaStream_t>(stream)));
}

int bd_attn_needed_gather(const void* x_local, const void* plan, int B, int C, int L, int D, int dtype, void* send,
                          int max_rows, int32_t* status, bd_stream_t stream) {
  if (!x_local || !plan || !send || !status) return BD_ERR_ARG;
  if (!aligned16(x_local) || !aligned16(plan) || !aligned16(send)) return BD_ERR_ARG;
  const int sh = exchange_vshift(B, C, L, D, dtype, max_rows);
  if (sh < 0) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  return cuda_rc(launch_needed_gather(x_local, static_cast<const int32_t*>(plan), B, C, L, sh, send, max_rows,
                                      status, static_cast<cudaStream_t>(stream)));
}

int bd_attn_needed_scatter_add(const void* grad_send, const void* plan, int B, int C, int L, int D, int dtype,
                               void* grad_local, int max_rows, int32_t* status, bd_stream_t stream) {
  if (!grad_send || !plan || !grad_local || !status) return BD_ERR_ARG;
  if (!aligned16(grad_send) || !aligned16(plan) || !aligned16(grad_local)) return BD_ERR_ARG;
  const int sh = exchange_vshift(B, C, L, D, dtype, max_rows);
  if (sh < 0) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  return cuda_rc(launch_needed_scatter_add(grad_send, static_cast<const int32_t*>(plan), B, C, L, sh,
                                           dtype == BD_DTYPE_BF16, grad_local, max_rows, status,
                                           static_cast<cudaStream_t>(stream)));
}

namespace {
int fwd_impl(const void* q, const void* k, const void* v, const void* seg, const bd_geom* gi, void* out, float* lse,
             int32_t* status, int merge, bd_stream_t stream) {
  Geom g;
  if (int rc = to_geom(gi, &g)) return rc;
  if (!q || !k || !v || !seg || !out || !lse || !status) return BD_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(seg)) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  if (!load_encode()) return BD_ERR_CUDA;
  CUtensorMap mq, mk, mv;
  if (make_map(&mq, q, g.D, g.L, g.B * g.Hq, kTile) || make_map_kv(&mk, k, g, kTile) ||
      make_map_kv(&mv, v, g, kTile))
    return BD_ERR_CUDA;
  if (g.D == 512)
    return cuda_rc(launch_fwd512(mq, mk, mv, static_cast<const int32_t*>(seg), g, out, lse, status, merge,
                                 static_cast<cudaStream_t>(stream)));
  return cuda_rc(launch_fwd(mq, mk, mv, static_cast<const int32_t*>(seg), g, out, lse, status, merge,
                            static_cast<cudaStream_t>(stream)));
}
}  // namespace

int bd_attn_fwd(const void* q, const void* k, const void* v, const void* seg, const bd_geom* gi, void* out,
                float* lse, int32_t* status, bd_stream_t stream) {
  return fwd_impl(q, k, v, seg, gi, out, lse, status, 0, stream);
}

int bd_attn_fwd_merge(const void* q, const void* k, const void* v, const void* seg, const bd_geom* gi, void* out,
                      float* lse, int32_t* status, bd_stream_t stream) {
  return fwd_impl(q, k, v, seg, gi, out, lse, status, 1, stream);
}

}  // extern "C"

namespace {
// The prep and main stages with the dq accumulator either in the workspace
// (dq_f32 == nullptr) or in the caller's fp32 dq buffer.
int bwd_prep_impl(const void* dout, const void* out, const bd_geom* gi, void* workspace, float* dq_f32,
                  int32_t* status, bd_stream_t stream) {
  Geom g;
  if (int rc = to_geom(gi, &g)) return rc;
  if (!dout || !out || !workspace || !status) return BD_ERR_ARG;
  if (!aligned16(dout) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return BD_ERR_ARG;
  if (dq_f32 && !aligned16(dq_f32)) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  return cuda_rc(launch_bwd_prep(g, dout, out, workspace, dq_f32, status, static_cast<cudaStream_t>(stream)));
}

int bwd_main_impl(const void* dout, const void* q, const void* k, const void* v, const float* lse, const void* seg,
                  const bd_geom* gi, int grad_dtype, void* dk, void* dv, void* workspace, float* dq_f32,
                  int32_t* status, bd_stream_t stream) {
  Geom g;
  if (int rc = to_geom(gi, &g)) return rc;
  if (!dout || !q || !k || !v || !lse || !seg || !dk || !dv || !workspace || !status) return BD_ERR_ARG;
  if (grad_dtype != BD_DTYPE_F32 && grad_dtype != BD_DTYPE_BF16) return BD_ERR_ARG;
  if (!aligned16(dout) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(seg) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return BD_ERR_ARG;
  if (dq_f32 && !aligned16(dq_f32)) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  if (!load_encode()) return BD_ERR_CUDA;
  CUtensorMap mq, mdo, mk, mv, mdq;
  const int qbox = bwd_q_box_rows(g.D);
  if (make_map(&mq, q, g.D, g.L, g.B * g.Hq, qbox) || make_map(&mdo, dout, g.D, g.L, g.B * g.Hq, qbox) ||
      make_map_kv(&mk, k, g, kTile) || make_map_kv(&mv, v, g, kTile) ||
      make_map_f32(&mdq, workspace, g.D, g.L, g.B * g.Hq))
    return BD_ERR_CUDA;
  return cuda_rc(launch_bwd_main(mq, mdo, mk, mv, mdq, static_cast<const int32_t*>(seg), g, lse, dk, dv,
                                 grad_dtype == BD_DTYPE_BF16, workspace, dq_f32, status,
                                 static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

int bd_attn_bwd_prep(const void* dout, const void* out, const bd_geom* gi, void* workspace, int32_t* status,
                     bd_stream_t stream) {
  return bwd_prep_impl(dout, out, gi, workspace, nullptr, status, stream);
}

int bd_attn_bwd_main(const void* dout, const void* q, const void* k, const void* v, const float* lse,
                     const void* seg, const bd_geom* gi, int grad_dtype, void* dk, void* dv, void* workspace,
                     int32_t* status, bd_stream_t stream) {
  return bwd_main_impl(dout, q, k, v, lse, seg, gi, grad_dtype, dk, dv, workspace, nullptr, status, stream);
}

int bd_attn_bwd_prep_dq(const void* dout, const void* out, const bd_geom* gi, void* workspace, float* dq,
                        int32_t* status, bd_stream_t stream) {
  if (!dq) return BD_ERR_ARG;
  return bwd_prep_impl(dout, out, gi, workspace, dq, status, stream);
}

int bd_attn_bwd_main_dq(const void* dout, const void* q, const void* k, const void* v, const float* lse,
                        const void* seg, const bd_geom* gi, int grad_dtype, float* dq, void* dk, void* dv,
                        void* workspace, int32_t* status, bd_stream_t stream) {
  if (!dq) return BD_ERR_ARG;
  return bwd_main_impl(dout, q, k, v, lse, seg, gi, grad_dtype, dk, dv, workspace, dq, status, stream);
}

int bd_attn_bwd_finalize(const bd_geom* gi, int grad_dtype, void* dq, void* workspace, int32_t* status,
                         bd_stream_t stream) {
  Geom g;
  if (int rc = to_geom(gi, &g)) return rc;
  if (!dq || !workspace || !status) return BD_ERR_ARG;
  if (grad_dtype != BD_DTYPE_F32 && grad_dtype != BD_DTYPE_BF16) return BD_ERR_ARG;
  if (!aligned16(dq) || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  return cuda_rc(launch_bwd_finalize(g, dq, grad_dtype == BD_DTYPE_BF16, workspace, status,
                                     static_cast<cudaStream_t>(stream)));
}

int bd_attn_bwd_deterministic(const void* dout, const void* q, const void* k, const void* v, const void* out,
                              const float* lse, const void* seg, const bd_geom* gi, int grad_dtype, void* dq,
                              void* dk, void* dv, void* workspace, int32_t* status, bd_stream_t stream) {
  Geom g;
  if (int rc = to_geom(gi, &g)) return rc;
  if (!dout || !q || !k || !v || !out || !lse || !seg || !dq || !dk || !dv || !workspace || !status)
    return BD_ERR_ARG;
  if (grad_dtype != BD_DTYPE_F32 && grad_dtype != BD_DTYPE_BF16) return BD_ERR_ARG;
  if (!aligned16(dout) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || !aligned16(seg) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  if (!load_encode()) return BD_ERR_CUDA;
  // the dq pass reads 128-row q / dout boxes; the dK / dV kernel's boxes follow its head dim
  CUtensorMap mq, mdo, mk, mv, mq_m, mdo_m;
  const int qbox = bwd_q_box_rows(g.D);
  if (make_map(&mq, q, g.D, g.L, g.B * g.Hq, kTile) || make_map(&mdo, dout, g.D, g.L, g.B * g.Hq, kTile) ||
      make_map(&mq_m, q, g.D, g.L, g.B * g.Hq, qbox) || make_map(&mdo_m, dout, g.D, g.L, g.B * g.Hq, qbox) ||
      make_map_kv(&mk, k, g, kTile) || make_map_kv(&mv, v, g, kTile))
    return BD_ERR_CUDA;
  const auto st = static_cast<cudaStream_t>(stream);
  const int32_t* sg = static_cast<const int32_t*>(seg);
  const int bf16 = grad_dtype == BD_DTYPE_BF16;
  if (int rc = cuda_rc(launch_bwd_delta(g, dout, out, workspace, status, st))) return rc;
  if (int rc = cuda_rc(launch_bwd_main_nodq(mq_m, mdo_m, mk, mv, sg, g, lse, dk, dv, bf16, workspace, status, st)))
    return rc;
  return cuda_rc(launch_bwd_dq(mq, mdo, mk, mv, sg, g, lse, bwd_delta_ptr(g, workspace), dq, bf16, status, st));
}

int bd_attn_bwd(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
                const void* seg, const bd_geom* gi, int grad_dtype, void* dq, void* dk, void* dv, void* workspace,
                int32_t* status, bd_stream_t stream) {
  Geom g;
  if (int rc = to_geom(gi, &g)) return rc;
  // check everything up front so that a bad argument enqueues nothing
  if (!dout || !q || !k || !v || !out || !lse || !seg || !dq || !dk || !dv || !workspace || !status)
    return BD_ERR_ARG;
  if (grad_dtype != BD_DTYPE_F32 && grad_dtype != BD_DTYPE_BF16) return BD_ERR_ARG;
  if (!aligned16(dout) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || !aligned16(seg) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return BD_ERR_ARG;
  if (grad_dtype == BD_DTYPE_F32) {
    // fp32 dq is its own accumulator: no finalize pass over it
    float* dqf = static_cast<float*>(dq);
    if (int rc = bwd_prep_impl(dout, out, gi, workspace, dqf, status, stream)) return rc;
    return bwd_main_impl(dout, q, k, v, lse, seg, gi, grad_dtype, dk, dv, workspace, dqf, status, stream);
  }
  if (int rc = bd_attn_bwd_prep(dout, out, gi, workspace, status, stream)) return rc;
  if (int rc = bd_attn_bwd_main(dout, q, k, v, lse, seg, gi, grad_dtype, dk, dv, workspace, status, stream))
    return rc;
  return bd_attn_bwd_finalize(gi, grad_dtype, dq, workspace, status, stream);
}

}  // extern "C"

// ------------------------------------------------- allocation-free backward
// The backward's scratch (fp32 dq accumulator + delta) for callers that cannot
// allocate device memory at call time: one array per GPU, shared by every
// bd_attn_bwd_noalloc call on that GPU and held until the process exits. The
// CUDA driver places it in device memory when it loads this file's code on a
// device: when the context is created under CUDA_MODULE_LOADING=EAGER, else
// (lazy loading, the default) at the first use of this file's code there,
// which is at the latest the set-up below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[BD_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Set-up, once per device with that device current: the device address of
// g_noalloc_scratch. Host code must never hand the symbol itself to a kernel;
// on the host it is only a stand-in. A failure here (typically the driver
// finding no room to load the array) is reported as BD_ERR_NOALLOC_SETUP.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // clear the (non-sticky) error so that later launches do not report it
      return BD_ERR_NOALLOC_SETUP;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return BD_OK;
}
}  // namespace

extern "C" {

int bd_attn_bwd_noalloc(const void* dout, const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* seg, const bd_geom* gi, int grad_dtype, void* dq, void* dk,
                        void* dv, int32_t* status, bd_stream_t stream) {
  // every pointer NULL: only the set-up of the current device, nothing enqueued
  if (!dout && !q && !k && !v && !out && !lse && !seg && !gi && !dq && !dk && !dv && !status) {
    if (int rc = check_device()) return rc;
    void* scratch = nullptr;
    return noalloc_scratch(&scratch);
  }
  Geom g;
  if (int rc = to_geom(gi, &g)) return rc;
  if (bwd_workspace_bytes(g) > BD_NOALLOC_SCRATCH_BYTES) return BD_ERR_SCRATCH_TOO_SMALL;
  if (int rc = check_device()) return rc;
  void* scratch = nullptr;
  if (int rc = noalloc_scratch(&scratch)) return rc;
  // same three stages as bd_attn_bwd; the prep stage zeroes the accumulator
  return bd_attn_bwd(dout, q, k, v, out, lse, seg, gi, grad_dtype, dq, dk, dv, scratch, status, stream);
}

const char* bd_attn_strerror(int code) {
  switch (code) {
    case BD_OK: return "ok";
    case BD_ERR_ARG: return "invalid argument (nothing enqueued)";
    case BD_ERR_CUDA: return "CUDA runtime or driver call failed";
    case BD_ERR_UNSUPPORTED: return "device is not a Blackwell sm_10x GPU";
    case BD_ERR_SCRATCH_TOO_SMALL:
      return "problem needs more backward scratch than bd_attn_bwd_noalloc's static 16 MiB (use bd_attn_bwd)";
    case BD_ERR_NOALLOC_SETUP:
      return "bd_attn_bwd_noalloc could not place its static 16 MiB scratch on this device (no free device memory "
             "when the library's code was loaded: do the set-up call before reserving memory, or run with "
             "CUDA_MODULE_LOADING=EAGER)";
    default: return "unknown bdattn error code";
  }
}

int bd_attn_selftest_wait_timeout(int32_t* status, uint64_t limit_ns, bd_stream_t stream) {
  if (!status || limit_ns > 2000000000ull) return BD_ERR_ARG;
  if (int rc = check_device()) return rc;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
  return cuda_rc(cudaGetLastError());
}

}  // extern "C"
