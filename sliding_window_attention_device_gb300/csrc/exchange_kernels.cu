// K6: the K/V exchange plans of block-diagonal context parallelism and the
// sender's local halves of the needed-only exchange (blockdiag_cp.exchange:
// the global left-halo plan, the all-to-all-v split sizes with the local
// gather index, and `_NeededKVExchange`'s forward gather / backward
// index-add), built on the device from the replicated doc ids.
//
//  plan_rows_kernel    one CTA per (rank, batch row): the rank's real local
//                      rows, the layout checks and the chunk's last run start;
//  plan_finish_kernel  one CTA: the run start holding each rank's first
//                      position (from the earlier chunks' run starts), the
//                      union over batch rows, back_r, use_halo,
//                      the (src, dst) counts, this rank's splits, their
//                      prefix sums and send_index;
//  needed_gather / needed_scatter_add: HBM-bound grid-stride copies in 16-byte
//                      vectors over the token-major send buffer.
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace bd {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kCopyThreads = 256;

struct SumI { __device__ int operator()(int a, int b) const { return a + b; } };
struct MinI { __device__ int operator()(int a, int b) const { return a < b ? a : b; } };
struct MaxI { __device__ int operator()(int a, int b) const { return a > b ? a : b; } };

// Every thread gets the reduction of v over the CTA (blockDim a multiple of 32).
template <class Op>
__device__ int cta_allreduce(int v, Op op, int* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();  // s_red may still be read by a previous call
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  v = s_red[0];
  for (int w = 1; w < n_warps; ++w) v = op(v, s_red[w]);
  return v;
}

__global__ void __launch_bounds__(kPlanThreads) plan_rows_kernel(const int32_t* __restrict__ doc, int B, int S, int W,
                                                                int L, int32_t* __restrict__ plan, int32_t* status) {
  pdl_begin();
  const int r = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, nthr = blockDim.x;
  int off[BD_PLAN_NOFF];
  plan_layout(B, W, L, off);
  const int32_t* row = doc + static_cast<size_t>(b) * S;
  const int lo = r * L;
  // real rows, layout checks, and the last position of the chunk where a run
  // of equal ids starts (position 0, or an id unlike its left neighbour)
  int n_real = 0, bad = 0, last_real = -1, first_pad = L, last_start = -1;
  for (int i = tid; i < L; i += nthr) {
    const int q = lo + i;
    const int d = row[q];
    if (d < 0) bad = 1;
    if (d != 0) {
      ++n_real;
      last_real = i;  // i grows along this thread's loop
    } else if (first_pad == L) {
      first_pad = i;
    }
    if (q == 0 || row[q - 1] != d) last_start = q;
  }
  // the five reductions share one round through shared memory
  const int lane = tid & 31, warp = tid >> 5, n_warps = nthr >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    n_real += __shfl_xor_sync(0xffffffffu, n_real, o);
    last_real = max(last_real, __shfl_xor_sync(0xffffffffu, last_real, o));
    first_pad = min(first_pad, __shfl_xor_sync(0xffffffffu, first_pad, o));
    last_start = max(last_start, __shfl_xor_sync(0xffffffffu, last_start, o));
    bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  }
  __shared__ int s_part[5][32];
  if (lane == 0) {
    s_part[0][warp] = n_real;
    s_part[1][warp] = last_real;
    s_part[2][warp] = first_pad;
    s_part[3][warp] = last_start;
    s_part[4][warp] = bad;
  }
  __syncthreads();
  if (tid != 0) return;  // one thread finishes
  for (int x = 1; x < n_warps; ++x) {
    n_real += s_part[0][x];
    last_real = max(last_real, s_part[1][x]);
    first_pad = min(first_pad, s_part[2][x]);
    last_start = max(last_start, s_part[3][x]);
    bad |= s_part[4][x];
  }
  bad |= last_real > first_pad ? 1 : 0;  // a real id after padding
  int32_t* rr = plan + off[BD_PLAN_OFF_ROW_RANGE] + 2 * (static_cast<size_t>(b) * W + r);
  rr[0] = last_start;
  rr[1] = lo + n_real;  // real_end
  if (bad) atomicOr(status, BD_STATUS_LAYOUT);
}

__device__ __forceinline__ int piece(int src, int L, int lo_dst, int hi_dst) {
  const int a = max(src * L, lo_dst), e = min((src + 1) * L, hi_dst);
  return e > a ? e - a : 0;
}

__global__ void __launch_bounds__(kPlanThreads) plan_finish_kernel(const int32_t* __restrict__ doc, int B, int S,
                                                                  int W, int L, int rank,
                                                                  int32_t* __restrict__ plan) {
  pdl_begin();
  __shared__ int s_red[32];
  __shared__ int s_lo[kPlanMaxRanks], s_hi[kPlanMaxRanks], s_soff[kPlanMaxRanks];
  const int tid = threadIdx.x, nthr = blockDim.x;
  int off[BD_PLAN_NOFF];
  plan_layout(B, W, L, off);
  const int32_t* rr = plan + off[BD_PLAN_OFF_ROW_RANGE];
  int fits = 1, halo = 0;
  for (int r = tid; r < W; r += nthr) {
    int lo = r * L, hi = r * L;
    bool any = false;
    for (int b = 0; b < B; ++b) {
      const int e = rr[2 * (b * W + r) + 1];
      if (e > r * L) {  // this batch row has real local rows
        // the run holding r L starts there when the id changes at r L, else at
        // the last run start of an earlier chunk (chunk 0 starts one at 0)
        const int32_t* row = doc + static_cast<size_t>(b) * S;
        int s = r * L;
        if (r > 0 && row[r * L - 1] == row[r * L]) {
          s = 0;  // the largest run start of the chunks before r (loads only: they overlap)
          for (int c = 0; c < r; ++c) s = max(s, rr[2 * (b * W + c)]);
        }
        lo = any ? min(lo, s) : s;
        hi = any ? max(hi, e) : e;
        any = true;
      }
    }
    s_lo[r] = lo;
    s_hi[r] = hi;
    plan[off[BD_PLAN_OFF_S_FIRST] + r] = lo;
    plan[off[BD_PLAN_OFF_REAL_END] + r] = hi;
    plan[off[BD_PLAN_OFF_BACK] + r] = r * L - lo;
    fits &= (r * L - lo <= L) ? 1 : 0;
    halo = max(halo, r * L - lo);
  }
  fits = cta_allreduce(fits, MinI(), s_red);  // also orders the s_lo / s_hi writes before the reads below
  halo = cta_allreduce(halo, MaxI(), s_red);
  for (int r = tid; r < W; r += nthr) plan[off[BD_PLAN_OFF_HALO_SEND] + r] = r + 1 < W ? (r + 1) * L - s_lo[r + 1] : 0;
  for (int x = tid; x < W * W; x += nthr) {
    const int src = x / W, dst = x - src * W;
    plan[off[BD_PLAN_OFF_COUNTS] + x] = piece(src, L, s_lo[dst], s_hi[dst]);
  }
  if (tid == 0) {
    int so = 0, ro = 0;
    for (int d = 0; d < W; ++d) {
      const int n_in = piece(rank, L, s_lo[d], s_hi[d]), n_out = piece(d, L, s_lo[rank], s_hi[rank]);
      plan[off[BD_PLAN_OFF_IN_SPLITS] + d] = n_in;
      plan[off[BD_PLAN_OFF_OUT_SPLITS] + d] = n_out;
      plan[off[BD_PLAN_OFF_SEND_OFF] + d] = so;
      plan[off[BD_PLAN_OFF_RECV_OFF] + d] = ro;
      s_soff[d] = so;
      so += n_in;
      ro += n_out;
    }
    int32_t* h = plan + off[BD_PLAN_OFF_HDR];
    for (int x = 0; x < BD_PLAN_HDR_WORDS; ++x) h[x] = 0;
    h[BD_PLAN_CP_SIZE] = W;
    h[BD_PLAN_L] = L;
    h[BD_PLAN_RANK] = rank;
    h[BD_PLAN_B] = B;
    h[BD_PLAN_USE_HALO] = fits;
    h[BD_PLAN_HALO_SIZE] = halo;
    h[BD_PLAN_TOTAL_SEND] = so;
    h[BD_PLAN_TOTAL_RECV] = ro;
    h[BD_PLAN_MAGIC] = kPlanMagic;
  }
  __syncthreads();
  int32_t* idx = plan + off[BD_PLAN_OFF_SEND_INDEX];
  for (int d = 0; d < W; ++d) {
    const int a = max(rank * L, s_lo[d]) - rank * L, n = piece(rank, L, s_lo[d], s_hi[d]), o = s_soff[d];
    for (int k = tid; k < n; k += nthr) idx[o + k] = a + k;
  }
}

// The plan header matches (B, L) and the send count fits max_rows; else BOUNDS.
__device__ bool plan_usable(const int32_t* plan, int B, int L, int max_rows, int32_t* status) {
  const int W = plan[BD_PLAN_CP_SIZE], n = plan[BD_PLAN_TOTAL_SEND];
  const bool ok = plan[BD_PLAN_MAGIC] == kPlanMagic && plan[BD_PLAN_B] == B && plan[BD_PLAN_L] == L && W >= 1 &&
                  W <= kPlanMaxRanks && n >= 0 && n <= max_rows && n <= static_cast<long long>(W) * L;
  if (!ok && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, BD_STATUS_BOUNDS);
  return ok;
}

// send[j][bc][v] = x[bc][send_index[j]][v], 16-byte vectors, vpr = 1 << vshift per row.
__global__ void __launch_bounds__(kCopyThreads) needed_gather_kernel(const uint4* __restrict__ x,
                                                                    const int32_t* __restrict__ plan, int B, int BC,
                                                                    int L, int vshift, uint4* __restrict__ send,
                                                                    int max_rows, int32_t* status) {
  pdl_begin();
  if (*reinterpret_cast<const volatile int32_t*>(status) != 0) return;
  if (!plan_usable(plan, B, L, max_rows, status)) return;
  const int W = plan[BD_PLAN_CP_SIZE], n = plan[BD_PLAN_TOTAL_SEND];
  int off[BD_PLAN_NOFF];
  plan_layout(B, W, L, off);
  const int32_t* idx = plan + off[BD_PLAN_OFF_SEND_INDEX];
  const int total = (n * BC) << vshift;  // the host bounds max_rows * BC * vpr below 2^31
  const int vmask = (1 << vshift) - 1, stride = gridDim.x * blockDim.x;
  // four independent elements per thread and pass: their index loads, then
  // their row loads, are in flight together
  int e = blockIdx.x * blockDim.x + threadIdx.x;
  for (; e + 3 * stride < total; e += 4 * stride) {
    int src[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int row = (e + u * stride) >> vshift;
      const int j = row / BC, bc = row - j * BC;
      const int t = __ldg(idx + j);
      src[u] = static_cast<unsigned>(t) < static_cast<unsigned>(L) ? (((bc * L + t) << vshift) + ((e + u * stride) & vmask)) : -1;
    }
    uint4 val[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) val[u] = src[u] >= 0 ? __ldg(x + src[u]) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (src[u] >= 0)
        send[e + u * stride] = val[u];
      else
        atomicOr(status, BD_STATUS_BOUNDS);
    }
  }
  for (; e < total; e += stride) {
    const int row = e >> vshift, v = e & vmask;
    const int j = row / BC, bc = row - j * BC;
    const int t = __ldg(idx + j);
    if (static_cast<unsigned>(t) >= static_cast<unsigned>(L)) {
      atomicOr(status, BD_STATUS_BOUNDS);
      continue;
    }
    // a source row may go to several destinations: keep it cacheable
    send[e] = __ldg(x + ((bc * L + t) << vshift) + v);
  }
}

__device__ __forceinline__ void acc_vec(float (&a)[8], uint4 g, bool bf16) {
  if (bf16) {
    const uint32_t w[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
      a[2 * k] += __low2float(h);
      a[2 * k + 1] += __high2float(h);
    }
  } else {
    a[0] += __uint_as_float(g.x);
    a[1] += __uint_as_float(g.y);
    a[2] += __uint_as_float(g.z);
    a[3] += __uint_as_float(g.w);
  }
}

// grad_local[bc][t][v] = sum over destinations d (in order) whose piece holds
// token t of grad_send[send_off[d] + (rank L + t - a_d)][bc][v]; 0 if none.
template <bool kBf16>
__global__ void __launch_bounds__(kCopyThreads) needed_scatter_add_kernel(const uint4* __restrict__ gsend,
                                                                         const int32_t* __restrict__ plan, int B,
                                                                         int BC, int L, int vshift,
                                                                         uint4* __restrict__ glocal, int max_rows,
                                                                         int32_t* status) {
  pdl_begin();
  __shared__ int s_a[kPlanMaxRanks], s_e[kPlanMaxRanks], s_o[kPlanMaxRanks];
  if (*reinterpret_cast<const volatile int32_t*>(status) != 0) return;
  if (!plan_usable(plan, B, L, max_rows, status)) return;
  const int W = plan[BD_PLAN_CP_SIZE], rank = plan[BD_PLAN_RANK];
  int off[BD_PLAN_NOFF];
  plan_layout(B, W, L, off);
  // each destination's piece as a local token range [a, e) and its first send row
  for (int d = threadIdx.x; d < W; d += blockDim.x) {
    const int lo = plan[off[BD_PLAN_OFF_S_FIRST] + d], hi = plan[off[BD_PLAN_OFF_REAL_END] + d];
    s_a[d] = max(rank * L, lo) - rank * L;
    s_e[d] = min((rank + 1) * L, hi) - rank * L;
    s_o[d] = plan[off[BD_PLAN_OFF_SEND_OFF] + d];
  }
  __syncthreads();
  const int total = (BC * L) << vshift;
  const int vmask = (1 << vshift) - 1, stride = gridDim.x * blockDim.x;
  // element order [t][bc][v]: a warp shares t, so the destination tests are
  // uniform; four independent elements per thread and pass
  int e = blockIdx.x * blockDim.x + threadIdx.x;
  for (; e < total; e += 4 * stride) {
    int t[4], bc[4];
    float a[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int row = (e + u * stride) >> vshift;
      t[u] = e + u * stride < total ? row / BC : -1;
      bc[u] = row - t[u] * BC;
#pragma unroll
      for (int k = 0; k < 8; ++k) a[u][k] = 0.f;
    }
    for (int d = 0; d < W; ++d) {
      const int lo = s_a[d], hi = s_e[d], o = s_o[d];
      uint4 g[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool in = t[u] >= lo && t[u] < hi;
        g[u] = in ? __ldcs(gsend + (((o + t[u] - lo) * BC + bc[u]) << vshift) + ((e + u * stride) & vmask))
                  : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (t[u] >= lo && t[u] < hi) acc_vec(a[u], g[u], kBf16);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (t[u] < 0) continue;
      uint4 o;
      if (kBf16) {
        o.x = pack_bf16x2(a[u][0], a[u][1]);
        o.y = pack_bf16x2(a[u][2], a[u][3]);
        o.z = pack_bf16x2(a[u][4], a[u][5]);
        o.w = pack_bf16x2(a[u][6], a[u][7]);
      } else {
        o = make_uint4(__float_as_uint(a[u][0]), __float_as_uint(a[u][1]), __float_as_uint(a[u][2]),
                       __float_as_uint(a[u][3]));
      }
      glocal[((bc[u] * L + t[u]) << vshift) + ((e + u * stride) & vmask)] = o;
    }
  }
}

// One full wave: resident CTAs per SM (from the occupancy query, made once per
// kernel) times the SM count, or fewer when the work is smaller.
template <auto kKernel>
unsigned copy_grid(long long elems) {
  static int per_sm = 0, sms = 0;
  if (per_sm == 0) {
    int dev = 0, n = 0, b = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) ==
                                                  cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kKernel, kCopyThreads, 0) == cudaSuccess && n > 0 && b > 0) {
      sms = n;
      per_sm = b;
    } else {
      sms = 152;
      per_sm = 4;
    }
  }
  const long long want = (elems + kCopyThreads - 1) / kCopyThreads;
  const long long wave = static_cast<long long>(sms) * per_sm;
  return static_cast<unsigned>(want < 1 ? 1 : (want < wave ? want : wave));
}

}  // namespace

cudaError_t launch_exchange_plan(const int32_t* doc, int B, int S, int W, int rank, int32_t* plan, int32_t* status,
                                 cudaStream_t st) {
  const int L = S / W;
  if (const cudaError_t le = launch_pdl(plan_rows_kernel, dim3(dim3(W, B)), dim3(kPlanThreads), 0, st, doc, B, S, W,
      L, plan, status); le != cudaSuccess) return le;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (const cudaError_t le = launch_pdl(plan_finish_kernel, dim3(1), dim3(kPlanThreads), 0, st, doc, B, S, W, L,
      rank, plan); le != cudaSuccess) return le;
  return cudaGetLastError();
}

cudaError_t launch_needed_gather(const void* x, const int32_t* plan, int B, int C, int L, int vshift, void* send,
                                 int max_rows, int32_t* status, cudaStream_t st) {
  const long long elems = (static_cast<long long>(max_rows) * B * C) << vshift;
  if (const cudaError_t le = launch_pdl(needed_gather_kernel, dim3(copy_grid<needed_gather_kernel>(elems)),
      dim3(kCopyThreads), 0, st, static_cast<const uint4*>(x), plan, B, B * C, L, vshift, static_cast<uint4*>(send),
      max_rows, status); le != cudaSuccess) return le;
  return cudaGetLastError();
}

cudaError_t launch_needed_scatter_add(const void* gsend, const int32_t* plan, int B, int C, int L, int vshift,
                                      int bf16, void* glocal, int max_rows, int32_t* status, cudaStream_t st) {
  const long long elems = (static_cast<long long>(B) * C * L) << vshift;
  const auto* g = static_cast<const uint4*>(gsend);
  auto* o = static_cast<uint4*>(glocal);
  const cudaError_t e =
      bf16 ? launch_pdl(needed_scatter_add_kernel<true>, dim3(copy_grid<needed_scatter_add_kernel<true>>(elems)),
                        dim3(kCopyThreads), 0, st, g, plan, B, B * C, L, vshift, o, max_rows, status)
           : launch_pdl(needed_scatter_add_kernel<false>, dim3(copy_grid<needed_scatter_add_kernel<false>>(elems)),
                        dim3(kCopyThreads), 0, st, g, plan, B, B * C, L, vshift, o, max_rows, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace bd
