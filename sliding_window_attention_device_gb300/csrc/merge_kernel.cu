// K5: log-sum-exp merge of one K/V chunk's forward result into a running
// result (gemma4_moe.cp_local_ring: per-chunk forward returning (out, lse)
// and the -inf-safe online softmax merge of chunk results):
//   lse = log(exp(lse_a) + exp(lse_b))
//   out = exp(lse_a - lse) out_a + exp(lse_b - lse) out_b
// A row whose two sides are both empty (lse = -inf) stays out = 0,
// lse = -inf; an empty side has weight 0 whatever its out holds.
//
// Memory bound: each thread blends 8 bf16 values (16 bytes) of one row, two
// such pieces for D = 512; the rows of a warp are whole (a row is at most one
// warp wide), and the loop bounds are the same for every lane, so a
// __syncwarp separates the reads of a row's lse from its single rewrite.
#include <cuda_bf16.h>
#include <cstdint>

#include "sm100_ptx.cuh"
#include "common.cuh"

namespace bd {

namespace {

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(__nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                    const __nv_bfloat16* __restrict__ out_c,
                                                    const float* __restrict__ lse_c, long long rows,
                                                    const int32_t* status) {
  pdl_begin();
  constexpr int kPerRow = D / 8 < 32 ? D / 8 : 32;  // lanes per row
  constexpr int kVec = D / 8 / kPerRow;             // 16-byte pieces per lane
  constexpr int kRowsPerWarp = 32 / kPerRow;
  static_assert(32 % kPerRow == 0 && kVec * kPerRow * 8 == D, "a warp holds whole rows");
  if (*reinterpret_cast<const volatile int32_t*>(status) != 0) return;
  const int lane = threadIdx.x & 31, part = lane % kPerRow;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r0 = warp0 * kRowsPerWarp; r0 < rows; r0 += n_warps * kRowsPerWarp) {
    const long long row = r0 + lane / kPerRow;
    const bool live = row < rows;
    float la = -INFINITY, lb = -INFINITY;
    uint4 a[kVec], b[kVec];
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
      a[u] = make_uint4(0, 0, 0, 0);
      b[u] = make_uint4(0, 0, 0, 0);
    }
    if (live) {
      la = lse[row];
      lb = lse_c[row];
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        a[u] = *reinterpret_cast<const uint4*>(out + row * D + (part + u * kPerRow) * 8);
        b[u] = *reinterpret_cast<const uint4*>(out_c + row * D + (part + u * kPerRow) * 8);
      }
    }
    __syncwarp();  // every lane has read its row's lse before it is rewritten
    const float m = fmaxf(la, lb);
    float wa = 0.f, wb = 0.f, l = -INFINITY;
    if (m != -INFINITY) {
      const float ea = expf(la - m), eb = expf(lb - m);  // an empty side gives exp(-inf) = 0
      const float tot = ea + eb;
      wa = ea / tot;
      wb = eb / tot;
      l = m + logf(tot);
    }
    if (live) {
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        const uint32_t av[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, bv[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
        uint32_t ov[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&av[e]);
          const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(&bv[e]);
          // an empty side contributes nothing even if its values are not finite
          const float lo = (wa > 0.f ? wa * __low2float(x) : 0.f) + (wb > 0.f ? wb * __low2float(y) : 0.f);
          const float hi = (wa > 0.f ? wa * __high2float(x) : 0.f) + (wb > 0.f ? wb * __high2float(y) : 0.f);
          ov[e] = pack_bf16x2(lo, hi);
        }
        *reinterpret_cast<uint4*>(out + row * D + (part + u * kPerRow) * 8) = make_uint4(ov[0], ov[1], ov[2], ov[3]);
      }
      if (part == 0) lse[row] = l;
    }
  }
}

}  // namespace

cudaError_t launch_merge(const Geom& g, void* out, float* lse, const void* out_c, const float* lse_c,
                         const int32_t* status, cudaStream_t st) {
  const long long rows = static_cast<long long>(g.B) * g.Hq * g.L;
  const long long threads = rows * (g.D / 8 < 32 ? g.D / 8 : 32);
  const long long want = (threads + 255) / 256;
  const unsigned grid = static_cast<unsigned>(want < 152 * 16 ? (want > 0 ? want : 1) : 152 * 16);
  auto* o = static_cast<__nv_bfloat16*>(out);
  auto* oc = static_cast<const __nv_bfloat16*>(out_c);
  switch (g.D) {
    case 64: if (const cudaError_t le = launch_pdl(merge_kernel<64>, dim3(grid), dim3(256), 0, st, o, lse, oc, lse_c,
        rows, status); le != cudaSuccess) return le; break;
    case 128: if (const cudaError_t le = launch_pdl(merge_kernel<128>, dim3(grid), dim3(256), 0, st, o, lse, oc,
        lse_c, rows, status); le != cudaSuccess) return le; break;
    case 256: if (const cudaError_t le = launch_pdl(merge_kernel<256>, dim3(grid), dim3(256), 0, st, o, lse, oc,
        lse_c, rows, status); le != cudaSuccess) return le; break;
    case 512: if (const cudaError_t le = launch_pdl(merge_kernel<512>, dim3(grid), dim3(256), 0, st, o, lse, oc,
        lse_c, rows, status); le != cudaSuccess) return le; break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace bd
