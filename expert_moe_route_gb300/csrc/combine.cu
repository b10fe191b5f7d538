// Combine: each token's R expert outputs come back to it and are averaged with
// the gate weights ("Enabling trillion-parameter models on AWS EFA", sections
// "Introduction" and "Dispatch and combine": accumulation at the receiving
// side).  y[t] = bf16( sum_r w[t,r] * o[slot_row[t*R+r]] ), fp32 in r order.
//
// One warp per token.  The warp stages the token's rows and weights in shared
// memory once, then each lane handles 16-byte vectors (8 bf16) of the hidden
// dimension: it issues the R row loads of a vector before accumulating them
// in order, so R independent 16-byte loads are in flight per lane.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int CW = 8;   // warps per block

// One warp per (token, column chunk of cv 16-byte vectors, a multiple of 32):
// with few tokens (small batches, e.g. decode) each row is cut into `chunks`
// pieces so that every SM gets several warps.
__global__ void __launch_bounds__(CW * 32) combine_kernel(const uint16_t* __restrict__ o,
                                                          const int32_t* __restrict__ slot_row,
                                                          const float* __restrict__ w, int T,
                                                          int d, int R, int N, int chunks, int cv,
                                                          const uint16_t* __restrict__ add,
                                                          uint16_t* __restrict__ y) {
  __shared__ int rows_s[CW][32];
  __shared__ float w_s[CW][32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nv = d / 8;
  const long long units = (long long)T * chunks;
  for (long long u = (long long)blockIdx.x * CW + wid; u < units; u += (long long)gridDim.x * CW) {
    const int t = (int)(u / chunks), c = (int)(u % chunks);
    const int vend = min(nv, (c + 1) * cv);
    if (lane < R) {
      const int row = slot_row[(size_t)t * R + lane];
      rows_s[wid][lane] = ((unsigned)row < (unsigned)N) ? row : -1;
      w_s[wid][lane] = w ? w[(size_t)t * R + lane] : 1.f;
    }
    __syncwarp();
    for (int v = c * cv + lane; v < vend; v += 32) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (add) unpack8(ldg_nc_v4(add + (size_t)t * d + (size_t)v * 8), acc);   // shared expert first
      for (int r0 = 0; r0 < R; r0 += 4) {
        uint4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int row = (r0 + u < R) ? rows_s[wid][r0 + u] : -1;
          q[u] = row >= 0 ? ldg_nc_v4(o + (size_t)row * d + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (r0 + u >= R) break;
          const float wr = w_s[wid][r0 + u];
          float f[8];
          unpack8(q[u], f);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = fmaf(wr, f[j], acc[j]);
        }
      }
      reinterpret_cast<uint4*>(y + (size_t)t * d)[v] = pack8(acc);
    }
    __syncwarp();
  }
}
// Failure-detection self-test: the barrier expects one arrival that never comes.
__global__ void selftest_wait_kernel(unsigned long long limit_ns, int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, err, limit_ns);
  __syncthreads();
}
}  // namespace

cudaError_t launch_selftest_wait(unsigned limit_us, int* err, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>((unsigned long long)limit_us * 1000ull, err);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* o, const int32_t* slot_row, const float* w, int T,
                           int d, int R, uint16_t* y, cudaStream_t s, const uint16_t* add) {
  if (T == 0) return cudaSuccess;
  // few tokens: cut each row into column chunks so that ~16 warps per SM work
  const int nv = d / 8;
  const long long want = 152LL * 16;
  int chunks = 1;
  if (T < want) {
    const long long c = (want + T - 1) / T;
    const int cmax = nv / 32 > 1 ? nv / 32 : 1;
    chunks = c < cmax ? (int)c : cmax;
  }
  const int cv = ceil_div(ceil_div(nv, chunks), 32) * 32;
  chunks = ceil_div(nv, cv);
  const long long units = (long long)T * chunks;
  const int blocks = (int)((units + CW - 1) / CW < 152 * 8 ? (units + CW - 1) / CW : 152 * 8);
  combine_kernel<<<blocks, CW * 32, 0, s>>>(o, slot_row, w, T, d, R, T * R, chunks, cv, add, y);
  count_launches(1);
  return cudaGetLastError();
}

namespace {
__global__ void one_expert_offsets_kernel(int32_t* offsets, int T) {
  offsets[0] = 0;
  offsets[1] = T;
}
}  // namespace

cudaError_t launch_one_expert_offsets(int32_t* offsets, int T, cudaStream_t s) {
  one_expert_offsets_kernel<<<1, 1, 0, s>>>(offsets, T);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
