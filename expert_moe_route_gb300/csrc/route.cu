// Router: gate projection logits = x W_g + bias (fp32 accumulation) and the
// per-token softmax top-R choice with the lowest-index tie-break.
// ("Enabling trillion-parameter models on AWS EFA", section "Introduction":
// a small linear routing layer picks the experts each token is sent to.)
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------- gate logits
// logits[T,E] = x[T,d] (bf16) * W_g[d,E] (fp32) + bias[E], fp32 FMA accumulation
// in ascending k.  64x64 output tile per 256-thread block, 4x4 per thread.
namespace {
constexpr int GL_BM = 64, GL_BN = 64, GL_BK = 32;

__global__ void __launch_bounds__(256) gate_logits_kernel(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ wg,
                                                          const float* __restrict__ bias, int T,
                                                          int d, int E,
                                                          float* __restrict__ logits) {
  __shared__ float xs[GL_BK][GL_BM + 4];
  __shared__ float ws[GL_BK][GL_BN + 4];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.y * GL_BM;
  const int e0 = blockIdx.x * GL_BN;
  const int ty = tid / 16, tx = tid % 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += GL_BK) {
    {  // x tile: 64 tokens x 32 k, one 16-byte vector per thread
      const int tok = tid / 4, kc = (tid % 4) * 8;
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (t0 + tok < T && k0 + kc < d) {
        uint4 q = ldg_nc_v4(x + (size_t)(t0 + tok) * d + k0 + kc);
        unpack8(q, v);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) xs[kc + j][tok] = v[j];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // W_g tile: 32 k x 64 experts, coalesced along e
      const int kk = tid / 64 + 4 * i, ee = tid % 64;
      ws[kk][ee] = (k0 + kk < d && e0 + ee < E) ? wg[(size_t)(k0 + kk) * E + e0 + ee] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < GL_BK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[k][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[k][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) logits[(size_t)t * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
    }
  }
}

// ---------------------------------------------------------------- top-R
// One warp per token.  Lane l holds the logits of experts l, l+32, ...; R rounds
// of a warp arg-max under the order (value desc, index asc) pick the experts in
// selection order.  Lane r keeps the r-th choice; the gate weights are the
// softmax of the chosen logits.
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int T, int E,
                                                   int R, int32_t* __restrict__ idx,
                                                   float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x / 32;
  for (int t = blockIdx.x * warps + threadIdx.x / 32; t < T; t += gridDim.x * warps) {
    float v[EPL];
    uint32_t taken = 0;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane + 32 * j;
      if (e < E) {
        v[j] = logits[(size_t)t * E + e];
      } else {
        v[j] = -FLT_MAX;
        taken |= 1u << j;
      }
    }
    float my_v = 0.f;
    int my_i = 0;
    for (int r = 0; r < R; ++r) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        if (!(taken & (1u << j)) && beats(v[j], e, bv, bi)) {
          bv = v[j];
          bi = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, off);
        const int oi = __shfl_xor_sync(kFull, bi, off);
        if (beats(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (bi != 0x7fffffff && (bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == r) {
        my_v = bv;
        my_i = bi;
      }
    }
    const float m = __shfl_sync(kFull, my_v, 0);
    const float ex = lane < R ? expf(my_v - m) : 0.f;
    float s = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
    if (lane < R) {
      idx[(size_t)t * R + lane] = my_i;
      w[(size_t)t * R + lane] = ex / s;
    }
  }
}
// W_g [d, E] fp32 -> W_gs [E, 3d] bf16 with W_gs[e, k] = hi, [e, d+k] = mid,
// [e, 2d+k] = lo: hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid).
// Both differences are exact in fp32 (Sterbenz), so hi + mid + lo carries
// w's 24-bit significand to within 2^-24 |w|, and x (bf16) times each term is
// exact in fp32: logits = x hi + x mid + x lo is a bf16 GEMM with K = 3d.
__global__ void wg_split_kernel(const float* __restrict__ wg, int d, int E,
                                uint16_t* __restrict__ wgs) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int k = k0 + i, e = e0 + threadIdx.x;
    tile[i][threadIdx.x] = (k < d && e < E) ? wg[(size_t)k * E + e] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int e = e0 + i, k = k0 + threadIdx.x;
    if (k >= d || e >= E) continue;
    const float w = tile[threadIdx.x][i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    uint16_t* row = wgs + (size_t)e * 3 * d;
    row[k] = *reinterpret_cast<const uint16_t*>(&hi);
    row[d + k] = *reinterpret_cast<const uint16_t*>(&mid);
    row[2 * d + k] = *reinterpret_cast<const uint16_t*>(&lo);
  }
}
}  // namespace

cudaError_t launch_wg_split(const float* wg, int d, int E, uint16_t* wgs, cudaStream_t s) {
  dim3 grid(ceil_div(d, 32), ceil_div(E, 32));
  wg_split_kernel<<<grid, dim3(32, 8), 0, s>>>(wg, d, E, wgs);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_gate_logits(const uint16_t* x, const float* wg, const float* bias, int T, int d,
                               int E, float* logits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dim3 grid(ceil_div(E, GL_BN), ceil_div(T, GL_BM));
  gate_logits_kernel<<<grid, 256, 0, s>>>(x, wg, bias, T, d, E, logits);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int T, int E, int R, int32_t* idx, float* w,
                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = ceil_div(T, 8) < 152 * 16 ? ceil_div(T, 8) : 152 * 16;
  const int epl = ceil_div(E, 32);
#define MOE_TOPK(N) topk_kernel<N><<<blocks, 256, 0, s>>>(logits, T, E, R, idx, w)
  if (epl <= 1) MOE_TOPK(1);
  else if (epl <= 2) MOE_TOPK(2);
  else if (epl <= 4) MOE_TOPK(4);
  else if (epl <= 8) MOE_TOPK(8);
  else if (epl <= 16) MOE_TOPK(16);
  else MOE_TOPK(32);
#undef MOE_TOPK
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
