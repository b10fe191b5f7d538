// Backward of the routing, dispatch and combine steps (the expert GEMMs'
// backward is in grouped_gemm.cu).  With y_t = sum_r w_r o_{row(t,r)} and the
// gate weights the softmax over the chosen logits:
//   dw_r = <dy_t, o_row>,  do_row = bf16(w_r dy_t)
//   dlogits at the chosen experts: w_q (dw_q - sum_r w_r dw_r); zero elsewhere
//   dW_g = x^T dlogits  (one dense contraction over the tokens, on the tensor cores)
//   dx_t = bf16( sum_r dx_perm[row(t,r)] + sum_r dlogits_{t,r} W_g[:, idx[t,r]] )
// All reductions run in a fixed order, so results are bitwise reproducible.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int BW = 8;  // warps per block

// One warp per token.  Lane l accumulates partial dot products for all R
// choices over its vectors, then the warp reduces them.
__global__ void __launch_bounds__(BW * 32) bwd_route_kernel(
    const uint16_t* __restrict__ dy, const uint16_t* __restrict__ o,
    const int32_t* __restrict__ slot_row, const float* __restrict__ w, int T, int d, int R, int N,
    uint16_t* __restrict__ dO, float* __restrict__ dsel_tok) {
  __shared__ int rows_s[BW][32];
  __shared__ float w_s[BW][32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nv = d / 8;
  for (int t = blockIdx.x * BW + wid; t < T; t += gridDim.x * BW) {
    if (lane < R) {
      const int row = slot_row[(size_t)t * R + lane];
      rows_s[wid][lane] = ((unsigned)row < (unsigned)N) ? row : -1;
      w_s[wid][lane] = w[(size_t)t * R + lane];
    }
    __syncwarp();
    float acc[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) acc[r] = 0.f;
    for (int v = lane; v < nv; v += 32) {
      float g[8];
      unpack8(ldg_nc_v4(dy + (size_t)t * d + (size_t)v * 8), g);
#pragma unroll
      for (int r0 = 0; r0 < 32; r0 += 4) {
        if (r0 >= R) break;
        uint4 q[4];   // four rows' loads in flight before any is used
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int row = (r0 + u < R) ? rows_s[wid][r0 + u] : -1;
          q[u] = row >= 0 ? ldg_nc_v4(o + (size_t)row * d + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = r0 + u;
          if (r >= R) break;
          const int row = rows_s[wid][r];
          if (row < 0) continue;
          float ov[8], dv[8];
          unpack8(q[u], ov);
          const float wr = w_s[wid][r];
          float s = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            s = fmaf(g[j], ov[j], s);
            dv[j] = wr * g[j];
          }
          acc[r] += s;
          reinterpret_cast<uint4*>(dO + (size_t)row * d)[v] = pack8(dv);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      if (r >= R) break;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(kFull, acc[r], off);
    }
    // every lane now holds all dw_r; lane r finishes choice r
    float wdw = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      if (r >= R) break;
      wdw = fmaf(w_s[wid][r], acc[r], wdw);
    }
    float mine = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r)
      if (r == lane) mine = acc[r];
    if (lane < R) {
      const float ds = w_s[wid][lane] * (mine - wdw);
      dsel_tok[(size_t)t * R + lane] = ds;
    }
    __syncwarp();
  }
}

// Router weight gradient on the tensor cores.  dW_g = x^T dlogits is one dense
// contraction over the T tokens (dlogits [T, E] is zero off each token's chosen
// experts).  dlogits is split into two bf16 terms, hi = bf16(v) and
// lo = bf16(v - hi) (v - hi is exact in fp32, so hi + lo carries 16 significant
// bits of v), laid out side by side as S = [hi | lo] [T, 2 Ep], Ep = E rounded up
// to 32.  One bf16 GEMM with fp32 accumulation, x^T S over chunks of the tokens,
// gives both products for every chunk (P[s] [d, 2 Ep]); a last pass adds each
// chunk's hi and lo columns, chunks in order.
//
// Operand pass: warp per token writes the token's row of S (zeros, then, after
// the warp's zero stores, its R hi and lo values); block 0 also writes the chunk
// offsets {0, c, 2c, ..., T}.
__global__ void __launch_bounds__(BW * 32) dwg_operand_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ dsel, int T, int E, int R, int Ep,
    int chunk, int S, uint16_t* __restrict__ Sm, int32_t* __restrict__ offs) {
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i <= S; i += blockDim.x) offs[i] = i < S ? min(i * chunk, T) : T;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nv = Ep / 4;   // 16-byte groups in a row of 2 Ep bf16
  for (int t = blockIdx.x * BW + wid; t < T; t += gridDim.x * BW) {
    uint4* row = reinterpret_cast<uint4*>(Sm + (size_t)t * 2 * Ep);
    for (int v = lane; v < nv; v += 32) row[v] = make_uint4(0, 0, 0, 0);
    __syncwarp();
    if (lane < R) {
      const int e = idx[(size_t)t * R + lane];
      if ((unsigned)e < (unsigned)E) {
        const float v = dsel[(size_t)t * R + lane];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
        Sm[(size_t)t * 2 * Ep + e] = __bfloat16_as_ushort(hi);
        Sm[(size_t)t * 2 * Ep + Ep + e] = __bfloat16_as_ushort(lo);
      }
    }
    __syncwarp();
  }
}

// dW_g[k, e] = sum over chunks s (ascending) of (P[s][k][e] + P[s][k][Ep + e]).
__global__ void dwg_sum_kernel(const float* __restrict__ P, int S, int d, int E, int Ep,
                               float* __restrict__ dW_gate) {
  const long long n = (long long)d * E;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int k = (int)(i / E), e = (int)(i % E);
    const float* p = P + (size_t)k * 2 * Ep + e;
    const size_t step = (size_t)d * 2 * Ep;
    float v = 0.f;
    for (int s = 0; s < S; ++s) v += p[s * step] + p[s * step + Ep];
    dW_gate[i] = v;
  }
}

__global__ void wg_transpose_kernel(const float* __restrict__ wg, int d, int E,
                                    float* __restrict__ wgT) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int k = k0 + i, e = e0 + threadIdx.x;
    tile[i][threadIdx.x] = (k < d && e < E) ? wg[(size_t)k * E + e] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int e = e0 + i, k = k0 + threadIdx.x;
    if (k < d && e < E) wgT[(size_t)e * d + k] = tile[threadIdx.x][i];
  }
}

// dx[t] = bf16( sum_r dx_perm[row_r] + sum_r dsel[t,r] * W_g^T[idx[t,r]] ), fp32 in r order.
__global__ void __launch_bounds__(BW * 32) dx_combine_kernel(
    const uint16_t* __restrict__ dx_perm, const int32_t* __restrict__ slot_row,
    const int32_t* __restrict__ idx, const float* __restrict__ dsel, const float* __restrict__ wgT,
    int T, int d, int E, int R, int N, const uint16_t* __restrict__ add,
    uint16_t* __restrict__ dx) {
  __shared__ int rows_s[BW][32];
  __shared__ int exp_s[BW][32];
  __shared__ float ds_s[BW][32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nv = d / 8;
  for (int t = blockIdx.x * BW + wid; t < T; t += gridDim.x * BW) {
    if (lane < R) {
      const int row = slot_row[(size_t)t * R + lane];
      rows_s[wid][lane] = ((unsigned)row < (unsigned)N) ? row : -1;
      const int e = idx[(size_t)t * R + lane];
      exp_s[wid][lane] = ((unsigned)e < (unsigned)E) ? e : -1;
      ds_s[wid][lane] = dsel[(size_t)t * R + lane];
    }
    __syncwarp();
    for (int v = lane; v < nv; v += 32) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int r0 = 0; r0 < R; r0 += 4) {       // sum of the token's dx_perm rows, r order
        uint4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int row = (r0 + u < R) ? rows_s[wid][r0 + u] : -1;
          q[u] = row >= 0 ? ldg_nc_v4(dx_perm + (size_t)row * d + (size_t)v * 8)
                          : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (r0 + u >= R) break;
          if (rows_s[wid][r0 + u] < 0) continue;
          float f[8];
          unpack8(q[u], f);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] += f[j];
        }
      }
      for (int r0 = 0; r0 < R; r0 += 4) {       // + dlogits_t W_g^T, r order
        float4 a[4], b[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = (r0 + u < R) ? exp_s[wid][r0 + u] : -1;
          if (e >= 0) {
            const float4* p = reinterpret_cast<const float4*>(wgT + (size_t)e * d + (size_t)v * 8);
            a[u] = p[0];
            b[u] = p[1];
          } else {
            a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (r0 + u >= R) break;
          if (exp_s[wid][r0 + u] < 0) continue;
          const float ds = ds_s[wid][r0 + u];
          acc[0] = fmaf(ds, a[u].x, acc[0]); acc[1] = fmaf(ds, a[u].y, acc[1]);
          acc[2] = fmaf(ds, a[u].z, acc[2]); acc[3] = fmaf(ds, a[u].w, acc[3]);
          acc[4] = fmaf(ds, b[u].x, acc[4]); acc[5] = fmaf(ds, b[u].y, acc[5]);
          acc[6] = fmaf(ds, b[u].z, acc[6]); acc[7] = fmaf(ds, b[u].w, acc[7]);
        }
      }
      if (add) {   // + the shared expert's dx
        float f[8];
        unpack8(ldg_nc_v4(add + (size_t)t * d + (size_t)v * 8), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += f[j];
      }
      reinterpret_cast<uint4*>(dx + (size_t)t * d)[v] = pack8(acc);
    }
    __syncwarp();
  }
}

int grid_for(int T, int per_block) {
  const int b = ceil_div(T, per_block);
  return b < 152 * 8 ? b : 152 * 8;
}

// Chunks of the router weight-gradient GEMM: whole 64-row k-blocks, about two
// waves of 76 CTA-pair items, at least 256 rows each.
DwgPlan plan_dwg(int T, int d, int E) {
  DwgPlan p;
  p.Ep = ceil_div(E, 32) * 32;
  const int tiles = ceil_div(d, 256) * ceil_div(2 * p.Ep, 256);
  int S = std::max(1, 152 / tiles);
  S = std::min(S, std::max(1, ceil_div(T, 256)));
  S = std::min(S, 64);
  p.chunk = std::max(64, ceil_div(ceil_div(std::max(T, 1), S), 64) * 64);
  p.S = std::max(1, ceil_div(T, p.chunk));
  return p;
}

}  // namespace

DwgPlan dwg_plan(int T, int d, int E) { return plan_dwg(T, d, E); }

size_t dwg_ws_bytes(int T, int d, int E) {
  const DwgPlan p = plan_dwg(T, d, E);
  return align_up((size_t)T * 2 * p.Ep * 2, 256) + align_up((size_t)p.S * d * 2 * p.Ep * 4, 256) +
         align_up((size_t)(p.S + 1) * 4, 256) + align_up((size_t)4 * p.S * 128, 256);
}

cudaError_t launch_bwd_route(const uint16_t* dy, const uint16_t* o, const int32_t* slot_row,
                             const float* w, int T, int d, int R, uint16_t* dO, float* dsel_tok,
                             cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  bwd_route_kernel<<<grid_for(T, BW), BW * 32, 0, s>>>(dy, o, slot_row, w, T, d, R, T * R, dO,
                                                      dsel_tok);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_wg_transpose(const float* wg, int d, int E, float* wgT, cudaStream_t s) {
  dim3 grid(ceil_div(d, 32), ceil_div(E, 32));
  wg_transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(wg, d, E, wgT);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dwg(const uint16_t* x, const int32_t* idx, const float* dsel_tok, int T, int d,
                       int E, int R, float* dW_gate, void* ws, int* err, bool cta_pairs,
                       cudaStream_t s) {
  const DwgPlan p = plan_dwg(T, d, E);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* Sm = reinterpret_cast<uint16_t*>(w);
  w += align_up((size_t)T * 2 * p.Ep * 2, 256);
  float* P = reinterpret_cast<float*>(w);
  w += align_up((size_t)p.S * d * 2 * p.Ep * 4, 256);
  int32_t* offs = reinterpret_cast<int32_t*>(w);
  w += align_up((size_t)(p.S + 1) * 4, 256);
  void* maps = w;
  dwg_operand_kernel<<<std::max(1, grid_for(T, BW)), BW * 32, 0, s>>>(idx, dsel_tok, T, E, R,
                                                                      p.Ep, p.chunk, p.S, Sm, offs);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_dwg_gemm(x, Sm, offs, T, d, 2 * p.Ep, p.S, P, maps, err, cta_pairs, s);
  if (e != cudaSuccess) return e;
  dwg_sum_kernel<<<std::min(ceil_div(d * E, 256), 152 * 8), 256, 0, s>>>(P, p.S, d, E, p.Ep,
                                                                        dW_gate);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dx_combine(const uint16_t* dx_perm, const int32_t* slot_row,
                              const int32_t* idx, const float* dsel_tok, const float* wgT, int T,
                              int d, int E, int R, uint16_t* dx, cudaStream_t s,
                              const uint16_t* add) {
  if (T == 0) return cudaSuccess;
  dx_combine_kernel<<<grid_for(T, BW), BW * 32, 0, s>>>(dx_perm, slot_row, idx, dsel_tok, wgT, T,
                                                       d, E, R, T * R, add, dx);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
