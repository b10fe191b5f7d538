// Backward of the routing, dispatch and combine steps (the expert GEMMs'
// backward is in grouped_gemm.cu).  With y_t = sum_r w_r o_{row(t,r)} and the
// gate weights the softmax over the chosen logits:
//   dw_r = <dy_t, o_row>,  do_row = bf16(w_r dy_t)
//   dlogits at the chosen experts: w_q (dw_q - sum_r w_r dw_r); zero elsewhere
//   dW_g = x^T dlogits  -> for expert e: sum over its rows of dlogits_row x_perm[row]
//   dx_t = bf16( sum_r dx_perm[row(t,r)] + sum_r dlogits_{t,r} W_g[:, idx[t,r]] )
// All reductions run in a fixed order, so results are bitwise reproducible.
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
    uint16_t* __restrict__ dO, float* __restrict__ dsel_tok, float* __restrict__ dsel_row) {
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
      for (int r = 0; r < 32; ++r) {
        if (r >= R) break;
        const int row = rows_s[wid][r];
        if (row < 0) continue;
        float ov[8], dv[8];
        unpack8(ldg_nc_v4(o + (size_t)row * d + (size_t)v * 8), ov);
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
      const int row = rows_s[wid][lane];
      if (row >= 0) dsel_row[row] = ds;
    }
    __syncwarp();
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

// dW_g[k, e] = sum over expert e's rows (ascending) of dsel_row[row] * x_perm[row, k].
// Block = (expert, 256-column chunk); thread = one column k.
__global__ void __launch_bounds__(256) dwg_kernel(const uint16_t* __restrict__ x_perm,
                                                  const int32_t* __restrict__ offsets,
                                                  const float* __restrict__ dsel_row, int d, int E,
                                                  float* __restrict__ dW_gate) {
  const int e = blockIdx.y;
  const int k = blockIdx.x * 256 + threadIdx.x;
  const int r0 = offsets[e], r1 = offsets[e + 1];
  float acc = 0.f;
  if (k < d) {
    const unsigned short* xp = reinterpret_cast<const unsigned short*>(x_perm);
    for (int row = r0; row < r1; ++row) {
      const float xv = __uint_as_float((uint32_t)xp[(size_t)row * d + k] << 16);
      acc = fmaf(dsel_row[row], xv, acc);
    }
    dW_gate[(size_t)k * E + e] = acc;
  }
}

// dx[t] = bf16( sum_r dx_perm[row_r] + sum_r dsel[t,r] * W_g^T[idx[t,r]] ), fp32 in r order.
__global__ void __launch_bounds__(BW * 32) dx_combine_kernel(
    const uint16_t* __restrict__ dx_perm, const int32_t* __restrict__ slot_row,
    const int32_t* __restrict__ idx, const float* __restrict__ dsel, const float* __restrict__ wgT,
    int T, int d, int E, int R, int N, uint16_t* __restrict__ dx) {
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
      for (int r = 0; r < R; ++r) {
        const int row = rows_s[wid][r];
        if (row < 0) continue;
        float f[8];
        unpack8(ldg_nc_v4(dx_perm + (size_t)row * d + (size_t)v * 8), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += f[j];
      }
      for (int r = 0; r < R; ++r) {
        const int e = exp_s[wid][r];
        if (e < 0) continue;
        const float ds = ds_s[wid][r];
        const float4* p = reinterpret_cast<const float4*>(wgT + (size_t)e * d + (size_t)v * 8);
        const float4 a = p[0], b = p[1];
        acc[0] = fmaf(ds, a.x, acc[0]); acc[1] = fmaf(ds, a.y, acc[1]);
        acc[2] = fmaf(ds, a.z, acc[2]); acc[3] = fmaf(ds, a.w, acc[3]);
        acc[4] = fmaf(ds, b.x, acc[4]); acc[5] = fmaf(ds, b.y, acc[5]);
        acc[6] = fmaf(ds, b.z, acc[6]); acc[7] = fmaf(ds, b.w, acc[7]);
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
}  // namespace

cudaError_t launch_bwd_route(const uint16_t* dy, const uint16_t* o, const int32_t* slot_row,
                             const float* w, int T, int d, int R, uint16_t* dO, float* dsel_tok,
                             float* dsel_row, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  bwd_route_kernel<<<grid_for(T, BW), BW * 32, 0, s>>>(dy, o, slot_row, w, T, d, R, T * R, dO,
                                                      dsel_tok, dsel_row);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_wg_transpose(const float* wg, int d, int E, float* wgT, cudaStream_t s) {
  dim3 grid(ceil_div(d, 32), ceil_div(E, 32));
  wg_transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(wg, d, E, wgT);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dwg(const uint16_t* x_perm, const int32_t* offsets, const float* dsel_row,
                       int d, int E, float* dW_gate, cudaStream_t s) {
  dim3 grid(ceil_div(d, 256), E);
  dwg_kernel<<<grid, 256, 0, s>>>(x_perm, offsets, dsel_row, d, E, dW_gate);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dx_combine(const uint16_t* dx_perm, const int32_t* slot_row,
                              const int32_t* idx, const float* dsel_tok, const float* wgT, int T,
                              int d, int E, int R, uint16_t* dx, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dx_combine_kernel<<<grid_for(T, BW), BW * 32, 0, s>>>(dx_perm, slot_row, idx, dsel_tok, wgT, T,
                                                       d, E, R, T * R, dx);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
