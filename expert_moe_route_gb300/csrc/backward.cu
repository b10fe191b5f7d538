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
// Pass 1: block = (1024-column chunk, expert, row chunk s of DWG_SPLIT); thread =
// 8 consecutive columns (16-byte loads), four rows' loads in flight per step,
// fp32 accumulation in row order -> part[s][e][k].  Pass 2 adds the DWG_SPLIT
// partials in s order and writes dW_g transposed through shared memory.
constexpr int DWG_THREADS = 128;
constexpr int DWG_SPLIT = 4;
// dW_g column e, split over DWG_SPLIT row ranges: sum over the expert's rows of
// dsel_row[row] * x[token(row)].  The rows are read from x through row_slot
// (x_perm[row] == x[row_slot[row] / R]): every expert walks its tokens in
// ascending order, so the R reads of a token's row come close together and
// mostly hit L2 -- x (T*d) is read from HBM about once instead of x_perm (N*d).
__global__ void __launch_bounds__(DWG_THREADS) dwg_partial_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ row_slot, int R,
    const int32_t* __restrict__ offsets, const float* __restrict__ dsel_row, int d, int E,
    float* __restrict__ part) {
  const int e = blockIdx.y, sp = blockIdx.z;
  const int k0 = (blockIdx.x * DWG_THREADS + threadIdx.x) * 8;
  if (k0 >= d) return;
  const int e0 = offsets[e], n = offsets[e + 1] - e0;
  const int r0 = e0 + (int)((long long)n * sp / DWG_SPLIT);
  const int r1 = e0 + (int)((long long)n * (sp + 1) / DWG_SPLIT);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  int row = r0;
  for (; row + 4 <= r1; row += 4) {
    uint4 q[4];
    float s[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      q[u] = ldg_nc_v4(x + (size_t)(row_slot[row + u] / R) * d + k0);
      s[u] = dsel_row[row + u];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float xv[8];
      unpack8(q[u], xv);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(s[u], xv[j], acc[j]);
    }
  }
  for (; row < r1; ++row) {
    float xv[8];
    unpack8(ldg_nc_v4(x + (size_t)(row_slot[row] / R) * d + k0), xv);
    const float s = dsel_row[row];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = fmaf(s, xv[j], acc[j]);
  }
  float4* dst = reinterpret_cast<float4*>(part + ((size_t)sp * E + e) * d + k0);
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

__global__ void dwg_reduce_kernel(const float* __restrict__ part, int d, int E,
                                  float* __restrict__ dW_gate) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {      // i: expert in tile, x: column
    const int e = e0 + i, k = k0 + threadIdx.x;
    float v = 0.f;
    if (e < E && k < d)
      for (int sp = 0; sp < DWG_SPLIT; ++sp) v += part[((size_t)sp * E + e) * d + k];
    tile[i][threadIdx.x] = v;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {      // i: column in tile, x: expert
    const int k = k0 + i, e = e0 + threadIdx.x;
    if (k < d && e < E) dW_gate[(size_t)k * E + e] = tile[threadIdx.x][i];
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

size_t dwg_ws_bytes(int d, int E) { return align_up((size_t)DWG_SPLIT * E * d * 4, 256); }

cudaError_t launch_dwg(const uint16_t* x, const int32_t* row_slot, int R, const int32_t* offsets,
                       const float* dsel_row, int d, int E, float* dW_gate, void* ws,
                       cudaStream_t s) {
  float* part = static_cast<float*>(ws);
  dim3 grid(ceil_div(d, DWG_THREADS * 8), E, DWG_SPLIT);
  dwg_partial_kernel<<<grid, DWG_THREADS, 0, s>>>(x, row_slot, R, offsets, dsel_row, d, E, part);
  dwg_reduce_kernel<<<dim3(ceil_div(d, 32), ceil_div(E, 32)), dim3(32, 8), 0, s>>>(part, d, E,
                                                                                  dW_gate);
  count_launches(2);
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
