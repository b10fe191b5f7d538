// Dispatch: group the T*R routed slots by expert into contiguous rows.
// ("Enabling trillion-parameter models on AWS EFA", section "Dispatch and
// combine": per-expert token counts, a cumulative sum of the counts for the
// offsets that pack each expert's tokens contiguously, and the shuffle of the
// tokens into the tensor the grouped GEMM reads.)
//
// Four kernels, all deterministic (no atomic decides an order):
//   1. expert_hist:  per block of CHUNK tokens, a shared-memory histogram of its
//      slots' experts -> blk_counts[e][b]; also flags out-of-range or repeated
//      expert indices.
//   2. expert_scan:  one CTA scans blk_counts in (expert, block) order ->
//      blk_base[e][b] = offsets[e] + rows of e in earlier blocks; counts, offsets.
//   3. slot_rank:    per block, warps walk their slots in order; __match_any_sync
//      gives each slot its rank among equal experts of its 32-slot group, so
//      row = blk_base + earlier warps + earlier groups + rank (stable order).
//   4. permute_rows: one warp per token reads x[t] once (16-byte vectors) and
//      writes it to its R rows of x_perm.
// With at most CHUNK tokens (one block of slots, e.g. a decode batch) one
// kernel does 1-3 (dispatch_plan_one_block): the same per-warp counts and
// ranks, with the per-expert totals scanned in shared memory.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int CHUNK = 256;     // tokens per block in hist / rank
constexpr int DWARPS = 8;      // warps per block in hist / rank

__global__ void __launch_bounds__(256) expert_hist_kernel(const int32_t* __restrict__ idx, int T,
                                                          int E, int R, int nblk,
                                                          int32_t* __restrict__ blk_counts,
                                                          int* __restrict__ err) {
  extern __shared__ int32_t cnt[];
  const int b = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int t0 = b * CHUNK;
  const int t1 = min(T, t0 + CHUNK);
  const int s0 = t0 * R, s1 = t1 * R;
  bool bad = false;
  for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
    const int e = idx[s];
    if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);
    else bad = true;
  }
  for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {  // repeated expert in a token
    const int32_t* row = idx + (size_t)t * R;
    for (int i = 1; i < R; ++i) {
      const int ei = row[i];
      for (int j = 0; j < i; ++j) bad |= (row[j] == ei);
    }
  }
  if (bad) atomicOr(err, kErrBadRouting);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blk_counts[(size_t)e * nblk + b] = cnt[e];
}

// Exclusive scan of L = E*nblk counts by one 1024-thread CTA, 4 values per thread per pass.
__global__ void __launch_bounds__(1024) expert_scan_kernel(const int32_t* __restrict__ blk_counts,
                                                            int E, int nblk,
                                                            int32_t* __restrict__ blk_base,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry_s;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const long long L = (long long)E * nblk;
  if (tid == 0) carry_s = 0;
  __syncthreads();
  for (long long base = 0; base < L; base += 4096) {
    int v[4];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long i = base + tid * 4 + j;
      v[j] = i < L ? blk_counts[i] : 0;
      sum += v[j];
    }
    int incl = sum;  // inclusive warp scan of per-thread sums
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int ws = warp_sums[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, ws, off);
        if (lane >= off) ws += o;
      }
      warp_sums[lane] = ws;  // inclusive over warps
    }
    __syncthreads();
    const int carry = carry_s;
    int run = carry + (wid > 0 ? warp_sums[wid - 1] : 0) + incl - sum;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long i = base + tid * 4 + j;
      if (i < L) blk_base[i] = run;
      run += v[j];
    }
    __syncthreads();
    if (tid == 0) carry_s = carry + warp_sums[31];
    __syncthreads();
  }
  const int total = carry_s;
  for (int e = tid; e < E; e += blockDim.x) {
    const int first = blk_base[(size_t)e * nblk];
    const int next = (e + 1 < E) ? blk_base[(size_t)(e + 1) * nblk] : total;
    offsets[e] = first;
    counts[e] = next - first;
  }
  if (tid == 0) offsets[E] = total;
}

__global__ void __launch_bounds__(256) slot_rank_kernel(const int32_t* __restrict__ idx, int T,
                                                        int E, int R, int nblk,
                                                        const int32_t* __restrict__ blk_base,
                                                        int32_t* __restrict__ row_slot,
                                                        int32_t* __restrict__ slot_row) {
  extern __shared__ int32_t sm[];
  int32_t* wcnt = sm;                       // [DWARPS][E]
  int32_t* keys = sm + DWARPS * E;          // [CHUNK*R]
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int t0 = b * CHUNK;
  const int t1 = min(T, t0 + CHUNK);
  const int s0 = t0 * R, ns = (t1 - t0) * R;
  for (int i = threadIdx.x; i < DWARPS * E; i += blockDim.x) wcnt[i] = 0;
  for (int i = threadIdx.x; i < ns; i += blockDim.x) {
    const int e = idx[s0 + i];
    keys[i] = ((unsigned)e < (unsigned)E) ? e : -1;
  }
  __syncthreads();
  // this warp's contiguous range of slots, in slot order
  const int per_warp = ceil_div(ns, DWARPS * 32) * 32;
  const int w0 = wid * per_warp;
  const int w1 = min(ns, w0 + per_warp);
  int32_t* my = wcnt + wid * E;
  for (int g = w0; g < w1; g += 32) {  // pass 1: per-warp counts
    const int i = g + lane;
    const int e = i < w1 ? keys[i] : -1;
    const unsigned peers = __match_any_sync(kFull, e);
    if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {  // warp bases for this block
    int run = blk_base[(size_t)e * nblk + b];
#pragma unroll
    for (int w = 0; w < DWARPS; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int g = w0; g < w1; g += 32) {  // pass 2: rows
    const int i = g + lane;
    const int e = i < w1 ? keys[i] : -1;
    const unsigned peers = __match_any_sync(kFull, e);
    int row = -1;
    if (e >= 0) row = my[e] + __popc(peers & lt);
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
    if (i < w1) {
      slot_row[s0 + i] = row;
      if (row >= 0) row_slot[row] = s0 + i;
    }
  }
}

// Steps 1-3 for T <= CHUNK in one block: validation, per-warp counts (pass 1 of
// slot_rank), per-expert totals, their exclusive scan (offsets), warp bases,
// and the rows (pass 2).  Same rows as the three-kernel path.
__global__ void __launch_bounds__(256) dispatch_plan_one_block_kernel(
    const int32_t* __restrict__ idx, int T, int E, int R, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ row_slot, int32_t* __restrict__ slot_row,
    int* __restrict__ err) {
  extern __shared__ int32_t sm[];
  int32_t* wcnt = sm;                       // [DWARPS][E]
  int32_t* keys = sm + DWARPS * E;          // [CHUNK*R]
  int32_t* tot = keys + CHUNK * R;          // [E]
  __shared__ int32_t warp_sums[DWARPS];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int ns = T * R;
  bool bad = false;
  for (int i = threadIdx.x; i < DWARPS * E; i += blockDim.x) wcnt[i] = 0;
  for (int i = threadIdx.x; i < ns; i += blockDim.x) {
    const int e = idx[i];
    const bool ok = (unsigned)e < (unsigned)E;
    bad |= !ok;
    keys[i] = ok ? e : -1;
  }
  for (int t = threadIdx.x; t < T; t += blockDim.x) {  // repeated expert in a token
    const int32_t* row = idx + (size_t)t * R;
    for (int i = 1; i < R; ++i) {
      const int ei = row[i];
      for (int j = 0; j < i; ++j) bad |= (row[j] == ei);
    }
  }
  if (bad) atomicOr(err, kErrBadRouting);
  __syncthreads();
  const int per_warp = ceil_div(ns, DWARPS * 32) * 32;
  const int w0 = wid * per_warp;
  const int w1 = min(ns, w0 + per_warp);
  int32_t* my = wcnt + wid * E;
  for (int g = w0; g < w1; g += 32) {  // per-warp counts
    const int i = g + lane;
    const int e = i < w1 ? keys[i] : -1;
    const unsigned peers = __match_any_sync(kFull, e);
    if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < DWARPS; ++w) c += wcnt[w * E + e];
    tot[e] = c;
  }
  __syncthreads();
  // exclusive scan of tot: each thread a contiguous range of experts
  const int per = ceil_div(E, (int)blockDim.x);
  const int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
  int sum = 0;
  for (int e = e0; e < e1; ++e) sum += tot[e];
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  int run = incl - sum;
  for (int w = 0; w < wid; ++w) run += warp_sums[w];
  for (int e = e0; e < e1; ++e) {   // offsets, counts and the warps' bases of expert e
    const int c = tot[e];
    offsets[e] = run;
    counts[e] = c;
    int wrun = run;
#pragma unroll
    for (int w = 0; w < DWARPS; ++w) {
      const int cw = wcnt[w * E + e];
      wcnt[w * E + e] = wrun;
      wrun += cw;
    }
    run += c;
  }
  if (threadIdx.x == blockDim.x - 1) offsets[E] = run;   // rows of valid slots
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int g = w0; g < w1; g += 32) {  // rows
    const int i = g + lane;
    const int e = i < w1 ? keys[i] : -1;
    const unsigned peers = __match_any_sync(kFull, e);
    int row = -1;
    if (e >= 0) row = my[e] + __popc(peers & lt);
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
    if (i < w1) {
      slot_row[i] = row;
      if (row >= 0) row_slot[row] = i;
    }
  }
}

// One warp per token; lanes move 16-byte vectors of x[t] to the token's R rows.
// One warp per (token, column chunk): a token's row is cut into `chunks`
// pieces of `cv` 16-byte vectors (a multiple of 128) when there are too few
// tokens to give every SM several warps (small batches, e.g. decode).
__global__ void __launch_bounds__(256) permute_rows_kernel(const uint16_t* __restrict__ x, int T,
                                                           int d, int R, int N, int chunks,
                                                           int cv,
                                                           const int32_t* __restrict__ slot_row,
                                                           uint16_t* __restrict__ x_perm) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x / 32;
  const int nv = d / 8;
  const long long units = (long long)T * chunks;
  for (long long u = (long long)blockIdx.x * warps + threadIdx.x / 32; u < units;
       u += (long long)gridDim.x * warps) {
    const int t = (int)(u / chunks), c = (int)(u % chunks);
    int my_row = lane < R ? slot_row[(size_t)t * R + lane] : -1;
    if ((unsigned)my_row >= (unsigned)N) my_row = -1;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const int vend = min(nv, (c + 1) * cv);
    for (int base = c * cv; base < vend; base += 32 * 4) {  // warp-uniform trip count
      const int v0 = base + lane;
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < vend) q[u] = ldg_nc_v4(src + v0 + 32 * u);
      for (int r = 0; r < R; ++r) {
        const int row = __shfl_sync(kFull, my_row, r);
        if (row < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)row * d);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (v0 + 32 * u < vend) dst[v0 + 32 * u] = q[u];
      }
    }
  }
}
// Block-scaled fp8 variant of permute_rows: one warp per token quantises each
// 128-channel block once (16 lanes x 8 channels: amax by half-warp shuffles,
// scale = amax / 448, codes = E4M3(x / scale) rounded to nearest even with
// saturation) and writes the 8-byte code groups and the block scales to the
// token's R rows.  An all-zero block gets scale 0 and zero codes.
__global__ void __launch_bounds__(256) permute_rows_fp8_kernel(
    const uint16_t* __restrict__ x, int T, int d, int R, int N,
    const int32_t* __restrict__ slot_row, uint8_t* __restrict__ xq, float* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x / 32;
  const int nb = d / 128;
  for (int t = blockIdx.x * warps + threadIdx.x / 32; t < T; t += gridDim.x * warps) {
    int my_row = lane < R ? slot_row[(size_t)t * R + lane] : -1;
    if ((unsigned)my_row >= (unsigned)N) my_row = -1;
    for (int base = 0; base < d; base += 256) {       // two blocks per pass, warp-uniform
      const int c = base + lane * 8;
      const bool valid = c < d;
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (valid) unpack8(ldg_nc_v4(x + (size_t)t * d + c), v);
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
      const float scale = amax / 448.f;
      uint32_t lo = 0, hi = 0;
      if (scale > 0.f) {
        __nv_fp8x2_storage_t p0 = __nv_cvt_float2_to_fp8x2(make_float2(v[0] / scale, v[1] / scale), __NV_SATFINITE, __NV_E4M3);
        __nv_fp8x2_storage_t p1 = __nv_cvt_float2_to_fp8x2(make_float2(v[2] / scale, v[3] / scale), __NV_SATFINITE, __NV_E4M3);
        __nv_fp8x2_storage_t p2 = __nv_cvt_float2_to_fp8x2(make_float2(v[4] / scale, v[5] / scale), __NV_SATFINITE, __NV_E4M3);
        __nv_fp8x2_storage_t p3 = __nv_cvt_float2_to_fp8x2(make_float2(v[6] / scale, v[7] / scale), __NV_SATFINITE, __NV_E4M3);
        lo = (uint32_t)p0 | ((uint32_t)p1 << 16);
        hi = (uint32_t)p2 | ((uint32_t)p3 << 16);
      }
      const int blk = c / 128;
      for (int r = 0; r < R; ++r) {
        const int row = __shfl_sync(kFull, my_row, r);
        if (row < 0 || !valid) continue;
        *reinterpret_cast<uint2*>(xq + (size_t)row * d + c) = make_uint2(lo, hi);
        if ((lane & 15) == 0) xs[(size_t)row * nb + blk] = scale;
      }
    }
  }
}

// Microscaled fp8 rows (mx_exponent, mx_codes4).  One warp per source row
// (token t of x, or row t of a weight matrix): each
// lane takes 8 channels, four lanes one 32-channel block (amax by shuffles
// within the four), codes = E4M3(v * 2^-k) rounded to nearest even (exact
// scaling), and writes the 8-byte code groups and the block's scale byte to
// the row's R destination rows (slot_row), or to row t itself when slot_row is
// null.  Scale rows are sk bytes apart (K/32 rounded up to 16).
__global__ void __launch_bounds__(256) quantize_mx_rows_kernel(
    const uint16_t* __restrict__ x, long long rows, int K, int R, int N,
    const int32_t* __restrict__ slot_row, uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
    int sk) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x / 32;
  for (long long t = blockIdx.x * (long long)warps + threadIdx.x / 32; t < rows;
       t += (long long)gridDim.x * warps) {
    int my_row = -1;                               // (unused when slot_row is null)
    if (slot_row != nullptr) {
      my_row = lane < R ? slot_row[(size_t)t * R + lane] : -1;
      if ((unsigned)my_row >= (unsigned)N) my_row = -1;
    }
    const int nr = slot_row == nullptr ? 1 : R;
    for (int base = 0; base < K; base += 256) {    // eight blocks per pass, warp-uniform
      const int c = base + lane * 8;
      const bool valid = c < K;
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (valid) unpack8(ldg_nc_v4(x + (size_t)t * K + c), v);
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
      const int k = mx_exponent(amax);
      const uint32_t w[2] = {mx_codes4(v, k), mx_codes4(v + 4, k)};
      for (int r = 0; r < nr; ++r) {
        const long long row = slot_row == nullptr ? t : (long long)__shfl_sync(kFull, my_row, r);
        if (row < 0 || !valid) continue;
        *reinterpret_cast<uint2*>(xq + (size_t)row * K + c) = make_uint2(w[0], w[1]);
        if ((lane & 3) == 0) xs[(size_t)row * sk + c / 32] = (uint8_t)(k + 127);
      }
    }
  }
}

// Identity expert for fp8-dispatched rows: out = bf16(code * scale).
__global__ void __launch_bounds__(256) dequant_fp8_kernel(const uint8_t* __restrict__ xq,
                                                          const float* __restrict__ xs, long long N,
                                                          int d, uint16_t* __restrict__ out) {
  const int nb = d / 128;
  const long long groups = N * (d / 8);
  for (long long gi = blockIdx.x * (long long)blockDim.x + threadIdx.x; gi < groups;
       gi += (long long)gridDim.x * blockDim.x) {
    const long long row = gi / (d / 8);
    const int c = (int)(gi % (d / 8)) * 8;
    const float scale = xs[row * nb + c / 128];
    const uint2 q = *reinterpret_cast<const uint2*>(xq + row * d + c);
    float f[8];
    e4m3x8_scaled(q, scale, f);
    *reinterpret_cast<uint4*>(out + row * d + c) = pack8(f);
  }
}
}  // namespace

size_t dispatch_ws_bytes(int T, int E) {
  const int nblk = ceil_div(T > 0 ? T : 1, CHUNK);
  return align_up((size_t)2 * E * nblk * sizeof(int32_t), 256);
}

cudaError_t launch_dispatch(const uint16_t* x, const int32_t* idx, int T, int d, int E, int R,
                            int32_t* counts, int32_t* offsets, int32_t* row_slot,
                            int32_t* slot_row, uint16_t* x_perm, void* ws, int* err,
                            cudaStream_t s) {
  const int nblk = ceil_div(T > 0 ? T : 1, CHUNK);
  int32_t* blk_counts = static_cast<int32_t*>(ws);
  int32_t* blk_base = blk_counts + (size_t)E * nblk;
  if (T == 0) {
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
    if (e != cudaSuccess) return e;
    return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
  }
  if (nblk == 1) {   // one block of slots: the plan in one kernel
    const size_t smem = sizeof(int32_t) * ((size_t)DWARPS * E + (size_t)CHUNK * R + E);
    dispatch_plan_one_block_kernel<<<1, 256, smem, s>>>(idx, T, E, R, counts, offsets, row_slot,
                                                        slot_row, err);
    count_launches(1);
  } else {
    expert_hist_kernel<<<nblk, 256, E * sizeof(int32_t), s>>>(idx, T, E, R, nblk, blk_counts,
                                                             err);
    expert_scan_kernel<<<1, 1024, 0, s>>>(blk_counts, E, nblk, blk_base, counts, offsets);
    const size_t rank_smem = sizeof(int32_t) * ((size_t)DWARPS * E + (size_t)CHUNK * R);
    slot_rank_kernel<<<nblk, 256, rank_smem, s>>>(idx, T, E, R, nblk, blk_base, row_slot,
                                                  slot_row);
    count_launches(3);
  }
  if (x != nullptr && x_perm != nullptr) {
    // few tokens: cut each row into column chunks so that ~16 warps per SM copy
    const int nv = d / 8;
    const long long want = 152LL * 16;
    int chunks = 1;
    if (T < want) {
      const long long c = (want + T - 1) / T;
      const int cmax = nv / 128 > 1 ? nv / 128 : 1;
      chunks = c < cmax ? (int)c : cmax;
    }
    const int cv = ceil_div(ceil_div(nv, chunks), 128) * 128;
    chunks = ceil_div(nv, cv);
    const long long units = (long long)T * chunks;
    const int blocks = (int)((units + 7) / 8 < 152 * 8 ? (units + 7) / 8 : 152 * 8);
    permute_rows_kernel<<<blocks, 256, 0, s>>>(x, T, d, R, T * R, chunks, cv, slot_row, x_perm);
    count_launches(1);
  }
  return cudaGetLastError();
}

cudaError_t launch_dispatch_fp8(const uint16_t* x, const int32_t* idx, int T, int d, int E, int R,
                                int32_t* counts, int32_t* offsets, int32_t* row_slot,
                                int32_t* slot_row, uint8_t* xq, float* xs, void* ws, int* err,
                                cudaStream_t s) {
  cudaError_t e = launch_dispatch(nullptr, idx, T, d, E, R, counts, offsets, row_slot, slot_row,
                                  nullptr, ws, err, s);
  if (e != cudaSuccess || T == 0) return e;
  const int blocks = ceil_div(T, 8) < 152 * 8 ? ceil_div(T, 8) : 152 * 8;
  permute_rows_fp8_kernel<<<blocks, 256, 0, s>>>(x, T, d, R, T * R, slot_row, xq, xs);
  count_launches(1);
  return cudaGetLastError();
}

int mx_scale_row_bytes(int K) { return ceil_div(K / 32, 16) * 16; }

cudaError_t launch_quantize_mx(const uint16_t* x, long long rows, int K, uint8_t* xq,
                               uint8_t* xs, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const long long want = (rows + 7) / 8;
  const int blocks = want < 152 * 8 ? (int)want : 152 * 8;
  quantize_mx_rows_kernel<<<blocks, 256, 0, s>>>(x, rows, K, 1, 0, nullptr, xq, xs,
                                                 mx_scale_row_bytes(K));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_mx(const uint16_t* x, const int32_t* idx, int T, int d, int E, int R,
                               int32_t* counts, int32_t* offsets, int32_t* row_slot,
                               int32_t* slot_row, uint8_t* xq, uint8_t* xs, void* ws, int* err,
                               cudaStream_t s) {
  cudaError_t e = launch_dispatch(nullptr, idx, T, d, E, R, counts, offsets, row_slot, slot_row,
                                  nullptr, ws, err, s);
  if (e != cudaSuccess || T == 0) return e;
  const int blocks = ceil_div(T, 8) < 152 * 8 ? ceil_div(T, 8) : 152 * 8;
  quantize_mx_rows_kernel<<<blocks, 256, 0, s>>>(x, T, d, R, T * R, slot_row, xq, xs,
                                                 mx_scale_row_bytes(d));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dequant_fp8(const uint8_t* xq, const float* xs, long long N, int d,
                               uint16_t* out, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  const long long groups = N * (d / 8);
  const long long want = (groups + 255) / 256;
  const int blocks = want < 152 * 16 ? (int)want : 152 * 16;
  dequant_fp8_kernel<<<blocks, 256, 0, s>>>(xq, xs, N, d, out);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t dispatch_set_smem_limits() {
  const int max_rank_smem = sizeof(int32_t) * (DWARPS * 1024 + CHUNK * 32);
  cudaError_t e = cudaFuncSetAttribute(slot_rank_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max_rank_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(dispatch_plan_one_block_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              max_rank_smem + (int)sizeof(int32_t) * 1024);
}

}  // namespace moe
