// Internal launchers shared by the C-ABI implementation (not exported).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Host-side checks and status handling shared by the C ABI's entry points.
// The shapes every routed entry point accepts (T tokens, hidden size d, E experts, top-R).
moe_status_t shape_check(int T, int d, int E, int R);
// Records e as this thread's last CUDA error (moe_last_cuda_error); returns MOE_ERR_CUDA.
moe_status_t cuda_failed(cudaError_t e);
// The status of a call whose work was enqueued with result `launched`; with
// MOE_CHECK in `flags`, waits for `s` and translates the device error word.
moe_status_t finish(cudaError_t launched, const int* err_dev, unsigned flags, cudaStream_t s);

// Adds n to the process-wide count of kernels launched by the library.
void count_launches(int n);
// Record the caller's trace events around stage `stage` (moe_stage_t), if tracing is on.
void trace_begin(int stage, cudaStream_t s);
void trace_end(int stage, cudaStream_t s);

// Arguments of the grouped tcgen05 GEMM kernel (one struct for all modes).
struct GemmArgs {
  int E, N, d, f;
  const int32_t* offsets;     // [E+1] expert row offsets
  const int2* tiles;          // ragged 128-row tiles {first row, expert}
  const int32_t* tile_count;  // number of valid entries in tiles
  int kblocks;                // 64-deep k-blocks per tile (row-ragged modes)
  int prepacked;              // forward weights in the tiled layout of moe_prepack_weights
  int n_tiles_n;              // output column tiles
  int n_tiles_m;              // output row tiles per expert (weight-gradient modes)
  uint16_t* out_bf16;
  uint16_t* save_a;
  uint16_t* save_b;
  const uint16_t* in_a;
  const uint16_t* in_b;
  float* out_f32;
  float* out_f32b;
  const float* bias;
  const float* row_scale;     // down epilogue: out[row] = bf16(row_scale[row] * acc), or null
  // weight-gradient modes: per expert e, tensor maps of A (entry 2e) and B
  // (2e+1) whose row extent ends at the expert's last row (CUtensorMap, 64-B aligned)
  const void* emaps;
  // gate: K split over ksplit (1 or 4) CTAs per tile, partials [4][T][E] fp32
  int ksplit;
  float* out_parts;
  int* err;
};

cudaError_t launch_gate_logits(const uint16_t* x, const float* wg, const float* bias, int T, int d,
                               int E, float* logits, cudaStream_t s);
cudaError_t launch_wg_split(const float* wg, int d, int E, uint16_t* wgs, cudaStream_t s);
// Gate projection on the tensor cores (needs d % 64 == 0): logits = x W_g + bias
// through the 3-term bf16 split of W_g; ws holds the split weights.
bool gate_tc_supported(int d);
size_t gate_tc_ws_bytes(int T, int d, int E);
cudaError_t launch_gate_tc(const uint16_t* x, const float* wg, const float* bias, int T, int d,
                           int E, float* logits, void* ws, int* err, cudaStream_t s);
// One block waits (bounded) on an mbarrier that nothing arrives on.
cudaError_t launch_selftest_wait(unsigned limit_us, int* err, cudaStream_t s);
cudaError_t launch_topk(const float* logits, int T, int E, int R, int32_t* idx, float* w,
                        cudaStream_t s);

size_t dispatch_ws_bytes(int T, int E);
cudaError_t launch_dispatch(const uint16_t* x, const int32_t* idx, int T, int d, int E, int R,
                            int32_t* counts, int32_t* offsets, int32_t* row_slot,
                            int32_t* slot_row, uint16_t* x_perm, void* ws, int* err,
                            cudaStream_t s);
cudaError_t dispatch_set_smem_limits();
cudaError_t launch_dispatch_fp8(const uint16_t* x, const int32_t* idx, int T, int d, int E, int R,
                                int32_t* counts, int32_t* offsets, int32_t* row_slot,
                                int32_t* slot_row, uint8_t* xq, float* xs, void* ws, int* err,
                                cudaStream_t s);
cudaError_t launch_dequant_fp8(const uint8_t* xq, const float* xs, long long N, int d,
                               uint16_t* out, cudaStream_t s);
// Microscaled fp8 (E4M3 codes, one UE8M0 scale per 32 elements along K; scale
// rows K/32 bytes rounded up to a multiple of 16).
int mx_scale_row_bytes(int K);
cudaError_t launch_quantize_mx(const uint16_t* x, long long rows, int K, uint8_t* xq,
                               uint8_t* xs, cudaStream_t s);
cudaError_t launch_dispatch_mx(const uint16_t* x, const int32_t* idx, int T, int d, int E, int R,
                               int32_t* counts, int32_t* offsets, int32_t* row_slot,
                               int32_t* slot_row, uint8_t* xq, uint8_t* xs, void* ws, int* err,
                               cudaStream_t s);
// Grouped SwiGLU FFN on microscaled fp8 rows and weights (d % 128 == 0, f % 128 == 0):
// h is quantised along f into hq / hs (or the workspace when null).
bool ffn_mx_supported(int d, int f);
size_t ffn_mx_ws_bytes(int N, int d, int f, int E);
cudaError_t launch_ffn_mx(const uint8_t* xq, const uint8_t* xs, const int32_t* offsets, int N,
                          int d, int f, int E, const uint8_t* W1q, const uint8_t* W1s,
                          const uint8_t* W3q, const uint8_t* W3s, const uint8_t* W2q,
                          const uint8_t* W2s, const float* row_scale, uint8_t* hq, uint8_t* hs,
                          uint16_t* out, void* ws, int* err, cudaStream_t s);

// y = bf16(add + sum_r w o); add (bf16 [T,d], the shared expert's output) may be null.
cudaError_t launch_combine(const uint16_t* o, const int32_t* slot_row, const float* w, int T,
                           int d, int R, uint16_t* y, cudaStream_t s,
                           const uint16_t* add = nullptr);
// offsets = {0, T}: every token in one expert (the shared expert).
cudaError_t launch_one_expert_offsets(int32_t* offsets, int T, cudaStream_t s);

size_t tiles_ws_bytes(int N, int E);
// The ragged tile lists in a tile workspace: {first row, expert} per tile_rows-row
// tile (and, with tail_rows > 0, experts' last tiles of at most tail_rows rows
// in a second list), their counts on the device.
struct TileLists {
  const int32_t* count;
  const int2* tiles;
  const int32_t* tail_count;
  const int2* tails;
};
TileLists tile_lists(void* ws, int E);
cudaError_t launch_build_tiles(const int32_t* offsets, int E, void* ws, cudaStream_t s,
                               int tile_rows = 128, int tail_rows = 0);
// A 2-D tensor map (CUtensorMap at `map`) of `outer` rows of `inner` elements of
// CUtensorMapDataType `dtype`, rows `row_bytes` apart, box {box_inner, box_outer}.
bool encode_map_2d(void* map, int dtype, const void* base, unsigned long long inner,
                   unsigned long long outer, unsigned long long row_bytes, unsigned box_inner,
                   unsigned box_outer, bool swizzle128);
cudaError_t launch_ffn_fwd(const uint16_t* x_perm, const int32_t* offsets, int N, int d, int f,
                           int E, const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                           uint16_t* a_save, uint16_t* b_save, uint16_t* h, uint16_t* out,
                           void* tiles_ws, int* err, bool prepacked, bool cta_pairs,
                           cudaStream_t s, const float* row_scale = nullptr);
// Weight tiles for the forward GEMMs: W1p, W3p [E][f/128][d/64][128][64] and
// W2p [E][d/256][f/64][256][64] (bf16), each tile one TMA box, contiguous.
bool prepack_supported(int d, int f);
cudaError_t launch_prepack(const uint16_t* W1, const uint16_t* W3, const uint16_t* W2, int E,
                           int d, int f, uint16_t* W1p, uint16_t* W3p, uint16_t* W2p,
                           cudaStream_t s);
cudaError_t launch_ffn_bwd(const uint16_t* x_perm, const int32_t* offsets, int N, int d, int f,
                           int E, const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                           const uint16_t* a_s, const uint16_t* b_s, const uint16_t* h,
                           const uint16_t* dO, uint16_t* dab, uint16_t* dx_perm, float* dW1,
                           float* dW3, float* dW2, void* tiles_ws, int* err, bool cta_pairs,
                           cudaStream_t s);

// backward of routing / dispatch / combine
cudaError_t launch_bwd_route(const uint16_t* dy, const uint16_t* o, const int32_t* slot_row,
                             const float* w, int T, int d, int R, uint16_t* dO, float* dsel_tok,
                             cudaStream_t s);
// dW_g = x^T dlogits on the tensor cores: dlogits split into bf16 hi and lo
// columns, S = [hi | lo] [T, 2 Ep], and the weight-gradient GEMM run over S
// chunks of the tokens (one partial [d, 2 Ep] per chunk), then summed.
struct DwgPlan {
  int Ep;      // E rounded up to 32
  int chunk;   // tokens per chunk (a multiple of 64)
  int S;       // chunks
};
DwgPlan dwg_plan(int T, int d, int E);
size_t dwg_ws_bytes(int T, int d, int E);
cudaError_t launch_dwg(const uint16_t* x, const int32_t* idx, const float* dsel_tok, int T, int d,
                       int E, int R, float* dW_gate, void* ws, int* err, bool cta_pairs,
                       cudaStream_t s);
// P[s] = x[rows of chunk s]^T S[rows of chunk s] for the chunks in offs[0..S]
// (S [T, n2] bf16, P [S, d, n2] fp32); maps_ws holds 4 * S tensor maps.
cudaError_t launch_dwg_gemm(const uint16_t* x, const uint16_t* Sm, const int32_t* offs, int T,
                            int d, int n2, int S, float* P, void* maps_ws, int* err,
                            bool cta_pairs, cudaStream_t s);
cudaError_t launch_wg_transpose(const float* wg, int d, int E, float* wgT, cudaStream_t s);
cudaError_t launch_dx_combine(const uint16_t* dx_perm, const int32_t* slot_row,
                              const int32_t* idx, const float* dsel_tok, const float* wgT, int T,
                              int d, int E, int R, uint16_t* dx, cudaStream_t s,
                              const uint16_t* add = nullptr);

}  // namespace moe
