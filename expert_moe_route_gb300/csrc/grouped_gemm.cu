// Grouped per-expert GEMMs on the 5th-generation tensor cores (tcgen05).
// ("Enabling trillion-parameter models on AWS EFA", section "MoE all-to-all
// over EFA": after dispatch, grouped GEMMs multiply each expert's tokens by its
// weights; the expert FFN here is SwiGLU.)
//
// One persistent, warp-specialised kernel template serves all six contractions
// of the layer:
//   GATEUP  [a|b] = x_perm W1[e]^T | x_perm W3[e]^T, epilogue h = bf16(silu(a) b)
//   DOWN    o = bf16(h W2[e]^T)
//   DH      dh = do W2[e], epilogue da = bf16(dh b silu'(a)), db = bf16(dh silu(a))
//   DX      dx_perm = bf16([da|db] [W1[e]; W3[e]])
//   WG2     dW2[e] = do^T h                     (K = the expert's rows, ragged)
//   WG13    [dW1[e]; dW3[e]] = [da|db]^T x_perm (K ragged)
// Roles (320 threads): warp 0 issues TMA loads into a shared-memory ring,
// warp 1 owns TMEM and issues tcgen05.mma (bf16 in, fp32 accumulate), warps
// 2-9 drain the accumulator (tcgen05.ld; two warps per TMEM lane quadrant,
// each taking half of the columns) and run the epilogue.  Two 256-column TMEM
// accumulators let the epilogue of one tile overlap the main loop of the next.
// By default a cluster of two CTAs computes 256 x 256 tiles with
// tcgen05.mma.cta_group::2 (each CTA stages 128 rows of A and 128 columns of
// B, six 32 KB stages; rank 0 issues the MMAs); single-CTA kernels compute
// 128 x 256 tiles from four 48 KB stages.  The weight-gradient modes contract
// over each expert's rows: an expert's last, partial k-block is loaded through
// tensor maps whose row extent ends at the expert's last row, so the rows of
// the next expert arrive as zeros.  Every wait is bounded
// (kWaitLimitNs); a timeout sets the error word and all roles return after
// their in-flight copies and MMAs have drained.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int BM = 128, BK = 64, BN = 256, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KiB
constexpr int B_BYTES = BN * BK * 2;            // 32 KiB
constexpr int ATOM_BYTES = 64 * BK * 2;         // MN-major block: 64 elements x 64 k-rows
constexpr int EPI_WARPS = 8;                      // two per TMEM lane quadrant
constexpr int EPI_WARP_BYTES = 32 * 128;          // one 32-row x 128-B fp32 staging box
constexpr int EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES;  // per CTA (weight-gradient modes only)
constexpr int CTL_BYTES = 256;

constexpr int THREADS = 64 + 32 * EPI_WARPS;     // TMA warp, MMA warp, epilogue warps
constexpr uint32_t TMEM_COLS = 512;

enum Mode : int { GATEUP = 0, DOWN = 1, DH = 2, DX = 3, WG2 = 4, WG13 = 5, GATE = 6,
                  GATEUP2 = 7, DOWN2 = 8 };

template <int M, bool C2 = false> struct Traits {
  static constexpr bool a_mn = (M == WG2 || M == WG13);
  static constexpr bool b_mn = (M == DH || M == DX || M == WG2 || M == WG13);
  static constexpr bool wgrad = (M == WG2 || M == WG13);
  // one 32-row x 128-B staging box per epilogue warp (all modes but the gate)
  // (the weight-gradient modes on pairs store from registers: their 32 KB go to
  // a seventh pipeline stage instead)
  static constexpr int epi_bytes = (M == GATE || (C2 && (M == WG2 || M == WG13))) ? 0 : EPI_BYTES;
  // GATE: 128-column tiles with four partial accumulators (K-blocks rotate over
  // them; the epilogue adds them in IEEE fp32), so each accumulator takes a
  // quarter of the tensor core's accumulation steps.  A stage holds one
  // 64-deep block of x and the same block of the three bf16 terms of W_g
  // (hi, mid, lo), so x is loaded once for the three products.
  static constexpr bool partials = (M == GATE);
  static constexpr int bn = partials ? 128 : BN;
  // GATEUP2 / DOWN2: each item is a 256-row block of one expert, computed as
  // two 128-row accumulators (TMEM columns 0-255 and 256-511) that share every
  // B (weight) stage: each weight tile is read once per 256 rows and each SM
  // keeps twice the distinct weight bytes in flight -- the weight-streaming
  // regime (few rows per expert).  No second accumulator set, so the epilogue
  // does not overlap the next item's main loop.
  static constexpr bool pair = (M == GATEUP2 || M == DOWN2);
  static constexpr bool is_gateup = (M == GATEUP || M == GATEUP2);
  static constexpr bool is_down = (M == DOWN || M == DOWN2);
  static constexpr bool single_acc = partials || pair;
  // C2: the CTA pair computes 256-row tiles; each CTA stages 128 rows of A
  // and half of B (128 of the 256 columns), so a stage is 32 KB and six fit.
  static constexpr int tile_m = C2 ? 2 * BM : BM;
  static constexpr int stages =
      (pair || partials) ? 3 : (C2 ? ((M == WG2 || M == WG13) ? 7 : 6) : STAGES);
  static constexpr int a_bytes = pair ? 2 * A_BYTES : A_BYTES;
  static constexpr int b_bytes = partials ? 3 * 128 * BK * 2 : (C2 ? B_BYTES / 2 : B_BYTES);
  static constexpr int stage_bytes = a_bytes + b_bytes;
  // bytes the full barrier expects per stage (rank 0's barrier counts both CTAs' loads)
  static constexpr uint32_t stage_tx =
      (uint32_t)(C2 ? 2 * stage_bytes : stage_bytes);
  // stages | epilogue staging | control block, plus slack for 1024-B alignment
  static constexpr int smem_bytes = stages * stage_bytes + epi_bytes + CTL_BYTES + 1024;
};

constexpr int MAX_STAGES = 7;

struct alignas(8) SharedCtl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

struct Item {
  int e, row0, row_end, mt, nt, kblocks, krow0, krows;   // krows: K rows (weight-gradient modes)
  int kb0 = 0, kstep = 1;   // GATE split over CTAs: this item's k-blocks are kb0, kb0 + kstep, ...
};

__device__ __forceinline__ bool decode_item(const GemmArgs& g, int mode, int item, Item& it) {
  if (mode == GATE) {  // one group of T rows: 128-row tiles x 128-expert column tiles
    // with g.ksplit = 4, four CTAs share a tile: CTA p takes the k-blocks
    // kb = p (mod 4), i.e. the tile's partial accumulator p
    const int S = g.ksplit > 1 ? g.ksplit : 1;
    const int tile = item / S, p = item - tile * S;
    const int mi = tile / g.n_tiles_n;
    it.nt = tile % g.n_tiles_n;
    it.row0 = mi * BM;
    it.row_end = g.N;
    it.e = 0;
    it.mt = 0;
    it.krow0 = it.krows = 0;
    it.kb0 = p;
    it.kstep = S;
    it.kblocks = (g.kblocks - p + S - 1) / S;
    return true;
  }
  if (mode == WG2 || mode == WG13) {
    const int per_e = g.n_tiles_m * g.n_tiles_n;
    it.e = item / per_e;
    const int rem = item % per_e;
    it.mt = rem / g.n_tiles_n;
    it.nt = rem % g.n_tiles_n;
    it.krow0 = g.offsets[it.e];
    it.krows = g.offsets[it.e + 1] - it.krow0;
    it.kblocks = ceil_div(it.krows, BK);
    it.row0 = it.row_end = 0;
    return true;
  }
  const int mi = item / g.n_tiles_n;
  it.nt = item % g.n_tiles_n;
  const int2 tl = g.tiles[mi];
  it.row0 = tl.x;
  it.e = tl.y;
  it.row_end = g.offsets[it.e + 1];
  it.mt = 0;
  it.krow0 = it.krows = 0;
  it.kblocks = g.kblocks;
  return true;
}

__device__ __forceinline__ int total_items(const GemmArgs& g, int mode) {
  if (mode == WG2 || mode == WG13) return g.E * g.n_tiles_m * g.n_tiles_n;
  if (mode == GATE) return g.n_tiles_m * g.n_tiles_n * (g.ksplit > 1 ? g.ksplit : 1);
  return (*g.tile_count) * g.n_tiles_n;
}

__device__ __forceinline__ float silu_f(float a) { return a / (1.f + expf(-a)); }

__device__ __forceinline__ void store_bf16x16(uint16_t* dst, const float* v, int ncols_left) {
  // ncols_left: columns still inside the row (multiple of 8)
  if (ncols_left >= 8) reinterpret_cast<uint4*>(dst)[0] = pack8(v);
  if (ncols_left >= 16) reinterpret_cast<uint4*>(dst)[1] = pack8(v + 8);
}

template <int MODE, bool C2>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmC2, const __grid_constant__ CUtensorMap tmC3,
                    const __grid_constant__ GemmArgs g) {
  using Tr = Traits<MODE, C2>;
  static_assert(Tr::stages <= MAX_STAGES, "stages");
  static_assert(!C2 || (!Tr::pair && !Tr::partials), "CTA pairs: 256-row modes only");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t tile_base = (raw_addr + 1023u) & ~1023u;       // 1024-B aligned stages
  uint8_t* tile_ptr = smem_raw + (tile_base - raw_addr);
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(tile_ptr + Tr::stages * Tr::stage_bytes + Tr::epi_bytes);
  static_assert(sizeof(SharedCtl) <= CTL_BYTES, "control block");
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // C2: rank 0 of the pair issues the MMAs; both CTAs walk the same items.
  const uint32_t rank = C2 ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  const int first_item = C2 ? (int)cluster_index() : (int)blockIdx.x;
  const int item_step = C2 ? (int)cluster_count() : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Tr::stages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&ctl->tfull[a]), 1);
      mbar_init(smem_u32(&ctl->tempty[a]), C2 ? 2 * EPI_WARPS : EPI_WARPS);
    }
    mbar_init(smem_u32(&ctl->mma_done), 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (Tr::is_gateup || MODE == DX) tma_prefetch_desc(&tmB2);
    if (MODE != GATE) tma_prefetch_desc(&tmC);
    if (MODE == WG13 || Tr::is_gateup) tma_prefetch_desc(&tmC2);
    if (Tr::is_gateup) tma_prefetch_desc(&tmC3);
  }
  if (warp == 1) {
    if (C2) {
      tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (C2) cluster_sync_all();   // both CTAs' barriers and tensor memory are ready
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  const int total = total_items(g, MODE);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it_count = 0;   // k-blocks issued so far (all items)
      bool ok = true;
      // C2: this CTA's loads land in its own shared memory and signal rank 0's barrier
      auto ld2 = [&](uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y) {
        if (C2) tma_load_2d_pair(dst, m, bar, x, y);
        else tma_load_2d(dst, m, bar, x, y);
      };
      auto ld4 = [&](uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y, int z, int w) {
        if (C2) tma_load_4d_pair(dst, m, bar, x, y, z, w);
        else tma_load_4d(dst, m, bar, x, y, z, w);
      };
      const int rrow = (int)rank * BM;        // this CTA's rows of a 256-row tile
      const int rcol = (int)rank * (BN / 2);  // this CTA's half of the B columns
      const CUtensorMap* emaps = static_cast<const CUtensorMap*>(g.emaps);
      int acquired_e = -1;   // weight gradients: the expert whose maps this thread acquired
      for (int item = first_item; item < total && ok; item += item_step) {
        Item it;
        decode_item(g, MODE, item, it);
        if (Tr::wgrad && (it.krows % BK) != 0 && it.e != acquired_e) {
          // the expert's own maps (written by an earlier kernel), fetched ahead
          // of the item's last k-block
          tensormap_acquire(emaps + 2 * it.e);
          tensormap_acquire(emaps + 2 * it.e + 1);
          tma_prefetch_desc(emaps + 2 * it.e);
          tma_prefetch_desc(emaps + 2 * it.e + 1);
          acquired_e = it.e;
        }
        for (int kb = 0; kb < it.kblocks; ++kb, ++it_count) {
          const int s = it_count % Tr::stages;
          const uint32_t ph = (it_count / Tr::stages) & 1u;
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, g.err)) {
            ok = false;
            break;
          }
          const uint32_t bar_local = smem_u32(&ctl->full[s]);
          const uint32_t bar = C2 ? mapa_shared(bar_local, 0) : bar_local;
          const uint32_t sa = tile_base + s * Tr::stage_bytes;
          const uint32_t sb = sa + Tr::a_bytes;
          if (leader) mbar_arrive_expect_tx(bar_local, Tr::stage_tx);
          const int kx = (it.kb0 + kb * it.kstep) * BK;
          if (Tr::pair) tma_load_2d(sa + A_BYTES, &tmA, bar, kx, it.row0 + BM);   // rows 128-255
          if (Tr::is_gateup) {
            ld2(sa, &tmA, bar, kx, it.row0 + rrow);
            // B = [W1 rows; W3 rows] of the column tile (C2: rank 0 W1, rank 1 W3)
            if (g.prepacked) {   // one contiguous 16 KB tile per box
              const int rt = it.e * (g.f / 128) + it.nt;
              if (C2) {
                ld4(sb, rank ? &tmB2 : &tmB, bar, 0, 0, kb, rt);
              } else {
                tma_load_4d(sb, &tmB, bar, 0, 0, kb, rt);
                tma_load_4d(sb + B_BYTES / 2, &tmB2, bar, 0, 0, kb, rt);
              }
            } else {
              const int brow = it.e * g.f + it.nt * 128;
              if (C2) {
                ld2(sb, rank ? &tmB2 : &tmB, bar, kx, brow);
              } else {
                tma_load_2d(sb, &tmB, bar, kx, brow);
                tma_load_2d(sb + B_BYTES / 2, &tmB2, bar, kx, brow);
              }
            }
          } else if (MODE == GATE) {
            // x's k-block, then W_g's hi, mid and lo terms of it (thirds of B's K)
            tma_load_2d(sa, &tmA, bar, kx, it.row0);
#pragma unroll
            for (int t = 0; t < 3; ++t)
              tma_load_2d(sb + t * 128 * BK * 2, &tmB, bar, t * g.d + kx, it.nt * Tr::bn);
          } else if (Tr::is_down) {
            ld2(sa, &tmA, bar, kx, it.row0 + rrow);
            if (g.prepacked) {   // one contiguous 32 KB tile (C2: each CTA its 128 rows)
              const int rt = it.e * (g.d / BN) + it.nt;
              ld4(sb, &tmB, bar, 0, rcol, kb, rt);
            } else {
              ld2(sb, &tmB, bar, kx, it.e * g.d + it.nt * BN + rcol);
            }
          } else if (MODE == DH) {
            ld2(sa, &tmA, bar, kx, it.row0 + rrow);
#pragma unroll
            for (int j = 0; j < Tr::b_bytes / ATOM_BYTES; ++j)
              ld2(sb + j * ATOM_BYTES, &tmB, bar, it.nt * BN + rcol + j * 64, it.e * g.d + kx);
          } else if (MODE == DX) {
            ld2(sa, &tmA, bar, kx, it.row0 + rrow);
            const bool first = kx < g.f;
            const int krow = it.e * g.f + (first ? kx : kx - g.f);
#pragma unroll
            for (int j = 0; j < Tr::b_bytes / ATOM_BYTES; ++j)
              ld2(sb + j * ATOM_BYTES, first ? &tmB : &tmB2, bar, it.nt * BN + rcol + j * 64, krow);
          } else {  // WG2 / WG13: both operands MN-major, K = rows of expert e
            const int krow = it.krow0 + kx;
            // the last k-block of an expert whose rows end inside it: the
            // expert's maps end at its last row, so the TMA fills the rest of
            // the box with zeros (the full box's bytes still arrive)
            const bool last = it.krows - kx < BK;
            const CUtensorMap* mA = last ? emaps + 2 * it.e : &tmA;
            const CUtensorMap* mB = last ? emaps + 2 * it.e + 1 : &tmB;
#pragma unroll
            for (int j = 0; j < 2; ++j)
              ld2(sa + j * ATOM_BYTES, mA, bar, it.mt * Tr::tile_m + rrow + j * 64, krow);
#pragma unroll
            for (int j = 0; j < Tr::b_bytes / ATOM_BYTES; ++j)
              ld2(sb + j * ATOM_BYTES, mB, bar, it.nt * BN + rcol + j * 64, krow);
          }
        }
      }
      if (!ok && C2) {
        // The pair's loads signal rank 0's barriers, which this CTA cannot
        // observe: give any load still in flight time to land (tens of us).
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 200000ull) {
        }
      } else if (!ok) {
        // drain: the last (up to STAGES) issued loads must land before the CTA exits
        const uint32_t n = it_count < (uint32_t)Tr::stages ? it_count : (uint32_t)Tr::stages;
        for (uint32_t q = 0; q < n; ++q) {
          const uint32_t c = it_count - 1 - q;
          volatile int never = 0;
          mbar_wait_bounded(smem_u32(&ctl->full[c % Tr::stages]), (c / Tr::stages) & 1u, &never,
                            nullptr);
        }
      }
    }
  } else if (warp == 1 && leader) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16(Tr::tile_m, Tr::bn, Tr::a_mn, Tr::b_mn);
    uint32_t it_count = 0;
    int j = 0;
    bool ok = true;
    bool issued_any = false;
    for (int item = first_item; item < total && ok; item += item_step, ++j) {
      Item it;
      decode_item(g, MODE, item, it);
      const int acc = Tr::single_acc ? 0 : (j & 1);
      const uint32_t aph = Tr::single_acc ? (j & 1u) : ((j >> 1) & 1u);
      // C2: both CTAs' epilogues arrive on this barrier
      ok = C2 ? mbar_wait_bounded_cluster(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort_flag, g.err)
              : mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort_flag, g.err);
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_base = tmem_base + acc * BN;
      for (int kb = 0; kb < it.kblocks; ++kb, ++it_count) {
        const int s = it_count % Tr::stages;
        const uint32_t ph = (it_count / Tr::stages) & 1u;
        ok = mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag, g.err);
        ok = __all_sync(kFull, ok);
        if (!ok) break;
        const uint32_t sa = tile_base + s * Tr::stage_bytes;
        const uint32_t sb = sa + Tr::a_bytes;
        int kk_end = BK / 16;
        if (Tr::wgrad) {
          // An expert's last K-block: MMAs only for the 16-row groups that
          // hold its rows (the rows past its end were loaded as zeros).
          const int rem = it.krows - kb * BK;
          if (rem < BK) kk_end = ceil_div(rem, 16);
        }
        const int kbg = it.kb0 + kb * it.kstep;   // the k-block's index in K
        const uint32_t d_tmem = Tr::partials ? tmem_base + (kbg & 3) * 128 : d_base;
        const bool first = Tr::partials ? kbg < 4 : kb == 0;
        auto issue = [&](int kk0, int kk1) {   // 16-deep K groups kk0 .. kk1-1 (one lane)
          if constexpr (Tr::partials) {   // the three W_g terms against the same x block
#pragma unroll
            for (int t = 0; t < 3; ++t)
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                tc_mma_bf16(d_tmem, smem_desc_sw128(sa + kk * 32, 16, 1024),
                            smem_desc_sw128(sb + t * 128 * BK * 2 + kk * 32, 16, 1024), idesc,
                            (!first || t > 0 || kk > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              if (kk < kk0) continue;
              if (kk >= kk1) break;
              const uint64_t ad = Tr::a_mn ? smem_desc_sw128(sa + kk * 2048, ATOM_BYTES, 1024)
                                           : smem_desc_sw128(sa + kk * 32, 16, 1024);
              const uint64_t bd = Tr::b_mn ? smem_desc_sw128(sb + kk * 2048, ATOM_BYTES, 1024)
                                           : smem_desc_sw128(sb + kk * 32, 16, 1024);
              if (C2) tc_mma_bf16_pair(d_tmem, ad, bd, idesc, (!first || kk > 0) ? 1u : 0u);
              else tc_mma_bf16(d_tmem, ad, bd, idesc, (!first || kk > 0) ? 1u : 0u);
              if (Tr::pair && it.row_end - it.row0 > BM)   // rows 128-255 share the B stage
                tc_mma_bf16(tmem_base + BN, smem_desc_sw128(sa + A_BYTES + kk * 32, 16, 1024),
                            bd, idesc, (!first || kk > 0) ? 1u : 0u);
            }
          }
        };
        if (lane == 0) {
          tc_fence_after();
          issue(0, kk_end);
          issued_any = true;
          // frees the stage (C2: in both CTAs) when these MMAs finish
          if (C2) tc_commit_pair(smem_u32(&ctl->empty[s]), 3);
          else tc_commit(smem_u32(&ctl->empty[s]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) {
        const uint32_t tf = smem_u32(&ctl->tfull[acc]);
        if (it.kblocks > 0) {
          if (C2) tc_commit_pair(tf, 3);
          else tc_commit(tf);
        } else {
          mbar_arrive(tf);
          if (C2) mbar_arrive_cluster(mapa_shared(tf, 1));
        }
      }
      __syncwarp();
    }
    // drain outstanding MMAs before TMEM is released
    if (lane == 0 && issued_any) {
      if (C2) tc_commit_pair(smem_u32(&ctl->mma_done), 1);
      else tc_commit(smem_u32(&ctl->mma_done));
      volatile int never = 0;
      mbar_wait_bounded(smem_u32(&ctl->mma_done), 0, &never, nullptr);
    }
    __syncwarp();
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quadrant this warp may access
    const int r_local = q * 32 + lane;   // accumulator row owned by this thread
    const int half = (warp - 2) >> 2;    // which half of the tile's columns this warp drains
    const int rrow = (int)rank * BM;     // C2: this CTA's rows of the 256-row tile
    // This warp's staging box: 32 rows (its TMEM lanes) x 128 B, 128-B swizzled
    // (16-B chunk j of row r at r * 128 + (j ^ (r & 7)) * 16), written by the
    // warp and sent to global memory by one bulk tensor store.
    const uint32_t sbox = tile_base + Tr::stages * Tr::stage_bytes + (warp - 2) * EPI_WARP_BYTES;
    uint8_t* sbox_row = tile_ptr + Tr::stages * Tr::stage_bytes + (warp - 2) * EPI_WARP_BYTES +
                        lane * 128;
    auto stage_begin = [&]() {   // the box is free once its previous store has read it
      if (lane == 0) bulk_wait_read_0();
      __syncwarp();
    };
    auto stage_put = [&](int j, uint4 v) {   // 16-B chunk j (8 bf16) of this lane's row
      *reinterpret_cast<uint4*>(sbox_row + ((j ^ (lane & 7)) * 16)) = v;
    };
    auto stage_end = [&](const CUtensorMap* m, int x, int y) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(m, sbox, x, y);
        bulk_commit();
      }
    };
    int j = 0;
    for (int item = first_item; item < total; item += item_step, ++j) {
      Item it;
      decode_item(g, MODE, item, it);
      const int acc = Tr::single_acc ? 0 : (j & 1);
      const uint32_t aph = Tr::single_acc ? (j & 1u) : ((j >> 1) & 1u);
      bool ok = mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), aph, abort_flag, g.err);
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      for (int hh = 0; hh < (Tr::pair ? 2 : 1); ++hh) {   // row halves of a 256-row item
      if (hh == 1 && it.row_end - it.row0 <= BM) break;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + hh * BN;
      const int grow0 = it.row0 + rrow + hh * BM + q * 32;   // this warp's first row
      // Whole 32-row groups of the expert go out as staged boxes; the group
      // holding the expert's last row (the next expert's rows follow it) is
      // written row by row.
      const bool boxed = grow0 + 32 <= it.row_end;
      if (Tr::is_gateup && boxed) {
        // h, then the saved a and b: 64 columns of this warp's 32 rows each
        const int c0 = half * 64;
        const int col0 = it.nt * 128 + c0;
        const int nout = g.save_a ? 3 : 1;
        for (int o = 0; o < nout && col0 < g.f; ++o) {
          stage_begin();
#pragma unroll 1
          for (int k = 0; k < 4; ++k) {
            float a[16], b[16];
            if (o != 2) tmem_ld16(t_row + c0 + 16 * k, a);
            if (o != 1) tmem_ld16(t_row + 128 + c0 + 16 * k, b);
            tmem_ld_wait();
            if (o == 0) {
#pragma unroll
              for (int u = 0; u < 16; ++u) a[u] = silu_f(a[u]) * b[u];
            }
            if (o == 2) {
              stage_put(2 * k, pack8(b));
              stage_put(2 * k + 1, pack8(b + 8));
            } else {
              stage_put(2 * k, pack8(a));
              stage_put(2 * k + 1, pack8(a + 8));
            }
          }
          stage_end(o == 0 ? &tmC : (o == 1 ? &tmC2 : &tmC3), col0, grow0);
        }
      } else if (Tr::is_gateup) {
        const int row = it.row0 + rrow + hh * BM + r_local;
        const bool valid = row < it.row_end;
        for (int c = half * 64; c < half * 64 + 64 && grow0 < it.row_end; c += 16) {
          float a[16], b[16];
          tmem_ld16(t_row + c, a);
          tmem_ld16(t_row + 128 + c, b);
          tmem_ld_wait();
          const int col = it.nt * 128 + c;
          if (valid && col < g.f) {
            float h[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) h[u] = silu_f(a[u]) * b[u];
            const size_t off = (size_t)row * g.f + col;
            store_bf16x16(g.out_bf16 + off, h, g.f - col);
            if (g.save_a) {
              store_bf16x16(g.save_a + off, a, g.f - col);
              store_bf16x16(g.save_b + off, b, g.f - col);
            }
          }
        }
      } else if (MODE == GATE && g.ksplit > 1) {
        // this CTA's partial accumulator (k-blocks kb0 (mod 4)) as it is; a
        // second kernel adds the four partials in order, with the bias
        const int row = it.row0 + r_local;
        const bool valid = row < it.row_end;
        for (int c = half * 64; c < half * 64 + 64; c += 16) {
          float v[16];
          tmem_ld16(t_row + it.kb0 * 128 + c, v);
          tmem_ld_wait();
          const int col = it.nt * 128 + c;
          if (valid && col < g.E) {
            float* dst = g.out_parts + ((size_t)it.kb0 * g.N + row) * g.E + col;
            const int n = g.E - col < 16 ? g.E - col : 16;
            for (int u = 0; u < n; ++u) dst[u] = v[u];
          }
        }
      } else if (MODE == GATE) {
        const int row = it.row0 + r_local;
        const bool valid = row < it.row_end;
        const int parts = it.kblocks < 4 ? it.kblocks : 4;
        for (int c = half * 64; c < half * 64 + 64; c += 16) {
          float v[16];
          tmem_ld16(t_row + c, v);
          tmem_ld_wait();
          for (int p = 1; p < parts; ++p) {
            float w[16];
            tmem_ld16(t_row + p * 128 + c, w);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] += w[u];
          }
          const int col = it.nt * 128 + c;
          if (valid && col < g.E) {
            float* dst = g.out_f32 + (size_t)row * g.E + col;
            const int n = g.E - col < 16 ? g.E - col : 16;
            for (int u = 0; u < n; ++u) dst[u] = v[u] + (g.bias ? g.bias[col + u] : 0.f);
          }
        }
      } else if ((Tr::is_down || MODE == DX) && boxed) {
        for (int bx = 0; bx < 2; ++bx) {   // two boxes of 64 columns
          const int c0 = half * (BN / 2) + bx * 64;
          const int col0 = it.nt * BN + c0;
          if (col0 >= g.d) break;
          float v[64];
#pragma unroll
          for (int k = 0; k < 4; ++k) tmem_ld16(t_row + c0 + 16 * k, v + 16 * k);
          tmem_ld_wait();
          if (Tr::is_down && g.row_scale) {   // this lane's row's scale, before rounding
            const float sc = g.row_scale[grow0 + lane];
#pragma unroll
            for (int u = 0; u < 64; ++u) v[u] *= sc;
          }
          stage_begin();
#pragma unroll
          for (int k = 0; k < 8; ++k) stage_put(k, pack8(v + 8 * k));
          stage_end(&tmC, col0, grow0);
        }
      } else if (Tr::is_down || MODE == DX) {
        const int row = it.row0 + rrow + hh * BM + r_local;
        const bool valid = row < it.row_end;
        for (int c = half * (BN / 2); c < (half + 1) * (BN / 2) && grow0 < it.row_end; c += 16) {
          float v[16];
          tmem_ld16(t_row + c, v);
          tmem_ld_wait();
          const int col = it.nt * BN + c;
          if (valid && col < g.d) {
            if (Tr::is_down && g.row_scale) {
              const float sc = g.row_scale[row];
#pragma unroll
              for (int u = 0; u < 16; ++u) v[u] *= sc;
            }
            store_bf16x16(g.out_bf16 + (size_t)row * g.d + col, v, g.d - col);
          }
        }
      } else if (MODE == DH) {
        const int row = it.row0 + rrow + r_local;
        const bool valid = row < it.row_end;
        const uint16_t* pa = g.in_a + (size_t)row * g.f;
        const uint16_t* pb = g.in_b + (size_t)row * g.f;
        // saved a, b for a 16-column chunk (zeros past the row's end)
        auto load_ab = [&](int c, uint4* a4, uint4* b4) {
          const int col = it.nt * BN + c;
          const uint4 z = make_uint4(0, 0, 0, 0);
          a4[0] = a4[1] = b4[0] = b4[1] = z;
          if (valid && col < g.f) {
            a4[0] = ldg_nc_v4(pa + col);
            b4[0] = ldg_nc_v4(pb + col);
            if (g.f - col >= 16) {
              a4[1] = ldg_nc_v4(pa + col + 8);
              b4[1] = ldg_nc_v4(pb + col + 8);
            }
          }
        };
        uint4 na[2], nb[2];
        auto dadb = [&](const float* dh, const uint4* ca, const uint4* cb, float* da, float* db) {
          float a[16], b[16];
          unpack8(ca[0], a);
          unpack8(ca[1], a + 8);
          unpack8(cb[0], b);
          unpack8(cb[1], b + 8);
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const float sg = 1.f / (1.f + expf(-a[u]));
            da[u] = dh[u] * b[u] * (sg * (1.f + a[u] * (1.f - sg)));
            db[u] = dh[u] * a[u] * sg;
          }
        };
        if (boxed) {
          // f % 64 == 0: a 64-column box lies wholly inside da (or db)
          for (int bx = 0; bx < 2; ++bx) {
            const int c0 = half * (BN / 2) + bx * 64;
            const int col0 = it.nt * BN + c0;
            if (col0 >= g.f) break;
            uint4 dbp[8];   // this box's db, packed, while da's box is stored
            load_ab(c0, na, nb);
            stage_begin();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint4 ca[2] = {na[0], na[1]}, cb[2] = {nb[0], nb[1]};
              if (k < 3) load_ab(c0 + 16 * (k + 1), na, nb);
              float dh[16], da[16], db[16];
              tmem_ld16(t_row + c0 + 16 * k, dh);
              tmem_ld_wait();
              dadb(dh, ca, cb, da, db);
              stage_put(2 * k, pack8(da));
              stage_put(2 * k + 1, pack8(da + 8));
              dbp[2 * k] = pack8(db);
              dbp[2 * k + 1] = pack8(db + 8);
            }
            stage_end(&tmC, col0, grow0);
            stage_begin();
#pragma unroll
            for (int k = 0; k < 8; ++k) stage_put(k, dbp[k]);
            stage_end(&tmC, g.f + col0, grow0);
          }
        }
        const int c0 = half * (BN / 2), c1 = boxed ? c0 : c0 + BN / 2;
        if (c0 < c1) load_ab(c0, na, nb);  // the next chunk's loads are in flight while this one computes
        for (int c = c0; c < c1; c += 16) {
          uint4 ca[2] = {na[0], na[1]}, cb[2] = {nb[0], nb[1]};
          if (c + 16 < c1) load_ab(c + 16, na, nb);
          float dh[16];
          tmem_ld16(t_row + c, dh);
          tmem_ld_wait();
          const int col = it.nt * BN + c;
          if (valid && col < g.f) {
            float da[16], db[16];
            dadb(dh, ca, cb, da, db);
            const size_t o2 = (size_t)row * (2 * g.f) + col;
            store_bf16x16(g.out_bf16 + o2, da, g.f - col);
            store_bf16x16(g.out_bf16 + o2 + g.f, db, g.f - col);
          }
        }
      } else {  // WG2 / WG13: fp32 weight gradients
        // This warp owns output rows m0 .. m0+31 of expert e and half of the
        // columns.  Each 32-column chunk goes TMEM -> registers -> (pairs) each
        // lane's 128 contiguous bytes of its row by plain 16-byte stores, or (one
        // CTA) a 128-B-swizzled 32x32 fp32 box in shared memory -> one bulk
        // tensor store.
        const int m0 = it.mt * Tr::tile_m + rrow + q * 32;
        const int mrows = (MODE == WG2) ? g.d : 2 * g.f;
        const int ncols = (MODE == WG2) ? g.f : g.d;
        const CUtensorMap* map = &tmC;
        int mrow = m0;
        if (MODE == WG13 && m0 >= g.f) {
          map = &tmC2;
          mrow = m0 - g.f;
        }
        const uint32_t box = tile_base + Tr::stages * Tr::stage_bytes + (warp - 2) * EPI_WARP_BYTES;
        uint8_t* box_ptr = tile_ptr + Tr::stages * Tr::stage_bytes + (warp - 2) * EPI_WARP_BYTES;
        for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32) {
          float v[32];
          if (it.kblocks > 0) {
            tmem_ld16(t_row + c, v);
            tmem_ld16(t_row + c + 16, v + 16);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int u = 0; u < 32; ++u) v[u] = 0.f;
          }
          const int col = it.nt * BN + c;
          if (m0 >= mrows || col >= ncols) continue;          // warp-uniform
          if (C2) {   // pairs: the lane's 32 values straight to its output row
            float* base = (MODE == WG13 && m0 >= g.f) ? g.out_f32b : g.out_f32;
            const int rows_e = (MODE == WG2) ? g.d : g.f;
            float* dst = base + ((size_t)it.e * rows_e + mrow + lane) * ncols + col;
            // a row starts 256-B aligned relative to base (ncols % 64 == 0), so
            // base's alignment decides, uniformly: whole 32-byte sectors when it
            // allows (twice fewer, full-sector L2 writes), else 16-byte stores
            if ((reinterpret_cast<uintptr_t>(base) & 31u) == 0) {
#pragma unroll
              for (int q8 = 0; q8 < 4; ++q8) st_global_v8(dst + 8 * q8, v + 8 * q8);
            } else {
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4)
                reinterpret_cast<float4*>(dst)[q4] =
                    make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
            }
            continue;
          }
          if (lane == 0) bulk_wait_read_0();                  // the box's last store has read it
          __syncwarp();
          uint8_t* bp = box_ptr;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const int phys = lane * 128 + ((ch ^ (lane & 7)) * 16);
            *reinterpret_cast<float4*>(bp + phys) =
                make_float4(v[4 * ch], v[4 * ch + 1], v[4 * ch + 2], v[4 * ch + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(map, box, col, mrow, it.e);
            bulk_commit();
          }
        }
      }
      }  // row halves
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t te = smem_u32(&ctl->tempty[acc]);
        if (C2 && !leader) mbar_arrive_cluster(mapa_shared(te, 0));
        else mbar_arrive(te);
      }
    }
    if (MODE != GATE) {
      if (lane == 0) bulk_wait_all();   // stores done before the CTA's shared memory goes away
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (C2) cluster_sync_all();   // the pair's MMAs, loads and remote arrivals are over
  if (warp == 1) {
    tc_fence_after();
    if (C2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Weight prepacking: W [E * rows_per_e, K] row-major -> tiles
// [E * rows_per_e / TR][K / 64][TR][64]; each (row tile, k-block) box of the
// forward GEMMs becomes one contiguous TR * 128-byte region.  One thread moves
// 16 bytes (8 bf16).
__global__ void prepack_kernel(const uint16_t* __restrict__ W, long long rows, int K, int TR,
                               uint16_t* __restrict__ Wp) {
  const long long chunks = rows * (K / 8);
  const int kb_n = K / 64;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < chunks;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / (K / 8);
    const int c8 = (int)(i % (K / 8));          // 16-byte chunk within the row
    const int kb = c8 / 8, cin = c8 % 8;
    const long long rt = r / TR;
    const int rin = (int)(r % TR);
    const size_t dst = (((size_t)rt * kb_n + kb) * TR + rin) * 64 + (size_t)cin * 8;
    reinterpret_cast<uint4*>(Wp)[dst / 8] = reinterpret_cast<const uint4*>(W)[i];
  }
}

// Per-expert operand maps of the weight-gradient GEMMs.  Thread i writes map
// i % 4 of expert e = i / 4: a copy of tmpl.m[i % 4] whose row extent (outer
// dimension) ends at the expert's last row offsets[e + 1], so that a box
// reaching past that row reads zeros.  Maps 0, 1 (WG2's A and B) go to
// out[2e], out[2e + 1]; maps 2, 3 (WG13's) to out[2E + 2e], out[2E + 2e + 1].
struct MapTemplates {
  CUtensorMap m[4];
};

__global__ void __launch_bounds__(256) expert_maps_kernel(const __grid_constant__ MapTemplates tmpl,
                                                          const int32_t* __restrict__ offsets,
                                                          int E, CUtensorMap* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 4 * E) return;
  const int e = i >> 2, m = i & 3;
  CUtensorMap* dst = out + (m >> 1) * 2 * E + 2 * e + (m & 1);
  const uint4* src = reinterpret_cast<const uint4*>(&tmpl.m[m]);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int k = 0; k < (int)(sizeof(CUtensorMap) / sizeof(uint4)); ++k) d4[k] = src[k];
  const int end = offsets[e + 1];
  tensormap_set_dim1(dst, end > 0 ? end : 1);   // (an empty leading expert's map is never used)
  tensormap_release();
}

// Exclusive prefix sum of v over the block's 1024 threads; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
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
    warp_sums[lane] = ws;
  }
  __syncthreads();
  const int excl = (wid > 0 ? warp_sums[wid - 1] : 0) + incl - v;
  *total = warp_sums[31];
  __syncthreads();
  return excl;
}

// Ragged M tiles: expert e's rows [offsets[e], offsets[e+1]) split into
// tile_rows-row tiles (128, or 256 for CTA pairs and the paired modes);
// tiles[i] = {first row, expert}, ordered by expert then row.  With
// tail_rows > 0, an expert's last tile goes to the second list `tails`
// instead when it holds at most tail_rows rows (the single-CTA kernels run
// those tiles: on a pair the other CTA would load and multiply a whole tile
// of rows that are not the expert's).
__global__ void __launch_bounds__(1024) build_tiles_kernel(const int32_t* __restrict__ offsets,
                                                           int E, int tile_rows, int tail_rows,
                                                           int2* __restrict__ tiles,
                                                           int32_t* __restrict__ tile_count,
                                                           int2* __restrict__ tails,
                                                           int32_t* __restrict__ tail_count) {
  __shared__ int warp_sums[32];
  int carry = 0, carry_t = 0;
  for (int e0 = 0; e0 < E; e0 += 1024) {
    const int e = e0 + threadIdx.x;
    int r0 = 0, n = 0, nt = 0;
    if (e < E) {
      r0 = offsets[e];
      const int rows = offsets[e + 1] - r0;
      n = ceil_div(rows, tile_rows);
      const int rem = rows % tile_rows;
      if (tail_rows > 0 && rem > 0 && rem <= tail_rows) {
        n -= 1;
        nt = 1;
      }
    }
    int tot = 0, tot_t = 0;
    const int start = carry + block_exclusive_scan(n, warp_sums, &tot);
    const int start_t = carry_t + block_exclusive_scan(nt, warp_sums, &tot_t);
    for (int i = 0; i < n; ++i) tiles[start + i] = make_int2(r0 + i * tile_rows, e);
    if (nt) tails[start_t] = make_int2(r0 + n * tile_rows, e);
    carry += tot;
    carry_t += tot_t;
  }
  if (threadIdx.x == 0) {
    *tile_count = carry;
    if (tail_count) *tail_count = carry_t;
  }
}
}  // namespace

// ------------------------------------------------------------------ host side
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// bf16 matrix [rows, cols] (row pitch = cols elements), box {64 cols, box_rows}, 128-B swizzle.
bool make_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [E, rows, cols] (dense), box {32 cols, 32 rows, 1}, 128-B swizzle: output
// of the weight-gradient epilogue's bulk tensor stores.
bool make_map_f32_3d(CUtensorMap* m, void* base, long long E, long long rows, long long cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)E};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)rows * cols * 4};
  cuuint32_t box[3] = {32u, 32u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Prepacked weight tiles [tiles][kb][rows][64] viewed 4-D: {64, rows, kblocks, tiles};
// a box is box_rows rows of one tile's k-block (all of them by default).
bool make_map_tiles(CUtensorMap* m, const void* base, long long tiles, long long kblocks,
                    int rows, int box_rows = 0) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)kblocks, (cuuint64_t)tiles};
  cuuint64_t strides[3] = {128, (cuuint64_t)rows * 128, (cuuint64_t)kblocks * rows * 128};
  cuuint32_t box[4] = {64u, (cuuint32_t)(box_rows > 0 ? box_rows : rows), 1u, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_map_2d(void* map, int dtype, const void* base, unsigned long long inner,
                   unsigned long long outer, unsigned long long row_bytes, unsigned box_inner,
                   unsigned box_outer, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(static_cast<CUtensorMap*>(map), static_cast<CUtensorMapDataType>(dtype), 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
int sm_count() {
  static int n[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (n[dev] == 0) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev] > 0 ? n[dev] : 148;
}

template <int MODE, bool C2 = false>
cudaError_t launch_mode(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2,
                        const CUtensorMap& c, const CUtensorMap& c2, const CUtensorMap& c3,
                        const GemmArgs& g, long long max_items, cudaStream_t s) {
  constexpr int SMEM_BYTES = Traits<MODE, C2>::smem_bytes;
  auto kernel = grouped_gemm_kernel<MODE, C2>;
  static bool attr_done[64] = {false};
  static int pair_slots[64] = {0};   // C2: clusters of two that fit on the GPU at once
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  if (C2) {
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (!attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (C2) {
      cfg.gridDim = dim3(2 * (sm_count() / 2));
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
      if (e != cudaSuccess) return e;
      if (n <= 0) return cudaErrorInvalidConfiguration;
      pair_slots[dev] = n;
    }
    attr_done[dev] = true;
  }
  if (max_items <= 0) return cudaSuccess;
  const long long ctas = C2 ? 2 * std::min<long long>(pair_slots[dev], max_items)
                            : std::min<long long>(sm_count(), max_items);
  cfg.gridDim = dim3((unsigned)ctas);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a, b, b2, c, c2, c3, g);
  count_launches(1);
  return e;
}
}  // namespace

bool gate_tc_supported(int d) { return d % 64 == 0; }

namespace {
// The gate splits each tile's K over four CTAs (one per partial accumulator)
// when the tiles alone would leave most SMs idle: at most 38 tiles (152 / 4)
// and at least four k-blocks.
bool gate_split(int T, int d, int E) {
  const int tiles = ceil_div(T, BM) * ceil_div(E, 128);
  return tiles * 4 <= 152 && d / BK >= 4;
}

// logits = ((P0 + P1) + P2) + P3 + bias, fp32, the order of the one-CTA epilogue
__global__ void gate_sum_kernel(const float* __restrict__ parts, const float* __restrict__ bias,
                                int T, int E, float* __restrict__ logits) {
  const long long n = (long long)T * E;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    float v = parts[i];
#pragma unroll
    for (int p = 1; p < 4; ++p) v += parts[p * n + i];
    logits[i] = v + (bias ? bias[i % E] : 0.f);
  }
}
}  // namespace

size_t gate_tc_ws_bytes(int T, int d, int E) {
  return align_up((size_t)E * 3 * d * 2, 256) +
         (gate_split(T, d, E) ? align_up((size_t)4 * T * E * 4, 256) : 0);
}

cudaError_t launch_gate_tc(const uint16_t* x, const float* wg, const float* bias, int T, int d,
                           int E, float* logits, void* ws, int* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  uint16_t* wgs = static_cast<uint16_t*>(ws);
  const bool split = gate_split(T, d, E);
  float* parts = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                          align_up((size_t)E * 3 * d * 2, 256));
  cudaError_t e = launch_wg_split(wg, d, E, wgs, s);
  if (e != cudaSuccess) return e;
  CUtensorMap ma, mb;
  if (!make_map(&ma, x, T, d, BM) || !make_map(&mb, wgs, E, 3LL * d, 128))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = E; g.N = T; g.d = d; g.f = 0;
  g.kblocks = d / BK;
  g.n_tiles_m = ceil_div(T, BM);
  g.n_tiles_n = ceil_div(E, 128);
  g.out_f32 = logits;
  g.bias = bias;
  g.err = err;
  g.ksplit = split ? 4 : 1;
  g.out_parts = parts;
  e = launch_mode<GATE>(ma, mb, mb, ma, ma, ma, g,
                        (long long)g.n_tiles_m * g.n_tiles_n * g.ksplit, s);
  if (e != cudaSuccess || !split) return e;
  const long long n = (long long)T * E;
  gate_sum_kernel<<<(int)std::min<long long>((n + 255) / 256, 152 * 8), 256, 0, s>>>(
      parts, bias, T, E, logits);
  count_launches(1);
  return cudaGetLastError();
}

bool prepack_supported(int d, int f) { return d % BN == 0 && f % 128 == 0; }

cudaError_t launch_prepack(const uint16_t* W1, const uint16_t* W3, const uint16_t* W2, int E,
                           int d, int f, uint16_t* W1p, uint16_t* W3p, uint16_t* W2p,
                           cudaStream_t s) {
  const int blocks = 152 * 8;
  prepack_kernel<<<blocks, 256, 0, s>>>(W1, (long long)E * f, d, 128, W1p);
  prepack_kernel<<<blocks, 256, 0, s>>>(W3, (long long)E * f, d, 128, W3p);
  prepack_kernel<<<blocks, 256, 0, s>>>(W2, (long long)E * d, f, BN, W2p);
  count_launches(3);
  return cudaGetLastError();
}

// Tile-list workspace: [tile count, tail count | E tail entries | tiles], then
// (128-B aligned) the weight-gradient GEMMs' per-expert maps, 4 per expert.
static size_t tile_list_bytes(int N, int E) {
  return align_up(16 + sizeof(int2) * ((size_t)E + ceil_div(N, BM) + E), 128);
}

size_t tiles_ws_bytes(int N, int E) {
  return align_up(tile_list_bytes(N, E) + 4 * sizeof(CUtensorMap) * (size_t)E, 256);
}

static CUtensorMap* expert_maps(void* ws, int N, int E) {
  return reinterpret_cast<CUtensorMap*>(static_cast<uint8_t*>(ws) + tile_list_bytes(N, E));
}

TileLists tile_lists(void* ws, int E) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  return {reinterpret_cast<const int32_t*>(b), reinterpret_cast<const int2*>(b + 16 + 8 * (size_t)E),
          reinterpret_cast<const int32_t*>(b + 4), reinterpret_cast<const int2*>(b + 16)};
}

cudaError_t launch_build_tiles(const int32_t* offsets, int E, void* ws, cudaStream_t s,
                               int tile_rows, int tail_rows) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  build_tiles_kernel<<<1, 1024, 0, s>>>(offsets, E, tile_rows, tail_rows,
                                        reinterpret_cast<int2*>(b + 16 + 8 * (size_t)E),
                                        reinterpret_cast<int32_t*>(b),
                                        reinterpret_cast<int2*>(b + 16),
                                        reinterpret_cast<int32_t*>(b + 4));
  count_launches(1);
  return cudaGetLastError();
}

// x_perm [N,d] -> h [N,f] (and a, b); h -> out [N,d].
cudaError_t launch_ffn_fwd(const uint16_t* x_perm, const int32_t* offsets, int N, int d, int f,
                           int E, const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                           uint16_t* a_save, uint16_t* b_save, uint16_t* h, uint16_t* out,
                           void* tiles_ws, int* err, bool prepacked, bool cta_pairs,
                           cudaStream_t s, const float* row_scale) {
  if (N == 0) return cudaSuccess;
  // cta_pairs: 256-row tiles on CTA pairs (tcgen05 .cta_group::2).  Otherwise
  // single-CTA tiles; with few rows per expert (on average at most two 128-row
  // tiles) the layer streams weights, so one CTA takes both 128-row halves of
  // a 256-row block to share each weight tile (GATEUP2 / DOWN2).
  const bool pair = !cta_pairs && (long long)N <= 2LL * BM * E;
  const int tile_rows = (pair || cta_pairs) ? 2 * BM : BM;
  // On pairs with few rows per expert (on average at most one 256-row tile),
  // an expert's last tile of at most 128 rows runs on one CTA after the pairs
  // (measured: it pays there; with more rows per expert the extra launch costs
  // more than the tails' second CTA).
  const bool split_tails = cta_pairs && (long long)N <= 2LL * BM * E;
  trace_begin(MOE_STAGE_GATEUP, s);
  cudaError_t e = launch_build_tiles(offsets, E, tiles_ws, s, tile_rows, split_tails ? BM : 0);
  if (e != cudaSuccess) return e;
  const TileLists tl = tile_lists(tiles_ws, E);
  GemmArgs g{};
  g.E = E; g.N = N; g.d = d; g.f = f;
  g.offsets = offsets;
  g.tile_count = tl.count;
  g.tiles = tl.tiles;
  g.err = err;
  GemmArgs gt = g;   // the tails' launch: one CTA per 128-row tile
  auto tails = [&](GemmArgs& gg) {
    gg = g;
    gg.tile_count = tl.tail_count;
    gg.tiles = tl.tails;
    return (long long)E * g.n_tiles_n;
  };
  const long long max_m_tiles = ceil_div(N, tile_rows) + E;
  CUtensorMap ma, mb, mb2;
  // gate-up: A = x_perm, B = W1 / W3 rows (128 per tile each)
  g.prepacked = prepacked ? 1 : 0;

  if (!make_map(&ma, x_perm, N, d, BM)) return cudaErrorInvalidValue;
  if (prepacked ? !(make_map_tiles(&mb, W1, (long long)E * f / 128, d / 64, 128) &&
                    make_map_tiles(&mb2, W3, (long long)E * f / 128, d / 64, 128))
                : !(make_map(&mb, W1, (long long)E * f, d, 128) &&
                    make_map(&mb2, W3, (long long)E * f, d, 128)))
    return cudaErrorInvalidValue;
  g.kblocks = ceil_div(d, BK);
  g.n_tiles_n = ceil_div(f, 128);
  g.out_bf16 = h; g.save_a = a_save; g.save_b = b_save;
  // epilogue outputs, stored in 32-row x 64-column boxes
  CUtensorMap mh, msa, msb;
  if (!make_map(&mh, h, N, f, 32)) return cudaErrorInvalidValue;
  msa = msb = mh;
  if (a_save && !(make_map(&msa, a_save, N, f, 32) && make_map(&msb, b_save, N, f, 32)))
    return cudaErrorInvalidValue;
  const long long items = max_m_tiles * g.n_tiles_n;
  e = cta_pairs ? launch_mode<GATEUP, true>(ma, mb, mb2, mh, msa, msb, g, items, s)
      : pair    ? launch_mode<GATEUP2>(ma, mb, mb2, mh, msa, msb, g, items, s)
                : launch_mode<GATEUP>(ma, mb, mb2, mh, msa, msb, g, items, s);
  if (e == cudaSuccess && split_tails) {
    // one CTA loads a whole 128-row W1 and W3 tile: the same maps as the pairs
    const long long n = tails(gt);
    e = launch_mode<GATEUP>(ma, mb, mb2, mh, msa, msb, gt, n, s);
  }
  trace_end(MOE_STAGE_GATEUP, s);
  if (e != cudaSuccess) return e;
  // down: A = h, B = W2 rows (256 per tile; each CTA of a pair loads 128)
  const int w2_box = cta_pairs ? BN / 2 : BN;
  if (!make_map(&ma, h, N, f, BM)) return cudaErrorInvalidValue;
  if (prepacked ? !make_map_tiles(&mb, W2, (long long)E * d / BN, f / 64, BN, w2_box)
                : !make_map(&mb, W2, (long long)E * d, f, w2_box))
    return cudaErrorInvalidValue;
  g.kblocks = ceil_div(f, BK);
  g.n_tiles_n = ceil_div(d, BN);
  g.out_bf16 = out; g.save_a = g.save_b = nullptr;
  g.row_scale = row_scale;
  CUtensorMap mo;
  if (!make_map(&mo, out, N, d, 32)) return cudaErrorInvalidValue;

  trace_begin(MOE_STAGE_DOWN, s);
  const long long items_down = max_m_tiles * g.n_tiles_n;
  e = cta_pairs ? launch_mode<DOWN, true>(ma, mb, mb, mo, mo, mo, g, items_down, s)
      : pair    ? launch_mode<DOWN2>(ma, mb, mb, mo, mo, mo, g, items_down, s)
                : launch_mode<DOWN>(ma, mb, mb, mo, mo, mo, g, items_down, s);
  if (e == cudaSuccess && split_tails) {
    // the tails' CTA loads all 256 W2 rows of a column tile
    CUtensorMap mb_full;
    if (prepacked ? !make_map_tiles(&mb_full, W2, (long long)E * d / BN, f / 64, BN, BN)
                  : !make_map(&mb_full, W2, (long long)E * d, f, BN))
      return cudaErrorInvalidValue;
    const long long n = tails(gt);
    e = launch_mode<DOWN>(ma, mb_full, mb_full, mo, mo, mo, gt, n, s);
  }
  trace_end(MOE_STAGE_DOWN, s);
  return e;
}

// Backward contractions.  d % 64 == 0 and f % 64 == 0 are required.
cudaError_t launch_ffn_bwd(const uint16_t* x_perm, const int32_t* offsets, int N, int d, int f,
                           int E, const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                           const uint16_t* a_s, const uint16_t* b_s, const uint16_t* h,
                           const uint16_t* dO, uint16_t* dab, uint16_t* dx_perm, float* dW1,
                           float* dW3, float* dW2, void* tiles_ws, int* err, bool cta_pairs,
                           cudaStream_t s) {
  cudaError_t e;
  const int tile_m = cta_pairs ? 2 * BM : BM;   // rows per M tile (pairs: 256)
  GemmArgs g{};
  g.E = E; g.N = N; g.d = d; g.f = f;
  g.offsets = offsets;
  const TileLists tl = tile_lists(tiles_ws, E);
  g.tile_count = tl.count;
  g.tiles = tl.tiles;
  g.err = err;
  GemmArgs gt;   // the tails' launches (pairs): one CTA per tile of at most 128 rows
  auto tails = [&]() {
    gt = g;
    gt.tile_count = tl.tail_count;
    gt.tiles = tl.tails;
    return (long long)E * g.n_tiles_n;
  };
  CUtensorMap ma, mb, mb2;
  const bool split_tails = cta_pairs && (long long)N <= 2LL * BM * E;   // as in the forward
  if (N > 0) {
    trace_begin(MOE_STAGE_BWD_DH, s);
    e = launch_build_tiles(offsets, E, tiles_ws, s, tile_m, split_tails ? BM : 0);
    if (e != cudaSuccess) return e;
    const long long max_m_tiles = ceil_div(N, tile_m) + E;
    // dh = do W2[e] (B MN-major: W2 viewed [E*d, f]); epilogue -> dab = [da | db]
    if (!make_map(&ma, dO, N, d, BM) || !make_map(&mb, W2, (long long)E * d, f, 64))
      return cudaErrorInvalidValue;
    g.kblocks = d / BK;
    g.n_tiles_n = ceil_div(f, BN);
    g.out_bf16 = dab; g.in_a = a_s; g.in_b = b_s;
    CUtensorMap mo;
    if (!make_map(&mo, dab, N, 2LL * f, 32)) return cudaErrorInvalidValue;
    e = cta_pairs ? launch_mode<DH, true>(ma, mb, mb, mo, mo, mo, g, max_m_tiles * g.n_tiles_n, s)
                  : launch_mode<DH>(ma, mb, mb, mo, mo, mo, g, max_m_tiles * g.n_tiles_n, s);
    if (e == cudaSuccess && split_tails) {
      const long long n = tails();
      e = launch_mode<DH>(ma, mb, mb, mo, mo, mo, gt, n, s);
    }
    trace_end(MOE_STAGE_BWD_DH, s);
    if (e != cudaSuccess) return e;
    // dx_perm = [da | db] [W1[e]; W3[e]] (B MN-major: W1, W3 viewed [E*f, d])
    if (!make_map(&ma, dab, N, 2LL * f, BM) || !make_map(&mb, W1, (long long)E * f, d, 64) ||
        !make_map(&mb2, W3, (long long)E * f, d, 64))
      return cudaErrorInvalidValue;
    g.kblocks = 2 * f / BK;
    g.n_tiles_n = ceil_div(d, BN);
    g.out_bf16 = dx_perm;
    if (!make_map(&mo, dx_perm, N, d, 32)) return cudaErrorInvalidValue;
    trace_begin(MOE_STAGE_BWD_DX, s);
    e = cta_pairs ? launch_mode<DX, true>(ma, mb, mb2, mo, mo, mo, g, max_m_tiles * g.n_tiles_n, s)
                  : launch_mode<DX>(ma, mb, mb2, mo, mo, mo, g, max_m_tiles * g.n_tiles_n, s);
    if (e == cudaSuccess && split_tails) {
      const long long n = tails();
      e = launch_mode<DX>(ma, mb, mb2, mo, mo, mo, gt, n, s);
    }
    trace_end(MOE_STAGE_BWD_DX, s);
    if (e != cudaSuccess) return e;
  }
  // dW2[e] = do^T h: A = do [N, d] MN-major, B = h [N, f] MN-major;
  // [dW1[e]; dW3[e]] = [da | db]^T x_perm: A = dab [N, 2f], B = x_perm [N, d].
  // Each expert also gets copies of the four operand maps whose rows end at its
  // last row (its last k-block then reads zeros past it).
  const long long rows = N > 0 ? N : 1;
  MapTemplates mt;
  if (!make_map(&mt.m[0], dO, rows, d, 64) || !make_map(&mt.m[1], h, rows, f, 64) ||
      !make_map(&mt.m[2], dab, rows, 2LL * f, 64) || !make_map(&mt.m[3], x_perm, rows, d, 64))
    return cudaErrorInvalidValue;
  CUtensorMap* emaps = expert_maps(tiles_ws, N, E);
  trace_begin(MOE_STAGE_BWD_WG2, s);
  expert_maps_kernel<<<ceil_div(4 * E, 256), 256, 0, s>>>(mt, offsets, E, emaps);
  count_launches(1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  g.n_tiles_m = ceil_div(d, tile_m);
  g.n_tiles_n = ceil_div(f, BN);
  g.out_f32 = dW2;
  g.emaps = emaps;
  CUtensorMap mc, mc2;
  if (!make_map_f32_3d(&mc, dW2, E, d, f)) return cudaErrorInvalidValue;
  const long long wg2_items = (long long)E * g.n_tiles_m * g.n_tiles_n;
  e = cta_pairs ? launch_mode<WG2, true>(mt.m[0], mt.m[1], mt.m[1], mc, mc, mc, g, wg2_items, s)
                : launch_mode<WG2>(mt.m[0], mt.m[1], mt.m[1], mc, mc, mc, g, wg2_items, s);
  trace_end(MOE_STAGE_BWD_WG2, s);
  if (e != cudaSuccess) return e;
  g.n_tiles_m = ceil_div(2 * f, tile_m);
  g.n_tiles_n = ceil_div(d, BN);
  g.out_f32 = dW1; g.out_f32b = dW3;
  g.emaps = emaps + 2 * E;
  if (!make_map_f32_3d(&mc, dW1, E, f, d) || !make_map_f32_3d(&mc2, dW3, E, f, d))
    return cudaErrorInvalidValue;
  trace_begin(MOE_STAGE_BWD_WG13, s);
  const long long wg13_items = (long long)E * g.n_tiles_m * g.n_tiles_n;
  e = cta_pairs ? launch_mode<WG13, true>(mt.m[2], mt.m[3], mt.m[3], mc, mc2, mc2, g, wg13_items, s)
                : launch_mode<WG13>(mt.m[2], mt.m[3], mt.m[3], mc, mc2, mc2, g, wg13_items, s);
  trace_end(MOE_STAGE_BWD_WG13, s);
  return e;
}

// The router weight gradient's GEMM: the weight-gradient kernel (mode WG2) with
// one "expert" per chunk of tokens, A = x [T, d] and B = S [T, n2], both
// MN-major, K = the chunk's tokens; each chunk's maps end at its last token.
cudaError_t launch_dwg_gemm(const uint16_t* x, const uint16_t* Sm, const int32_t* offs, int T,
                            int d, int n2, int S, float* P, void* maps_ws, int* err,
                            bool cta_pairs, cudaStream_t s) {
  if (T == 0 || S == 0) return cudaSuccess;
  const int tile_m = cta_pairs ? 2 * BM : BM;
  MapTemplates mt;
  if (!make_map(&mt.m[0], x, T, d, 64) || !make_map(&mt.m[1], Sm, T, n2, 64))
    return cudaErrorInvalidValue;
  mt.m[2] = mt.m[0];
  mt.m[3] = mt.m[1];
  CUtensorMap* emaps = static_cast<CUtensorMap*>(maps_ws);
  expert_maps_kernel<<<ceil_div(4 * S, 256), 256, 0, s>>>(mt, offs, S, emaps);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  GemmArgs g{};
  g.E = S; g.N = T; g.d = d; g.f = n2;
  g.offsets = offs;
  g.err = err;
  g.n_tiles_m = ceil_div(d, tile_m);
  g.n_tiles_n = ceil_div(n2, BN);
  g.out_f32 = P;
  g.emaps = emaps;
  CUtensorMap mc;
  if (!make_map_f32_3d(&mc, P, S, d, n2)) return cudaErrorInvalidValue;
  const long long items = (long long)S * g.n_tiles_m * g.n_tiles_n;
  return cta_pairs ? launch_mode<WG2, true>(mt.m[0], mt.m[1], mt.m[1], mc, mc, mc, g, items, s)
                   : launch_mode<WG2>(mt.m[0], mt.m[1], mt.m[1], mc, mc, mc, g, items, s);
}

}  // namespace moe
