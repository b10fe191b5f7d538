// Grouped per-expert SwiGLU FFN on microscaled fp8 operands, on the 5th-generation
// tensor cores (tcgen05.mma kind::mxf8f6f4 with UE8M0 block scales).
// ("Enabling trillion-parameter models on AWS EFA", section "Evaluation": the
// tokens travel as block-scaled fp8; here the expert GEMMs consume them as they
// are, with weights quantised the same way.)
//
// Operands: E4M3 codes, K contiguous, one power-of-two scale per 32 elements
// along K (scale rows padded to 16 bytes).  Two modes of one kernel:
//   GATEUP  [a | b] = x W1[e]^T | x W3[e]^T;  epilogue h = silu(a) b (fp32),
//           written as microscaled fp8 along f (codes + scales)
//   DOWN    o = bf16(s_row * (h W2[e]^T))
// One CTA per SM, 128-row tiles of an expert's rows (ragged, from the tile
// list), 256 output columns (GATEUP: 128 of W1 and the same 128 of W3).  Roles
// (448 threads): warp 0 issues TMA loads of 128-deep k-blocks (A 16 KB, B 32 KB)
// into four stages, and two groups ahead the scales of each group of four
// k-blocks (16 bytes per row of A and of B) into a ring of three slots; warp 1
// issues the MMAs (four 32-deep steps per k-block) into one 256-column TMEM
// accumulator; warps 10-13 move each group's scales from shared to tensor
// memory (tcgen05.st) into one of three buffers; warps 2-9 drain the
// accumulator and write the outputs.  Every wait is bounded.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int BM = 128, BK = 128, BN = 256, STAGES = 4;
constexpr int A_BYTES = BM * BK;              // 16 KB of codes
constexpr int B_BYTES = BN * BK;              // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SFA_BYTES = BM * 16;            // scales of 4 k-blocks: 16 bytes per row
constexpr int SFB_BYTES = BN * 16;
constexpr int SF_BYTES = SFA_BYTES + SFB_BYTES;
constexpr int EPI_WARPS = 8, SF_WARPS = 4;
constexpr int THREADS = 64 + 32 * (EPI_WARPS + SF_WARPS);
constexpr int SF_WARP0 = 2 + EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
// Scale groups: three slots in shared memory and three buffers in tensor memory,
// so that the scales of a group are loaded two groups ahead of its operands and
// written while the MMAs of the two groups before it run.
constexpr uint32_t NBUF = 3;
// tensor-memory columns: accumulator 0-255; per scale buffer b, k-block j of its
// group of four: A scales at 256 + 16b + 4j (+ m/32), B scales at 304 + 32b + 8j
constexpr uint32_t SFA_COL = 256, SFB_COL = 256 + 16 * NBUF;
static_assert(SFB_COL + 32 * NBUF <= TMEM_COLS, "tensor memory");
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + (int)NBUF * SF_BYTES + 256 + 1024;

enum Mode : int { GATEUP = 0, DOWN = 1 };

struct alignas(8) Ctl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t sfs_full[NBUF];    // a group's scales landed in its shared-memory slot
  uint64_t sfs_free[NBUF];    // the scale warps have read the slot
  uint64_t sf_full[NBUF];     // the group's scales are in tensor memory
  uint64_t sf_empty[NBUF];    // the MMAs that read a tensor-memory scale buffer are done
  uint64_t tfull, tempty, mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Ctl) <= 256, "control block");

struct MxArgs {
  int E, N, d, f;
  const int32_t* offsets;
  const int2* tiles;           // 128-row tiles {first row, expert}
  const int32_t* tile_count;
  int n_tiles_n;               // 256-column output tiles (GATEUP: 128-column h tiles)
  int kblocks;                 // 128-deep k-blocks
  uint8_t* hq;                 // GATEUP: h codes [N, f] and scales [N, hs_stride]
  uint8_t* hs;
  int hs_stride;
  uint16_t* out;               // DOWN: o [N, d]
  const float* row_scale;      // DOWN: per-row output scale, or null
  int* err;
};

__device__ __forceinline__ float silu_mx(float a) { return a / (1.f + expf(-a)); }

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmSA,
                       const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                       const __grid_constant__ CUtensorMap tmSB, const __grid_constant__ CUtensorMap tmSB2,
                       const __grid_constant__ MxArgs g) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t tile_base = (raw_addr + 1023u) & ~1023u;
  uint8_t* tile_ptr = smem_raw + (tile_base - raw_addr);
  const uint32_t sf_base = tile_base + STAGES * STAGE_BYTES;   // the scale slots
  Ctl* ctl = reinterpret_cast<Ctl*>(tile_ptr + STAGES * STAGE_BYTES + NBUF * SF_BYTES);
  volatile int* abort_flag = &ctl->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < (int)NBUF; ++b) {
      mbar_init(smem_u32(&ctl->sfs_full[b]), 1);
      mbar_init(smem_u32(&ctl->sfs_free[b]), SF_WARPS);
      mbar_init(smem_u32(&ctl->sf_full[b]), SF_WARPS);
      mbar_init(smem_u32(&ctl->sf_empty[b]), 1);
    }
    mbar_init(smem_u32(&ctl->tfull), 1);
    mbar_init(smem_u32(&ctl->tempty), EPI_WARPS);
    mbar_init(smem_u32(&ctl->mma_done), 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmSA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSB);
    if (MODE == GATEUP) {
      tma_prefetch_desc(&tmB2);
      tma_prefetch_desc(&tmSB2);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  const int total = (*g.tile_count) * g.n_tiles_n;
  const int nkb = g.kblocks;

  auto decode = [&](int item, int& row0, int& e, int& row_end, int& nt) {
    const int2 tl = g.tiles[item / g.n_tiles_n];
    nt = item % g.n_tiles_n;
    row0 = tl.x;
    e = tl.y;
    row_end = g.offsets[e + 1];
  };
  // B rows of a tile: GATEUP W1 (and W3) rows nt*128..; DOWN W2 rows nt*256..
  auto b_row = [&](int e, int nt) { return MODE == GATEUP ? e * g.f + nt * 128 : e * g.d + nt * BN; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it_count = 0;
      // scale group G (four k-blocks) is item blockIdx.x + (G / gpi) * gridDim.x,
      // k-blocks 4 (G % gpi) ..; groups are loaded kAhead ahead of the operands
      const int gpi = (nkb + 3) / 4;
      uint32_t g_sf = 0, g_op = 0;
      constexpr uint32_t kAhead = 2;
      bool ok = true;
      auto load_scales = [&](uint32_t G) -> bool {
        const int item = blockIdx.x + (int)(G / gpi) * gridDim.x;
        if (item >= total) return true;
        const uint32_t b = G % NBUF;
        if (!mbar_wait_bounded(smem_u32(&ctl->sfs_free[b]), ((G / NBUF) & 1u) ^ 1u, abort_flag,
                               g.err))
          return false;
        int row0, e, row_end, nt;
        decode(item, row0, e, row_end, nt);
        const int brow = b_row(e, nt);
        const int x = (int)(G % gpi) * 16;   // bytes 16 (G % gpi) .. of each scale row
        const uint32_t lb = smem_u32(&ctl->sfs_full[b]);
        const uint32_t ssa = sf_base + b * SF_BYTES;
        const uint32_t ssb = ssa + SFA_BYTES;
        mbar_arrive_expect_tx(lb, SF_BYTES);
        tma_load_2d(ssa, &tmSA, lb, x, row0);
        if (MODE == GATEUP) {
          tma_load_2d(ssb, &tmSB, lb, x, brow);
          tma_load_2d(ssb + SFB_BYTES / 2, &tmSB2, lb, x, brow);
        } else {
          tma_load_2d(ssb, &tmSB, lb, x, brow);
        }
        return true;
      };
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        int row0, e, row_end, nt;
        decode(item, row0, e, row_end, nt);
        const int brow = b_row(e, nt);
        for (int kb = 0; kb < nkb; ++kb, ++it_count) {
          if ((kb & 3) == 0) {
            for (; ok && g_sf <= g_op + kAhead; ++g_sf) ok = load_scales(g_sf);
            ++g_op;
            if (!ok) break;
          }
          const int s = it_count % STAGES;
          const uint32_t ph = (it_count / STAGES) & 1u;
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, g.err)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&ctl->full[s]);
          const uint32_t sa = tile_base + s * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          mbar_arrive_expect_tx(bar, STAGE_BYTES);
          tma_load_2d(sa, &tmA, bar, kb * BK, row0);
          if (MODE == GATEUP) {
            tma_load_2d(sb, &tmB, bar, kb * BK, brow);
            tma_load_2d(sb + B_BYTES / 2, &tmB2, bar, kb * BK, brow);
          } else {
            tma_load_2d(sb, &tmB, bar, kb * BK, brow);
          }
        }
      }
      if (!ok) {   // the loads still in flight land before the CTA exits
        const uint32_t n = it_count < (uint32_t)STAGES ? it_count : (uint32_t)STAGES;
        for (uint32_t q = 0; q < n; ++q) {
          const uint32_t c = it_count - 1 - q;
          volatile int never = 0;
          mbar_wait_bounded(smem_u32(&ctl->full[c % STAGES]), (c / STAGES) & 1u, &never, nullptr);
        }
        for (uint32_t G = g_sf > NBUF ? g_sf - NBUF : 0; G < g_sf; ++G) {
          volatile int never = 0;
          mbar_wait_bounded(smem_u32(&ctl->sfs_full[G % NBUF]), (G / NBUF) & 1u, &never, nullptr,
                            200000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t it_count = 0, grp = 0;
    bool ok = true, issued_any = false;
    int j = 0;
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++j) {
      ok = mbar_wait_bounded(smem_u32(&ctl->tempty), (j & 1u) ^ 1u, abort_flag, g.err);
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t gcur = 0;
      for (int kb = 0; kb < nkb; ++kb, ++it_count) {
        const int s = it_count % STAGES;
        const uint32_t ph = (it_count / STAGES) & 1u;
        ok = mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag, g.err);
        if (ok && (kb & 3) == 0) {   // this group's scales are in tensor memory
          gcur = grp++;
          ok = mbar_wait_bounded(smem_u32(&ctl->sf_full[gcur % NBUF]), (gcur / NBUF) & 1u,
                                 abort_flag, g.err);
        }
        ok = __all_sync(kFull, ok);
        if (!ok) break;
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sa = tile_base + s * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          const uint32_t buf = gcur % NBUF, jj = kb & 3;
          const uint32_t sfa = tmem_base + SFA_COL + 16 * buf + 4 * jj;
          const uint32_t sfb = tmem_base + SFB_COL + 32 * buf + 8 * jj;
#pragma unroll
          for (int ks = 0; ks < BK / 32; ++ks)
            tc_mma_mxf8(tmem_base, smem_desc_sw128(sa + ks * 32, 16, 1024),
                        smem_desc_sw128(sb + ks * 32, 16, 1024), idesc_mxf8(BM, BN, ks, ks), sfa,
                        sfb, (kb > 0 || ks > 0) ? 1u : 0u);
          issued_any = true;
          tc_commit(smem_u32(&ctl->empty[s]));
          if (jj == 3 || kb == nkb - 1) tc_commit(smem_u32(&ctl->sf_empty[buf]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(smem_u32(&ctl->tfull));
      __syncwarp();
    }
    if (lane == 0 && issued_any) {
      tc_commit(smem_u32(&ctl->mma_done));
      volatile int never = 0;
      mbar_wait_bounded(smem_u32(&ctl->mma_done), 0, &never, nullptr);
    }
    __syncwarp();
  } else if (warp >= SF_WARP0) {
    // ------------------------------------------------------------ scales -> tensor memory
    // This warp's lanes are TMEM lanes 32q .. 32q+31: A row m = 32q + lane, and
    // (a copy of) the B scales that lane quadrant reads.
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    uint32_t grp = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
      for (int kb0 = 0; kb0 < nkb; kb0 += 4, ++grp) {
        const uint32_t buf = grp % NBUF;
        // the group's scales landed in their slot, and the MMAs of the group that
        // used this tensor-memory buffer NBUF groups ago are done
        ok = mbar_wait_bounded(smem_u32(&ctl->sfs_full[buf]), (grp / NBUF) & 1u, abort_flag,
                               g.err);
        ok = ok && mbar_wait_bounded(smem_u32(&ctl->sf_empty[buf]), ((grp / NBUF) & 1u) ^ 1u,
                                     abort_flag, g.err);
        ok = __all_sync(kFull, ok);
        if (!ok) break;
        const uint8_t* ssa = tile_ptr + STAGES * STAGE_BYTES + buf * SF_BYTES;
        const uint8_t* ssb = ssa + SFA_BYTES;
        // A: row m's four k-blocks, each word copied to the four columns of its k-block
        const uint4 wa = *reinterpret_cast<const uint4*>(ssa + m * 16);
        const uint32_t av[4] = {wa.x, wa.y, wa.z, wa.w};
        uint32_t r[16];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) r[jj * 4 + cc] = av[jj];
        tmem_st16(lane_base + SFA_COL + 16 * buf, r);
        // B: column 8 jj + t of k-block jj holds B row 32 t + lane
        uint32_t bv[8][4];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const uint4 w = *reinterpret_cast<const uint4*>(ssb + (32 * t + lane) * 16);
          bv[t][0] = w.x; bv[t][1] = w.y; bv[t][2] = w.z; bv[t][3] = w.w;
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int jj = 0; jj < 2; ++jj)
#pragma unroll
            for (int t = 0; t < 8; ++t) r[jj * 8 + t] = bv[t][half * 2 + jj];
          tmem_st16(lane_base + SFB_COL + 32 * buf + 16 * half, r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&ctl->sfs_free[buf]));   // the slot may be reloaded
          mbar_arrive(smem_u32(&ctl->sf_full[buf]));
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-9)
    const int q = warp & 3;                 // TMEM lane quadrant
    const int half = (warp - 2) >> 2;       // which half of the columns
    int j = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++j) {
      int row0, e, row_end, nt;
      decode(item, row0, e, row_end, nt);
      bool ok = mbar_wait_bounded(smem_u32(&ctl->tfull), j & 1u, abort_flag, g.err);
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16);
      const int row = row0 + q * 32 + lane;
      const bool valid = row < row_end;
      const bool any = row0 + q * 32 < row_end;   // warp-uniform: rows of the expert here
      // the accumulator is released as soon as this warp's last TMEM load has
      // landed: the math and the stores of its last block then overlap the
      // next item's MMAs
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty));
      };
      if (MODE == GATEUP) {
        // 64 columns of h, two 32-element scale blocks: a at c, b at 128 + c.
        // Block 0 is turned into codes while block 1's loads are in flight; both
        // blocks' stores come after the release.
        auto codes = [&](float* a, const float* b, uint32_t* w) {
          float amax = 0.f;
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            a[u] = silu_mx(a[u]) * b[u];
            amax = fmaxf(amax, fabsf(a[u]));
          }
          const int k = mx_exponent(amax);
#pragma unroll
          for (int u = 0; u < 8; ++u) w[u] = mx_codes4(a + 4 * u, k);
          return k;
        };
        auto put = [&](int c, const uint32_t* w, int k) {
          if (!valid) return;
          const int col = nt * 128 + c;
          uint4* dst = reinterpret_cast<uint4*>(g.hq + (size_t)row * g.f + col);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          g.hs[(size_t)row * g.hs_stride + col / 32] = (uint8_t)(k + 127);
        };
        const int c0 = half * 64, c1 = c0 + 32;
        uint32_t w0[8], w1[8];
        int k0 = 0;
        float a[32], b[32];
        if (any) {
          tmem_ld16(t_row + c0, a);
          tmem_ld16(t_row + c0 + 16, a + 16);
          tmem_ld16(t_row + 128 + c0, b);
          tmem_ld16(t_row + 128 + c0 + 16, b + 16);
          tmem_ld_wait();
          k0 = codes(a, b, w0);
          tmem_ld16(t_row + c1, a);
          tmem_ld16(t_row + c1 + 16, a + 16);
          tmem_ld16(t_row + 128 + c1, b);
          tmem_ld16(t_row + 128 + c1 + 16, b + 16);
          tmem_ld_wait();
        }
        release();
        if (any) {
          put(c0, w0, k0);
          const int k1 = codes(a, b, w1);
          put(c1, w1, k1);
        }
      } else {
        // 128 columns in two batches of 64 (four TMEM loads per wait); batch 0
        // is packed to bf16 while batch 1 loads, and both are stored after the
        // release
        const float sc = (valid && g.row_scale) ? g.row_scale[row] : 1.f;
        const int c0 = half * 128;
        auto pack64 = [&](float* v, uint32_t* p) {
          if (g.row_scale) {
#pragma unroll
            for (int t = 0; t < 64; ++t) v[t] *= sc;
          }
#pragma unroll
          for (int t = 0; t < 32; ++t) p[t] = pack_bf16(v[2 * t], v[2 * t + 1]);
        };
        auto put64 = [&](int c, const uint32_t* p) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int col = nt * BN + c + 16 * u;
            if (valid && col < g.d) {
              uint4* dst = reinterpret_cast<uint4*>(g.out + (size_t)row * g.d + col);
              dst[0] = make_uint4(p[8 * u], p[8 * u + 1], p[8 * u + 2], p[8 * u + 3]);
              dst[1] = make_uint4(p[8 * u + 4], p[8 * u + 5], p[8 * u + 6], p[8 * u + 7]);
            }
          }
        };
        uint32_t p0[32], p1[32];
        float v[64];
        if (any) {
#pragma unroll
          for (int u = 0; u < 4; ++u) tmem_ld16(t_row + c0 + 16 * u, v + 16 * u);
          tmem_ld_wait();
          pack64(v, p0);
#pragma unroll
          for (int u = 0; u < 4; ++u) tmem_ld16(t_row + c0 + 64 + 16 * u, v + 16 * u);
          tmem_ld_wait();
        }
        release();
        if (any) {
          put64(c0, p0);
          pack64(v, p1);
          put64(c0 + 64, p1);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

constexpr int kU8 = (int)CU_TENSOR_MAP_DATA_TYPE_UINT8;

int sms() {
  static int n[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (n[dev] == 0) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev] > 0 ? n[dev] : 148;
}

template <int MODE>
cudaError_t launch_mx(const CUtensorMap& a, const CUtensorMap& sa, const CUtensorMap& b,
                      const CUtensorMap& b2, const CUtensorMap& sb, const CUtensorMap& sb2,
                      const MxArgs& g, long long max_items, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_mx_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  if (max_items <= 0) return cudaSuccess;
  const int grid = (int)(max_items < sms() ? max_items : sms());
  grouped_gemm_mx_kernel<MODE><<<grid, THREADS, SMEM_BYTES, s>>>(a, sa, b, b2, sb, sb2, g);
  count_launches(1);
  return cudaGetLastError();
}
}  // namespace

bool ffn_mx_supported(int d, int f) { return d % 128 == 0 && f % 128 == 0; }

size_t ffn_mx_ws_bytes(int N, int d, int f, int E) {
  (void)d;
  return tiles_ws_bytes(N, E) + align_up((size_t)N * f, 256) +
         align_up((size_t)N * mx_scale_row_bytes(f), 256);
}

cudaError_t launch_ffn_mx(const uint8_t* xq, const uint8_t* xs, const int32_t* offsets, int N,
                          int d, int f, int E, const uint8_t* W1q, const uint8_t* W1s,
                          const uint8_t* W3q, const uint8_t* W3s, const uint8_t* W2q,
                          const uint8_t* W2s, const float* row_scale, uint8_t* hq, uint8_t* hs,
                          uint16_t* out, void* ws, int* err, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  uint8_t* w = static_cast<uint8_t*>(ws);
  void* tws = w;
  w += tiles_ws_bytes(N, E);
  const int skd = mx_scale_row_bytes(d), skf = mx_scale_row_bytes(f);
  if (!hq) hq = w;
  w += align_up((size_t)N * f, 256);
  if (!hs) hs = w;
  trace_begin(MOE_STAGE_GATEUP, s);
  cudaError_t e = launch_build_tiles(offsets, E, tws, s, BM, 0);
  if (e != cudaSuccess) return e;
  const TileLists tl = tile_lists(tws, E);
  MxArgs g{};
  g.E = E; g.N = N; g.d = d; g.f = f;
  g.offsets = offsets;
  g.tiles = tl.tiles;
  g.tile_count = tl.count;
  g.err = err;
  g.hq = hq; g.hs = hs; g.hs_stride = skf;
  g.out = out;
  g.row_scale = row_scale;
  const long long m_tiles = ceil_div(N, BM) + E;
  CUtensorMap ma, msa, mb, mb2, msb, msb2;
  // gate-up: A = x codes [N, d], B = W1 / W3 codes [E f, d] (128 rows each per tile)
  if (!encode_map_2d(&ma, kU8, xq, d, N, d, BK, BM, true) ||
      !encode_map_2d(&msa, kU8, xs, skd, N, skd, 16, BM, false) ||
      !encode_map_2d(&mb, kU8, W1q, d, (unsigned long long)E * f, d, BK, 128, true) ||
      !encode_map_2d(&mb2, kU8, W3q, d, (unsigned long long)E * f, d, BK, 128, true) ||
      !encode_map_2d(&msb, kU8, W1s, skd, (unsigned long long)E * f, skd, 16, 128, false) ||
      !encode_map_2d(&msb2, kU8, W3s, skd, (unsigned long long)E * f, skd, 16, 128, false))
    return cudaErrorInvalidValue;
  g.n_tiles_n = f / 128;
  g.kblocks = d / BK;
  e = launch_mx<GATEUP>(ma, msa, mb, mb2, msb, msb2, g, m_tiles * g.n_tiles_n, s);
  trace_end(MOE_STAGE_GATEUP, s);
  if (e != cudaSuccess) return e;
  // down: A = h codes [N, f], B = W2 codes [E d, f] (256 rows per tile)
  trace_begin(MOE_STAGE_DOWN, s);
  if (!encode_map_2d(&ma, kU8, hq, f, N, f, BK, BM, true) ||
      !encode_map_2d(&msa, kU8, hs, skf, N, skf, 16, BM, false) ||
      !encode_map_2d(&mb, kU8, W2q, f, (unsigned long long)E * d, f, BK, BN, true) ||
      !encode_map_2d(&msb, kU8, W2s, skf, (unsigned long long)E * d, skf, 16, BN, false))
    return cudaErrorInvalidValue;
  g.n_tiles_n = ceil_div(d, BN);
  g.kblocks = f / BK;
  e = launch_mx<DOWN>(ma, msa, mb, mb, msb, msb, g, m_tiles * g.n_tiles_n, s);
  trace_end(MOE_STAGE_DOWN, s);
  return e;
}

}  // namespace moe
