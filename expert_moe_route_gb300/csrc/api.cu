// C ABI of the MoE layer hot path (declared in include/moe.h): argument
// checks, workspace layout, kernel sequencing on the caller's stream.
#include <stdio.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
static std::atomic<unsigned long long> g_launches{0};
static std::atomic<void* const*> g_trace{nullptr};
// > 0 while this thread launches the shared expert's GEMMs, whose per-GEMM
// stages would otherwise overwrite the routed GEMMs' trace events.
static thread_local int g_trace_mute = 0;
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
// A failed trace record must not surface later as a launch error: clear it.
static void trace_record(int slot, cudaStream_t s) {
  if (g_trace_mute) return;
  void* const* ev = g_trace.load(std::memory_order_relaxed);
  if (ev && ev[slot] && cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[slot]), s) != cudaSuccess)
    (void)cudaGetLastError();
}
void trace_begin(int stage, cudaStream_t s) { trace_record(2 * stage, s); }
void trace_end(int stage, cudaStream_t s) { trace_record(2 * stage + 1, s); }

moe_status_t shape_check(int T, int d, int E, int R) {
  if (T < 0 || d <= 0 || E <= 0 || R <= 0) return MOE_ERR_INVALID_ARG;
  if (R > E) return MOE_ERR_INVALID_ARG;
  if (R > 32 || E > 1024 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * R >= (1LL << 31) || (long long)T * d >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// The CUDA error behind this thread's last MOE_ERR_CUDA (moe_last_cuda_error).
static thread_local int g_last_cuda = 0;

moe_status_t cuda_failed(cudaError_t e) {
  g_last_cuda = (int)e;
  return MOE_ERR_CUDA;
}

// Optionally wait for the stream and translate the device error word.
moe_status_t finish(cudaError_t launched, const int* err_dev, unsigned flags, cudaStream_t s) {
  if (launched != cudaSuccess) return cuda_failed(launched);
  if (!(flags & MOE_CHECK)) return MOE_OK;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_failed(e);
  if (!err_dev) return MOE_OK;
  int h = 0;
  e = cudaMemcpy(&h, err_dev, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_failed(e);
  if (h & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (h & kErrBadRouting) return MOE_ERR_BAD_ROUTING;
  return MOE_OK;
}
}  // namespace moe

using namespace moe;

namespace {

constexpr size_t kErrBytes = 256;   // device error word, at the start of every workspace

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

inline cudaStream_t S(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

bool init_once() {
  static int done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev < 0 || dev >= 64) return false;
  if (!done[dev]) {
    if (dispatch_set_smem_limits() != cudaSuccess) return false;
    done[dev] = 1;
  }
  return true;
}

struct Carve {
  uint8_t* base;
  size_t off = 0;
  explicit Carve(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    void* p = base ? base + off : nullptr;
    off += align_up(bytes, 256);
    return p;
  }
};

// Records the stage-boundary events of moe_trace_events, when enabled.
struct Stage {
  cudaStream_t s;
  int i;
  Stage(cudaStream_t s_, int stage) : s(s_), i(stage) { trace_begin(i, s); }
  ~Stage() { trace_end(i, s); }
};

struct TraceMute {
  TraceMute() { ++g_trace_mute; }
  ~TraceMute() { --g_trace_mute; }
};

// The shared expert's stream: one per device, created on first use and kept
// for the life of the process.
cudaStream_t side_stream() {
  static std::mutex mu;
  static cudaStream_t st[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!st[dev] && cudaStreamCreateWithFlags(&st[dev], cudaStreamNonBlocking) != cudaSuccess)
    st[dev] = nullptr;
  return st[dev];
}

// `to` waits for the work enqueued on `from` so far.
cudaError_t stream_wait(cudaStream_t to, cudaStream_t from) {
  if (to == from) return cudaSuccess;
  cudaEvent_t ev;
  cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(ev, from);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(to, ev, 0);
  cudaEventDestroy(ev);   // released once the recorded work completes
  return e;
}

// Joins the side stream back into the caller's stream when it goes out of
// scope, so that no return path leaves shared-expert work unordered with
// the caller's later work.
struct Join {
  cudaStream_t to, from;
  bool armed = false;
  ~Join() {
    if (armed) (void)stream_wait(to, from);
  }
  cudaError_t now() {
    armed = false;
    return stream_wait(to, from);
  }
};

#define MOE_TRY(expr)                        \
  do {                                       \
    cudaError_t e_ = (expr);                 \
    if (e_ != cudaSuccess) return finish(e_, nullptr, 0, nullptr); \
  } while (0)

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_BAD_ROUTING: return "MOE_ERR_BAD_ROUTING";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
  }
  return "unknown moe_status_t";
}

int moe_version(void) { return 100; }

int moe_last_cuda_error(void) { return g_last_cuda; }

moe_status_t moe_trace_events(void* const* events) {
  g_trace.store(events, std::memory_order_relaxed);
  return MOE_OK;
}

unsigned long long moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status_t moe_selftest_wait_timeout(unsigned limit_us, void* ws, moe_stream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u || !ws) return MOE_ERR_INVALID_ARG;
  if (!al256(ws)) return MOE_ERR_WORKSPACE;
  if (!init_once()) return MOE_ERR_CUDA;
  cudaStream_t s = S(stream);
  int* err = static_cast<int*>(ws);
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(int), s));
  return finish(launch_selftest_wait(limit_us, err, s), err, MOE_CHECK, s);
}

static size_t gate_ws_bytes(int T, int d, int E) {
  return gate_tc_supported(d) ? gate_tc_ws_bytes(T, d, E) : 0;
}

// Gate projection: tensor-core split path when d % 64 == 0, else fp32 FMA.
static cudaError_t launch_gate(const uint16_t* x, const float* w_gate, const float* bias, int T,
                               int d, int E, float* logits, void* gws, int* err, cudaStream_t s) {
  if (gate_tc_supported(d)) return launch_gate_tc(x, w_gate, bias, T, d, E, logits, gws, err, s);
  return launch_gate_logits(x, w_gate, bias, T, d, E, logits, s);
}

moe_status_t moe_route(const uint16_t* x, const float* w_gate, const float* bias, int T, int d,
                       int E, int R, float* logits, int32_t* topk_idx, float* topk_w, void* ws,
                       size_t* ws_bytes, unsigned flags, moe_stream_t stream) {
  const bool logits_in = flags & MOE_LOGITS_IN;
  if (logits_in) {
    if (T < 0 || E <= 0 || R <= 0 || R > E) return MOE_ERR_INVALID_ARG;
    if (R > 32 || E > 1024) return MOE_ERR_UNSUPPORTED;
  } else {
    moe_status_t st = shape_check(T, d, E, R);
    if (st != MOE_OK) return st;
    if (!ws_bytes) return MOE_ERR_INVALID_ARG;
    const size_t need = kErrBytes + gate_ws_bytes(T, d, E);
    if (!ws) {
      *ws_bytes = need;
      return MOE_OK;
    }
    if (*ws_bytes < need || !al256(ws)) return MOE_ERR_WORKSPACE;
  }
  if (T == 0) return MOE_OK;
  if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!logits_in) {
    if (!x || !w_gate) return MOE_ERR_INVALID_ARG;
    if (!al16(x)) return MOE_ERR_UNSUPPORTED;
  }
  if (!init_once()) return MOE_ERR_CUDA;
  cudaStream_t s = S(stream);
  int* err = nullptr;
  if (!logits_in) {
    err = static_cast<int*>(ws);
    MOE_TRY(cudaMemsetAsync(err, 0, sizeof(int), s));
    Stage st_(s, MOE_STAGE_GATE);
    MOE_TRY(launch_gate(x, w_gate, bias, T, d, E, logits, static_cast<uint8_t*>(ws) + kErrBytes,
                        err, s));
  }
  cudaError_t e;
  {
    Stage st_(s, MOE_STAGE_TOPK);
    e = launch_topk(logits, T, E, R, topk_idx, topk_w, s);
  }
  return finish(e, err, flags, s);
}

moe_status_t moe_dispatch(const uint16_t* x, const int32_t* topk_idx, int T, int d, int E, int R,
                          int32_t* counts, int32_t* offsets, int32_t* row_slot, int32_t* slot_row,
                          uint16_t* x_perm, void* ws, size_t* ws_bytes, unsigned flags,
                          moe_stream_t stream) {
  moe_status_t st = shape_check(T, d, E, R);
  if (st != MOE_OK) return st;
  if (!ws_bytes) return MOE_ERR_INVALID_ARG;
  const size_t need = kErrBytes + dispatch_ws_bytes(T, E);
  if (!ws) {
    *ws_bytes = need;
    return MOE_OK;
  }
  if (*ws_bytes < need || !al256(ws)) return MOE_ERR_WORKSPACE;
  if (!counts || !offsets || (T > 0 && (!topk_idx || !row_slot || !slot_row)))
    return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if (x && (!al16(x) || !al16(x_perm))) return MOE_ERR_UNSUPPORTED;
  if (!init_once()) return MOE_ERR_CUDA;
  cudaStream_t s = S(stream);
  int* err = static_cast<int*>(ws);
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(int), s));
  cudaError_t e;
  {
    Stage st_(s, MOE_STAGE_DISPATCH);
    e = launch_dispatch(x, topk_idx, T, d, E, R, counts, offsets, row_slot, slot_row, x_perm,
                        static_cast<uint8_t*>(ws) + kErrBytes, err, s);
  }
  return finish(e, err, flags, s);
}

moe_status_t moe_dispatch_fp8(const uint16_t* x, const int32_t* topk_idx, int T, int d, int E,
                              int R, int32_t* counts, int32_t* offsets, int32_t* row_slot,
                              int32_t* slot_row, uint8_t* xq_perm, float* xscale_perm, void* ws,
                              size_t* ws_bytes, unsigned flags, moe_stream_t stream) {
  moe_status_t st = shape_check(T, d, E, R);
  if (st != MOE_OK) return st;
  if (d % 128) return MOE_ERR_UNSUPPORTED;
  if (!ws_bytes) return MOE_ERR_INVALID_ARG;
  const size_t need = kErrBytes + dispatch_ws_bytes(T, E);
  if (!ws) {
    *ws_bytes = need;
    return MOE_OK;
  }
  if (*ws_bytes < need || !al256(ws)) return MOE_ERR_WORKSPACE;
  if (!counts || !offsets || (T > 0 && (!x || !topk_idx || !row_slot || !slot_row || !xq_perm ||
                                        !xscale_perm)))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!al16(x) || ((uintptr_t)xq_perm & 7) || ((uintptr_t)xscale_perm & 3)))
    return MOE_ERR_UNSUPPORTED;
  if (!init_once()) return MOE_ERR_CUDA;
  cudaStream_t s = S(stream);
  int* err = static_cast<int*>(ws);
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(int), s));
  cudaError_t e;
  {
    Stage st_(s, MOE_STAGE_DISPATCH);
    e = launch_dispatch_fp8(x, topk_idx, T, d, E, R, counts, offsets, row_slot, slot_row, xq_perm,
                            xscale_perm, static_cast<uint8_t*>(ws) + kErrBytes, err, s);
  }
  return finish(e, err, flags, s);
}

moe_status_t moe_dequant_fp8(const uint8_t* xq, const float* xscale, int N, int d, uint16_t* out,
                             moe_stream_t stream) {
  if (N < 0 || d <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 128) return MOE_ERR_UNSUPPORTED;
  if (N == 0) return MOE_OK;
  if (!xq || !xscale || !out) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)xq & 7) || ((uintptr_t)xscale & 3) || !al16(out)) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = S(stream);
  return finish(launch_dequant_fp8(xq, xscale, N, d, out, s), nullptr, 0, s);
}

moe_status_t moe_grouped_ffn(const uint16_t* x_perm, const int32_t* offsets, int N, int d, int f,
                             int E, const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                             const float* row_scale, uint16_t* a_save, uint16_t* b_save,
                             uint16_t* h, uint16_t* out, void* ws, size_t* ws_bytes,
                             unsigned flags, moe_stream_t stream) {
  if (N < 0 || d <= 0 || f <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 8 || f % 8 || E > 1024) return MOE_ERR_UNSUPPORTED;
  if ((flags & MOE_WEIGHTS_PREPACKED) && !prepack_supported(d, f)) return MOE_ERR_UNSUPPORTED;
  if (!ws_bytes) return MOE_ERR_INVALID_ARG;
  const size_t need = kErrBytes + tiles_ws_bytes(N, E);
  if (!ws) {
    *ws_bytes = need;
    return MOE_OK;
  }
  if (*ws_bytes < need || !al256(ws)) return MOE_ERR_WORKSPACE;
  if (!offsets || !W1 || !W3 || !W2) return MOE_ERR_INVALID_ARG;
  if (N > 0 && (!x_perm || !h || !out)) return MOE_ERR_INVALID_ARG;
  if ((a_save == nullptr) != (b_save == nullptr)) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {x_perm, W1, W3, W2, a_save, b_save, h, out};
  for (const void* p : ps)
    if (p && !al16(p)) return MOE_ERR_UNSUPPORTED;
  if (!init_once()) return MOE_ERR_CUDA;
  cudaStream_t s = S(stream);
  int* err = static_cast<int*>(ws);
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(int), s));
  cudaError_t e = launch_ffn_fwd(x_perm, offsets, N, d, f, E, W1, W3, W2, a_save, b_save, h, out,
                                 static_cast<uint8_t*>(ws) + kErrBytes, err,
                                 (flags & MOE_WEIGHTS_PREPACKED) != 0,
                                 !(flags & MOE_SINGLE_CTA_TILES), s, row_scale);
  return finish(e, err, flags, s);
}

moe_status_t moe_grouped_ffn_fp8(const uint8_t* xq_perm, const float* xscale_perm,
                                 const int32_t* offsets, int N, int d, int f, int E,
                                 const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                                 const float* row_scale, uint16_t* a_save, uint16_t* b_save,
                                 uint16_t* h, uint16_t* out, void* ws, size_t* ws_bytes,
                                 unsigned flags, moe_stream_t stream) {
  if (N < 0 || d <= 0 || f <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 128 || f % 8 || E > 1024) return MOE_ERR_UNSUPPORTED;
  if ((flags & MOE_WEIGHTS_PREPACKED) && !prepack_supported(d, f)) return MOE_ERR_UNSUPPORTED;
  if (!ws_bytes) return MOE_ERR_INVALID_ARG;
  const size_t tws = tiles_ws_bytes(N, E);
  const size_t need = kErrBytes + tws + align_up((size_t)N * d * 2, 256);
  if (!ws) {
    *ws_bytes = need;
    return MOE_OK;
  }
  if (*ws_bytes < need || !al256(ws)) return MOE_ERR_WORKSPACE;
  if (!offsets || !W1 || !W3 || !W2) return MOE_ERR_INVALID_ARG;
  if (N > 0 && (!xq_perm || !xscale_perm || !h || !out)) return MOE_ERR_INVALID_ARG;
  if ((a_save == nullptr) != (b_save == nullptr)) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {xq_perm, W1, W3, W2, a_save, b_save, h, out};
  for (const void* p : ps)
    if (p && !al16(p)) return MOE_ERR_UNSUPPORTED;
  if ((uintptr_t)xscale_perm & 3) return MOE_ERR_UNSUPPORTED;
  if (!init_once()) return MOE_ERR_CUDA;
  cudaStream_t s = S(stream);
  int* err = static_cast<int*>(ws);
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(int), s));
  // Each element is converted once, into the workspace: a gate-up GEMM that
  // converted its fp8 A tiles in shared memory would convert every element
  // once per 128-column tile of W1 / W3, more than the SM's conversion rate
  // can feed to the tensor cores.
  uint16_t* x_perm = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + kErrBytes + tws);
  cudaError_t e = N > 0 ? launch_dequant_fp8(xq_perm, xscale_perm, N, d, x_perm, s) : cudaSuccess;
  if (e == cudaSuccess)
    e = launch_ffn_fwd(x_perm, offsets, N, d, f, E, W1, W3, W2, a_save, b_save, h, out,
                       static_cast<uint8_t*>(ws) + kErrBytes, err,
                       (flags & MOE_WEIGHTS_PREPACKED) != 0, !(flags & MOE_SINGLE_CTA_TILES), s,
                       row_scale);
  return finish(e, err, flags, s);
}

moe_status_t moe_quantize_mx(const uint16_t* W, long long rows, int K, uint8_t* codes,
                             uint8_t* scales, moe_stream_t stream) {
  if (rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 32) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (!W || !codes || !scales) return MOE_ERR_INVALID_ARG;
  if (!al16(W) || !al16(codes) || !al16(scales)) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = S(stream);
  return finish(launch_quantize_mx(W, rows, K, codes, scales, s), nullptr, 0, s);
}

moe_status_t moe_dispatch_mx(const uint16_t* x, const int32_t* topk_idx, int T, int d, int E, int R,
                             int32_t* counts, int32_t* offsets, int32_t* row_slot,
                             int32_t* slot_row, uint8_t* xq_perm, uint8_t* xscale_perm, void* ws,
                             size_t* ws_bytes, unsigned flags, moe_stream_t stream) {
  moe_status_t st = shape_check(T, d, E, R);
  if (st != MOE_OK) return st;
  if (d % 128) return MOE_ERR_UNSUPPORTED;
  if (!ws_bytes) return MOE_ERR_INVALID_ARG;
  const size_t need = kErrBytes + dispatch_ws_bytes(T, E);
  if (!ws) {
    *ws_bytes = need;
    return MOE_OK;
  }
  if (*ws_bytes < need || !al256(ws)) return MOE_ERR_WORKSPACE;
  if (!counts || !offsets || (T > 0 && (!x || !topk_idx || !row_slot || !slot_row || !xq_perm ||
                                        !xscale_perm)))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!al16(x) || !al16(xq_perm) || !al16(xscale_perm))) return MOE_ERR_UNSUPPORTED;
  if (!init_once()) return MOE_ERR_CUDA;
  cudaStream_t s = S(stream);
  int* err = static_cast<int*>(ws);
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(int), s));
  cudaError_t e;
  {
    Stage st_(s, MOE_STAGE_DISPATCH);
    e = launch_dispatch_mx(x, topk_idx, T, d, E, R, counts, offsets, row_slot, slot_row, xq_perm,
                           xscale_perm, static_cast<uint8_t*>(ws) + kErrBytes, err, s);
  }
  return finish(e, err, flags, s);
}

moe_status_t moe_grouped_ffn_mx(const uint8_t* xq, const uint8_t* xs, const int32_t* offsets,
                                int N, int d, int f, int E, const uint8_t* W1q,
                                const uint8_t* W1s, const uint8_t* W3q, const uint8_t* W3s,
                                const uint8_t* W2q, const uint8_t* W2s, const float* row_scale,
                                uint8_t* hq, uint8_t* hs, uint16_t* out, void* ws,
                                size_t* ws_bytes, unsigned flags, moe_stream_t stream) {
  if (N < 0 || d <= 0 || f <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (!ffn_mx_supported(d, f) || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (!ws_bytes) return MOE_ERR_INVALID_ARG;
  const size_t need = kErrBytes + ffn_mx_ws_bytes(N, d, f, E);
  if (!ws) {
    *ws_bytes = need;
    return MOE_OK;
  }
  if (*ws_bytes < need || !al256(ws)) return MOE_ERR_WORKSPACE;
  if (!offsets || !W1q || !W1s || !W3q || !W3s || !W2q || !W2s) return MOE_ERR_INVALID_ARG;
  if (N > 0 && (!xq || !xs || !out)) return MOE_ERR_INVALID_ARG;
  if ((hq == nullptr) != (hs == nullptr)) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {xq, xs, W1q, W1s, W3q, W3s, W2q, W2s, hq, hs, out};
  for (const void* p : ps)
    if (p && !al16(p)) return MOE_ERR_UNSUPPORTED;
  if (!init_once()) return MOE_ERR_CUDA;
  cudaStream_t s = S(stream);
  int* err = static_cast<int*>(ws);
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(int), s));
  cudaError_t e = launch_ffn_mx(xq, xs, offsets, N, d, f, E, W1q, W1s, W3q, W3s, W2q, W2s,
                                row_scale, hq, hs, out, static_cast<uint8_t*>(ws) + kErrBytes, err,
                                s);
  return finish(e, err, flags, s);
}

moe_status_t moe_prepack_weights(const uint16_t* W1, const uint16_t* W3, const uint16_t* W2, int E,
                                 int d, int f, uint16_t* W1p, uint16_t* W3p, uint16_t* W2p,
                                 moe_stream_t stream) {
  if (E <= 0 || d <= 0 || f <= 0) return MOE_ERR_INVALID_ARG;
  if (!prepack_supported(d, f) || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (!W1 || !W3 || !W2 || !W1p || !W3p || !W2p) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {W1, W3, W2, W1p, W3p, W2p};
  for (const void* p : ps)
    if (!al16(p)) return MOE_ERR_UNSUPPORTED;
  if (!init_once()) return MOE_ERR_CUDA;
  cudaStream_t s = S(stream);
  return finish(launch_prepack(W1, W3, W2, E, d, f, W1p, W3p, W2p, s), nullptr, 0, s);
}

moe_status_t moe_combine(const uint16_t* expert_out, const int32_t* slot_row, const float* topk_w,
                         int T, int d, int R, uint16_t* y, moe_stream_t stream) {
  if (T < 0 || d <= 0 || R <= 0) return MOE_ERR_INVALID_ARG;
  if (R > 32 || d % 8) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * R >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!expert_out || !slot_row || !y) return MOE_ERR_INVALID_ARG;
  if (!al16(expert_out) || !al16(y)) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = S(stream);
  cudaError_t e;
  {
    Stage st_(s, MOE_STAGE_COMBINE);
    e = launch_combine(expert_out, slot_row, topk_w, T, d, R, y, s);
  }
  return finish(e, nullptr, 0, s);
}

static moe_status_t check_layer(const moe_layer_t* L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  moe_status_t st = shape_check(L->T, L->d, L->E, L->R);
  if (st != MOE_OK) return st;
  if (L->f <= 0) return MOE_ERR_INVALID_ARG;
  if (L->f % 8) return MOE_ERR_UNSUPPORTED;
  if (!L->w_gate || !L->W1 || !L->W3 || !L->W2) return MOE_ERR_INVALID_ARG;
  if (!al16(L->W1) || !al16(L->W3) || !al16(L->W2)) return MOE_ERR_UNSUPPORTED;
  if (const moe_shared_t* sh = L->shared) {
    if (sh->fs <= 0 || !sh->W1 || !sh->W3 || !sh->W2) return MOE_ERR_INVALID_ARG;
    if (sh->fs % 8 || !al16(sh->W1) || !al16(sh->W3) || !al16(sh->W2)) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

// Workspace of the shared expert's forward: offsets {0, T}, its tile list,
// its output rows [T,d] and (inference) its hidden rows [T,fs].
static size_t shared_fwd_ws(const moe_layer_t* L) {
  if (!L->shared) return 0;
  const size_t T = L->T, d = L->d, fs = L->shared->fs;
  return 256 + tiles_ws_bytes((int)T, 1) + align_up(T * d * 2, 256) + align_up(T * fs * 2, 256);
}

// fp8 dispatch (MOE_FP8_DISPATCH): the rows' E4M3 codes and their scales.
static size_t fp8_rows_ws(const moe_layer_t* L) {
  const size_t N = (size_t)L->T * L->R, d = L->d;
  return align_up(N * d, 256) + align_up(N * (d / 128) * 4, 256);
}

// microscaled fp8 (MOE_FP8_MX): the rows' codes and scales, then the grouped FFN's own workspace
static size_t mx_rows_ws(const moe_layer_t* L) {
  const size_t N = (size_t)L->T * L->R, d = L->d;
  return align_up(N * d, 256) + align_up(N * mx_scale_row_bytes(L->d), 256) +
         ffn_mx_ws_bytes((int)N, L->d, L->f, L->E);
}

static size_t layer_fwd_ws(const moe_layer_t* L, unsigned flags) {
  const int N = L->T * L->R;
  return kErrBytes + align_up(dispatch_ws_bytes(L->T, L->E), 256) + tiles_ws_bytes(N, L->E) +
         align_up(gate_ws_bytes(L->T, L->d, L->E), 256) + shared_fwd_ws(L) +
         ((flags & MOE_FP8_DISPATCH) ? fp8_rows_ws(L) : 0) +
         ((flags & MOE_FP8_MX) ? mx_rows_ws(L) : 0);
}

moe_status_t moe_layer_fwd(const moe_layer_t* L, const uint16_t* x, uint16_t* y,
                           const moe_saved_t* sv, void* ws, size_t* ws_bytes, unsigned flags,
                           moe_stream_t stream) {
  moe_status_t st = check_layer(L);
  if (st != MOE_OK) return st;
  if ((flags & MOE_WEIGHTS_PREPACKED) && !prepack_supported(L->d, L->f)) return MOE_ERR_UNSUPPORTED;
  const bool fp8 = (flags & MOE_FP8_DISPATCH) != 0;
  if (fp8 && L->d % 128) return MOE_ERR_UNSUPPORTED;
  const bool mx = (flags & MOE_FP8_MX) != 0;
  if (mx && (fp8 || (flags & MOE_WEIGHTS_PREPACKED) || !ffn_mx_supported(L->d, L->f)))
    return MOE_ERR_UNSUPPORTED;
  if (!ws_bytes) return MOE_ERR_INVALID_ARG;
  const size_t need = layer_fwd_ws(L, flags);
  if (!ws) {
    *ws_bytes = need;
    return MOE_OK;
  }
  if (*ws_bytes < need || !al256(ws)) return MOE_ERR_WORKSPACE;
  if (L->T == 0) return MOE_OK;   // nothing to route: no buffer is touched
  if (!sv || !x || !y) return MOE_ERR_INVALID_ARG;
  if (!sv->logits || !sv->topk_idx || !sv->topk_w || !sv->counts || !sv->offsets ||
      !sv->row_slot || !sv->slot_row || !sv->o || (!mx && (!sv->x_perm || !sv->h)))
    return MOE_ERR_INVALID_ARG;
  const moe_mx_weights_t* MX = L->mx;
  if (mx && (!MX || !MX->W1q || !MX->W1s || !MX->W3q || !MX->W3s || !MX->W2q || !MX->W2s))
    return MOE_ERR_INVALID_ARG;
  if (mx) {
    const void* qs[] = {MX->W1q, MX->W1s, MX->W3q, MX->W3s, MX->W2q, MX->W2s};
    for (const void* p : qs)
      if (!al16(p)) return MOE_ERR_UNSUPPORTED;
  }
  if ((sv->a == nullptr) != (sv->b == nullptr)) return MOE_ERR_INVALID_ARG;
  const moe_shared_t* SH = L->shared;
  if (SH && ((sv->sa == nullptr) != (sv->sb == nullptr) || (sv->sa && !sv->sh)))
    return MOE_ERR_INVALID_ARG;
  const void* ps[] = {x, y, sv->x_perm, sv->a, sv->b, sv->h, sv->o,
                      SH ? sv->sa : nullptr, SH ? sv->sb : nullptr, SH ? sv->sh : nullptr};
  for (const void* p : ps)
    if (p && !al16(p)) return MOE_ERR_UNSUPPORTED;
  if (!init_once()) return MOE_ERR_CUDA;
  const int T = L->T, d = L->d, E = L->E, R = L->R, f = L->f, N = T * R;
  const bool pairs = !(flags & MOE_SINGLE_CTA_TILES);
  cudaStream_t s = S(stream);
  const bool side = SH && !(flags & MOE_SHARED_SERIAL);
  cudaStream_t s2 = side ? side_stream() : s;
  if (side && !s2) return MOE_ERR_CUDA;   // (the caller's stream may be the null stream)
  Carve c(ws);
  int* err = static_cast<int*>(c.take(kErrBytes));
  void* dws = c.take(dispatch_ws_bytes(T, E));
  void* tws = c.take(tiles_ws_bytes(N, E));
  void* gws = c.take(gate_ws_bytes(T, d, E));
  uint8_t* xq = nullptr;
  float* xs = nullptr;
  if (fp8) {
    xq = static_cast<uint8_t*>(c.take((size_t)N * d));
    xs = static_cast<float*>(c.take((size_t)N * (d / 128) * 4));
  }
  uint8_t *mq = nullptr, *ms = nullptr;
  void* mws = nullptr;
  if (mx) {
    mq = static_cast<uint8_t*>(c.take((size_t)N * d));
    ms = static_cast<uint8_t*>(c.take((size_t)N * mx_scale_row_bytes(d)));
    mws = c.take(ffn_mx_ws_bytes(N, d, f, E));
  }
  int32_t* s_off = nullptr;
  void* s_tws = nullptr;
  uint16_t *s_out = nullptr, *s_h = nullptr;
  if (SH) {
    s_off = static_cast<int32_t*>(c.take(256));
    s_tws = c.take(tiles_ws_bytes(T, 1));
    s_out = static_cast<uint16_t*>(c.take((size_t)T * d * 2));
    s_h = static_cast<uint16_t*>(c.take((size_t)T * SH->fs * 2));
    if (sv->sh) s_h = sv->sh;
  }
  // the shared expert: SwiGLU of every token (one expert holding all T rows)
  auto shared_fwd = [&]() -> cudaError_t {
    Stage st_(s2, MOE_STAGE_SHARED_FWD);
    TraceMute mute_;
    cudaError_t e = launch_one_expert_offsets(s_off, T, s2);
    if (e == cudaSuccess)
      e = launch_ffn_fwd(x, s_off, T, d, SH->fs, 1, SH->W1, SH->W3, SH->W2, sv->sa, sv->sb, s_h,
                         s_out, s_tws, err, false, pairs, s2);
    return e;
  };
  Join join{s, s2};
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(int), s));
  {
    Stage st_(s, MOE_STAGE_GATE);
    MOE_TRY(launch_gate(x, L->w_gate, L->bias, T, d, E, sv->logits, gws, err, s));
  }
  if (side) {   // fork: the shared expert overlaps top-R, dispatch and the routed FFN
    MOE_TRY(stream_wait(s2, s));
    join.armed = true;
    MOE_TRY(shared_fwd());
  }
  {
    Stage st_(s, MOE_STAGE_TOPK);
    MOE_TRY(launch_topk(sv->logits, T, E, R, sv->topk_idx, sv->topk_w, s));
  }
  {
    Stage st_(s, MOE_STAGE_DISPATCH);
    if (fp8) {   // the rows travel as fp8 codes and scales; the GEMMs read them dequantised
      MOE_TRY(launch_dispatch_fp8(x, sv->topk_idx, T, d, E, R, sv->counts, sv->offsets,
                                  sv->row_slot, sv->slot_row, xq, xs, dws, err, s));
      MOE_TRY(launch_dequant_fp8(xq, xs, N, d, sv->x_perm, s));
    } else if (mx) {   // microscaled fp8 rows, multiplied as they are by the fp8 tensor cores
      MOE_TRY(launch_dispatch_mx(x, sv->topk_idx, T, d, E, R, sv->counts, sv->offsets,
                                 sv->row_slot, sv->slot_row, mq, ms, dws, err, s));
    } else {
      MOE_TRY(launch_dispatch(x, sv->topk_idx, T, d, E, R, sv->counts, sv->offsets, sv->row_slot,
                              sv->slot_row, sv->x_perm, dws, err, s));
    }
  }
  if (mx)
    MOE_TRY(launch_ffn_mx(mq, ms, sv->offsets, N, d, f, E, MX->W1q, MX->W1s, MX->W3q, MX->W3s,
                          MX->W2q, MX->W2s, nullptr, nullptr, nullptr, sv->o, mws, err, s));
  else
    MOE_TRY(launch_ffn_fwd(sv->x_perm, sv->offsets, N, d, f, E, L->W1, L->W3, L->W2, sv->a,
                           sv->b, sv->h, sv->o, tws, err, (flags & MOE_WEIGHTS_PREPACKED) != 0,
                           pairs, s));
  if (SH && !side) MOE_TRY(shared_fwd());
  if (side) MOE_TRY(join.now());
  cudaError_t e;
  {
    Stage st_(s, MOE_STAGE_COMBINE);
    e = launch_combine(sv->o, sv->slot_row, sv->topk_w, T, d, R, y, s, s_out);
  }
  return finish(e, err, flags, s);
}

static size_t layer_bwd_ws(const moe_layer_t* L) {
  const size_t T = L->T, d = L->d, E = L->E, R = L->R, f = L->f, N = T * R;
  size_t n = kErrBytes;
  n += tiles_ws_bytes((int)N, (int)E);
  n += align_up(N * d * 2, 256);        // do
  n += align_up(N * 2 * f * 2, 256);    // [da | db]
  n += align_up(N * d * 2, 256);        // dx_perm
  n += align_up(N * 4, 256);            // dlogits per slot (token order)
  n += align_up(E * d * 4, 256);        // W_g^T
  n += dwg_ws_bytes((int)T, (int)d, (int)E);   // router weight gradient: S, partials, maps
  if (L->shared) {                      // shared expert: offsets, tiles, [das | dbs], dxs
    const size_t fs = L->shared->fs;
    n += 256 + tiles_ws_bytes((int)T, 1) + align_up(T * 2 * fs * 2, 256) + align_up(T * d * 2, 256);
  }
  return n;
}

moe_status_t moe_layer_bwd(const moe_layer_t* L, const uint16_t* x, const moe_saved_t* sv,
                           const uint16_t* dy, uint16_t* dx, float* dW_gate, float* dW1,
                           float* dW3, float* dW2, void* ws, size_t* ws_bytes, unsigned flags,
                           moe_stream_t stream) {
  moe_status_t st = check_layer(L);
  if (st != MOE_OK) return st;
  if (L->d % 64 || L->f % 64 || (flags & MOE_WEIGHTS_PREPACKED)) return MOE_ERR_UNSUPPORTED;
  const moe_shared_t* SH = L->shared;
  if (SH && SH->fs % 64) return MOE_ERR_UNSUPPORTED;
  if (!ws_bytes) return MOE_ERR_INVALID_ARG;
  const size_t need = layer_bwd_ws(L);
  if (!ws) {
    *ws_bytes = need;
    return MOE_OK;
  }
  if (*ws_bytes < need || !al256(ws)) return MOE_ERR_WORKSPACE;
  if (!dW_gate || !dW1 || !dW3 || !dW2) return MOE_ERR_INVALID_ARG;
  if (SH && (!SH->dW1 || !SH->dW3 || !SH->dW2)) return MOE_ERR_INVALID_ARG;
  if (SH && (!al16(SH->dW1) || !al16(SH->dW3) || !al16(SH->dW2))) return MOE_ERR_UNSUPPORTED;
  if (L->T == 0) {   // no tokens: every gradient is zero
    if (!al16(dW_gate) || !al16(dW1) || !al16(dW3) || !al16(dW2)) return MOE_ERR_UNSUPPORTED;
    if (!init_once()) return MOE_ERR_CUDA;
    cudaStream_t s0 = S(stream);
    const size_t d = L->d, E = L->E, f = L->f;
    if (SH) {
      const size_t fs = SH->fs;
      MOE_TRY(cudaMemsetAsync(SH->dW1, 0, sizeof(float) * fs * d, s0));
      MOE_TRY(cudaMemsetAsync(SH->dW3, 0, sizeof(float) * fs * d, s0));
      MOE_TRY(cudaMemsetAsync(SH->dW2, 0, sizeof(float) * fs * d, s0));
    }
    MOE_TRY(cudaMemsetAsync(dW_gate, 0, sizeof(float) * d * E, s0));
    MOE_TRY(cudaMemsetAsync(dW1, 0, sizeof(float) * E * f * d, s0));
    MOE_TRY(cudaMemsetAsync(dW3, 0, sizeof(float) * E * f * d, s0));
    return finish(cudaMemsetAsync(dW2, 0, sizeof(float) * E * f * d, s0), nullptr, flags, s0);
  }
  if (!sv || !x || !dy || !dx) return MOE_ERR_INVALID_ARG;
  if (!sv->a || !sv->b || !sv->h || !sv->o || !sv->x_perm || !sv->topk_idx || !sv->topk_w ||
      !sv->offsets || !sv->slot_row || !sv->row_slot)
    return MOE_ERR_INVALID_ARG;
  if (SH && (!sv->sa || !sv->sb || !sv->sh)) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {x, dy, dx, dW_gate, dW1, dW3, dW2, sv->a, sv->b, sv->h, sv->o, sv->x_perm};
  for (const void* p : ps)
    if (!al16(p)) return MOE_ERR_UNSUPPORTED;
  if (SH && (!al16(sv->sa) || !al16(sv->sb) || !al16(sv->sh))) return MOE_ERR_UNSUPPORTED;
  if (!init_once()) return MOE_ERR_CUDA;
  const int T = L->T, d = L->d, E = L->E, R = L->R, f = L->f, N = T * R;
  const bool pairs = !(flags & MOE_SINGLE_CTA_TILES);
  cudaStream_t s = S(stream);
  const bool side = SH && !(flags & MOE_SHARED_SERIAL);
  cudaStream_t s2 = side ? side_stream() : s;
  if (side && !s2) return MOE_ERR_CUDA;   // (the caller's stream may be the null stream)
  Carve c(ws);
  int* err = static_cast<int*>(c.take(kErrBytes));
  void* tws = c.take(tiles_ws_bytes(N, E));
  uint16_t* dO = static_cast<uint16_t*>(c.take((size_t)N * d * 2));
  uint16_t* dab = static_cast<uint16_t*>(c.take((size_t)N * 2 * f * 2));
  uint16_t* dxp = static_cast<uint16_t*>(c.take((size_t)N * d * 2));
  float* dsel_tok = static_cast<float*>(c.take((size_t)N * 4));
  float* wgT = static_cast<float*>(c.take((size_t)E * d * 4));
  void* dwg_ws = c.take(dwg_ws_bytes(T, d, E));
  int32_t* s_off = nullptr;
  void* s_tws = nullptr;
  uint16_t *s_dab = nullptr, *s_dx = nullptr;
  if (SH) {
    s_off = static_cast<int32_t*>(c.take(256));
    s_tws = c.take(tiles_ws_bytes(T, 1));
    s_dab = static_cast<uint16_t*>(c.take((size_t)T * 2 * SH->fs * 2));
    s_dx = static_cast<uint16_t*>(c.take((size_t)T * d * 2));
  }
  // the shared expert's backward, with dy as its output gradient
  auto shared_bwd = [&]() -> cudaError_t {
    Stage st_(s2, MOE_STAGE_SHARED_BWD);
    TraceMute mute_;
    cudaError_t e = launch_one_expert_offsets(s_off, T, s2);
    if (e == cudaSuccess)
      e = launch_ffn_bwd(x, s_off, T, d, SH->fs, 1, SH->W1, SH->W3, SH->W2, sv->sa, sv->sb, sv->sh,
                         dy, s_dab, s_dx, SH->dW1, SH->dW3, SH->dW2, s_tws, err, pairs, s2);
    return e;
  };
  Join join{s, s2};
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(int), s));
  if (side) {   // fork: the shared expert's backward overlaps the routed one
    MOE_TRY(stream_wait(s2, s));
    join.armed = true;
    MOE_TRY(shared_bwd());
  }
  if (N == 0) {
    MOE_TRY(cudaMemsetAsync(dW_gate, 0, sizeof(float) * d * E, s));
    MOE_TRY(cudaMemsetAsync(dW1, 0, sizeof(float) * E * f * d, s));
    MOE_TRY(cudaMemsetAsync(dW3, 0, sizeof(float) * E * f * d, s));
    return finish(cudaMemsetAsync(dW2, 0, sizeof(float) * E * f * d, s), err, flags, s);
  }
  {
    Stage st_(s, MOE_STAGE_BWD_ROUTE);
    MOE_TRY(launch_bwd_route(dy, sv->o, sv->slot_row, sv->topk_w, T, d, R, dO, dsel_tok, s));
  }
  MOE_TRY(launch_ffn_bwd(sv->x_perm, sv->offsets, N, d, f, E, L->W1, L->W3, L->W2, sv->a, sv->b,
                         sv->h, dO, dab, dxp, dW1, dW3, dW2, tws, err, pairs, s));
  {
    Stage st_(s, MOE_STAGE_BWD_DWG);
    MOE_TRY(launch_dwg(x, sv->topk_idx, dsel_tok, T, d, E, R, dW_gate, dwg_ws, err, pairs, s));
  }
  if (SH && !side) MOE_TRY(shared_bwd());
  if (side) MOE_TRY(join.now());
  cudaError_t e;
  {
    Stage st_(s, MOE_STAGE_BWD_DXC);
    e = launch_wg_transpose(L->w_gate, d, E, wgT, s);
    if (e == cudaSuccess)
      e = launch_dx_combine(dxp, sv->slot_row, sv->topk_idx, dsel_tok, wgT, T, d, E, R, dx, s,
                            s_dx);
  }
  return finish(e, err, flags, s);
}

}  // extern "C"
