// moe_dispatch_noalloc: the dispatch step for callers that cannot allocate
// device memory, using scratch that the library reserves statically.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// embedded in a host application or framework whose allocator owns all device
// memory (a caching allocator or a fixed memory budget that forbids raw
// allocations), and latency-critical loops where cudaMalloc's implicit device
// synchronisation is not acceptable.  For them this variant of moe_dispatch
// keeps its scratch (per-block expert histograms, their scan and the device
// error word) in a file-scope device array of fixed size, which every GPU that
// loads the library holds until the process exits.  Its argument checks,
// status codes, recorded CUDA errors and trace events are those of
// moe_dispatch.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

// Scratch reserved per device: 4 MiB.
constexpr size_t kNoAllocScratchBytes = 4u << 20;
constexpr size_t kErrBytes = 256;

static __device__ __align__(256) unsigned char g_dispatch_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {nullptr};

// Set-up, once per device with that device current: the device address of
// g_dispatch_scratch (in host code the symbol is only a host-side stand-in, not
// a device address) and the dispatch kernels' shared-memory limit.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    e = moe::dispatch_set_smem_limits();
    if (e != cudaSuccess) return e;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return cudaSuccess;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status_t moe_dispatch_noalloc(const uint16_t* x, const int32_t* topk_idx, int T,
                                             int d, int E, int R, int32_t* counts,
                                             int32_t* offsets, int32_t* row_slot,
                                             int32_t* slot_row, uint16_t* x_perm, unsigned flags,
                                             moe_stream_t stream) {
  moe_status_t st = moe::shape_check(T, d, E, R);
  if (st != MOE_OK) return st;
  // the static scratch must hold the error word and the histograms of this call
  if (kErrBytes + moe::dispatch_ws_bytes(T, E) > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
  if (!counts || !offsets || (T > 0 && (!topk_idx || !row_slot || !slot_row)))
    return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if (x && (!al16(x) || !al16(x_perm))) return MOE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return moe::cuda_failed(e);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(scratch);
  // the array keeps the previous call's contents: the error word must start at zero
  e = cudaMemsetAsync(err, 0, sizeof(int), s);
  if (e != cudaSuccess) return moe::cuda_failed(e);
  moe::trace_begin(MOE_STAGE_DISPATCH, s);
  e = moe::launch_dispatch(x, topk_idx, T, d, E, R, counts, offsets, row_slot, slot_row, x_perm,
                           static_cast<uint8_t*>(scratch) + kErrBytes, err, s);
  moe::trace_end(MOE_STAGE_DISPATCH, s);
  return moe::finish(e, err, flags, s);
}
