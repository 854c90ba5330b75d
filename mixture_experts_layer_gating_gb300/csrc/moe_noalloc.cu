// moe_permute_noalloc: moe_permute for callers that cannot allocate device
// memory.
//
// Some hosts give an operator nothing but its input and output buffers and
// forbid device allocation while a request runs -- a serving runtime that
// plans all device memory once at start-up, or a plugin interface with no
// workspace argument.  Such a caller cannot hand moe_permute the workspace it
// uses for its per-segment expert histograms.  This entry point keeps that
// scratch in a fixed array in the library's own device memory instead, so the
// caller passes only the inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kMaxScratchInts * 4 bytes, 256 KiB) until the process
// exits.  Host code cannot use the variable's name as a device address, so
// the first call on each device looks the address up with
// cudaGetSymbolAddress, with that device current, and reuses it afterwards.
#include <cuda_runtime.h>

#include <mutex>

#include "moe_internal.h"

namespace {

// Per-(expert, routing segment) histogram entries the array holds: at most
// 512 experts times 128 segments.  One more int at the front is the error word
// the routing kernels write to.
constexpr int kMaxScratchInts = 65536;

static __device__ __align__(256) int32_t g_permute_scratch[1 + kMaxScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_permute_scratch on the current device (nullptr on error).
int32_t* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int moe_permute_noalloc(const moe_config_t* cfg, const int32_t* topk_ids,
                                   const void* x, int32_t* counts, int32_t* offsets,
                                   int32_t* sorted_rows, int32_t* dest, void* x_perm,
                                   void* stream) {
  // the same configuration checks as moe_permute, then the scratch-size guard
  if (!moe::cfg_valid(cfg)) return MOE_ERR_INVALID_ARG;
  if (!moe::combo_supported(cfg)) return MOE_ERR_UNSUPPORTED;
  if (!topk_ids || !counts || !offsets || !sorted_rows || !dest) return MOE_ERR_INVALID_ARG;
  if (x && (!x_perm || (reinterpret_cast<uintptr_t>(x) & 15u) ||
            (reinterpret_cast<uintptr_t>(x_perm) & 15u)))
    return MOE_ERR_INVALID_ARG;
  const long long R = static_cast<long long>(cfg->T) * cfg->k;  // <= 2^30 (cfg_valid)
  // the histogram needs E * route_segments(R) entries (never more than the
  // array holds while R <= 2^30); the check stays as a guard
  if (static_cast<long long>(cfg->E) * moe::route_segments(R) > kMaxScratchInts)
    return MOE_ERR_INVALID_ARG;
  int32_t* scratch = scratch_on_current_device();
  if (!scratch) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the error word keeps the last call's flags: start each call from zero
  // (every histogram entry is overwritten by the call, so it needs no clearing)
  if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* err = scratch;
  int32_t* seg = scratch + 1;
  if (moe::launch_init_routing(topk_ids, static_cast<int>(R), cfg->E, counts, offsets,
                               sorted_rows, dest, seg, err, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (x && R > 0 &&
      moe::launch_permute_gather(x, sorted_rows, static_cast<int>(R), cfg->k, cfg->T,
                                 static_cast<size_t>(cfg->D) * moe::act_bytes(cfg->act_dtype),
                                 x_perm, err, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
