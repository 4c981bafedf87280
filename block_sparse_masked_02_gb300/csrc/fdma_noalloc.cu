// Allocation-free forward entry point.
//
// Some callers cannot allocate device memory at the point where they need
// attention: code running inside a custom allocator or memory-pool callback,
// plugins of host frameworks that hand out only fixed buffers, and processes
// that must not grow their device footprint after start-up.  For them,
// fdma_fwd_noalloc() runs the same classification + forward as fdma_fwd(),
// but its workspace is a fixed-size array compiled into this library instead
// of a caller-provided buffer.  The caller still passes the inputs and the
// outputs (out, lse).
//
// The array lives in device global memory of every GPU that loads the
// library and stays there until the process exits.  Its address is looked up
// on the host once per device (cudaGetSymbolAddress, with that device
// current) on the first call made on that device.
#include <mutex>
#include <unordered_map>

#include "fdma_internal.h"

namespace fdma {
namespace {

// 16 MiB: enough for the forward workspace of about 4000 tiles of 128 x 128
// (for example B * Hkv * ceil(Nq/128) * ceil(Nk/128) <= 4095).
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(16) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device (nullptr on failure).
void* noalloc_scratch_address() {
  static std::mutex mu;
  static std::unordered_map<int, void*> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
  cache[dev] = ptr;
  return ptr;
}

}  // namespace
}  // namespace fdma

extern "C" {

int fdma_fwd_noalloc(const fdma_args* args, void* out, float* lse, void* stream) {
  if (args == nullptr) return FDMA_ERR_INVALID;
  const size_t need = fdma_workspace_size(args, 0);
  if (need == 0) {
    fdma_args probe = *args;
    probe.workspace = nullptr;
    probe.workspace_bytes = 0;
    return fdma_fwd(&probe, out, lse, stream);  // reports the argument error; launches nothing
  }
  if (need > fdma::kNoAllocScratchBytes) return FDMA_ERR_WORKSPACE;
  void* scratch = fdma::noalloc_scratch_address();
  if (scratch == nullptr) return FDMA_ERR_CUDA;
  fdma_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = fdma::kNoAllocScratchBytes;
  a.flags &= ~FDMA_FLAG_REUSE_CLASSIFICATION;  // the shared array may hold another call's classes
  return fdma_fwd(&a, out, lse, stream);
}

}  // extern "C"
