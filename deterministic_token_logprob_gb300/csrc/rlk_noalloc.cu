// rlk_noalloc.cu -- rlk_linear_logp_fwd_noalloc: the forward without a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// The forward's only scratch is the per-(leaf, token) statistics array. Here it
// lives in one file-scope device array of fixed size, created when the module is
// loaded on a GPU and held by every GPU that loads the library until the process
// exits. Host code cannot use the array's name as a device address (on the host it
// names a shadow variable), so the device address is looked up once per device
// with cudaGetSymbolAddress and cached for the life of the process (after a
// cudaDeviceReset the module is loaded anew and the cached address would be stale:
// calling this entry point after a reset is not supported).
//
// All calls on a device share this one array and it keeps the previous call's
// contents. The one part that must start at zero, the tile kernel's work-item
// counter at the end of the workspace, is zeroed on the stream by every call before
// its kernel runs; the tile kernel writes every (leaf, token) entry that the merge
// kernel then reads. Two calls whose work
// overlaps on the GPU (e.g. on different streams without ordering between them)
// race on the array and produce wrong results; order them.
#include <cuda_runtime.h>

#include <mutex>

#include "rlk.h"

namespace {

constexpr size_t kScratchBytes = RLK_FWD_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_fwd_scratch on the current device (looked up on the first
// call per device, with that device current).
rlk_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RLK_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return RLK_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || !p) return RLK_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return RLK_OK;
}

}  // namespace

extern "C" rlk_status rlk_linear_logp_fwd_noalloc(const void* h, const void* W, const int64_t* y,
                                                  int64_t T, int64_t H, int64_t V_local,
                                                  int64_t vocab_start, int64_t V_true,
                                                  float* logp, float* lse,
                                                  rlk_lse_partial* partial, int32_t* err_flag,
                                                  void* stream) {
  const size_t need = rlk_linear_logp_fwd_workspace(T, H, V_local);
  if (need > kScratchBytes) return RLK_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const rlk_status st = scratch_address(&scratch);
    if (st != RLK_OK) return st;
  }
  return rlk_linear_logp_fwd(h, W, y, T, H, V_local, vocab_start, V_true, logp, lse, partial,
                             err_flag, scratch, kScratchBytes, stream);
}
