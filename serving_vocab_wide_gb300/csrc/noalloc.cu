// noalloc.cu -- spec_verify for callers that cannot allocate device memory.
//
// spec_verify needs a device workspace from its caller.  Some callers have no
// way to provide one: a plain C serving loop that owns no device allocator, a
// plug-in that runs inside a host engine which forbids allocation once its
// memory pool is sized (a cudaMalloc there would also synchronise the whole
// device in the middle of a decode step), or a kernel-launch wrapper that only
// forwards tensors it was given.  For them this file keeps one fixed scratch
// area in the library itself and runs the same verification kernels on it.
//
// The scratch is a file-scope __device__ array of SVW_NOALLOC_SCRATCH_BYTES.
// It exists on every GPU that loads this library, for the life of the process.
// Host code cannot use the array's name as a device address, so the address is
// looked up once per device with cudaGetSymbolAddress (with that device
// current) and cached; the first call on a device does that lookup.
//
// Every call shares the one array and leaves its contents behind.  Nothing in
// it needs to start at zero: the verification prologue kernel resets every
// counter and flag it relies on at the start of each call.  Two calls whose
// kernels overlap on the GPU (different streams, no ordering between them)
// race on the array and corrupt each other's results.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "svw_internal.h"

namespace {

constexpr size_t kScratchBytes = SVW_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// device address of g_scratch on the current device (looked up once per device)
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" svw_status spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                                          svw_dtype dtype, int32_t V, int32_t N, const int32_t *cu_draft,
                                          int64_t total_draft_rows, int32_t max_len,
                                          const int32_t *draft_tokens, float temperature, uint64_t seed,
                                          int32_t *accept_len, int32_t *next_token, int32_t *status,
                                          void *stream) {
  const size_t need = svw_verify_workspace_size(N, total_draft_rows, V, dtype);
  if (need == 0) {
    // invalid shape: let spec_verify's own validation name the problem
    return spec_verify(target_logits, draft_logits, dtype, V, N, cu_draft, total_draft_rows, max_len,
                       draft_tokens, temperature, seed, accept_len, next_token, status, nullptr, 0, stream);
  }
  if (need > kScratchBytes) return SVW_ERR_UNSUPPORTED;  // batch too large for the fixed scratch
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SVW_ERR_CUDA;
  return spec_verify(target_logits, draft_logits, dtype, V, N, cu_draft, total_draft_rows, max_len,
                     draft_tokens, temperature, seed, accept_len, next_token, status, scratch, kScratchBytes,
                     stream);
}
