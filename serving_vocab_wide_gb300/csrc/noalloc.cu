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
// it needs to start at zero: every slot the finalize kernel reads (each
// warp's chunk partial, each stats CTA's CSR flag) is written by the stats
// kernel of the same call before it is read, so stale contents never reach a
// result.  Two calls whose kernels overlap on the GPU (different streams, no
// ordering between them) race on the array and corrupt each other's results.
//
// The scratch used is the current device's, so the stream must belong to
// that device: a stream of another GPU would run the kernels there with an
// address of this GPU's array.  Such a call is rejected before any launch.
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

namespace svw {
svw_status verify_check_args(const void *target_logits, const void *draft_logits, svw_dtype dtype, int32_t V,
                             int32_t N, const int32_t *cu_draft, int64_t total_draft_rows, int32_t max_len,
                             const int32_t *draft_tokens, float temperature, int32_t *accept_len,
                             int32_t *next_token, int32_t *status);
}

extern "C" svw_status spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                                          svw_dtype dtype, int32_t V, int32_t N, const int32_t *cu_draft,
                                          int64_t total_draft_rows, int32_t max_len,
                                          const int32_t *draft_tokens, float temperature, uint64_t seed,
                                          int32_t *accept_len, int32_t *next_token, int32_t *status,
                                          void *stream) {
  // spec_verify's own argument checks first, so that the codes are the same
  const svw_status st = svw::verify_check_args(target_logits, draft_logits, dtype, V, N, cu_draft,
                                               total_draft_rows, max_len, draft_tokens, temperature, accept_len,
                                               next_token, status);
  if (st != SVW_OK) return st;
  const size_t need = svw_verify_workspace_size(N, total_draft_rows, V, dtype);
  if (need == 0) return SVW_ERR_INVALID_ARG;
  if (need > kScratchBytes) return SVW_ERR_UNSUPPORTED;  // batch too large for the fixed scratch
  // the scratch is the current device's: the stream must run on that device
  int cur = 0, sdev = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return SVW_ERR_CUDA;
  if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) return SVW_ERR_INVALID_ARG;
  if (sdev != cur) return SVW_ERR_INVALID_ARG;
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SVW_ERR_CUDA;
  return spec_verify(target_logits, draft_logits, dtype, V, N, cu_draft, total_draft_rows, max_len,
                     draft_tokens, temperature, seed, accept_len, next_token, status, scratch, kScratchBytes,
                     stream);
}
