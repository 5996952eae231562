// mtp_chain_loss_noalloc: mtp_chain_loss for callers that cannot allocate
// device memory.
//
// Its workspace is a fixed array in this library's device image instead of a
// caller buffer.  Every GPU that loads the library holds the array until the
// process exits.  The array's device address is looked up once per device
// (cudaGetSymbolAddress with that device current) on the first call made
// while the device is current; that first call should therefore come before
// any stream capture.  The entry point itself allocates nothing: no
// cudaMalloc, cudaFree or allocating library routine.  All calls share the
// one array, so calls that overlap on the GPU (other streams, other threads)
// race on it; the chain rewrites every scratch element it reads, so no part
// of the array has to start at zero.  The cached address belongs to the
// device's primary context: after cudaDeviceReset (or anything else that
// destroys that context) it is stale, so a process that resets a device must
// not call this entry point on that device again.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = MTP_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[mtp::kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
mtp_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MTP_ERR_CUDA;
  if (dev < 0 || dev >= mtp::kMaxDevices) return MTP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      (void)cudaGetLastError();
      return MTP_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return MTP_OK;
}

}  // namespace

extern "C" mtp_status mtp_chain_loss_noalloc(const mtp_dims* dims, const mtp_weights* w, const int32_t* tokens,
                                             const int32_t* seg, const int32_t* pos, const void* h0, float lambda,
                                             int den, int with_main, double* sums_counts, float* losses,
                                             float* row_loss, void* h_out, cudaStream_t stream) {
  if (!dims) return MTP_ERR_INVALID_ARG;
  const size_t need = mtp_chain_workspace_bytes(dims);
  // invalid or unsupported dimensions: the workspace entry point's own checks
  // give the status (they fail before any launch)
  if (need == 0)
    return mtp_chain_loss(dims, w, tokens, seg, pos, h0, lambda, den, with_main, sums_counts, losses, row_loss,
                          h_out, nullptr, 0, stream);
  if (need > kScratchBytes) return MTP_ERR_WORKSPACE;
  void* scratch = nullptr;
  const mtp_status st = scratch_for_current_device(&scratch);
  if (st != MTP_OK) return st;
  return mtp_chain_loss(dims, w, tokens, seg, pos, h0, lambda, den, with_main, sums_counts, losses, row_loss,
                        h_out, scratch, kScratchBytes, stream);
}
