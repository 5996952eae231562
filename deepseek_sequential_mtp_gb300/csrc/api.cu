// Library-wide entry points: status strings, ABI version and the device
// error-word check that ORs the words of every kernel file.
#include "common.cuh"

unsigned int mtp_take_errors_chain();
unsigned int mtp_take_errors_gemm();
unsigned int mtp_take_errors_attn();

extern "C" const char* mtp_status_string(int s) {
  switch (s) {
    case MTP_OK: return "ok";
    case MTP_ERR_INVALID_ARG: return "invalid argument";
    case MTP_ERR_SHAPE: return "inconsistent shapes";
    case MTP_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case MTP_ERR_WORKSPACE: return "workspace too small";
    case MTP_ERR_CUDA: return "CUDA call failed";
    case MTP_ERR_DEVICE: return "device error word set";
    case MTP_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    default: return "unknown status";
  }
}

extern "C" int mtp_abi_version(void) { return MTP_ABI_VERSION; }

extern "C" mtp_status mtp_check_errors(cudaStream_t stream, unsigned int* flags) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MTP_ERR_CUDA;
  unsigned int v = mtp_take_errors_chain() | mtp_take_errors_gemm() | mtp_take_errors_attn();
  if (flags) *flags = v;
  return v ? MTP_ERR_DEVICE : MTP_OK;
}
