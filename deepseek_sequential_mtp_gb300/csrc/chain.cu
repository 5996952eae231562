#include "common.cuh"
MTP_DEFINE_ERROR_WORD(mtp_take_errors_chain)
extern "C" size_t mtp_chain_workspace_bytes(const mtp_dims*) { return 0; }
extern "C" mtp_status mtp_chain_forward(const mtp_dims*, const mtp_weights*, const int32_t*, const int32_t*,
                                        const int32_t*, const void*, void*, void*, size_t, cudaStream_t) {
  return MTP_ERR_UNSUPPORTED;
}
extern "C" mtp_status mtp_chain_loss(const mtp_dims*, const mtp_weights*, const int32_t*, const int32_t*,
                                     const int32_t*, const void*, float, int, int, double*, float*, float*,
                                     void*, void*, size_t, cudaStream_t) {
  return MTP_ERR_UNSUPPORTED;
}
