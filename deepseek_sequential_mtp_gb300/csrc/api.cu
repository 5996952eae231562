// Library-wide entry points: status strings, ABI version and the device
// error-word check that ORs the words of every kernel file.
#include <atomic>

#include "common.cuh"

namespace mtp {
namespace {
std::atomic<unsigned long long> g_launches{0};
struct Hook {
  cudaEvent_t* ev = nullptr;
  int n = 0;
  int* recorded = nullptr;
  int open = -1;  // index of the pair whose start has been recorded
};
Hook g_hooks[MTP_KC_COUNT];
}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void prof_begin(int kernel_class, cudaStream_t stream) {
  if (kernel_class < 0 || kernel_class >= MTP_KC_COUNT) return;
  Hook& h = g_hooks[kernel_class];
  if (!h.ev || *h.recorded >= h.n) return;
  h.open = *h.recorded;
  cudaEventRecord(h.ev[2 * h.open], stream);
}

void prof_end(int kernel_class, cudaStream_t stream) {
  if (kernel_class < 0 || kernel_class >= MTP_KC_COUNT) return;
  Hook& h = g_hooks[kernel_class];
  if (!h.ev || h.open < 0) return;
  cudaEventRecord(h.ev[2 * h.open + 1], stream);
  *h.recorded = h.open + 1;
  h.open = -1;
}
}  // namespace mtp

extern "C" mtp_status mtp_profile_kernel(int kernel_class, cudaEvent_t* events, int n_pairs, int* recorded) {
  if (kernel_class < 0 || kernel_class >= MTP_KC_COUNT) return MTP_ERR_INVALID_ARG;
  mtp::Hook& h = mtp::g_hooks[kernel_class];
  if (!events) {
    h = mtp::Hook{};
    return MTP_OK;
  }
  if (n_pairs < 0 || !recorded) return MTP_ERR_INVALID_ARG;
  h.ev = events;
  h.n = n_pairs;
  h.recorded = recorded;
  h.open = -1;
  *recorded = 0;
  return MTP_OK;
}

extern "C" unsigned long long mtp_kernel_launches(void) { return mtp::g_launches.load(); }

unsigned int mtp_take_errors_chain();
unsigned int mtp_take_errors_gemm();
unsigned int mtp_take_errors_attn();
unsigned int mtp_take_errors_verify();
unsigned int mtp_take_errors_draft();
unsigned int mtp_take_errors_fp8();
unsigned int mtp_take_errors_dgemm();

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
  const unsigned int parts[7] = {mtp_take_errors_chain(), mtp_take_errors_gemm(), mtp_take_errors_attn(),
                                 mtp_take_errors_verify(), mtp_take_errors_draft(), mtp_take_errors_fp8(),
                                 mtp_take_errors_dgemm()};
  const unsigned int from[7] = {MTP_DEVERR_FROM_CHAIN, MTP_DEVERR_FROM_GEMM, MTP_DEVERR_FROM_ATTN,
                                MTP_DEVERR_FROM_VERIFY, MTP_DEVERR_FROM_DRAFT, MTP_DEVERR_FROM_FP8,
                                MTP_DEVERR_FROM_DGEMM};
  unsigned int v = 0;
  for (int i = 0; i < 7; ++i)
    if (parts[i]) v |= parts[i] | from[i];
  if (flags) *flags = v;
  return v ? MTP_ERR_DEVICE : MTP_OK;
}
