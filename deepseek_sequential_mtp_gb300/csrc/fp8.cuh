// Internal interface of the FP8 block-scaled weight GEMM (fp8.cu) used by the
// draft step.
#pragma once

#include "common.cuh"

namespace mtp {

// One weight matrix of a grouped call: q [n, K] e4m3 codes (row-major, row
// stride K bytes), scale [ceil(n/128), ceil(K/128)] fp32 row-major (one
// factor per 128 x 128 block), out: fp32 [R, ldo] whose columns [0, n)
// receive x̃ · (q ⊙ scale)^T added in.
struct Fp8Seg {
  const uint8_t* q = nullptr;
  const float* scale = nullptr;
  int n = 0;
  float* out = nullptr;
};

// out_s[r, n] += Σ_k x̃[r, k] · e4m3(q_s[n, k]) · scale_s[n / 128, k / 128] for
// every segment s (1..3 segments sharing x [R, K] bf16, row stride K), where
// x̃ is x in its two-term e4m3 form per 128-wide k-tile (exact for elements
// within 2^10 of the tile's largest).  R in [1, 32], K % 16 == 0, q_s 16-byte
// aligned, ldo >= every n; ws: fp8w_workspace_bytes(K) bytes, 16-byte aligned
// (the split activations and their scales).
size_t fp8w_workspace_bytes(int K);
mtp_status fp8w_gemm_launch(const Fp8Seg* segs, int nseg, int K, const __nv_bfloat16* x, int R, int ldo, void* ws,
                            size_t ws_bytes, cudaStream_t stream);

}  // namespace mtp
