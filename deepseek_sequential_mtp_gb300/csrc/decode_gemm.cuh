// Internal interface of the bf16 decode-shaped GEMM (decode_gemm.cu) used by
// the draft step's linear maps.
#pragma once

#include "common.cuh"

namespace mtp {

// One weight matrix of a grouped call: w [n, K] bf16 row-major (row stride
// K); out: fp32 [R, ldo] whose columns [0, n) receive x · w^T added in.
struct DecSeg {
  const __nv_bfloat16* w = nullptr;
  int n = 0;
  float* out = nullptr;
};

// out_s[r, :] += x[r, :] · w_s^T for 1..3 segments sharing x [R, K] bf16 (row
// stride K).  R in [1, 32], K % 8 == 0, x and w_s 16-byte aligned, ldo >= n.
mtp_status dgemm_bf16_launch(const DecSeg* segs, int nseg, int K, const __nv_bfloat16* x, int R, int ldo,
                             cudaStream_t stream);

}  // namespace mtp
