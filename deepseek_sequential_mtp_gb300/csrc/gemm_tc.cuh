// Internal interface of the tcgen05 GEMM core (gemm_tc.cu) used by the chain.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mtp {

enum GemmEpilogue : int {
  EPI_STORE = 0,   // out = acc
  EPI_RESID = 1,   // out = resid + acc
  EPI_ROPE = 2,    // out = RoPE(acc) on columns < rope_cols, acc elsewhere
  EPI_SWIGLU = 3,  // out[:, j] = silu(gate_j) * up_j; B = (gate, up) stacked per tile
  EPI_CE = 4,      // no output: per (row, vocab tile) online max / sum-exp and the label logit
  // swap-AB (decode-shaped) variants: A = weights [features, K] on the
  // 128-row side, B = activations [tokens <= 32, K]; the accumulator tile is
  // [128 features, 32 tokens] and is written transposed, out[token, feature]
  EPI_T_STORE = 5,  // out_f32[token * ldo + feature] = acc (no split-K)
  // cross-entropy backward from recomputed logits z (rows = tokens, columns =
  // vocabulary entries ce_offset + col): out = bf16((exp(z - lse[row]) -
  // [ce_offset + col == labels[row]]) * ce_scale[0]), 0 for rows without a label
  EPI_CE_GRAD = 7,
  EPI_F32_ACC = 9  // out_f32[row * ldo + col] += acc (read-modify-write; with split-K, vector atomics)
};

// Epilogues that write bf16 boxes through the shared-memory staging buffers.
constexpr bool epi_uses_staging(int epi) {
  return epi == EPI_STORE || epi == EPI_RESID || epi == EPI_ROPE || epi == EPI_SWIGLU || epi == EPI_CE_GRAD;
}

// C-side description of one GEMM  acc[M, N] = A[M, K] · B[N, K]^T  (bf16 in,
// fp32 accumulate).  a_mn / b_mn (EPI_F32_ACC; b_mn also EPI_STORE): the operand is stored
// MN-major, i.e. as [K rows][M] (resp. [K rows][N]) with row stride lda (ldb),
// so A^T or B^T of a row-major matrix is read without a transposed copy.  B may be given as up to three row segments of
// `seg_rows` rows each (q/k/v weights); for EPI_SWIGLU B[0] = gate [N, K]
// and B[1] = up [N, K] and N counts output columns.
struct GemmDesc {
  int M = 0, N = 0, K = 0;
  const __nv_bfloat16* A = nullptr;
  int lda = 0;
  const __nv_bfloat16* B[3] = {nullptr, nullptr, nullptr};
  int ldb = 0;
  int nseg = 1;
  int seg_rows = 0;
  int epi = EPI_STORE;
  bool a_mn = false, b_mn = false;
  // EPI_F32_ACC with one split: store instead of adding (the output's first product)
  bool f32_overwrite = false;
  // programmatic dependent launch: the kernel's setup may overlap the stream's previous
  // kernel.  Only for launches whose stream predecessor is a kernel (not a memset or copy).
  bool pdl = false;
  // with pdl: B's first k-blocks are prefetched into L2 while the previous kernel still runs
  // (an L2 prefetch stays coherent with writes that follow it, so this is safe for any B; it
  // pays where B is not the previous kernel's output, e.g. weights)
  bool b_early = false;
  // release the stream's next kernel (a programmatic dependent that waits with pdl_wait)
  // when each CTA starts its last tile, so that its launch and setup overlap this one's tail
  bool trigger_early = false;
  __nv_bfloat16* out = nullptr;
  int ldo = 0;
  const __nv_bfloat16* resid = nullptr;
  int ldr = 0;
  // RoPE: pos [M] in [0, rope_len), table [rope_len, head_dim/2] of (cos, sin)
  const int32_t* pos = nullptr;
  const float2* rope = nullptr;
  int rope_len = 0, rope_cols = 0, head_dim = 0;
  // CE: labels [M] (-1 = none); ce_part [M, n_vtiles] (max, sumexp); z_tgt [M]
  const int32_t* labels = nullptr;
  float2* ce_part = nullptr;
  float* z_tgt = nullptr;
  // swap-AB variants and EPI_F32_ACC: fp32 output; the number of K splits
  float* out_f32 = nullptr;
  int splits = 1;
  // CE backward: per-token log-sum-exp and the scale dL/dl of a supervised row
  const float* lse = nullptr;
  const float* ce_scale = nullptr;
  int ce_offset = 0;
};

// Tile width along N the launcher will use for this descriptor (CE partial
// buffers are sized by ceil(N / ce_tile_n)).
int gemm_ce_tile_n();

mtp_status gemm_bf16_launch(const GemmDesc& g, cudaStream_t stream);

// Tensor map of a row-major bf16 matrix [rows, cols] (row stride ld
// elements, a multiple of 8) for tiled loads of box_cols x box_rows, either
// unswizzled or with the 128-byte swizzle (box_cols * 2 <= 128); false if
// the encoder is unavailable or rejects the description.
bool tensor_map_bf16_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                        uint32_t box_cols, uint32_t box_rows, bool swizzle128);

// Tensor map of a row-major byte matrix [rows, cols] (row stride ld bytes, a
// multiple of 16) for tiled loads of box_cols x box_rows with the 128-byte
// swizzle (box_cols <= 128).
bool tensor_map_u8_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_cols,
                      uint32_t box_rows);

}  // namespace mtp
