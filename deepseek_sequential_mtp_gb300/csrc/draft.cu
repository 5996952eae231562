// mtp_draft_step: one decode-shaped MTP proposal per request.
//
// "M7.6 - DeepSeek MTP: Sequential Modules, Teacher Forcing, and Speculative
// Runtime" §0x09 (a carried-frontier round proposes y from the saved parent
// hidden state and E(f), retaining q for verification) and §0x09A (the MTP
// block serves attention from its own K/V cache).  For request r:
//   c = [RMSNorm_h(parent_hidden_r); RMSNorm_e(E[f_r])], u = M c,
//   a = u + Attn(RMSNorm_a u) over the cached rows [0, ctx_len_r) and the new
//   row at position pos_r, h = a + SwiGLU(RMSNorm_f a),
//   q_r = softmax(W_U RMSNorm_out(h)), y_r = smallest v with Σ_{i<=v} q_i > u·Σq
//   where u = word 2 of Philox4x32-10(key = seed, counter = (0, r, offset)).
//
// Every weight-streaming product is a skinny GEMM (R <= 32 tokens).  The
// block's linear maps run on the decode GEMM (decode_gemm.cu: weights on the
// N = 256 side of the tcgen05 MMA, equal weight streams per SM), the head on
// the swap-AB mode of the tcgen05 core (weights on the 128-row side, logits
// stored transposed); partial tiles accumulate into an fp32 buffer with
// atomics and small "finish" kernels round to bf16 with the fused RoPE /
// residual / SwiGLU / RMSNorm.
// Attention is split-K decoding: persistent CTAs stream the cache with TMA
// and write partial (max, sum, output) records per (request, head, key
// split) that a combine kernel merges with the new row's key.  The head writes logits into q_out, which a per-request
// kernel turns into probabilities in place and samples from.
// With the module's linear maps in FP8 block-scaled form (mtp_draft_round_fp8)
// the same products run on the FP8 weight GEMM of fp8.cu, which streams half
// the bytes; the head stays bf16.
#include <cooperative_groups.h>

#include <algorithm>
#include <cmath>
#include <initializer_list>

#include "decode_gemm.cuh"
#include "fp8.cuh"
#include "gemm_tc.cuh"
#include "mbarrier.cuh"

namespace cg = cooperative_groups;

MTP_DEFINE_ERROR_WORD(mtp_take_errors_draft)

namespace {

constexpr int kMaxR = 32;


// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11) -- the draw uses word 2
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// block-wide sum of one float per thread (blockDim.x multiple of 32, <= 1024)
__device__ float block_sum(float v, float* sh) {
  v = mtp::warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < (blockDim.x >> 5); ++i) t += sh[i];
  return t;
}

// ---------------------------------------------------------------------------
// Row kernels: one 1024-thread CTA per request row, vector accesses (d is a
// multiple of 64), so a row takes one or two memory round trips per pass.
// ---------------------------------------------------------------------------
constexpr int kRowThreads = 1024;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 v = __bfloat1622float2(b[t]);
    f[2 * t] = v.x;
    f[2 * t + 1] = v.y;
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int t = 0; t < 4; ++t) b[t] = __floats2bfloat162_rn(f[2 * t], f[2 * t + 1]);
  return u;
}

// c = [RMSNorm_h(parent_hidden); RMSNorm_e(E[frontier])]
__global__ void __launch_bounds__(kRowThreads)
draft_prologue_kernel(const __nv_bfloat16* __restrict__ hp, int ld_h, const int32_t* __restrict__ frontier, int f_stride,
                      const __nv_bfloat16* __restrict__ embed, const __nv_bfloat16* __restrict__ gh,
                      const __nv_bfloat16* __restrict__ ge, __nv_bfloat16* __restrict__ c, int d, int V,
                      float eps) {
  __shared__ float sh[32];
  const int r = blockIdx.x;
  int tok = frontier[static_cast<size_t>(r) * f_stride];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) atomicOr(&g_mtp_error_word, MTP_DEVERR_TOKEN_RANGE);
    tok = min(max(tok, 0), V - 1);
  }
  const uint4* h8 = reinterpret_cast<const uint4*>(hp + static_cast<size_t>(r) * ld_h);
  const uint4* e8 = reinterpret_cast<const uint4*>(embed + static_cast<size_t>(tok) * d);
  const int n8 = d / 8;
  float a = 0.f, b = 0.f;
  for (int i = threadIdx.x; i < n8; i += kRowThreads) {
    float x[8], y[8];
    bf16x8_to_f32(h8[i], x);
    bf16x8_to_f32(e8[i], y);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      a += x[t] * x[t];
      b += y[t] * y[t];
    }
  }
  a = block_sum(a, sh);
  b = block_sum(b, sh);
  const float rh = 1.0f / sqrtf(a / d + eps), re = 1.0f / sqrtf(b / d + eps);
  uint4* out = reinterpret_cast<uint4*>(c + static_cast<size_t>(r) * 2 * d);
  for (int i = threadIdx.x; i < n8; i += kRowThreads) {
    float x[8], y[8], g1[8], g2[8];
    bf16x8_to_f32(h8[i], x);
    bf16x8_to_f32(e8[i], y);
    bf16x8_to_f32(reinterpret_cast<const uint4*>(gh)[i], g1);
    bf16x8_to_f32(reinterpret_cast<const uint4*>(ge)[i], g2);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      x[t] = g1[t] * (x[t] * rh);
      y[t] = g2[t] * (y[t] * re);
    }
    out[i] = f32_to_bf16x8(x);
    out[n8 + i] = f32_to_bf16x8(y);
  }
}

// y = bf16(acc [+ resid]); optionally norm_out = bf16(RMSNorm_g(y))
__global__ void __launch_bounds__(kRowThreads)
finish_row_kernel(const float* __restrict__ acc, const __nv_bfloat16* __restrict__ resid,
                  __nv_bfloat16* __restrict__ y, int ld_y, const __nv_bfloat16* __restrict__ g,
                  __nv_bfloat16* __restrict__ norm_out, int d, float eps) {
  __shared__ float sh[32];
  const int r = blockIdx.x;
  const int n8 = d / 8;
  const float4* a4 = reinterpret_cast<const float4*>(acc + static_cast<size_t>(r) * d);
  uint4* y8 = reinterpret_cast<uint4*>(y + static_cast<size_t>(r) * ld_y);
  float ss = 0.f;
  for (int i = threadIdx.x; i < n8; i += kRowThreads) {
    const float4 lo = a4[2 * i], hi = a4[2 * i + 1];
    float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    if (resid) {
      float rv[8];
      bf16x8_to_f32(reinterpret_cast<const uint4*>(resid + static_cast<size_t>(r) * d)[i], rv);
#pragma unroll
      for (int t = 0; t < 8; ++t) v[t] += rv[t];
    }
    const uint4 vb = f32_to_bf16x8(v);
    y8[i] = vb;
    float vf[8];
    bf16x8_to_f32(vb, vf);
#pragma unroll
    for (int t = 0; t < 8; ++t) ss += vf[t] * vf[t];
  }
  if (!norm_out) return;
  ss = block_sum(ss, sh);
  const float rn = 1.0f / sqrtf(ss / d + eps);
  uint4* o8 = reinterpret_cast<uint4*>(norm_out + static_cast<size_t>(r) * d);
  for (int i = threadIdx.x; i < n8; i += kRowThreads) {
    float vf[8], gf[8];
    bf16x8_to_f32(y8[i], vf);
    bf16x8_to_f32(reinterpret_cast<const uint4*>(g)[i], gf);
#pragma unroll
    for (int t = 0; t < 8; ++t) vf[t] = gf[t] * (vf[t] * rn);
    o8[i] = f32_to_bf16x8(vf);
  }
}

// qkv = bf16(RoPE(q), RoPE(k), v) at the request's position pos[r] + step;
// the new row's rotated key and its value also go to slot `step` of the
// staging rows [R, n_slots, d] that later draft steps attend to.  CTA (x, r)
// covers pairs / v columns [x*1024, x*1024 + 1024) of row r; the row's
// (cos, sin) per frequency index is computed once per CTA: angle formed and
// reduced modulo 2*pi in double, sine/cosine taken in fp32.
constexpr int kQkvCols = 1024;
__global__ void __launch_bounds__(256)
finish_qkv_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ qkv, const int32_t* __restrict__ pos,
                  int step, int d, int hd, float base, int pos_max, __nv_bfloat16* __restrict__ stage_k,
                  __nv_bfloat16* __restrict__ stage_v, int n_slots) {
  __shared__ float2 cs[64];  // hd / 2 <= 64
  const int r = blockIdx.y;
  const int half = hd / 2;
  if (threadIdx.x < half) {
    float c = 1.f, s = 0.f;
    if (base > 0.f) {
      int p = pos[r];
      if (p < 0 || p > pos_max) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(&g_mtp_error_word, MTP_DEVERR_TOKEN_RANGE);
        p = min(max(p, 0), pos_max);
      }
      p += step;
      const int j = threadIdx.x;
      const double ang = static_cast<double>(p) * exp2(-2.0 * j / hd * log2(static_cast<double>(base)));
      const double two_pi = 6.283185307179586;
      sincosf(static_cast<float>(ang - rint(ang / two_pi) * two_pi), &s, &c);
    }
    cs[threadIdx.x] = make_float2(c, s);
  }
  __syncthreads();
  const float* a = acc + static_cast<size_t>(r) * 3 * d;
  __nv_bfloat16* o = qkv + static_cast<size_t>(r) * 3 * d;
  __nv_bfloat16* sk = stage_k + (static_cast<size_t>(r) * n_slots + step) * d;
  __nv_bfloat16* sv = stage_v + (static_cast<size_t>(r) * n_slots + step) * d;
  const int i0 = blockIdx.x * kQkvCols;
  const int i1 = min(i0 + kQkvCols, d);
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    // pair i: head i / half over the 2H q and k heads, (j, j + half) within it
    const int head = i / half, j = i % half;
    const int col = head * hd + j;
    const float x1 = a[col], x2 = a[col + half];
    const float2 t = cs[j];
    const __nv_bfloat16 y1 = __float2bfloat16_rn(x1 * t.x - x2 * t.y);
    const __nv_bfloat16 y2 = __float2bfloat16_rn(x2 * t.x + x1 * t.y);
    o[col] = y1;
    o[col + half] = y2;
    if (col >= d) {  // a key head: stage the rotated key
      sk[col - d] = y1;
      sk[col - d + half] = y2;
    }
    const __nv_bfloat16 vv = __float2bfloat16_rn(a[2 * d + i]);
    o[2 * d + i] = vv;
    sv[i] = vv;
  }
}

// g = bf16(silu(gate) * up) from acc [R, 2*ffn] (gate then up)
__global__ void finish_swiglu_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ g, int ffn) {
  const int r = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= ffn) return;
  const float gt = acc[static_cast<size_t>(r) * 2 * ffn + j], up = acc[static_cast<size_t>(r) * 2 * ffn + ffn + j];
  g[static_cast<size_t>(r) * ffn + j] = __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * up);
}

// ---------------------------------------------------------------------------
// Decode attention over the module's K/V cache, streamed by TMA.
// Persistent CTAs (one per SM) walk work units u -> (head h, key split sp,
// request r), heads fastest so that concurrently running units read
// neighbouring pieces of the same cache rows.  A producer warp streams
// [64 keys x head_dim] tiles of K and V into a shared-memory ring as
// [64 x 64] boxes with the 128-byte swizzle; each of the 8 consumer warps
// takes 8 keys of every tile (so every consumer waits on every ring phase in
// order) and keeps its own online-softmax state.  Both products run on
// mma.sync.m16n8k16 with the single query as the one real row of the 16-row
// operand: scores S[1 x 8] = q K^T (K rows loaded by ldmatrix as the
// column-major B operand) and O[1 x hd] += P V (V by ldmatrix.trans); the
// score accumulator's lanes 0-3 already hold P in the A-operand layout.  P
// enters the P V product as two bf16 rows, p_hi = bf16(p) and
// p_lo = bf16(p - p_hi), whose output rows are added once per unit, so the
// weights are exact to ~2^-17 relative.  At the end of a unit the warps' (m, l, o) states merge
// into one record part[r, h, sp] = (max, sum, o[head_dim]).
// ---------------------------------------------------------------------------
constexpr int kAttnTileKeys = 64;
constexpr int kAttnWarps = 8;
constexpr int kAttnKeysPerWarp = kAttnTileKeys / kAttnWarps;
constexpr int kAttnThreads = (kAttnWarps + 1) * 32;
constexpr int kAttnRingBytes = 192 * 1024;
constexpr int kAttnSplitKeys = 1024;  // target keys per work unit
constexpr int kAttnBoxBytes = kAttnTileKeys * 64 * 2;  // [64 keys x 64 dims] bf16, 128-byte swizzled
static_assert(kAttnKeysPerWarp == 8, "one n8 MMA tile of keys per warp");

template <int HD>
struct AttnCfg {
  static constexpr int kBoxes = HD / 64;                   // boxes per K (or V) tile
  static constexpr int kTileBytes = kBoxes * kAttnBoxBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;       // K tile then V tile
  static constexpr int kStages = kAttnRingBytes / kStageBytes;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
};

template <int KD>
__device__ __forceinline__ void load_bf16x(const void* p, float (&f)[KD]) {
  if constexpr (KD == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    f[0] = f0.x; f[1] = f0.y; f[2] = f1.x; f[3] = f1.y;
  } else {
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
    f[0] = f0.x; f[1] = f0.y;
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// c += A(16x16, row) * B(16x8, col), bf16 in, fp32 accumulate; A rows 8..15 are zero here
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// shared address of 16-byte row piece (row, col..col+7) of a [64 x 64] box with the 128-byte swizzle
__device__ __forceinline__ uint32_t swz(uint32_t box, int row, int col) {
  return box + row * 128 + ((((col >> 3) ^ row) & 7) << 4);
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1)
decode_attn_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __nv_bfloat16* __restrict__ qkv, const int32_t* __restrict__ ctx_len,
                   float* __restrict__ part, int H, int T, int n_split, int split_keys, int n_units, float scale) {
  using C = AttnCfg<HD>;
  constexpr int S = C::kStages;
  constexpr int kKSteps = HD / 16;  // score MMAs per 8 keys
  constexpr int kNTiles = HD / 8;   // P V MMAs per 8 keys
  extern __shared__ uint8_t attn_smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * S];
  __shared__ float s_m[2][kAttnWarps], s_l[2][kAttnWarps];
  __shared__ float s_o[2][kAttnWarps][HD];
  __shared__ int s_abort;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(attn_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t ring_s = mtp::smem_u32(ring);
  const uint32_t full0 = mtp::smem_u32(bars), empty0 = full0 + 8u * S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = H * HD;
  volatile int* abort_flag = &s_abort;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mtp::mbar_init(full0 + 8u * i, 1);
      mtp::mbar_init(empty0 + 8u * i, kAttnWarps);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  auto unit = [&](int u, int& r, int& h, int& sp, int& lo, int& hi) {
    h = u % H;
    const int rest = u / H;
    sp = rest % n_split;
    r = rest / n_split;
    const int len = min(max(ctx_len[r], 0), T);
    lo = sp * split_keys;
    hi = min(lo + split_keys, len);
  };

  if (warp == kAttnWarps) {
    // ------------------------------ producer ------------------------------
    uint32_t g = 0;  // tiles issued
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      int r, h, sp, lo, hi;
      unit(u, r, h, sp, lo, hi);
      for (int s = lo; s < hi; s += kAttnTileKeys) {
        const uint32_t slot = g % S, use = g / S;
        // warp-uniform outcome: every lane waits, all must have seen the phase
        if (use > 0 && !__all_sync(0xffffffffu, mtp::mbar_wait_bounded(empty0 + 8u * slot, (use - 1) & 1))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full = full0 + 8u * slot;
          const uint32_t dst = ring_s + slot * C::kStageBytes;
          mtp::mbar_expect_tx(full, C::kStageBytes);
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx) {
            mtp::tma_tile_2d(dst + bx * kAttnBoxBytes, &tmK, h * HD + bx * 64, r * T + s, full);
            mtp::tma_tile_2d(dst + C::kTileBytes + bx * kAttnBoxBytes, &tmV, h * HD + bx * 64, r * T + s, full);
          }
        }
        __syncwarp();
        ++g;
      }
    }
    if (lane == 0) {
      if (!ok) {
        atomicOr(&g_mtp_error_word, MTP_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // no copy may still be landing in shared memory when the CTA leaves
      for (uint32_t t = g > static_cast<uint32_t>(S) ? g - S : 0; t < g; ++t)
        if (!mtp::mbar_wait_bounded(full0 + 8u * (t % S), (t / S) & 1)) {
          atomicOr(&g_mtp_error_word, MTP_DEVERR_TIMEOUT);
          break;
        }
    }
    return;
  }

  // ------------------------------ consumers ------------------------------
  // lanes 0-3 carry the real row of every fragment: key pair 2t, 2t+1 of the
  // warp's 8 keys, head_dim pairs 8j + 2t, 8j + 2t + 1 of the output
  const int t4 = lane & 3;
  const bool row0 = lane < 4;
  const int key_row = warp * kAttnKeysPerWarp + (lane & 7);  // ldmatrix row address of this lane
  const int col_sel = 8 * (lane >> 3);                       // ... and its column offset in a 32-column group
  uint32_t g = 0;
  int k = 0;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++k) {
    int r, h, sp, lo, hi;
    unit(u, r, h, sp, lo, hi);
    // q as the A operand: row 0 real (lanes 0-3), pairs 16kk + 2t (a0) and 16kk + 8 + 2t (a2)
    uint32_t qa[kKSteps][2];
    {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qkv + static_cast<size_t>(r) * 3 * d + h * HD);
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
        qa[kk][0] = row0 ? qrow[8 * kk + t4] : 0u;
        qa[kk][1] = row0 ? qrow[8 * kk + 4 + t4] : 0u;
      }
    }
    float m = -INFINITY, l = 0.f;
    float o[kNTiles][4];
#pragma unroll
    for (int j = 0; j < kNTiles; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    for (int s = lo; s < hi; s += kAttnTileKeys, ++g) {
      const uint32_t slot = g % S, use = g / S;
      // the skip decision is warp-uniform (lane 0's view of the flag)
      bool skip = __shfl_sync(0xffffffffu, *abort_flag, 0) != 0;
      if (!skip && !__all_sync(0xffffffffu, mtp::mbar_wait_bounded(full0 + 8u * slot, use & 1))) {
        if (lane == 0) {
          atomicOr(&g_mtp_error_word, MTP_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        skip = true;
      }
      if (skip) continue;
      const uint32_t kbase = ring_s + slot * C::kStageBytes, vbase = kbase + C::kTileBytes;
      // scores: two independent accumulation chains over the head_dim steps
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t b[4];
        const int col = 32 * c + col_sel;
        ldsm_x4(swz(kbase + (col >> 6) * kAttnBoxBytes, key_row, col & 63), b);
        mma_16816(sc[0], qa[2 * c][0], qa[2 * c][1], b[0], b[1]);
        mma_16816(sc[1], qa[2 * c + 1][0], qa[2 * c + 1][1], b[2], b[3]);
      }
      const int key0 = s + warp * kAttnKeysPerWarp + 2 * t4;
      const float s0 = key0 < hi ? (sc[0][0] + sc[1][0]) * scale : -INFINITY;
      const float s1 = key0 + 1 < hi ? (sc[0][1] + sc[1][1]) * scale : -INFINITY;
      float mx = fmaxf(s0, s1);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m, __shfl_sync(0xffffffffu, mx, 0));  // warp-uniform
      if (m_new != -INFINITY) {
        if (m_new > m) {
          const float alpha = __expf(m - m_new);
          l *= alpha;
#pragma unroll
          for (int j = 0; j < kNTiles; ++j) {
            o[j][0] *= alpha;
            o[j][1] *= alpha;
          }
          m = m_new;
        }
        // P = p_hi + p_lo (two bf16 parts, ~2^-17 relative): row 0 of the A
        // operand carries p_hi (lanes 0-3), row 1 carries p_lo (lanes 4-7)
        const float p0 = __expf(s0 - m), p1 = __expf(s1 - m);
        const uint32_t ph = pack_bf16x2(p0, p1);
        const float2 phf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ph));
        const uint32_t pl = __shfl_sync(0xffffffffu, pack_bf16x2(p0 - phf.x, p1 - phf.y), lane & 3);
        l += p0 + p1;
        const uint32_t pa = row0 ? ph : (lane < 8 ? pl : 0u);
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t b[4];
          const int col = 32 * c + col_sel;
          ldsm_x4_t(swz(vbase + (col >> 6) * kAttnBoxBytes, key_row, col & 63), b);
#pragma unroll
          for (int i = 0; i < 4; ++i) mma_16816(o[4 * c + i], pa, 0u, b[i], 0u);
        }
      }
      __syncwarp();
      if (lane == 0) mtp::mbar_arrive_cnt(empty0 + 8u * slot, 1);
    }
    // this warp's sum over its keys lives in lanes 0-3; its output in rows 0
    // (lanes 0-3, p_hi part) and 1 (lanes 4-7, p_lo part) of the accumulators
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
#pragma unroll
    for (int j = 0; j < kNTiles; ++j) {
      o[j][0] += __shfl_xor_sync(0xffffffffu, o[j][0], 4);
      o[j][1] += __shfl_xor_sync(0xffffffffu, o[j][1], 4);
    }
    // merge the 8 warps' states of this unit (double-buffered: one barrier per unit)
    const int b = k & 1;
    if (lane == 0) {
      s_m[b][warp] = m;
      s_l[b][warp] = l;
    }
    if (row0) {
#pragma unroll
      for (int j = 0; j < kNTiles; ++j) {
        s_o[b][warp][8 * j + 2 * t4] = o[j][0];
        s_o[b][warp][8 * j + 2 * t4 + 1] = o[j][1];
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kAttnWarps * 32) : "memory");
    if (threadIdx.x < HD) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[b][w]);
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) {
          const float e = __expf(s_m[b][w] - M);
          L += e * s_l[b][w];
          O += e * s_o[b][w][threadIdx.x];
        }
      }
      float* rec = part + ((static_cast<size_t>(r) * H + h) * n_split + sp) * (HD + 2);
      if (threadIdx.x == 0) {
        rec[0] = M;
        rec[1] = L;
      }
      rec[2 + threadIdx.x] = O;
    }
  }
}

// merge the split records with the staged rows 0..n_staged-1 (the rows of
// earlier draft steps and, last, the new row itself); one warp per (request,
// head): lane j scores staged row j, lanes read the records' (max, sum) in
// parallel, then the weighted outputs, lanes owning head_dim slices
template <int HD>
__global__ void decode_attn_combine_kernel(const __nv_bfloat16* __restrict__ qkv,
                                           const __nv_bfloat16* __restrict__ stage_k,
                                           const __nv_bfloat16* __restrict__ stage_v, int n_slots, int n_staged,
                                           const float* __restrict__ part, __nv_bfloat16* __restrict__ out, int R,
                                           int H, int n_split, float scale) {
  const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (item >= R * H) return;
  const int r = item / H, h = item % H;
  const int d = H * HD;
  constexpr int kDim = HD / 32;
  constexpr int kRec = HD + 2;
  float qv[kDim];
  load_bf16x<kDim>(qkv + static_cast<size_t>(r) * 3 * d + h * HD + lane * kDim, qv);
  const __nv_bfloat16* sk = stage_k + static_cast<size_t>(r) * n_slots * d + h * HD + lane * kDim;
  const __nv_bfloat16* sv = stage_v + static_cast<size_t>(r) * n_slots * d + h * HD + lane * kDim;
  float s_own = -INFINITY;  // lane j: score of staged row j
  for (int j = 0; j < n_staged; ++j) {
    float kv[kDim];
    load_bf16x<kDim>(sk + static_cast<size_t>(j) * d, kv);
    float qk = 0.f;
#pragma unroll
    for (int t = 0; t < kDim; ++t) qk = fmaf(qv[t], kv[t], qk);
    qk = mtp::warp_sum(qk) * scale;
    if (lane == j) s_own = qk;
  }
  const float* rec0 = part + (static_cast<size_t>(r) * H + h) * n_split * kRec;
  float m = s_own;
  for (int c = lane; c < n_split; c += 32) m = fmaxf(m, rec0[static_cast<size_t>(c) * kRec]);
  m = mtp::warp_max(m);
  const float w_own = lane < n_staged ? __expf(s_own - m) : 0.f;
  float l = w_own, o[kDim];
#pragma unroll
  for (int t = 0; t < kDim; ++t) o[t] = 0.f;
  for (int j = 0; j < n_staged; ++j) {
    const float wj = __shfl_sync(0xffffffffu, w_own, j);
    float vv[kDim];
    load_bf16x<kDim>(sv + static_cast<size_t>(j) * d, vv);
#pragma unroll
    for (int t = 0; t < kDim; ++t) o[t] = fmaf(wj, vv[t], o[t]);
  }
  for (int cb = 0; cb < n_split; cb += 32) {
    const int c = cb + lane;
    float wc = 0.f;
    if (c < n_split) {
      const float mc = rec0[static_cast<size_t>(c) * kRec], lc = rec0[static_cast<size_t>(c) * kRec + 1];
      if (lc > 0.f) {
        wc = __expf(mc - m);
        l += wc * lc;
      }
    }
    const int nc = min(32, n_split - cb);
#pragma unroll 8
    for (int k = 0; k < nc; ++k) {
      const float wk = __shfl_sync(0xffffffffu, wc, k);
      if (wk != 0.f) {  // warp-uniform
        float pv[kDim];
        const float* src = rec0 + static_cast<size_t>(cb + k) * kRec + 2 + lane * kDim;
#pragma unroll
        for (int t = 0; t < kDim; ++t) pv[t] = src[t];
#pragma unroll
        for (int t = 0; t < kDim; ++t) o[t] = fmaf(wk, pv[t], o[t]);
      }
    }
  }
  l = mtp::warp_sum(l);
  const float inv = 1.0f / l;
  __nv_bfloat16* dst = out + static_cast<size_t>(r) * d + h * HD + lane * kDim;
#pragma unroll
  for (int t = 0; t < kDim; ++t) dst[t] = __float2bfloat16_rn(o[t] * inv);
}

// ---------------------------------------------------------------------------
// q = softmax(z) in place and y ~ q by inverse CDF.  A cluster of 8 CTAs
// per request: CTA `rank` owns chunks [rank*cpc, rank*cpc + cpc) of 1024
// vocabulary entries.  Pass A: online (max, sum exp) per CTA, combined in
// CTA 0 through distributed shared memory.  Pass B: q written in place and
// compensated (hi, lo) chunk sums pushed into CTA 0.  CTA 0 takes the fp64
// prefix over chunks to find the chunk holding u * mass; the CTA owning that
// chunk rescans it in index order for the smallest index whose running sum
// exceeds the target.
// ---------------------------------------------------------------------------
constexpr int kSampleCluster = 8;
constexpr int kSampleThreads = 512;
constexpr int kSampleChunk = 1024;
constexpr int kMaxSampleChunks = 512;

// (m, s) <- the pair describing the union of two sets, s = sum exp(x - m)
__device__ __forceinline__ void merge_max_sum(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  s = s * __expf(m - M) + s2 * __expf(m2 - M);
  m = M;
}

__global__ void __cluster_dims__(kSampleCluster, 1, 1) __launch_bounds__(kSampleThreads)
softmax_sample_kernel(float* __restrict__ q, int V, size_t ldq, uint2 key, uint32_t step, uint32_t off_lo,
                      uint32_t off_hi, int32_t* __restrict__ y_out, int y_stride) {
  __shared__ float2 s_red[kSampleThreads / 32];
  __shared__ float2 s_ms[kSampleCluster];         // CTA 0: (max, sum) of every CTA
  __shared__ float2 s_chunk[kMaxSampleChunks];    // CTA 0: compensated chunk sums
  __shared__ float s_w[kSampleChunk];
  __shared__ int s_cstar;
  __shared__ double s_before, s_target;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int r = blockIdx.x / kSampleCluster;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* z = q + static_cast<size_t>(r) * ldq;
  int32_t* y_dst = y_out + static_cast<size_t>(r) * y_stride;
  const int n_chunks = (V + kSampleChunk - 1) / kSampleChunk;
  const int cpc = (n_chunks + kSampleCluster - 1) / kSampleCluster;
  const int c0 = min(n_chunks, rank * cpc), c1 = min(n_chunks, c0 + cpc);
  const int v0 = c0 * kSampleChunk, v1 = min(V, c1 * kSampleChunk);

  // pass A: online max / sum-exp
  float m = -INFINITY, sm = 0.f;
  for (int v = v0 + threadIdx.x; v < v1; v += kSampleThreads) {
    const float x = z[v];
    if (x > m) {
      sm = sm * __expf(m - x) + 1.f;
      m = x;
    } else {
      sm += __expf(x - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    merge_max_sum(m, sm, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, sm, o));
  if (lane == 0) s_red[warp] = make_float2(m, sm);
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kSampleThreads / 32; ++w) merge_max_sum(m, sm, s_red[w].x, s_red[w].y);
    *cluster.map_shared_rank(&s_ms[rank], 0) = make_float2(m, sm);
  }
  cluster.sync();
  float M = -INFINITY, S = 0.f;
  {
    const float2* all = cluster.map_shared_rank(s_ms, 0);
#pragma unroll
    for (int k = 0; k < kSampleCluster; ++k) {
      const float2 t = all[k];
      merge_max_sum(M, S, t.x, t.y);
    }
  }
  const float inv = 1.0f / S;

  // pass B: q in place and compensated chunk sums (warp per chunk)
  float2* chunk0 = cluster.map_shared_rank(s_chunk, 0);
  for (int c = c0 + warp; c < c1; c += kSampleThreads / 32) {
    float hi = 0.f, lo = 0.f;
    for (int i = lane; i < kSampleChunk; i += 32) {
      const int v = c * kSampleChunk + i;
      if (v < V) {
        const float pv = __expf(z[v] - M) * inv;
        z[v] = pv;
        float t, e;
        two_sum(hi, pv, t, e);
        hi = t;
        lo += e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ohi = __shfl_xor_sync(0xffffffffu, hi, o), olo = __shfl_xor_sync(0xffffffffu, lo, o);
      float t, e;
      two_sum(hi, ohi, t, e);
      hi = t;
      lo = (lo + olo) + e;
    }
    if (lane == 0) chunk0[c] = make_float2(hi, lo);
  }
  cluster.sync();

  // CTA 0: the chunk holding u * mass
  if (rank == 0 && warp == 0) {
    const uint4 w = philox4x32_10(make_uint4(step, static_cast<uint32_t>(r), off_lo, off_hi), key);
    const double u = static_cast<double>(w.z >> 8) * (1.0 / 16777216.0);
    const int per = (n_chunks + 31) / 32;
    double own = 0.0;
    for (int c = lane * per; c < min(n_chunks, (lane + 1) * per); ++c)
      own += static_cast<double>(s_chunk[c].x) + static_cast<double>(s_chunk[c].y);
    const double incl = mtp::warp_inclusive_scan(own);
    const double mass = __shfl_sync(0xffffffffu, incl, 31);
    const double target = u * mass;
    const unsigned over = __ballot_sync(0xffffffffu, incl > target);
    const unsigned has = __ballot_sync(0xffffffffu, own > 0.0);
    const int src = over ? __ffs(over) - 1 : (has ? 31 - __clz(has) : 0);
    int cstar = -1;
    double before = 0.0;
    if (lane == src) {
      double run = incl - own;
      int last = -1;
      double before_last = run;
      for (int c = lane * per; c < min(n_chunks, (lane + 1) * per); ++c) {
        const double cv = static_cast<double>(s_chunk[c].x) + static_cast<double>(s_chunk[c].y);
        if (cv > 0.0) { last = c; before_last = run; }
        if (over && run + cv > target) { cstar = c; before = run; break; }
        run += cv;
      }
      if (cstar < 0) { cstar = last; before = before_last; }
    }
    cstar = __shfl_sync(0xffffffffu, cstar, src);
    before = __shfl_sync(0xffffffffu, before, src);
    if (lane == 0) {
      s_cstar = cstar;
      s_before = before;
      s_target = target;
      if (cstar < 0) *y_dst = -1;
    }
  }
  cluster.sync();
  const int cstar = *cluster.map_shared_rank(&s_cstar, 0);
  const double before = *cluster.map_shared_rank(&s_before, 0);
  const double target = *cluster.map_shared_rank(&s_target, 0);
  // CTA 0's shared memory is read above; nobody touches it after this barrier
  cluster.sync();
  if (cstar < 0 || cstar / cpc != rank) return;
  // the owning CTA rescans the chosen chunk (its own writes of pass B)
  for (int i = threadIdx.x; i < kSampleChunk; i += kSampleThreads) {
    const int v = cstar * kSampleChunk + i;
    s_w[i] = v < V ? z[v] : 0.f;
  }
  __syncthreads();
  if (warp != 0) return;
  float lhi = 0.f, llo = 0.f;
  for (int i = 0; i < 32; ++i) {
    float s, e;
    two_sum(lhi, s_w[32 * lane + i], s, e);
    lhi = s;
    llo += e;
  }
  const double lane_sum = static_cast<double>(lhi) + static_cast<double>(llo);
  const double lincl = mtp::warp_inclusive_scan(lane_sum) + before;
  const unsigned lover = __ballot_sync(0xffffffffu, lincl > target);
  const unsigned lpos = __ballot_sync(0xffffffffu, lane_sum > 0.0);
  const int lsrc = lover ? __ffs(lover) - 1 : (lpos ? 31 - __clz(lpos) : 0);
  const double delta = __shfl_sync(0xffffffffu, target - (lincl - lane_sum), lsrc);
  const float wv = s_w[32 * lsrc + lane];
  float phi = wv, plo = 0.f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float nhi = __shfl_up_sync(0xffffffffu, phi, o), nlo = __shfl_up_sync(0xffffffffu, plo, o);
    if (lane >= o) {
      float s, e;
      two_sum(phi, nhi, s, e);
      phi = s;
      plo = (plo + nlo) + e;
    }
  }
  const unsigned eover = __ballot_sync(0xffffffffu, lover && (static_cast<double>(phi) + static_cast<double>(plo)) > delta);
  const unsigned epos = __ballot_sync(0xffffffffu, wv > 0.0f);
  if (lane == 0) {
    const int base = cstar * kSampleChunk + 32 * lsrc;
    *y_dst = eover ? base + __ffs(eover) - 1 : (epos ? base + 31 - __clz(epos) : -1);
  }
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------
inline size_t align_up(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

constexpr int kMaxRoundGamma = 31;  // draft steps per round (spec_verify takes gamma <= 31)

struct DraftLayout {
  size_t c, acc, u, x, qkv, o, a, g, h, part, stage_k, stage_v, f8ws, f8ws_bytes, total;
  int n_chunks;
};

// h holds two [R, d] rows (the state of the step and of the previous one);
// stage_k / stage_v hold the rotated key and the value of every step's row
DraftLayout draft_layout(const mtp_dims& D, int gamma) {
  DraftLayout L{};
  const size_t R = D.B, d = D.d;
  L.n_chunks = std::max(1, (D.T + kAttnSplitKeys - 1) / kAttnSplitKeys);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  L.c = take(R * 2 * d * 2);
  const size_t acc_cols = std::max<size_t>(3 * d, 2 * static_cast<size_t>(D.ffn));
  L.acc = take(R * acc_cols * 4);
  L.u = take(R * d * 2);
  L.x = take(R * d * 2);
  L.qkv = take(R * 3 * d * 2);
  L.o = take(R * d * 2);
  L.a = take(R * d * 2);
  L.g = take(R * static_cast<size_t>(D.ffn) * 2);
  L.h = take(2 * R * d * 2);
  L.part = take(R * static_cast<size_t>(D.n_heads) * L.n_chunks * (D.head_dim + 2) * 4);
  L.stage_k = take(R * static_cast<size_t>(gamma) * d * 2);
  L.stage_v = take(R * static_cast<size_t>(gamma) * d * 2);
  // the FP8 linear maps' split activations (largest reduction length: 2d or ffn)
  L.f8ws_bytes = mtp::fp8w_workspace_bytes(std::max(2 * D.d, D.ffn));
  L.f8ws = take(L.f8ws_bytes);
  L.total = off;
  return L;
}

bool draft_dims_ok(const mtp_dims& D) {
  return D.B > 0 && D.B <= kMaxR && D.T > 0 && D.d > 0 && D.d % 64 == 0 && D.n_heads > 0 &&
         (D.head_dim == 64 || D.head_dim == 128) && D.n_heads * D.head_dim == D.d && D.ffn > 0 && D.ffn % 8 == 0 &&
         D.V > 0 && D.V <= kMaxSampleChunks * kSampleChunk && D.D == 1 && D.dtype == MTP_BF16 && D.eps >= 0.f &&
         D.rope_base >= 0.f;
}

int sm_count() {
  return mtp::sm_count_current();
}

// out[R, ldo] (fp32) = X[R, K] · W[features, K]^T: the swap-AB tcgen05 GEMM (weights on the
// 128-row side, the <= 32 tokens as N, the logits stored transposed)
mtp_status skinny_gemm(const __nv_bfloat16* W, int features, int K, const __nv_bfloat16* X, int R, float* out,
                       int ldo, cudaStream_t st) {
  mtp::GemmDesc g;
  g.M = features;
  g.N = R;
  g.K = K;
  g.A = W;
  g.lda = K;
  g.B[0] = X;
  g.ldb = K;
  g.nseg = 1;
  g.seg_rows = R;
  g.out_f32 = out;
  g.ldo = ldo;
  g.splits = 1;
  g.epi = mtp::EPI_T_STORE;
  return mtp::gemm_bf16_launch(g, st);
}

#define TRY(expr)                \
  do {                           \
    mtp_status s_ = (expr);      \
    if (s_ != MTP_OK) return s_; \
  } while (0)

}  // namespace

namespace {

// One draft step s of a round: reads the parent state (row stride ld_parent)
// and the frontier token (stride f_stride), writes the step's state h_s (row
// stride ld_h), logits/q into q_s (row stride ldq), the draw into y_s (stride
// y_stride) and the step's key/value into staging slot s.
mtp_status draft_one_step(const mtp_dims& D, const mtp_weights* w, const mtp_block_fp8* f8, const DraftLayout& L,
                          uint8_t* base,
                          const __nv_bfloat16* parent, int ld_parent, const int32_t* frontier, int f_stride,
                          const int32_t* pos, const void* kv_k, const void* kv_v, const int32_t* ctx_len, int step,
                          int gamma, uint2 key, uint64_t offset, float* q_s, size_t ldq, int32_t* y_s, int y_stride,
                          __nv_bfloat16* h_s, int ld_h, cudaStream_t st) {
  const int R = D.B, d = D.d, ffn = D.ffn, V = D.V, H = D.n_heads, hd = D.head_dim;
  auto bfp = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(base + off); };
  float* acc = reinterpret_cast<float*>(base + L.acc);
  auto W0 = [&](const void* const* l) { return static_cast<const __nv_bfloat16*>(l[0]); };
  const __nv_bfloat16* E = static_cast<const __nv_bfloat16*>(w->embed);
  __nv_bfloat16 *c = bfp(L.c), *u = bfp(L.u), *x = bfp(L.x), *qkv = bfp(L.qkv), *o = bfp(L.o), *a = bfp(L.a),
                *g = bfp(L.g), *sk = bfp(L.stage_k), *sv = bfp(L.stage_v);
  // acc[:, col + (0..n)] += xin · W^T for one to three linear maps of the
  // block that share their input, in one grouped launch: bf16 weights on the
  // decode GEMM (decode_gemm.cu), FP8 block-scaled ones on the FP8 GEMM
  struct Map {
    const void* const* bf;
    const mtp_fp8_matrix* q8;
    int n, col;
  };
  auto linear = [&](std::initializer_list<Map> maps, int K, const __nv_bfloat16* xin, int ldo) -> mtp_status {
    if (f8) {
      mtp::Fp8Seg segs[3];
      int i = 0;
      for (const Map& m : maps) {
        segs[i].q = static_cast<const uint8_t*>(m.q8->q);
        segs[i].scale = m.q8->scale;
        segs[i].n = m.n;
        segs[i].out = acc + m.col;
        ++i;
      }
      return mtp::fp8w_gemm_launch(segs, i, K, xin, R, ldo, base + L.f8ws, L.f8ws_bytes, st);
    }
    mtp::DecSeg segs[3];
    int i = 0;
    for (const Map& m : maps) {
      segs[i].w = W0(m.bf);
      segs[i].n = m.n;
      segs[i].out = acc + m.col;
      ++i;
    }
    return mtp::dgemm_bf16_launch(segs, i, K, xin, R, ldo, st);
  };
  auto q8 = [&](const mtp_fp8_matrix mtp_block_fp8::*field) { return f8 ? &(f8->*field) : nullptr; };

  // c, u = M c, x = RMSNorm_a(u)
  draft_prologue_kernel<<<R, kRowThreads, 0, st>>>(parent, ld_parent, frontier, f_stride, E, W0(w->hnorm),
                                                   W0(w->enorm), c, d, V, D.eps);
  mtp::note_launch();
  MTP_CUDA_TRY(cudaMemsetAsync(acc, 0, static_cast<size_t>(R) * d * 4, st));
  TRY(linear({{w->eh_proj, q8(&mtp_block_fp8::eh_proj), d, 0}}, 2 * d, c, d));
  finish_row_kernel<<<R, kRowThreads, 0, st>>>(acc, nullptr, u, d, W0(w->attn_norm), x, d, D.eps);
  mtp::note_launch();
  // q, k, v with RoPE on q, k at pos + step; the row's k, v staged in slot `step`
  MTP_CUDA_TRY(cudaMemsetAsync(acc, 0, static_cast<size_t>(R) * 3 * d * 4, st));
  TRY(linear({{w->wq, q8(&mtp_block_fp8::wq), d, 0},
              {w->wk, q8(&mtp_block_fp8::wk), d, d},
              {w->wv, q8(&mtp_block_fp8::wv), d, 2 * d}},
             d, x, 3 * d));
  finish_qkv_kernel<<<dim3((d + kQkvCols - 1) / kQkvCols, R), 256, 0, st>>>(acc, qkv, pos, step, d, hd, D.rope_base,
                                                                            D.T, sk, sv, gamma);
  mtp::note_launch();
  // attention over the module's own cache, the rows staged by earlier steps and the new row
  const float scale = 1.0f / sqrtf(static_cast<float>(hd));
  float* part = reinterpret_cast<float*>(base + L.part);
  const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(kv_k);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(kv_v);
  const int n_split = L.n_chunks;
  const int split_keys = ((D.T + n_split - 1) / n_split + kAttnTileKeys - 1) / kAttnTileKeys * kAttnTileKeys;
  const int n_units = R * H * n_split;
  const int agrid = std::min(n_units, sm_count());
  CUtensorMap tmk, tmv;
  const uint64_t cache_rows = static_cast<uint64_t>(R) * D.T;
  if (cache_rows > 0x7FFFFFFFull) return MTP_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
  if (!mtp::tensor_map_bf16_2d(&tmk, kc, cache_rows, d, d, 64, kAttnTileKeys, true) ||
      !mtp::tensor_map_bf16_2d(&tmv, vc, cache_rows, d, d, 64, kAttnTileKeys, true))
    return MTP_ERR_CUDA;
  mtp::prof_begin(MTP_KC_ATTENTION, st);
  if (hd == 128) {
    static mtp::PerDevice attr;
    if (!mtp::smem_limit(attr, decode_attn_kernel<128>, AttnCfg<128>::kSmemBytes)) return MTP_ERR_CUDA;
    decode_attn_kernel<128><<<agrid, kAttnThreads, AttnCfg<128>::kSmemBytes, st>>>(
        tmk, tmv, qkv, ctx_len, part, H, D.T, n_split, split_keys, n_units, scale);
    mtp::note_launch();
    decode_attn_combine_kernel<128><<<(R * H + 7) / 8, 256, 0, st>>>(qkv, sk, sv, gamma, step + 1, part, o, R, H,
                                                                     n_split, scale);
  } else {
    static mtp::PerDevice attr;
    if (!mtp::smem_limit(attr, decode_attn_kernel<64>, AttnCfg<64>::kSmemBytes)) return MTP_ERR_CUDA;
    decode_attn_kernel<64><<<agrid, kAttnThreads, AttnCfg<64>::kSmemBytes, st>>>(
        tmk, tmv, qkv, ctx_len, part, H, D.T, n_split, split_keys, n_units, scale);
    mtp::note_launch();
    decode_attn_combine_kernel<64><<<(R * H + 7) / 8, 256, 0, st>>>(qkv, sk, sv, gamma, step + 1, part, o, R, H,
                                                                    n_split, scale);
  }
  mtp::note_launch();
  mtp::prof_end(MTP_KC_ATTENTION, st);
  // a = u + o Wo^T, x = RMSNorm_f(a)
  MTP_CUDA_TRY(cudaMemsetAsync(acc, 0, static_cast<size_t>(R) * d * 4, st));
  TRY(linear({{w->wo, q8(&mtp_block_fp8::wo), d, 0}}, d, o, d));
  finish_row_kernel<<<R, kRowThreads, 0, st>>>(acc, u, a, d, W0(w->ffn_norm), x, d, D.eps);
  mtp::note_launch();
  // g = silu(x Wg^T) * (x Wu^T)
  MTP_CUDA_TRY(cudaMemsetAsync(acc, 0, static_cast<size_t>(R) * 2 * ffn * 4, st));
  TRY(linear({{w->w_gate, q8(&mtp_block_fp8::w_gate), ffn, 0}, {w->w_up, q8(&mtp_block_fp8::w_up), ffn, ffn}}, d, x,
             2 * ffn));
  finish_swiglu_kernel<<<dim3((ffn + 255) / 256, R), 256, 0, st>>>(acc, g, ffn);
  mtp::note_launch();
  // h = a + g Wd^T, x = RMSNorm_out(h)
  MTP_CUDA_TRY(cudaMemsetAsync(acc, 0, static_cast<size_t>(R) * d * 4, st));
  TRY(linear({{w->w_down, q8(&mtp_block_fp8::w_down), d, 0}}, ffn, g, d));
  finish_row_kernel<<<R, kRowThreads, 0, st>>>(acc, a, h_s, ld_h, static_cast<const __nv_bfloat16*>(w->out_norm),
                                               x, d, D.eps);
  mtp::note_launch();
  // logits into q, then softmax and the draw
  mtp::prof_begin(MTP_KC_HEAD_CE_GEMM, st);
  if (ldq > 0x7FFFFFFFull) return MTP_ERR_UNSUPPORTED;
  TRY(skinny_gemm(static_cast<const __nv_bfloat16*>(w->head), V, d, x, R, q_s, static_cast<int>(ldq), st));
  mtp::prof_end(MTP_KC_HEAD_CE_GEMM, st);
  softmax_sample_kernel<<<R * kSampleCluster, kSampleThreads, 0, st>>>(
      q_s, V, ldq, key, static_cast<uint32_t>(step), static_cast<uint32_t>(offset & 0xFFFFFFFFu),
      static_cast<uint32_t>(offset >> 32), y_s, y_stride);
  mtp::note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

}  // namespace

extern "C" size_t mtp_draft_round_workspace_bytes(const mtp_dims* dims, int gamma) {
  if (!dims || !draft_dims_ok(*dims) || gamma < 1 || gamma > kMaxRoundGamma) return 0;
  return draft_layout(*dims, gamma).total;
}

extern "C" size_t mtp_draft_workspace_bytes(const mtp_dims* dims) { return mtp_draft_round_workspace_bytes(dims, 1); }

namespace {

mtp_status draft_round_impl(const mtp_dims* dims, const mtp_weights* w, const mtp_block_fp8* f8,
                            const void* parent_hidden, const int32_t* frontier, const int32_t* pos, const void* kv_k,
                            const void* kv_v, const int32_t* ctx_len, int gamma, uint64_t seed, uint64_t offset,
                            float* q_out, int32_t* y_out, void* h_out, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (!dims || !w) return MTP_ERR_INVALID_ARG;
  const mtp_dims& D = *dims;
  if (!draft_dims_ok(D)) return D.dtype != MTP_BF16 || D.D != 1 || D.B > kMaxR ? MTP_ERR_UNSUPPORTED : MTP_ERR_SHAPE;
  if (gamma < 1) return MTP_ERR_INVALID_ARG;
  if (gamma > kMaxRoundGamma) return MTP_ERR_UNSUPPORTED;
  if (!parent_hidden || !frontier || !pos || !kv_k || !kv_v || !ctx_len || !q_out || !y_out || !ws)
    return MTP_ERR_INVALID_ARG;
  if (!w->embed || !w->head || !w->out_norm) return MTP_ERR_INVALID_ARG;
  const void* const* norms[] = {w->hnorm, w->enorm, w->attn_norm, w->ffn_norm};
  for (auto l : norms)
    if (!l || !l[0] || !mtp::aligned16(l[0])) return l && l[0] ? MTP_ERR_ALIGNMENT : MTP_ERR_INVALID_ARG;
  if (f8) {
    if (D.ffn % 16) return MTP_ERR_UNSUPPORTED;  // 16-byte rows of the e4m3 down projection
    const mtp_fp8_matrix* mats[] = {&f8->eh_proj, &f8->wq, &f8->wk, &f8->wv, &f8->wo,
                                    &f8->w_gate, &f8->w_up, &f8->w_down};
    for (auto m : mats) {
      if (!m->q || !m->scale) return MTP_ERR_INVALID_ARG;
      if (!mtp::aligned16(m->q) || (reinterpret_cast<uintptr_t>(m->scale) & 3u)) return MTP_ERR_ALIGNMENT;
    }
  } else {
    const void* const* lists[] = {w->eh_proj, w->wq, w->wk, w->wv, w->wo, w->w_gate, w->w_up, w->w_down};
    for (auto l : lists)
      if (!l || !l[0] || !mtp::aligned16(l[0])) return l && l[0] ? MTP_ERR_ALIGNMENT : MTP_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {parent_hidden, kv_k, kv_v, static_cast<const void*>(q_out), ws, w->embed, w->head,
                        w->out_norm};
  for (const void* p : ptrs)
    if (!mtp::aligned16(p)) return MTP_ERR_ALIGNMENT;
  if (h_out && !mtp::aligned16(h_out)) return MTP_ERR_ALIGNMENT;
  const DraftLayout L = draft_layout(D, gamma);
  if (ws_bytes < L.total) return MTP_ERR_WORKSPACE;

  const int R = D.B, d = D.d;
  uint8_t* base = static_cast<uint8_t*>(ws);
  __nv_bfloat16* hbuf = reinterpret_cast<__nv_bfloat16*>(base + L.h);
  const uint2 key = make_uint2(static_cast<uint32_t>(seed & 0xFFFFFFFFu), static_cast<uint32_t>(seed >> 32));
  const size_t ldq = static_cast<size_t>(gamma) * D.V;
  for (int s = 0; s < gamma; ++s) {
    // the step's state: into h_out [R, gamma, d] if given, else a workspace ping-pong row
    __nv_bfloat16* h_s = h_out ? static_cast<__nv_bfloat16*>(h_out) + static_cast<size_t>(s) * d
                               : hbuf + static_cast<size_t>(s & 1) * R * d;
    const int ld_h = h_out ? gamma * d : d;
    const __nv_bfloat16* parent = static_cast<const __nv_bfloat16*>(parent_hidden);
    int ld_parent = d;
    const int32_t* f = frontier;
    int f_stride = 1;
    if (s > 0) {  // recurrent reuse: the previous step's state and draw
      parent = h_out ? static_cast<const __nv_bfloat16*>(h_out) + static_cast<size_t>(s - 1) * d
                     : hbuf + static_cast<size_t>((s - 1) & 1) * R * d;
      ld_parent = ld_h;
      f = y_out + (s - 1);
      f_stride = gamma;
    }
    TRY(draft_one_step(D, w, f8, L, base, parent, ld_parent, f, f_stride, pos, kv_k, kv_v, ctx_len, s, gamma, key,
                       offset, q_out + static_cast<size_t>(s) * D.V, ldq, y_out + s, gamma, h_s, ld_h, st));
  }
  return MTP_OK;
}

}  // namespace

extern "C" mtp_status mtp_draft_round(const mtp_dims* dims, const mtp_weights* w, const void* parent_hidden,
                                      const int32_t* frontier, const int32_t* pos, const void* kv_k,
                                      const void* kv_v, const int32_t* ctx_len, int gamma, uint64_t seed,
                                      uint64_t offset, float* q_out, int32_t* y_out, void* h_out, void* ws,
                                      size_t ws_bytes, cudaStream_t st) {
  return draft_round_impl(dims, w, nullptr, parent_hidden, frontier, pos, kv_k, kv_v, ctx_len, gamma, seed, offset,
                          q_out, y_out, h_out, ws, ws_bytes, st);
}

extern "C" mtp_status mtp_draft_round_fp8(const mtp_dims* dims, const mtp_weights* w, const mtp_block_fp8* f8,
                                          const void* parent_hidden, const int32_t* frontier, const int32_t* pos,
                                          const void* kv_k, const void* kv_v, const int32_t* ctx_len, int gamma,
                                          uint64_t seed, uint64_t offset, float* q_out, int32_t* y_out, void* h_out,
                                          void* ws, size_t ws_bytes, cudaStream_t st) {
  if (!f8) return MTP_ERR_INVALID_ARG;
  return draft_round_impl(dims, w, f8, parent_hidden, frontier, pos, kv_k, kv_v, ctx_len, gamma, seed, offset, q_out,
                          y_out, h_out, ws, ws_bytes, st);
}

extern "C" mtp_status mtp_draft_step(const mtp_dims* dims, const mtp_weights* w, const void* parent_hidden,
                                     const int32_t* frontier, const int32_t* pos, const void* kv_k, const void* kv_v,
                                     const int32_t* ctx_len, uint64_t seed, uint64_t offset, float* q_out,
                                     int32_t* y_out, void* h_out, void* ws, size_t ws_bytes, cudaStream_t st) {
  return mtp_draft_round(dims, w, parent_hidden, frontier, pos, kv_k, kv_v, ctx_len, 1, seed, offset, q_out, y_out,
                         h_out, ws, ws_bytes, st);
}
