// The teacher-forced sequential MTP chain and its masked cross-entropy loss.
//
// "M7.6 - DeepSeek MTP: Sequential Modules, Teacher Forcing, and Speculative
// Runtime": module equations (§0x03, §0x03C), depth alignment (§0x04), the
// row compiler's state/label support (§0x04C), the per-depth objective and
// L = L_main + λ/D Σ_k L^(k) (§0x05); "M7.4 - Multi-Token Prediction
// Foundations": label ownership on packed batches (§0x01A, §0x03A) and the
// max / sum-exp / target-logit form of the vocabulary cross-entropy (§0x06F).
//
// Dense layout: every depth keeps the [B, T, d] row = base-position identity.
// Row t of depth k reads h^{k-1}[t] and E[x_{t+k}].  With contiguous segments
// the row compiler's "t..t+k active and in one segment" is t+k < seg_end(t),
// and its label condition is t+k+1 < seg_end(t); a segment-causal key range
// [seg_start(t), t] only ever reaches rows that are themselves valid, so the
// dense rows carry exactly the compact rows' values.  Rows without state are
// computed on clamped inputs and never read by valid rows.
//
// Per depth (bf16): prologue (gather, dual RMSNorm, concat) -> eh_proj GEMM ->
// RMSNorm_a -> QKV GEMM + RoPE epilogue -> flash attention -> O GEMM +
// residual -> RMSNorm_f -> gate/up GEMM + SwiGLU epilogue -> down GEMM +
// residual = h^k -> RMSNorm_out -> head GEMM with online max/sum-exp
// epilogue (logits never stored) -> per-row CE and per-term sums.
// GEMMs run on the tcgen05 core (gemm_tc.cu); the f32 specialisation (small
// shapes) runs the same steps on SIMT kernels in fp32.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "gemm_tc.cuh"

MTP_DEFINE_ERROR_WORD(mtp_take_errors_chain)

namespace mtp {
mtp_status attn_bwd_launch(const __nv_bfloat16* qkv, const __nv_bfloat16* o, const __nv_bfloat16* dO,
                           const float* lse2, const int32_t* seg_start, const int32_t* seg_end, float* dqkv,
                           float* dsum, int B, int T, int H, int hd, cudaStream_t stream);
// work_ctr (bf16): a device int that is 0 on entry and is used up by the launch (one per launch)
mtp_status attn_launch(int dtype, const void* qkv, void* out, const int32_t* seg_start, int B, int T, int H,
                       int hd, cudaStream_t stream, float* lse2_out = nullptr, int* work_ctr = nullptr);
}

namespace {

using mtp::from_f32;
using mtp::load_f32;

// ---------------------------------------------------------------------------
// Segments: seg_start / seg_end (exclusive) of every position, token checks.
// One CTA per packed row; a block-wide max-scan of run starts and a reverse
// min-scan of run ends.  Pads get seg_start = seg_end = t.
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 1024;

// Inclusive max-scan over threadIdx order (blockDim a multiple of 32, at most 1024): within
// each warp by shuffles, then over the warp totals; the result is also left in sh[threadIdx.x].
__device__ int block_scan_max(int v, int* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = max(v, n);
  }
  if (lane == 31) sh[w] = v;
  __syncthreads();
  if (w == 0) {
    int t = lane < static_cast<int>(blockDim.x >> 5) ? sh[lane] : INT_MIN;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t = max(t, n);
    }
    sh[lane] = t;
  }
  __syncthreads();
  if (w > 0) v = max(v, sh[w - 1]);
  __syncthreads();
  sh[threadIdx.x] = v;
  __syncthreads();
  return v;
}

// (cos, sin) table entry i = p * half + j of the angle p * base^(-2j/hd) (rope_table_kernel)
__device__ __forceinline__ float2 rope_entry(int p, double inv_freq) {
  const double ang = static_cast<double>(p) * inv_freq;
  const double two_pi = 6.283185307179586;
  const double red = ang - rint(ang / two_pi) * two_pi;
  float s, c;
  sincosf(static_cast<float>(red), &s, &c);
  return make_float2(c, s);
}

struct SetupArgs {
  double* sums = nullptr;  // the loss (sum, count) pairs to zero (null: none)
  int n_sums = 0;
  float2* rope = nullptr;  // [T, half]
  int half = 0, hd = 0;
  double base = 0.0;       // 0: RoPE off, the table is zeroed
};

// The call's setup in one launch.  Blocks [0, B) find the segment bounds of packed row b
// (block 0 also zeroes the loss sums and the attention work counters); the blocks after them
// fill the RoPE table, each computing its frequencies base^(-2j/hd) once.
__global__ void __launch_bounds__(kScanThreads)
segments_kernel(const int32_t* __restrict__ seg, const int32_t* __restrict__ tokens, int T, int V,
                int32_t* __restrict__ seg_start, int32_t* __restrict__ seg_end, int* __restrict__ work_ctrs,
                int n_ctrs, int B, SetupArgs A) {
  __shared__ int sh[kScanThreads];
  __shared__ double inv_freq[64];
  const int b = blockIdx.x;
  if (b >= B) {  // RoPE table
    if (A.base > 0.0 && threadIdx.x < A.half) inv_freq[threadIdx.x] = exp2(-2.0 * threadIdx.x / A.hd * log2(A.base));
    __syncthreads();
    const int i = (b - B) * blockDim.x + threadIdx.x;
    if (i < T * A.half) A.rope[i] = A.base > 0.0 ? rope_entry(i / A.half, inv_freq[i % A.half]) : make_float2(0.f, 0.f);
    return;
  }
  if (b == 0) {
    // the attention launches of this call claim their work items from these counters
    for (int i = threadIdx.x; i < n_ctrs; i += blockDim.x) work_ctrs[i] = 0;
    for (int i = threadIdx.x; i < A.n_sums; i += blockDim.x) A.sums[i] = 0.0;
  }
  const int32_t* s = seg + static_cast<size_t>(b) * T;
  const int32_t* x = tokens + static_cast<size_t>(b) * T;
  int32_t* out_start = seg_start + static_cast<size_t>(b) * T;
  int32_t* out_end = seg_end + static_cast<size_t>(b) * T;
  const int per = (T + kScanThreads - 1) / kScanThreads;
  auto run_begins = [&](int t) { return t == 0 || s[t] != s[t - 1]; };
  auto run_ends = [&](int t) { return t == T - 1 || s[t] != s[t + 1]; };

  // forward pass over chunk [t0, t1): carry = last run start / largest id to the left
  const int t0 = min(T, threadIdx.x * per), t1 = min(T, t0 + per);
  int last_start = INT_MIN, max_id = INT_MIN;
  for (int t = t0; t < t1; ++t) {
    if (run_begins(t)) last_start = t;
    if (s[t] != -1) max_id = max(max_id, s[t]);
  }
  block_scan_max(last_start, sh);
  int cur_start = threadIdx.x ? sh[threadIdx.x - 1] : INT_MIN;
  __syncthreads();
  block_scan_max(max_id, sh);
  int prev_max = threadIdx.x ? sh[threadIdx.x - 1] : INT_MIN;
  __syncthreads();
  bool bad_seg = false, bad_tok = false;
  for (int t = t0; t < t1; ++t) {
    const bool nr = run_begins(t);
    if (nr) cur_start = t;
    if (s[t] != -1) {
      if (nr && prev_max != INT_MIN && s[t] <= prev_max) bad_seg = true;  // an id re-appears
      prev_max = max(prev_max, s[t]);
    }
    out_start[t] = s[t] == -1 ? t : cur_start;
    if (x[t] < 0 || x[t] >= V) bad_tok = true;
  }

  // backward pass: thread i owns chunk (kScanThreads-1-i), so thread order runs
  // right to left; carry = nearest run end to the right, scanned as max of -(end)
  const int rc = kScanThreads - 1 - threadIdx.x;
  const int r0 = min(T, rc * per), r1 = min(T, r0 + per);
  int first_end = INT_MIN;
  for (int t = r0; t < r1; ++t)
    if (run_ends(t)) { first_end = -(t + 1); break; }
  block_scan_max(first_end, sh);
  int cur_end = threadIdx.x ? sh[threadIdx.x - 1] : INT_MIN;
  __syncthreads();
  for (int t = r1 - 1; t >= r0; --t) {
    if (run_ends(t)) cur_end = -(t + 1);
    out_end[t] = s[t] == -1 ? t : -cur_end;
  }
  if (bad_seg) atomicOr(&g_mtp_error_word, MTP_DEVERR_SEGMENTS);
  if (bad_tok) atomicOr(&g_mtp_error_word, MTP_DEVERR_TOKEN_RANGE);
}

__device__ __forceinline__ int clamp_token(int v, int V) { return min(max(v, 0), V - 1); }

// ---------------------------------------------------------------------------
// Prologue: c = [RMSNorm_h(h^{k-1}); RMSNorm_e(E[x_{t+k}])] (one warp per row)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void prologue_kernel(const T* __restrict__ h_prev, const int32_t* __restrict__ tokens,
                                const T* __restrict__ embed, const T* __restrict__ g_h, const T* __restrict__ g_e,
                                T* __restrict__ c, int M, int Tlen, int d, int V, int k, float eps) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= M) return;
  const int m = warp;
  const int t = m % Tlen;
  const int src_t = min(t + k, Tlen - 1);
  const int tok = clamp_token(tokens[m - t + src_t], V);
  const T* h = h_prev + static_cast<size_t>(m) * d;
  const T* e = embed + static_cast<size_t>(tok) * d;
  float sh = 0.f, se = 0.f;
  for (int i = lane; i < d; i += 32) {
    const float a = load_f32(h + i), b = load_f32(e + i);
    sh += a * a;
    se += b * b;
  }
  sh = mtp::warp_sum(sh);
  se = mtp::warp_sum(se);
  const float rh = 1.0f / sqrtf(sh / d + eps);
  const float re = 1.0f / sqrtf(se / d + eps);
  T* out = c + static_cast<size_t>(m) * 2 * d;
  for (int i = lane; i < d; i += 32) {
    out[i] = from_f32<T>(load_f32(g_h + i) * (load_f32(h + i) * rh));
    out[d + i] = from_f32<T>(load_f32(g_e + i) * (load_f32(e + i) * re));
  }
}

// 8 bf16 <-> 8 floats
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}
__device__ __forceinline__ float sumsq8(const uint4& u) {
  float f[8];
  unpack8(u, f);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += f[i] * f[i];
  return s;
}
// out = bf16(g * x * r) for one 8-element chunk
__device__ __forceinline__ uint4 norm8(const uint4& x, const uint4& g, float r) {
  float fx[8], fg[8];
  unpack8(x, fx);
  unpack8(g, fg);
#pragma unroll
  for (int i = 0; i < 8; ++i) fx[i] = fg[i] * (fx[i] * r);
  return pack8(fx);
}

// bf16 prologue with 16-byte accesses (d % 8 == 0); same arithmetic order as above
__global__ void prologue_bf16_kernel(const uint4* __restrict__ h_prev, const int32_t* __restrict__ tokens,
                                     const uint4* __restrict__ embed, const uint4* __restrict__ g_h,
                                     const uint4* __restrict__ g_e, uint4* __restrict__ c, int M, int Tlen, int d8,
                                     int V, int k, float eps) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  mtp::pdl_wait();     // launched as a dependent of the kernel before it
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= M) return;
  const int m = warp;
  const int t = m % Tlen;
  const int tok = clamp_token(tokens[m - t + min(t + k, Tlen - 1)], V);
  const uint4* h = h_prev + static_cast<size_t>(m) * d8;
  const uint4* e = embed + static_cast<size_t>(tok) * d8;
  float sh = 0.f, se = 0.f;
  for (int i = lane; i < d8; i += 32) {
    sh += sumsq8(h[i]);
    se += sumsq8(e[i]);
  }
  sh = mtp::warp_sum(sh);
  se = mtp::warp_sum(se);
  const float d = 8.0f * d8;
  const float rh = 1.0f / sqrtf(sh / d + eps);
  const float re = 1.0f / sqrtf(se / d + eps);
  uint4* out = c + static_cast<size_t>(m) * 2 * d8;
  for (int i = lane; i < d8; i += 32) {
    out[i] = norm8(h[i], g_h[i], rh);
    out[d8 + i] = norm8(e[i], g_e[i], re);
  }
}

// y = RMSNorm_g(x) row-wise (one warp per row)
template <typename T>
__global__ void rmsnorm_kernel(const T* __restrict__ x, const T* __restrict__ g, T* __restrict__ y, int M, int d,
                               float eps) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= M) return;
  const T* xr = x + static_cast<size_t>(warp) * d;
  float ss = 0.f;
  for (int i = lane; i < d; i += 32) {
    const float a = load_f32(xr + i);
    ss += a * a;
  }
  ss = mtp::warp_sum(ss);
  const float r = 1.0f / sqrtf(ss / d + eps);
  T* yr = y + static_cast<size_t>(warp) * d;
  for (int i = lane; i < d; i += 32) yr[i] = from_f32<T>(load_f32(g + i) * (load_f32(xr + i) * r));
}

// bf16 RMSNorm with 16-byte accesses; when `labels` is given it also writes
// the label of term k for the row (x_{t+k+1} if t..t+k+1 share t's segment,
// else -1), which the head GEMM's CE epilogue consumes.
__global__ void rmsnorm_bf16_kernel(const uint4* __restrict__ x, const uint4* __restrict__ g, uint4* __restrict__ y,
                                    int M, int d8, float eps, const int32_t* __restrict__ tokens,
                                    const int32_t* __restrict__ seg, const int32_t* __restrict__ seg_end,
                                    int32_t* __restrict__ labels, int Tlen, int k, int V) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  mtp::pdl_wait();     // launched as a dependent of the kernel before it
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= M) return;
  const uint4* xr = x + static_cast<size_t>(warp) * d8;
  float ss = 0.f;
  for (int i = lane; i < d8; i += 32) ss += sumsq8(xr[i]);
  ss = mtp::warp_sum(ss);
  const float r = 1.0f / sqrtf(ss / (8.0f * d8) + eps);
  uint4* yr = y + static_cast<size_t>(warp) * d8;
  for (int i = lane; i < d8; i += 32) yr[i] = norm8(xr[i], g[i], r);
  if (labels && lane == 0) {
    const int m = warp, t = m % Tlen;
    const bool ok = seg[m] != -1 && t + k + 1 < seg_end[m];
    labels[m] = ok ? clamp_token(tokens[m + k + 1], V) : -1;
  }
}

// labels of term k (0 = main): x_{t+k+1} where t..t+k+1 lie in t's segment, else -1
__global__ void labels_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ seg,
                              const int32_t* __restrict__ seg_end, int32_t* __restrict__ labels, int M, int Tlen,
                              int k, int V) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  const int t = m % Tlen;
  const bool ok = seg[m] != -1 && t + k + 1 < seg_end[m];
  labels[m] = ok ? clamp_token(tokens[m + k + 1], V) : -1;
}

// ---------------------------------------------------------------------------
// f32 SIMT kernels (small shapes)
// ---------------------------------------------------------------------------
// C[M,N] = A[M,K] B[N,K]^T (+ R), 64x64 tiles, 16x16 threads, 4x4 per thread
__global__ void gemm_f32_kernel(const float* __restrict__ A, int lda, const float* __restrict__ B, int ldb,
                                float* __restrict__ C, int ldc, const float* __restrict__ R, int ldr, int M, int N,
                                int K) {
  __shared__ float As[16][65], Bs[16][65];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
      const int r = i / 16, kk = i % 16;
      As[kk][r] = (m0 + r < M && k0 + kk < K) ? A[static_cast<size_t>(m0 + r) * lda + k0 + kk] : 0.f;
      Bs[kk][r] = (n0 + r < N && k0 + kk < K) ? B[static_cast<size_t>(n0 + r) * ldb + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += As[kk][ty * 4 + i] * Bs[kk][tx * 4 + j];
    __syncthreads();
  }
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < M && n < N)
        C[static_cast<size_t>(m) * ldc + n] = acc[i][j] + (R ? R[static_cast<size_t>(m) * ldr + n] : 0.f);
    }
}

__global__ void rope_f32_kernel(float* __restrict__ qkv, const int32_t* __restrict__ pos,
                                const float2* __restrict__ tab, int M, int d, int hd, int Tlen) {
  const int half = hd / 2;
  const int per_row = 2 * d / 2;  // pairs over q and k
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= M * per_row) return;
  const int m = i / per_row, pr = i % per_row;
  const int head = pr / half, j = pr % half;  // head index over q then k (2*H heads)
  int p = pos[m];
  if (p < 0 || p >= Tlen) {
    atomicOr(&g_mtp_error_word, MTP_DEVERR_TOKEN_RANGE);
    p = min(max(p, 0), Tlen - 1);
  }
  const float2 cs = tab[static_cast<size_t>(p) * half + j];
  float* base = qkv + static_cast<size_t>(m) * 3 * d + head * hd;
  const float a = base[j], b = base[j + half];
  base[j] = a * cs.x - b * cs.y;
  base[j + half] = b * cs.x + a * cs.y;
}

__global__ void swiglu_f32_kernel(const float* __restrict__ G, const float* __restrict__ U, float* __restrict__ out,
                                  size_t n) {
  const size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  if (i >= n) return;
  const float g = G[i];
  out[i] = g / (1.0f + expf(-g)) * U[i];
}

// head logits of one row against a 256-wide vocabulary tile, reduced to the
// tile's (max, sum-exp) and the label logit; same partial format as the
// tcgen05 CE epilogue
__global__ void head_ce_f32_kernel(const float* __restrict__ x, const float* __restrict__ W, int d, int V,
                                   const int32_t* __restrict__ labels, float2* __restrict__ part, float* __restrict__ zt,
                                   int nvt) {
  __shared__ float red[256];
  const int m = blockIdx.y, tile = blockIdx.x;
  const int v = tile * 256 + threadIdx.x;
  float z = -INFINITY;
  if (v < V) {
    float acc = 0.f;
    const float* xr = x + static_cast<size_t>(m) * d;
    const float* wr = W + static_cast<size_t>(v) * d;
    for (int i = 0; i < d; ++i) acc += xr[i] * wr[i];
    z = acc;
    if (labels[m] == v) zt[m] = z;
  }
  red[threadIdx.x] = z;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + o]);
    __syncthreads();
  }
  const float mx = red[0];
  __syncthreads();
  red[threadIdx.x] = v < V ? expf(z - mx) : 0.f;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[static_cast<size_t>(m) * nvt + tile] = make_float2(mx, red[0]);
}

// ---------------------------------------------------------------------------
// CE reduction and loss assembly
// ---------------------------------------------------------------------------
// ℓ_t = max + log Σ_tiles s_j exp(m_j - max) - z_label for supervised rows;
// one warp per row (rows strided over the grid), one (sum, count) atomic pair per block
__global__ void ce_reduce_kernel(int M, int nvt, const float2* __restrict__ part, const float* __restrict__ zt,
                                 const int32_t* __restrict__ labels, float* __restrict__ row_loss,
                                 double* __restrict__ sum_count, float* __restrict__ lse_out) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  mtp::pdl_wait();     // launched as a dependent of the kernel before it
  __shared__ double s_sum[8];
  __shared__ int s_cnt[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  double wsum = 0.0;
  int wcnt = 0;
  for (int m = blockIdx.x * 8 + warp; m < M; m += gridDim.x * 8) {
    float loss = NAN;
    if (labels[m] >= 0) {
      const float2* p = part + static_cast<size_t>(m) * nvt;
      float mx = -INFINITY;
      for (int j = lane; j < nvt; j += 32) mx = fmaxf(mx, p[j].x);
      mx = mtp::warp_max(mx);
      float sum = 0.f;
      for (int j = lane; j < nvt; j += 32) {
        const float2 v = p[j];
        sum += v.y * expf(v.x - mx);
      }
      sum = mtp::warp_sum(sum);
      const float lse = mx + logf(sum);
      loss = lse - zt[m];
      if (lse_out && lane == 0) lse_out[m] = lse;
      wsum += loss;
      ++wcnt;
    }
    if (lane == 0 && row_loss) row_loss[m] = loss;
  }
  if (lane == 0) {
    s_sum[warp] = wsum;
    s_cnt[warp] = wcnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double a = 0.0;
    int c = 0;
    for (int w = 0; w < 8; ++w) {
      a += s_sum[w];
      c += s_cnt[w];
    }
    if (c) {
      atomicAdd(sum_count, a);
      atomicAdd(sum_count + 1, static_cast<double>(c));
    }
  }
}

// ce_reduce_kernel with the partials of G rows held in registers (nvt <= 32 NPL): a warp
// issues the loads of its G rows at once and reads each partial once.  Per row the same
// lane-strided maximum and sum as ce_reduce_kernel, so the same results bit for bit.
template <int NPL, int G>
__global__ void ce_reduce_reg_kernel(int M, int nvt, const float2* __restrict__ part, const float* __restrict__ zt,
                                     const int32_t* __restrict__ labels, float* __restrict__ row_loss,
                                     double* __restrict__ sum_count, float* __restrict__ lse_out) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  mtp::pdl_wait();     // launched as a dependent of the kernel before it
  __shared__ double s_sum[8];
  __shared__ int s_cnt[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  double wsum = 0.0;
  int wcnt = 0;
  const int stride = gridDim.x * 8;
  for (int m0 = blockIdx.x * 8 + warp; m0 < M; m0 += G * stride) {
    float2 v[G][NPL];
    int lab[G];
#pragma unroll
    for (int r = 0; r < G; ++r) {
      const int m = m0 + r * stride;
      lab[r] = m < M ? labels[m] : -1;
      const float2* p = part + static_cast<size_t>(m < M ? m : 0) * nvt;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int j = lane + 32 * i;
        v[r][i] = (lab[r] >= 0 && j < nvt) ? p[j] : make_float2(-INFINITY, 0.f);
      }
    }
#pragma unroll
    for (int r = 0; r < G; ++r) {
      const int m = m0 + r * stride;
      if (m >= M) continue;
      float loss = NAN;
      if (lab[r] >= 0) {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < NPL; ++i)
          if (lane + 32 * i < nvt) mx = fmaxf(mx, v[r][i].x);
        mx = mtp::warp_max(mx);
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < NPL; ++i)
          if (lane + 32 * i < nvt) sum += v[r][i].y * expf(v[r][i].x - mx);
        sum = mtp::warp_sum(sum);
        const float lse = mx + logf(sum);
        loss = lse - zt[m];
        if (lse_out && lane == 0) lse_out[m] = lse;
        wsum += loss;
        ++wcnt;
      }
      if (lane == 0 && row_loss) row_loss[m] = loss;
    }
  }
  if (lane == 0) {
    s_sum[warp] = wsum;
    s_cnt[warp] = wcnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double a = 0.0;
    int c = 0;
    for (int w = 0; w < 8; ++w) {
      a += s_sum[w];
      c += s_cnt[w];
    }
    if (c) {
      atomicAdd(sum_count, a);
      atomicAdd(sum_count + 1, static_cast<double>(c));
    }
  }
}

// losses = [L, L_main, L^(1..D)] from (sum, count) pairs
// Per-depth weights of the loss assembly (uniform lambda/D unless given).
constexpr int kMaxDepthWeights = 32;
struct DepthWeights {
  float w[kMaxDepthWeights];
  float lambda;
  int uniform;
};

// L^(k) and the total under reduction `den` (the enum's definitions in
// include/mtp.h): sums_counts holds (S_k, N_k), k = 0 main, 1..D depths.
__global__ void loss_assemble_kernel(const double* __restrict__ sc, float* __restrict__ losses, int D, double n_pos,
                                     DepthWeights W, int den, int with_main) {
  mtp::pdl_wait();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  auto weight = [&](int k) -> double {
    return W.uniform ? static_cast<double>(W.lambda) / D : static_cast<double>(W.w[k - 1]);
  };
  double n_all = 0.0, wn_all = 0.0;
  for (int k = 1; k <= D; ++k) {
    n_all += sc[2 * k + 1];
    wn_all += weight(k) * sc[2 * k + 1];
  }
  auto div = [](double a, double b) { return b > 0.0 ? a / b : 0.0; };
  auto term = [&](int i) -> double {
    if (den == MTP_DEN_FIXED) return sc[2 * i] / n_pos;
    if (den == MTP_DEN_SUM) return sc[2 * i];
    if (den == MTP_DEN_MASKED_MEAN || i == 0) return div(sc[2 * i], sc[2 * i + 1]);
    if (den == MTP_DEN_GLOBAL) return div(sc[2 * i], n_all);
    return div(sc[2 * i], wn_all);
  };
  const double main = with_main ? term(0) : 0.0;
  double mtp = 0.0;
  for (int k = 1; k <= D; ++k) {
    const double lk = term(k);
    losses[1 + k] = static_cast<float>(lk);
    mtp += weight(k) * lk;
  }
  losses[1] = static_cast<float>(main);
  losses[0] = static_cast<float>(main + mtp);
}

inline bool valid_den(int den) { return den >= MTP_DEN_FIXED && den <= MTP_DEN_WEIGHTED_PAIR; }

// ---------------------------------------------------------------------------
// Host orchestration
// ---------------------------------------------------------------------------
inline size_t align_up(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct Layout {
  size_t seg_start, seg_end, labels, c, u, x, qkv, o, a, g, g2, h0buf, h1buf, rope, ce_part, zt, work_ctrs, total;
  int nvt;
};

bool valid_dims(const mtp_dims& D) {
  if (D.B <= 0 || D.T <= 0 || D.d <= 0 || D.n_heads <= 0 || D.head_dim <= 0 || D.ffn <= 0 || D.V <= 0 || D.D <= 0)
    return false;
  if (D.n_heads * D.head_dim != D.d || D.head_dim % 2) return false;
  if (D.dtype != MTP_F32 && D.dtype != MTP_BF16) return false;
  if (!(D.eps >= 0.f) || !(D.rope_base >= 0.f)) return false;
  return true;
}

mtp_status supported(const mtp_dims& D) {
  if (D.dtype == MTP_BF16) {
    if (D.d % 128 || (D.head_dim != 64 && D.head_dim != 128) || D.ffn % 8) return MTP_ERR_UNSUPPORTED;
  } else {
    if (D.head_dim > 128 || static_cast<size_t>(D.T) * 16 > 200 * 1024) return MTP_ERR_UNSUPPORTED;
  }
  if (static_cast<long long>(D.B) * D.T > (1ll << 30)) return MTP_ERR_UNSUPPORTED;
  if (static_cast<long long>(D.T) * (D.head_dim / 2) > (1ll << 30)) return MTP_ERR_UNSUPPORTED;  // RoPE table
  return MTP_OK;
}

Layout make_layout(const mtp_dims& D) {
  Layout L{};
  const size_t M = static_cast<size_t>(D.B) * D.T;
  const size_t es = D.dtype == MTP_BF16 ? 2 : 4;
  L.nvt = (D.V + mtp::gemm_ce_tile_n() - 1) / mtp::gemm_ce_tile_n();
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  L.seg_start = take(M * 4);
  L.seg_end = take(M * 4);
  L.labels = take(M * 4);
  L.c = take(M * 2 * D.d * es);
  L.u = take(M * D.d * es);
  L.x = take(M * D.d * es);
  L.qkv = take(M * 3 * D.d * es);
  L.o = take(M * D.d * es);
  L.a = take(M * D.d * es);
  L.g = take(M * D.ffn * es);
  L.g2 = D.dtype == MTP_F32 ? take(M * D.ffn * es) : off;
  L.h0buf = take(M * D.d * es);
  L.h1buf = take(M * D.d * es);
  L.rope = take(static_cast<size_t>(D.T) * (D.head_dim / 2) * sizeof(float2));
  L.ce_part = take(M * L.nvt * sizeof(float2));
  L.zt = take(M * 4);
  L.work_ctrs = take(static_cast<size_t>(D.D) * sizeof(int));  // one per depth's attention launch
  L.total = off;
  return L;
}

// per-depth activations a training step keeps (offsets inside one depth's slot)
struct SaveOff {
  size_t c, u, x, qkv, o, a, y, lse2, bytes;
};

struct Ctx {
  const mtp_dims& D;
  const mtp_weights& W;
  const int32_t* tokens;
  const int32_t* seg;
  const int32_t* pos;
  uint8_t* ws;
  Layout L;
  cudaStream_t st;
  int M;
  float* lse_save = nullptr;  // training: per-term log-sum-exp of every supervised row, [(D+1), M]
  uint8_t* save = nullptr;     // training: depth i's activations at save + i * so.bytes
  SaveOff so{};
  // loss calls: a second stream for the row kernels off the chain of blocks (the next depth's
  // prologue, each term's CE reduction) and the events that order it against st (kEv*)
  cudaStream_t side = nullptr;
  cudaEvent_t* ev = nullptr;
  mutable bool red_pending = false;  // a CE reduction was enqueued on `side` (kEvRed recorded)
  template <typename T>
  T* buf(size_t off) const {
    return reinterpret_cast<T*>(ws + off);
  }
};

inline int warp_blocks(int rows) { return (rows + 7) / 8; }  // 8 warps (256 threads) per block

// Events of a loss call's second stream: the next prologue done, the head's norm enqueued (h^k
// ready), a head GEMM done, a CE reduction done.
enum { kEvPro = 0, kEvH, kEvHead, kEvRed, kSideEvents };
struct SideStream {
  std::mutex mu;
  cudaStream_t s = nullptr;
  cudaEvent_t ev[kSideEvents] = {};
  bool ready = false;
};
SideStream g_side[mtp::kMaxDevices];

// The current device's second stream, locked into `lock` for the call that enqueues on it
// (concurrent calls on one device take turns); null if it cannot be created, in which case
// the call runs on its own stream alone.
SideStream* side_stream(std::unique_lock<std::mutex>& lock) {
  const int dev = mtp::current_device();
  if (dev < 0 || dev >= mtp::kMaxDevices) return nullptr;
  SideStream& S = g_side[dev];
  lock = std::unique_lock<std::mutex>(S.mu);
  if (!S.ready) {
    bool ok = cudaStreamCreateWithFlags(&S.s, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < kSideEvents; ++i) ok = cudaEventCreateWithFlags(&S.ev[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return nullptr;
    }
    S.ready = true;
  }
  return &S;
}

// pdl = false: the stream's previous operation is not a kernel (e.g. an event wait)
template <typename T>
mtp_status gemm(const Ctx& C, const T* A, int lda, const T* const* Bs, int nseg, int seg_rows, int K, int N,
                T* out, int ldo, int epi, const T* resid = nullptr, int ldr = 0, const T* B2 = nullptr,
                bool pdl = true);

// bf16: the tcgen05 core
template <>
mtp_status gemm<__nv_bfloat16>(const Ctx& C, const __nv_bfloat16* A, int lda, const __nv_bfloat16* const* Bs,
                               int nseg, int seg_rows, int K, int N, __nv_bfloat16* out, int ldo, int epi,
                               const __nv_bfloat16* resid, int ldr, const __nv_bfloat16* B2, bool pdl) {
  mtp::GemmDesc g;
  g.M = C.M;
  g.N = N;
  g.K = K;
  g.A = A;
  g.lda = lda;
  for (int i = 0; i < nseg; ++i) g.B[i] = Bs[i];
  if (epi == mtp::EPI_SWIGLU) g.B[1] = B2;
  g.ldb = K;
  g.nseg = nseg;
  g.seg_rows = seg_rows;
  g.epi = epi;
  g.out = out;
  g.ldo = ldo;
  g.resid = resid;
  g.ldr = ldr;
  g.pdl = pdl;  // every forward-chain GEMM follows one of this library's kernels unless told otherwise
  g.b_early = true;  // B is a weight matrix
  g.trigger_early = true;  // the next kernel of the chain is a programmatic dependent
  if (epi == mtp::EPI_ROPE) {
    g.pos = C.pos;
    g.rope = C.buf<float2>(C.L.rope);
    g.rope_len = C.D.T;
    g.rope_cols = 2 * C.D.d;
    g.head_dim = C.D.head_dim;
  }
  return mtp::gemm_bf16_launch(g, C.st);
}

// f32: SIMT tiles; RoPE and SwiGLU as separate elementwise kernels
template <>
mtp_status gemm<float>(const Ctx& C, const float* A, int lda, const float* const* Bs, int nseg, int seg_rows, int K,
                       int N, float* out, int ldo, int epi, const float* resid, int ldr, const float* B2, bool) {
  auto run = [&](const float* B, float* o, int n, int ldo_, const float* R, int ldr_) {
    const dim3 grid((n + 63) / 64, (C.M + 63) / 64);
    gemm_f32_kernel<<<grid, 256, 0, C.st>>>(A, lda, B, K, o, ldo_, R, ldr_, C.M, n, K);
    mtp::note_launch();
  };
  if (epi == mtp::EPI_SWIGLU) {
    float* U = C.buf<float>(C.L.g2);
    run(Bs[0], out, N, ldo, nullptr, 0);
    run(B2, U, N, N, nullptr, 0);
    const size_t n = static_cast<size_t>(C.M) * N;
    swiglu_f32_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, C.st>>>(out, U, out, n);
    mtp::note_launch();
  } else {
    for (int s = 0; s < nseg; ++s) run(Bs[s], out + static_cast<size_t>(s) * seg_rows, seg_rows, ldo, resid, ldr);
    if (epi == mtp::EPI_ROPE && C.D.rope_base > 0.f) {
      const int n = C.M * C.D.d;
      rope_f32_kernel<<<(n + 255) / 256, 256, 0, C.st>>>(out, C.pos, C.buf<float2>(C.L.rope), C.M, C.D.d,
                                                          C.D.head_dim, C.D.T);
      mtp::note_launch();
    }
  }
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

#define TRY(expr)                          \
  do {                                     \
    mtp_status s_ = (expr);                \
    if (s_ != MTP_OK) return s_;           \
  } while (0)

// RMSNorm launch; with `labels` it also writes term k's labels (bf16 fuses
// them into the norm kernel, f32 uses a separate kernel).
// Register-resident forms of the two bf16 row kernels for d = 256 * NPL: every
// lane loads its NPL 16-byte chunks of the row at once, so a warp has the whole
// row in flight and reads it once.  Same summation order as the looped kernels
// (lane-strided chunks, then the warp sum), hence the same results bit for bit.
template <int NPL>
__global__ void rmsnorm_bf16_reg_kernel(const uint4* __restrict__ x, const uint4* __restrict__ g,
                                        uint4* __restrict__ y, int M, float eps, const int32_t* __restrict__ tokens,
                                        const int32_t* __restrict__ seg, const int32_t* __restrict__ seg_end,
                                        int32_t* __restrict__ labels, int Tlen, int k, int V) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  mtp::pdl_wait();     // launched as a dependent of the kernel before it
  constexpr int d8 = 32 * NPL;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= M) return;
  const uint4* xr = x + static_cast<size_t>(warp) * d8;
  uint4 v[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) v[i] = xr[lane + 32 * i];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) ss += sumsq8(v[i]);
  ss = mtp::warp_sum(ss);
  const float r = 1.0f / sqrtf(ss / (8.0f * d8) + eps);
  uint4* yr = y + static_cast<size_t>(warp) * d8;
#pragma unroll
  for (int i = 0; i < NPL; ++i) yr[lane + 32 * i] = norm8(v[i], g[lane + 32 * i], r);
  if (labels && lane == 0) {
    const int m = warp, t = m % Tlen;
    const bool ok = seg[m] != -1 && t + k + 1 < seg_end[m];
    labels[m] = ok ? clamp_token(tokens[m + k + 1], V) : -1;
  }
}

template <int NPL>
__global__ void prologue_bf16_reg_kernel(const uint4* __restrict__ h_prev, const int32_t* __restrict__ tokens,
                                         const uint4* __restrict__ embed, const uint4* __restrict__ g_h,
                                         const uint4* __restrict__ g_e, uint4* __restrict__ c, int M, int Tlen, int V,
                                         int k, float eps) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  mtp::pdl_wait();     // launched as a dependent of the kernel before it
  constexpr int d8 = 32 * NPL;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= M) return;
  const int m = warp;
  const int t = m % Tlen;
  const int tok = clamp_token(tokens[m - t + min(t + k, Tlen - 1)], V);
  const uint4* h = h_prev + static_cast<size_t>(m) * d8;
  const uint4* e = embed + static_cast<size_t>(tok) * d8;
  uint4 hv[NPL], ev[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    hv[i] = h[lane + 32 * i];
    ev[i] = e[lane + 32 * i];
  }
  float sh = 0.f, se = 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    sh += sumsq8(hv[i]);
    se += sumsq8(ev[i]);
  }
  sh = mtp::warp_sum(sh);
  se = mtp::warp_sum(se);
  const float d = 8.0f * d8;
  const float rh = 1.0f / sqrtf(sh / d + eps);
  const float re = 1.0f / sqrtf(se / d + eps);
  uint4* out = c + static_cast<size_t>(m) * 2 * d8;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    out[lane + 32 * i] = norm8(hv[i], g_h[lane + 32 * i], rh);
    out[d8 + lane + 32 * i] = norm8(ev[i], g_e[lane + 32 * i], re);
  }
}

// pdl: launch as a programmatic dependent (the stream's previous operation is a kernel)
template <typename T>
void launch_rmsnorm(const Ctx& C, const T* x, const T* g, T* y, int32_t* labels = nullptr, int k = 0,
                    bool pdl = false) {
  const mtp_dims& D = C.D;
  if constexpr (sizeof(T) == 2) {
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    const uint4* gv = reinterpret_cast<const uint4*>(g);
    uint4* yv = reinterpret_cast<uint4*>(y);
    const int32_t* se = C.buf<int32_t>(C.L.seg_end);
    const dim3 grid(warp_blocks(C.M)), block(256);
    auto go = [&](auto kern) {
      if (pdl)
        mtp::launch_pdl(kern, grid, block, 0, C.st, xv, gv, yv, C.M, D.eps, C.tokens, C.seg, se, labels, D.T, k, D.V);
      else
        kern<<<grid, block, 0, C.st>>>(xv, gv, yv, C.M, D.eps, C.tokens, C.seg, se, labels, D.T, k, D.V);
    };
    switch (D.d) {
      case 256: go(rmsnorm_bf16_reg_kernel<1>); break;
      case 512: go(rmsnorm_bf16_reg_kernel<2>); break;
      case 1024: go(rmsnorm_bf16_reg_kernel<4>); break;
      case 2048: go(rmsnorm_bf16_reg_kernel<8>); break;
      default:
        if (pdl)
          mtp::launch_pdl(rmsnorm_bf16_kernel, grid, block, 0, C.st, xv, gv, yv, C.M, D.d / 8, D.eps, C.tokens, C.seg,
                          se, labels, D.T, k, D.V);
        else
          rmsnorm_bf16_kernel<<<grid, block, 0, C.st>>>(xv, gv, yv, C.M, D.d / 8, D.eps, C.tokens, C.seg, se, labels,
                                                        D.T, k, D.V);
    }
    mtp::note_launch();
  } else {
    rmsnorm_kernel<T><<<warp_blocks(C.M), 256, 0, C.st>>>(x, g, y, C.M, D.d, D.eps);
    mtp::note_launch();
    if (labels) {
      labels_kernel<<<(C.M + 255) / 256, 256, 0, C.st>>>(C.tokens, C.seg, C.buf<int32_t>(C.L.seg_end), labels, C.M,
                                                         D.T, k, D.V);
      mtp::note_launch();
    }
  }
}

template <typename T>
void launch_prologue(const Ctx& C, const T* h_prev, int k, T* c, cudaStream_t st, bool pdl);

// head + CE for term `k` (0 = main) on hidden state h.  With the second stream and next_c, the
// prologue of depth k + 1 (which reads the same h) runs there beside this head's GEMM.
template <typename T>
mtp_status head_ce(const Ctx& C, const T* h, int k, float* row_loss_term, double* sum_count, T* next_c = nullptr) {
  const mtp_dims& D = C.D;
  T* x = C.buf<T>(C.L.x);
  int32_t* labels = C.buf<int32_t>(C.L.labels);
  float2* part = C.buf<float2>(C.L.ce_part);
  float* zt = C.buf<float>(C.L.zt);
  // its predecessor is a kernel (the previous depth's down projection or the setup kernel) unless
  // the previous term's CE reduction, on the second stream, must first finish reading the labels,
  // the partials and the target logits that this term overwrites
  bool norm_pdl = true;
  if (C.side && C.red_pending) {
    cudaStreamWaitEvent(C.st, C.ev[kEvRed], 0);
    norm_pdl = false;
  }
  launch_rmsnorm<T>(C, h, static_cast<const T*>(C.W.out_norm), x, labels, k, norm_pdl);
  MTP_LAUNCH_CHECK();
  if (C.side && next_c) {  // after the norm, so that it shares the SMs with the head GEMM rather than the norm
    cudaEventRecord(C.ev[kEvH], C.st);
    cudaStreamWaitEvent(C.side, C.ev[kEvH], 0);
    mtp::prof_begin(MTP_KC_PROLOGUE, C.side);
    launch_prologue<T>(C, h, k + 1, next_c, C.side, false);
    mtp::prof_end(MTP_KC_PROLOGUE, C.side);
    cudaEventRecord(C.ev[kEvPro], C.side);
    MTP_LAUNCH_CHECK();
  }
  if constexpr (sizeof(T) == 2) {
    mtp::GemmDesc g;
    g.M = C.M;
    g.N = D.V;
    g.K = D.d;
    g.A = x;
    g.lda = D.d;
    g.B[0] = static_cast<const __nv_bfloat16*>(C.W.head);
    g.ldb = D.d;
    g.nseg = 1;
    g.seg_rows = D.V;
    g.epi = mtp::EPI_CE;
    g.labels = labels;
    g.ce_part = part;
    g.z_tgt = zt;
    g.pdl = true;  // follows the RMSNorm kernel
    g.b_early = true;  // B = W_U
    g.trigger_early = true;  // the CE reduction that follows is a programmatic dependent
    mtp::prof_begin(MTP_KC_HEAD_CE_GEMM, C.st);
    TRY(mtp::gemm_bf16_launch(g, C.st));
    mtp::prof_end(MTP_KC_HEAD_CE_GEMM, C.st);
  } else {
    head_ce_f32_kernel<<<dim3(C.L.nvt, C.M), 256, 0, C.st>>>(x, static_cast<const float*>(C.W.head), D.d, D.V, labels,
                                                             part, zt, C.L.nvt);
    mtp::note_launch();
  }
  {
    const int grid = std::min((C.M + 7) / 8, 256);
    float* lse_out = C.lse_save ? C.lse_save + static_cast<size_t>(k) * C.M : nullptr;
    const int nvt = C.L.nvt;
    // on the second stream after the head (nothing on the chain of blocks reads its results), or
    // a programmatic dependent of the head GEMM (bf16) or of the f32 head kernel
    if (C.side) {
      cudaEventRecord(C.ev[kEvHead], C.st);
      cudaStreamWaitEvent(C.side, C.ev[kEvHead], 0);
    }
    auto go = [&](auto kern) {
      if (C.side)
        kern<<<grid, 256, 0, C.side>>>(C.M, nvt, part, zt, labels, row_loss_term, sum_count, lse_out);
      else
        mtp::launch_pdl(kern, dim3(grid), dim3(256), 0, C.st, C.M, nvt, part, zt, labels, row_loss_term, sum_count,
                        lse_out);
    };
    if (nvt <= 128)
      go(ce_reduce_reg_kernel<4, 4>);
    else if (nvt <= 256)
      go(ce_reduce_reg_kernel<8, 2>);
    else if (nvt <= 512)
      go(ce_reduce_reg_kernel<16, 1>);
    else
      go(ce_reduce_kernel);
    if (C.side) {
      cudaEventRecord(C.ev[kEvRed], C.side);
      C.red_pending = true;
    }
  }
  mtp::note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

// prologue input c of depth k from h^(k-1): [RMSNorm_hnorm(h); RMSNorm_enorm(E[x_{t+k}])] on `st`
// (pdl: the stream's previous operation is a kernel)
template <typename T>
void launch_prologue(const Ctx& C, const T* h_prev, int k, T* c, cudaStream_t st, bool pdl) {
  const mtp_dims& D = C.D;
  const int M = C.M, d = D.d, i = k - 1;
  if constexpr (sizeof(T) == 2) {
    const uint4* hp = reinterpret_cast<const uint4*>(h_prev);
    const uint4* ev = static_cast<const uint4*>(C.W.embed);
    const uint4* gh = static_cast<const uint4*>(C.W.hnorm[i]);
    const uint4* ge = static_cast<const uint4*>(C.W.enorm[i]);
    uint4* cv = reinterpret_cast<uint4*>(c);
    auto go = [&](auto kern) {
      if (pdl)
        mtp::launch_pdl(kern, dim3(warp_blocks(M)), dim3(256), 0, st, hp, C.tokens, ev, gh, ge, cv, M, D.T, D.V, k,
                        D.eps);
      else
        kern<<<warp_blocks(M), 256, 0, st>>>(hp, C.tokens, ev, gh, ge, cv, M, D.T, D.V, k, D.eps);
    };
    switch (d) {
      case 256: go(prologue_bf16_reg_kernel<1>); break;
      case 512: go(prologue_bf16_reg_kernel<2>); break;
      case 1024: go(prologue_bf16_reg_kernel<4>); break;
      default:
        prologue_bf16_kernel<<<warp_blocks(M), 256, 0, st>>>(hp, C.tokens, ev, gh, ge, cv, M, D.T, d / 8, D.V, k,
                                                             D.eps);
    }
  } else {
    prologue_kernel<T><<<warp_blocks(M), 256, 0, st>>>(h_prev, C.tokens, static_cast<const T*>(C.W.embed),
                                                       static_cast<const T*>(C.W.hnorm[i]),
                                                       static_cast<const T*>(C.W.enorm[i]), c, M, D.T, d, D.V, k,
                                                       D.eps);
  }
  mtp::note_launch();
}

template <typename T>
mtp_status run_chain(const Ctx& C, const T* h0, T* h_out, bool with_loss, float lambda, int den, int with_main,
                     double* sums_counts, float* losses, float* row_loss) {
  const mtp_dims& D = C.D;
  const int M = C.M, d = D.d;
  const size_t Md = static_cast<size_t>(M) * d;
  // loss calls with a second stream: depth k's prologue runs there beside the head GEMM of term
  // k - 1 (it needs only h^(k-1) and the tokens), and each term's CE reduction after its head
  const bool split = C.side != nullptr && with_loss;
  auto c_buf = [&](int k) -> T* {
    return C.save ? reinterpret_cast<T*>(C.save + static_cast<size_t>(k - 1) * C.so.bytes + C.so.c)
                  : C.buf<T>(C.L.c);
  };
  const int half = D.head_dim / 2;
  SetupArgs sa;
  sa.sums = with_loss ? sums_counts : nullptr;
  sa.n_sums = with_loss ? 2 * (D.D + 1) : 0;
  sa.rope = C.buf<float2>(C.L.rope);
  sa.half = half;
  sa.hd = D.head_dim;
  sa.base = D.rope_base > 0.f ? static_cast<double>(D.rope_base) : 0.0;
  const int rope_blocks = (D.T * half + kScanThreads - 1) / kScanThreads;
  segments_kernel<<<D.B + rope_blocks, kScanThreads, 0, C.st>>>(C.seg, C.tokens, D.T, D.V,
                                                                C.buf<int32_t>(C.L.seg_start),
                                                                C.buf<int32_t>(C.L.seg_end),
                                                                C.buf<int>(C.L.work_ctrs), D.D, D.B, sa);
  mtp::note_launch();
  MTP_LAUNCH_CHECK();
  if (with_loss) {
    if (with_main) TRY(head_ce<T>(C, h0, 0, row_loss, sums_counts, split ? c_buf(1) : nullptr));
    else if (row_loss)
      cudaMemsetAsync(row_loss, 0xff, static_cast<size_t>(M) * sizeof(float), C.st);  // NaN
  }
  T* c = C.buf<T>(C.L.c);
  T* u = C.buf<T>(C.L.u);
  T* x = C.buf<T>(C.L.x);
  T* qkv = C.buf<T>(C.L.qkv);
  T* o = C.buf<T>(C.L.o);
  T* a = C.buf<T>(C.L.a);
  T* g = C.buf<T>(C.L.g);
  T* y = x;  // the FFN norm's output (its own saved buffer in a training step)
  const T* h_prev = h0;
  for (int k = 1; k <= D.D; ++k) {
    const int i = k - 1;
    if (C.save) {
      uint8_t* sv = C.save + static_cast<size_t>(i) * C.so.bytes;
      c = reinterpret_cast<T*>(sv + C.so.c);
      u = reinterpret_cast<T*>(sv + C.so.u);
      x = reinterpret_cast<T*>(sv + C.so.x);
      qkv = reinterpret_cast<T*>(sv + C.so.qkv);
      o = reinterpret_cast<T*>(sv + C.so.o);
      a = reinterpret_cast<T*>(sv + C.so.a);
      y = reinterpret_cast<T*>(sv + C.so.y);
    }
    T* h_k = h_out ? h_out + static_cast<size_t>(i) * Md : C.buf<T>((k & 1) ? C.L.h1buf : C.L.h0buf);
    auto wt = [&](const void* const* arr) { return static_cast<const T*>(arr[i]); };
    if (split && (k > 1 || with_main)) {
      cudaStreamWaitEvent(C.st, C.ev[kEvPro], 0);  // this depth's c, from the second stream
    } else {
      // from the second depth on the previous operation is a kernel (the head's CE reduction
      // or the down projection): launch as its programmatic dependent
      mtp::prof_begin(MTP_KC_PROLOGUE, C.st);
      // (the first depth's follows a kernel unless the main term's row losses were just filled)
      launch_prologue<T>(C, h_prev, k, c, C.st, k > 1 || !(with_loss && !with_main && row_loss));
      mtp::prof_end(MTP_KC_PROLOGUE, C.st);
    }
    MTP_LAUNCH_CHECK();
    const T* proj[1] = {wt(C.W.eh_proj)};
    mtp::prof_begin(MTP_KC_PROJ_GEMM, C.st);
    TRY(gemm<T>(C, c, 2 * d, proj, 1, d, 2 * d, d, u, d, mtp::EPI_STORE, nullptr, 0, nullptr,
                !(split && (k > 1 || with_main))));
    mtp::prof_end(MTP_KC_PROJ_GEMM, C.st);
    launch_rmsnorm<T>(C, u, wt(C.W.attn_norm), x, nullptr, 0, true);
    const T* wqkv[3] = {wt(C.W.wq), wt(C.W.wk), wt(C.W.wv)};
    mtp::prof_begin(MTP_KC_QKV_GEMM, C.st);
    TRY(gemm<T>(C, x, d, wqkv, 3, d, d, 3 * d, qkv, 3 * d, D.rope_base > 0.f ? mtp::EPI_ROPE : mtp::EPI_STORE));
    mtp::prof_end(MTP_KC_QKV_GEMM, C.st);
    mtp::prof_begin(MTP_KC_ATTENTION, C.st);
    float* lse2 = C.save ? reinterpret_cast<float*>(C.save + static_cast<size_t>(i) * C.so.bytes + C.so.lse2) : nullptr;
    TRY(mtp::attn_launch(D.dtype, qkv, o, C.buf<int32_t>(C.L.seg_start), D.B, D.T, D.n_heads, D.head_dim, C.st,
                         lse2, C.buf<int>(C.L.work_ctrs) + i));
    mtp::prof_end(MTP_KC_ATTENTION, C.st);
    const T* wo[1] = {wt(C.W.wo)};
    mtp::prof_begin(MTP_KC_O_GEMM, C.st);
    TRY(gemm<T>(C, o, d, wo, 1, d, d, d, a, d, mtp::EPI_RESID, u, d));
    mtp::prof_end(MTP_KC_O_GEMM, C.st);
    launch_rmsnorm<T>(C, a, wt(C.W.ffn_norm), y, nullptr, 0, true);
    const T* wg[1] = {wt(C.W.w_gate)};
    mtp::prof_begin(MTP_KC_GATE_UP_GEMM, C.st);
    TRY(gemm<T>(C, y, d, wg, 1, D.ffn, d, D.ffn, g, D.ffn, mtp::EPI_SWIGLU, nullptr, 0, wt(C.W.w_up)));
    mtp::prof_end(MTP_KC_GATE_UP_GEMM, C.st);
    const T* wd[1] = {wt(C.W.w_down)};
    mtp::prof_begin(MTP_KC_DOWN_GEMM, C.st);
    TRY(gemm<T>(C, g, D.ffn, wd, 1, d, D.ffn, d, h_k, d, mtp::EPI_RESID, a, d));
    mtp::prof_end(MTP_KC_DOWN_GEMM, C.st);
    if (with_loss)
      TRY(head_ce<T>(C, h_k, k, row_loss ? row_loss + static_cast<size_t>(k) * M : nullptr, sums_counts + 2 * k,
                     split && k < D.D ? c_buf(k + 1) : nullptr));
    h_prev = h_k;
  }
  if (with_loss) {
    DepthWeights W{};
    W.lambda = lambda;
    W.uniform = 1;
    if (split && C.red_pending) {  // every reduction on the second stream has finished
      cudaStreamWaitEvent(C.st, C.ev[kEvRed], 0);
      loss_assemble_kernel<<<1, 32, 0, C.st>>>(sums_counts, losses, D.D, static_cast<double>(M), W, den, with_main);
    } else {  // a programmatic dependent of the last head's CE reduction
      mtp::launch_pdl(loss_assemble_kernel, dim3(1), dim3(32), 0, C.st, sums_counts, losses, D.D,
                      static_cast<double>(M), W, den, with_main);
    }
    mtp::note_launch();
    MTP_LAUNCH_CHECK();
  }
  return MTP_OK;
}

mtp_status check_common(const mtp_dims* dims, const mtp_weights* w, const int32_t* tokens, const int32_t* seg,
                        const int32_t* pos, const void* h0, void* ws, size_t ws_bytes) {
  if (!dims || !w || !tokens || !seg || !pos || !h0) return MTP_ERR_INVALID_ARG;
  if (!valid_dims(*dims)) return MTP_ERR_SHAPE;
  TRY(supported(*dims));
  if (!w->embed || !w->head || !w->out_norm) return MTP_ERR_INVALID_ARG;
  const void* const* lists[] = {w->hnorm, w->enorm, w->eh_proj, w->attn_norm, w->wq, w->wk, w->wv,
                                w->wo, w->ffn_norm, w->w_gate, w->w_up, w->w_down};
  for (auto l : lists) {
    if (!l) return MTP_ERR_INVALID_ARG;
    for (int k = 0; k < dims->D; ++k) {
      if (!l[k]) return MTP_ERR_INVALID_ARG;
      if (!mtp::aligned16(l[k])) return MTP_ERR_ALIGNMENT;
    }
  }
  for (const void* p : {static_cast<const void*>(tokens), static_cast<const void*>(seg),
                        static_cast<const void*>(pos), h0, w->embed, w->head, w->out_norm})
    if (!mtp::aligned16(p)) return MTP_ERR_ALIGNMENT;
  if (!ws || !mtp::aligned16(ws)) return ws ? MTP_ERR_ALIGNMENT : MTP_ERR_WORKSPACE;
  if (ws_bytes < make_layout(*dims).total) return MTP_ERR_WORKSPACE;
  return MTP_OK;
}

}  // namespace

extern "C" size_t mtp_chain_workspace_bytes(const mtp_dims* dims) {
  if (!dims || !valid_dims(*dims) || supported(*dims) != MTP_OK) return 0;
  return make_layout(*dims).total;
}

extern "C" mtp_status mtp_chain_forward(const mtp_dims* dims, const mtp_weights* w, const int32_t* tokens,
                                        const int32_t* seg, const int32_t* pos, const void* h0, void* h_out, void* ws,
                                        size_t ws_bytes, cudaStream_t stream) {
  TRY(check_common(dims, w, tokens, seg, pos, h0, ws, ws_bytes));
  if (!h_out) return MTP_ERR_INVALID_ARG;
  if (!mtp::aligned16(h_out)) return MTP_ERR_ALIGNMENT;
  Ctx C{*dims, *w, tokens, seg, pos, static_cast<uint8_t*>(ws), make_layout(*dims), stream, dims->B * dims->T};
  if (dims->dtype == MTP_BF16)
    return run_chain<__nv_bfloat16>(C, static_cast<const __nv_bfloat16*>(h0), static_cast<__nv_bfloat16*>(h_out),
                                    false, 0.f, 0, 0, nullptr, nullptr, nullptr);
  return run_chain<float>(C, static_cast<const float*>(h0), static_cast<float*>(h_out), false, 0.f, 0, 0, nullptr,
                          nullptr, nullptr);
}

extern "C" mtp_status mtp_chain_loss(const mtp_dims* dims, const mtp_weights* w, const int32_t* tokens,
                                     const int32_t* seg, const int32_t* pos, const void* h0, float lambda, int den,
                                     int with_main, double* sums_counts, float* losses, float* row_loss, void* h_out,
                                     void* ws, size_t ws_bytes, cudaStream_t stream) {
  TRY(check_common(dims, w, tokens, seg, pos, h0, ws, ws_bytes));
  if (!sums_counts || !losses) return MTP_ERR_INVALID_ARG;
  if (!valid_den(den)) return MTP_ERR_INVALID_ARG;
  if (h_out && !mtp::aligned16(h_out)) return MTP_ERR_ALIGNMENT;
  Ctx C{*dims, *w, tokens, seg, pos, static_cast<uint8_t*>(ws), make_layout(*dims), stream, dims->B * dims->T};
  std::unique_lock<std::mutex> side_lock;
  if (SideStream* S = side_stream(side_lock)) {
    C.side = S->s;
    C.ev = S->ev;
  }
  if (dims->dtype == MTP_BF16)
    return run_chain<__nv_bfloat16>(C, static_cast<const __nv_bfloat16*>(h0), static_cast<__nv_bfloat16*>(h_out),
                                    true, lambda, den, with_main, sums_counts, losses, row_loss);
  return run_chain<float>(C, static_cast<const float*>(h0), static_cast<float*>(h_out), true, lambda, den, with_main,
                          sums_counts, losses, row_loss);
}

extern "C" mtp_status mtp_loss_assemble_weighted(int D, const double* sums_counts, double n_positions,
                                                 const float* depth_weights, float lambda, int den, int with_main,
                                                 float* losses, cudaStream_t stream) {
  if (D <= 0 || !sums_counts || !losses || !(n_positions > 0)) return MTP_ERR_INVALID_ARG;
  if (!valid_den(den)) return MTP_ERR_INVALID_ARG;
  if (depth_weights && D > kMaxDepthWeights) return MTP_ERR_UNSUPPORTED;
  DepthWeights W{};
  W.lambda = lambda;
  W.uniform = depth_weights ? 0 : 1;
  if (depth_weights)
    for (int k = 0; k < D; ++k) W.w[k] = depth_weights[k];
  loss_assemble_kernel<<<1, 32, 0, stream>>>(sums_counts, losses, D, n_positions, W, den, with_main);
  mtp::note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

extern "C" mtp_status mtp_loss_assemble(int D, const double* sums_counts, double n_positions, float lambda, int den,
                                        int with_main, float* losses, cudaStream_t stream) {
  return mtp_loss_assemble_weighted(D, sums_counts, n_positions, nullptr, lambda, den, with_main, losses, stream);
}

// ---------------------------------------------------------------------------
// Training step: the forward with its states saved, then gradients.
// "M7.6 - DeepSeek MTP" §0x05: the shared head (and embedding) receive the
// main term's and every depth's gradient; depth k's states receive the
// gradients of terms k..D through the recurrence.
// ---------------------------------------------------------------------------
namespace {

// dL/dl of one supervised row of each term (the loss assembly's definitions)
__global__ void term_scale_kernel(const double* __restrict__ sc, float* __restrict__ scale, int D, double n_pos,
                                  DepthWeights W, int den, int with_main) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  auto weight = [&](int k) -> double {
    return W.uniform ? static_cast<double>(W.lambda) / D : static_cast<double>(W.w[k - 1]);
  };
  double n_all = 0.0, wn_all = 0.0;
  for (int k = 1; k <= D; ++k) {
    n_all += sc[2 * k + 1];
    wn_all += weight(k) * sc[2 * k + 1];
  }
  auto inv = [](double b) { return b > 0.0 ? 1.0 / b : 0.0; };
  auto term_inv = [&](int t) -> double {
    if (den == MTP_DEN_FIXED) return 1.0 / n_pos;
    if (den == MTP_DEN_SUM) return 1.0;
    if (den == MTP_DEN_MASKED_MEAN || t == 0) return inv(sc[2 * t + 1]);
    if (den == MTP_DEN_GLOBAL) return inv(n_all);
    return inv(wn_all);
  };
  scale[0] = with_main ? static_cast<float>(term_inv(0)) : 0.f;
  for (int k = 1; k <= D; ++k) scale[k] = static_cast<float>(weight(k) * term_inv(k));
}


// RMSNorm backward for y = g * h * r, r = (mean(h^2) + eps)^(-1/2), given
// dy: dh += r (g dy - xh * mean(g dy xh)) with xh = h r; dg += sum over rows
// of dy xh.  Row m reads h row h_rows[m] (or m) and adds its dh into row
// dh_rows[m] with atomics (or row m plainly); dh may be null.  A block takes
// kNormBwdRows rows (16: twice the blocks of 32, 0.18 ms less per training step):
// its warps first form each row's r and mean(g dy xh), then each
// thread sweeps 4 adjacent columns down the rows (16-byte loads and stores),
// summing the gain gradient in registers; the block writes that column sum to
// its row of dg_part and a second kernel adds the blocks' rows into dg, so no
// two blocks contend for the same dg entry.  Requires d % 4 == 0.
constexpr int kNormBwdRows = 16;
__global__ void __launch_bounds__(256)
rmsnorm_bwd_kernel(const __nv_bfloat16* __restrict__ h, int ld_h, const int32_t* __restrict__ h_rows,
                   const __nv_bfloat16* __restrict__ g, const float* __restrict__ dy, int ld_dy, float* __restrict__ dh,
                   int ld_dh, const int32_t* __restrict__ dh_rows, const float* __restrict__ dh_base,
                   bool dh_store, __nv_bfloat16* __restrict__ dh_bf16, float* __restrict__ dg_part, int M, int d,
                   float eps) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  __shared__ float s_r[kNormBwdRows], s_mean[kNormBwdRows];
  __shared__ int s_hrow[kNormBwdRows], s_dhrow[kNormBwdRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kNormBwdRows;
  const int rows = min(kNormBwdRows, M - m0);
  // row statistics: r = (mean(h^2) + eps)^(-1/2) and mean(g dy xh) (4 rows per warp)
  for (int j = warp; j < rows; j += 8) {
    const int m = m0 + j;
    const int hrow = h_rows ? h_rows[m] : m;
    const __nv_bfloat16* hr = h + static_cast<size_t>(hrow) * ld_h;
    const float* dyr = dy + static_cast<size_t>(m) * ld_dy;
    float ss = 0.f, dot = 0.f;
    for (int i = 4 * lane; i < d; i += 128) {
      const uint2 hv = *reinterpret_cast<const uint2*>(hr + i);
      const uint2 gv = *reinterpret_cast<const uint2*>(g + i);
      const float4 dv = *reinterpret_cast<const float4*>(dyr + i);
      const float2 h01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hv.x));
      const float2 h23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hv.y));
      const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv.x));
      const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv.y));
      ss += h01.x * h01.x + h01.y * h01.y + h23.x * h23.x + h23.y * h23.y;
      dot += g01.x * dv.x * h01.x + g01.y * dv.y * h01.y + g23.x * dv.z * h23.x + g23.y * dv.w * h23.y;
    }
    ss = mtp::warp_sum(ss);
    dot = mtp::warp_sum(dot);
    if (lane == 0) {
      const float r = 1.0f / sqrtf(ss / d + eps);
      s_r[j] = r;
      s_mean[j] = dot * r / d;
      s_hrow[j] = hrow;
      s_dhrow[j] = dh_rows ? dh_rows[m] : m;
    }
  }
  __syncthreads();
  for (int i = 4 * threadIdx.x; i < d; i += 4 * blockDim.x) {
    const uint2 gv = *reinterpret_cast<const uint2*>(g + i);
    const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv.x));
    const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv.y));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int j = 0; j < rows; ++j) {
      const float r = s_r[j], mean = s_mean[j];
      const uint2 hv = *reinterpret_cast<const uint2*>(h + static_cast<size_t>(s_hrow[j]) * ld_h + i);
      const float2 h01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hv.x));
      const float2 h23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hv.y));
      const float4 dv = *reinterpret_cast<const float4*>(dy + static_cast<size_t>(m0 + j) * ld_dy + i);
      const float4 xh = make_float4(h01.x * r, h01.y * r, h23.x * r, h23.y * r);
      acc.x += dv.x * xh.x;
      acc.y += dv.y * xh.y;
      acc.z += dv.z * xh.z;
      acc.w += dv.w * xh.w;
      if (dh || dh_bf16) {
        const float4 v = make_float4(r * (g01.x * dv.x - xh.x * mean), r * (g01.y * dv.y - xh.y * mean),
                                     r * (g23.x * dv.z - xh.z * mean), r * (g23.y * dv.w - xh.w * mean));
        float4* dst = dh ? reinterpret_cast<float4*>(dh + static_cast<size_t>(s_dhrow[j]) * ld_dh + i) : nullptr;
        if (dh_rows) {
          atomicAdd(dst, v);
        } else {
          // dh = [dh +] [dh_base +] v: without dh_store (or without dh) the sum starts from
          // dh's own value, with dh_store it is dh's first writer; dh_bf16 gets the result's
          // bf16 copy ([M, d], the next GEMM's operand)
          float4 o = (dh_store || !dh) ? make_float4(0.f, 0.f, 0.f, 0.f) : *dst;
          if (dh_base) {
            const float4 b = *reinterpret_cast<const float4*>(dh_base + static_cast<size_t>(s_dhrow[j]) * ld_dh + i);
            o.x += b.x;
            o.y += b.y;
            o.z += b.z;
            o.w += b.w;
          }
          o.x += v.x;
          o.y += v.y;
          o.z += v.z;
          o.w += v.w;
          if (dh) *dst = o;
          if (dh_bf16)
            *reinterpret_cast<uint2*>(dh_bf16 + static_cast<size_t>(s_dhrow[j]) * d + i) =
                make_uint2(mtp::pack2_bf16(o.x, o.y), mtp::pack2_bf16(o.z, o.w));
        }
      }
    }
    if (dg_part) *reinterpret_cast<float4*>(dg_part + static_cast<size_t>(blockIdx.x) * d + i) = acc;
  }
}

// dg[i] += Σ_b part[b][i] over the row blocks of rmsnorm_bwd_kernel: a block
// takes 32 columns, its 8 warps stride over the rows (coalesced 128-byte row
// pieces) and combine their sums in shared memory
__global__ void __launch_bounds__(256) colsum_add_kernel(const float* __restrict__ part, int nb, int d,
                                                         float* __restrict__ dg) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  __shared__ float s_sum[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 32 + lane;
  float acc = 0.f;
  if (i < d)
    for (int b = warp; b < nb; b += 8) acc += part[static_cast<size_t>(b) * d + i];
  s_sum[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && i < d) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += s_sum[w][lane];
    dg[i] += t;
  }
}

void rmsnorm_bwd(const __nv_bfloat16* h, int ld_h, const int32_t* h_rows, const __nv_bfloat16* g, const float* dy,
                 int ld_dy, float* dh, int ld_dh, const int32_t* dh_rows, float* dg, float* dg_part, int M, int d,
                 float eps, cudaStream_t st, const float* dh_base = nullptr, bool dh_store = false,
                 __nv_bfloat16* dh_bf16 = nullptr) {
  const int nb = (M + kNormBwdRows - 1) / kNormBwdRows;
  rmsnorm_bwd_kernel<<<nb, 256, 0, st>>>(h, ld_h, h_rows, g, dy, ld_dy, dh, ld_dh, dh_rows, dh_base, dh_store, dh_bf16,
                                         dg ? dg_part : nullptr, M, d, eps);
  mtp::note_launch();
  if (dg) {
    colsum_add_kernel<<<(d + 31) / 32, 256, 0, st>>>(dg_part, nb, d, dg);
    mtp::note_launch();
  }
}


inline int round_up8(int v) { return (v + 7) / 8 * 8; }

struct TrainLayout {
  size_t hs, lse, scale, dz, dx, dgp, dstate, save, total;
  int vc, vp, mp;
};

SaveOff make_save_off(const mtp_dims& D);

// after the forward's own workspace: the saved states h^1..h^D, the per-term
// log-sum-exp, the per-term row scales and the head-backward buffers
TrainLayout make_train_layout(const mtp_dims& D) {
  TrainLayout T{};
  const size_t M = static_cast<size_t>(D.B) * D.T, d = D.d;
  T.vp = round_up8(D.V);
  T.mp = round_up8(static_cast<int>(M));
  T.vc = std::min(32768, T.vp);  // vocabulary chunk of the head backward
  size_t off = make_layout(D).total;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  T.hs = take(static_cast<size_t>(D.D) * M * d * 2);
  T.lse = take(static_cast<size_t>(D.D + 1) * M * 4);
  T.scale = take(static_cast<size_t>(D.D + 1) * 4);
  T.dz = take(M * T.vc * 2);
  T.dx = take(M * d * 4);
  T.dgp = take(static_cast<size_t>((M + kNormBwdRows - 1) / kNormBwdRows) * d * 4);  // RMSNorm gain partials
  T.dstate = take(static_cast<size_t>(D.D + 1) * M * d * 4);
  T.save = take(static_cast<size_t>(D.D) * make_save_off(D).bytes);
  T.total = off;
  return T;
}

// out (+)= A B^T in fp32 (declared here, defined with the block backward).  The
// GEMM is launched for programmatic dependent launch, so the stream's previous
// operation must be a kernel (not a memset or a copy).
mtp_status gemm_acc(int M, int N, int K, const __nv_bfloat16* A, int lda, bool a_mn, const __nv_bfloat16* B, int ldb,
                    bool b_mn, float* out, int ldo, cudaStream_t st, bool overwrite = false);

mtp::GemmDesc gdesc(int M, int N, int K, const __nv_bfloat16* A, int lda, const __nv_bfloat16* B, int ldb) {
  mtp::GemmDesc g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.A = A;
  g.lda = lda;
  g.B[0] = B;
  g.ldb = ldb;
  g.nseg = 1;
  g.seg_rows = N;
  return g;
}

// gradients through the shared head and the final norm of term t (state h_t):
// per vocabulary chunk the logits are recomputed by one GEMM whose epilogue
// writes dz = (softmax - onehot) dL/dl (the logits are never stored whole);
// then dX += dz W_U[chunk] and, reading dz MN-major as dz^T, d_head[chunk] +=
// dz^T X; finally the final RMSNorm's backward writes d h_t into dstate[t] (its
// first writer: the heads run before the blocks, whose backward then adds the
// next depth's contribution), and its bf16 copy into dstate_bf16 when given, and
// accumulates d_out_norm.
mtp_status head_backward(const Ctx& C, const TrainLayout& T, int t, const __nv_bfloat16* h_t, float* d_head,
                         float* d_out_norm, __nv_bfloat16* dstate_bf16) {
  using bf = __nv_bfloat16;
  const mtp_dims& D = C.D;
  const int M = C.M, d = D.d, V = D.V;
  bf* x = C.buf<bf>(C.L.x);
  int32_t* labels = C.buf<int32_t>(C.L.labels);
  const bf* WU = static_cast<const bf*>(C.W.head);
  const bf* out_norm = static_cast<const bf*>(C.W.out_norm);
  bf* dz = C.buf<bf>(T.dz);
  float* dx = C.buf<float>(T.dx);
  const float* lse = C.buf<float>(T.lse) + static_cast<size_t>(t) * M;
  const float* scale = C.buf<float>(T.scale) + t;
  launch_rmsnorm<bf>(C, h_t, out_norm, x, labels, t);
  for (int v0 = 0; v0 < V; v0 += T.vc) {
    const int vc = std::min(T.vc, V - v0);
    mtp::GemmDesc g = gdesc(M, vc, d, x, d, WU + static_cast<size_t>(v0) * d, d);
    g.epi = mtp::EPI_CE_GRAD;
    g.out = dz;
    g.ldo = T.vc;
    g.labels = labels;
    g.lse = lse;
    g.ce_scale = scale;
    g.ce_offset = v0;
    g.pdl = true;  // follows the RMSNorm kernel or the previous chunk's GEMM
    g.b_early = true;  // B = W_U
    TRY(mtp::gemm_bf16_launch(g, C.st));
    // dX += dz W_U[v0 : v0 + vc] (W_U rows read as the MN-major B operand)
    TRY(gemm_acc(M, d, vc, dz, T.vc, false, WU + static_cast<size_t>(v0) * d, d, true, dx, d, C.st, v0 == 0));
    if (!d_head) continue;
    // dW_U[v0 : v0 + vc] += dz^T X (both operands read MN-major)
    TRY(gemm_acc(vc, d, M, dz, T.vc, true, x, d, true, d_head + static_cast<size_t>(v0) * d, d, C.st));
  }
  float* dstate_t = C.buf<float>(T.dstate) + static_cast<size_t>(t) * M * d;
  rmsnorm_bwd(h_t, d, nullptr, out_norm, dx, d, dstate_t, d, nullptr, d_out_norm, C.buf<float>(T.dgp), M, d, D.eps,
              C.st, nullptr, true, dstate_bf16);
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

// ---- block backward -------------------------------------------------------

// SwiGLU backward from the recomputed pre-activations pq = [p | q] ([M, 2 ffn]
// bf16) and dg ([M, ffn] fp32): g = silu(p) q, dp = dg q silu'(p), dq = dg silu(p).
// VEC: 8 columns per thread step with 16-byte accesses (ffn a multiple of 8,
// 16-byte aligned bases).
__device__ __forceinline__ void swiglu_bwd1(float p, float q, float dgv, float& g, float& dp, float& dq) {
  const float sg = 1.0f / (1.0f + __expf(-p));
  const float silu = p * sg;
  g = silu * q;
  dp = dgv * q * (sg * (1.0f + p * (1.0f - sg)));
  dq = dgv * silu;
}
template <bool VEC>
__global__ void swiglu_bwd_kernel(const __nv_bfloat16* __restrict__ pq, const float* __restrict__ dg,
                                  __nv_bfloat16* __restrict__ g, __nv_bfloat16* __restrict__ dpq, int M, int ffn) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  for (int m = blockIdx.x; m < M; m += gridDim.x) {
    const __nv_bfloat16* pr = pq + static_cast<size_t>(m) * 2 * ffn;
    const float* dgr = dg + static_cast<size_t>(m) * ffn;
    __nv_bfloat16* gr = g + static_cast<size_t>(m) * ffn;
    __nv_bfloat16* dr = dpq + static_cast<size_t>(m) * 2 * ffn;
    if constexpr (VEC) {
      for (int j = 8 * threadIdx.x; j < ffn; j += 8 * blockDim.x) {
        const uint4 pv = *reinterpret_cast<const uint4*>(pr + j);
        const uint4 qv = *reinterpret_cast<const uint4*>(pr + ffn + j);
        const float4 d0 = *reinterpret_cast<const float4*>(dgr + j);
        const float4 d1 = *reinterpret_cast<const float4*>(dgr + j + 4);
        const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w}, qw[4] = {qv.x, qv.y, qv.z, qv.w};
        const float dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
        uint32_t go[4], dpo[4], dqo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 p2 = mtp::unpack2_bf16(pw[i]), q2 = mtp::unpack2_bf16(qw[i]);
          float g0, g1, dp0, dp1, dq0, dq1;
          swiglu_bwd1(p2.x, q2.x, dv[2 * i], g0, dp0, dq0);
          swiglu_bwd1(p2.y, q2.y, dv[2 * i + 1], g1, dp1, dq1);
          go[i] = mtp::pack2_bf16(g0, g1);
          dpo[i] = mtp::pack2_bf16(dp0, dp1);
          dqo[i] = mtp::pack2_bf16(dq0, dq1);
        }
        *reinterpret_cast<uint4*>(gr + j) = make_uint4(go[0], go[1], go[2], go[3]);
        *reinterpret_cast<uint4*>(dr + j) = make_uint4(dpo[0], dpo[1], dpo[2], dpo[3]);
        *reinterpret_cast<uint4*>(dr + ffn + j) = make_uint4(dqo[0], dqo[1], dqo[2], dqo[3]);
      }
    } else {
      for (int j = threadIdx.x; j < ffn; j += blockDim.x) {
        float gv, dp, dq;
        swiglu_bwd1(__bfloat162float(pr[j]), __bfloat162float(pr[ffn + j]), dgr[j], gv, dp, dq);
        gr[j] = __float2bfloat16_rn(gv);
        dr[j] = __float2bfloat16_rn(dp);
        dr[ffn + j] = __float2bfloat16_rn(dq);
      }
    }
  }
}

// RoPE backward: the forward rotated (x1, x2) -> (x1 c - x2 s, x2 c + x1 s) at
// the row's position; the gradient rotates back: (d1 c + d2 s, d2 c - d1 s).
// dqkv [M, 3d] fp32 -> out [M, 3d] bf16 (v copied)
__global__ void rope_bwd_kernel(const float* __restrict__ dqkv, const float2* __restrict__ rope,
                                const int32_t* __restrict__ pos, __nv_bfloat16* __restrict__ out, int M, int d, int hd,
                                int Tlen, int use_rope) {
  mtp::pdl_trigger();  // a GEMM that follows may start its setup
  const int half = hd / 2;
  for (int m = blockIdx.x; m < M; m += gridDim.x) {
    const float* src = dqkv + static_cast<size_t>(m) * 3 * d;
    __nv_bfloat16* dst = out + static_cast<size_t>(m) * 3 * d;
    const float2* cs_row = rope + static_cast<size_t>(min(max(pos[m], 0), Tlen - 1)) * half;
    for (int pi = threadIdx.x; pi < d; pi += blockDim.x) {  // d pairs of the q and k heads, then v column pi
      const int head = pi / half, j = pi - head * half;
      const int col = head * hd + j;
      const float d1 = src[col], d2 = src[col + half];
      float c = 1.f, sn = 0.f;
      if (use_rope) {
        const float2 cs = cs_row[j];
        c = cs.x;
        sn = cs.y;
      }
      dst[col] = __float2bfloat16_rn(d1 * c + d2 * sn);
      dst[col + half] = __float2bfloat16_rn(d2 * c - d1 * sn);
      dst[2 * d + pi] = __float2bfloat16_rn(src[2 * d + pi]);
    }
  }
}

// token gathered by row m at depth k (the forward prologue's clamped rule)
__global__ void shifted_tokens_kernel(const int32_t* __restrict__ tokens, int32_t* __restrict__ out, int M, int Tlen,
                                      int k, int V) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  const int t = m % Tlen;
  out[m] = clamp_token(tokens[m - t + min(t + k, Tlen - 1)], V);
}

// scratch of the block backward (reused depth after depth)
struct BwdLayout {
  size_t dhb, pq, gb, dgf, dpq, dyf, daf, dab, dob, dqkvf, dqkvb, dxf, duf, dub, dcf, adsum, tok, total;
};

BwdLayout make_bwd_layout(const mtp_dims& D, size_t start, int mp) {
  BwdLayout B{};
  const size_t M = static_cast<size_t>(D.B) * D.T, d = D.d, f = D.ffn;
  size_t off = start;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  B.dhb = take(M * d * 2);
  B.pq = take(M * 2 * f * 2);
  B.gb = take(M * f * 2);
  B.dgf = take(M * f * 4);
  B.dpq = take(M * 2 * f * 2);
  B.dyf = take(M * d * 4);
  B.daf = take(M * d * 4);
  B.dab = take(M * d * 2);
  B.dob = take(M * d * 2);
  B.dqkvf = take(M * 3 * d * 4);
  B.dqkvb = take(M * 3 * d * 2);
  B.dxf = take(M * d * 4);
  B.duf = take(M * d * 4);
  B.dub = take(M * d * 2);
  B.dcf = take(M * 2 * d * 4);
  B.adsum = take(M * D.n_heads * 4);
  B.tok = take(M * 4);
  B.total = off;
  return B;
}

SaveOff make_save_off(const mtp_dims& D) {
  SaveOff S{};
  const size_t M = static_cast<size_t>(D.B) * D.T, d = D.d;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  S.c = take(M * 2 * d * 2);
  S.u = take(M * d * 2);
  S.x = take(M * d * 2);
  S.qkv = take(M * 3 * d * 2);
  S.o = take(M * d * 2);
  S.a = take(M * d * 2);
  S.y = take(M * d * 2);
  S.lse2 = take(M * D.n_heads * 4);
  S.bytes = off;
  return S;
}

// C += A B^T (C = A B^T with `overwrite`) into fp32; A is [M, K] (a_mn: stored [K, M]) and B is [N, K]
// (b_mn: stored [K, N]), so transposes of row-major operands are read in
// place.  K is split (partial tiles added with vector atomics) when the cost
// model below says the better-filled waves pay for the atomics (at most 16
// splits, at least 8 k-blocks per split).
mtp_status gemm_acc(int M, int N, int K, const __nv_bfloat16* A, int lda, bool a_mn, const __nv_bfloat16* B, int ldb,
                    bool b_mn, float* out, int ldo, cudaStream_t st, bool overwrite) {
  const int sms = mtp::sm_count_current();
  mtp::GemmDesc g = gdesc(M, N, K, A, lda, B, ldb);
  g.epi = mtp::EPI_F32_ACC;
  g.a_mn = a_mn;
  g.b_mn = b_mn;
  g.out_f32 = out;
  g.ldo = ldo;
  // K splits by a cost model: waves of (tile, split) units times the k-blocks of a unit
  // (~655 cycles each on a 256 x 256 CTA-pair tile), plus the split-K atomics (the fp32
  // output added once per split at ~680 B per cycle of L2 atomic throughput) and, for an
  // overwrite, the zeroing memset.  Measured on GB300: the head's dX (8192 x 1024, K = 32000)
  // took 345 us unsplit and 400 us in 4 splits although 4 splits balance the waves better.
  const bool pair = M > 128;
  const int units1 = (pair ? (M + 255) / 256 : (M + 127) / 128) * ((N + 255) / 256);
  const int slots = pair ? sms / 2 : sms;
  const int nk = (K + 63) / 64;
  const int max_split = std::max(1, std::min(16, nk / 8));
  const double out_bytes = 4.0 * M * N;
  int splits = 1;
  double best = 1e300;
  for (int sp = 1; sp <= max_split; ++sp) {
    const long long units = static_cast<long long>(units1) * sp;
    const double waves = static_cast<double>((units + slots - 1) / slots);
    double cyc = waves * ((nk + sp - 1) / sp) * 655.0;
    if (sp > 1) cyc += sp * out_bytes / 680.0 + (overwrite ? out_bytes / 3400.0 : 0.0);
    if (cyc < best * 0.98) {  // a split must win by 2%
      best = cyc;
      splits = sp;
    }
  }
  g.splits = splits;
  g.pdl = true;
  g.b_early = true;  // an L2 prefetch is coherent with later writes, so any B may be fetched early
  if (overwrite) {  // out = A B^T: one split stores directly, several add into a zeroed output
    if (splits == 1) {
      g.f32_overwrite = true;
    } else {
      MTP_CUDA_TRY(cudaMemset2DAsync(out, static_cast<size_t>(ldo) * 4, 0, static_cast<size_t>(N) * 4, M, st));
      g.pdl = false;  // a memset precedes the GEMM
    }
  }
  return mtp::gemm_bf16_launch(g, st);
}

// gradients of depth k's module given dstate[k] = dL/dh_k (complete): weight
// gradients into `grads` (those given), dL/dh_{k-1} added into dstate[k-1],
// the embedding rows' gradient scattered into grads->embed.
mtp_status block_backward(const Ctx& C, const TrainLayout& T, const BwdLayout& B, int k, const __nv_bfloat16* h_prev,
                          const mtp_grads* G, bool with_main) {
  using bf = __nv_bfloat16;
  const mtp_dims& D = C.D;
  const int M = C.M, d = D.d, f = D.ffn, H = D.n_heads, hd = D.head_dim, i = k - 1;
  const size_t Md = static_cast<size_t>(M) * d;
  cudaStream_t st = C.st;
  auto wt = [&](const void* const* arr) { return static_cast<const bf*>(arr[i]); };
  auto gp = [&](float* const* arr) -> float* { return arr ? arr[i] : nullptr; };
  auto bb = [&](size_t off) { return C.buf<bf>(off); };
  auto fb = [&](size_t off) { return C.buf<float>(off); };
  uint8_t* sv = C.save + static_cast<size_t>(i) * C.so.bytes;
  const bf *c = reinterpret_cast<const bf*>(sv + C.so.c), *u = reinterpret_cast<const bf*>(sv + C.so.u),
           *x = reinterpret_cast<const bf*>(sv + C.so.x), *qkv = reinterpret_cast<const bf*>(sv + C.so.qkv),
           *o = reinterpret_cast<const bf*>(sv + C.so.o), *a = reinterpret_cast<const bf*>(sv + C.so.a),
           *y = reinterpret_cast<const bf*>(sv + C.so.y);
  const float* dh = fb(T.dstate) + static_cast<size_t>(k) * Md;
  float* dh_prev = fb(T.dstate) + static_cast<size_t>(k - 1) * Md;
  // Input gradients dX = dY W read the row-major weights W [out, in] as the
  // MN-major B operand; weight gradients dW = dY^T X read both activations
  // as MN-major operands.  Nothing is transposed in memory.

  // h = a + g W_d^T: dW_d += dh^T g; dg = dh W_d; da = dh (+ the FFN path below).  dh's bf16
  // copy (B.dhb) was written by the kernel that completed dh: the next depth's backward, or
  // the last term's head backward for the deepest depth
  {  // recompute the gate and up pre-activations p = y Wg^T, q = y Wu^T into pq = [p | q]
    mtp::GemmDesc g = gdesc(M, f, d, y, d, wt(C.W.w_gate), d);
    g.epi = mtp::EPI_STORE;
    g.out = bb(B.pq);
    g.ldo = 2 * f;
    g.pdl = true;  // follows a row kernel (RMSNorm or gain reduction)
    g.b_early = true;
    TRY(mtp::gemm_bf16_launch(g, st));
    g = gdesc(M, f, d, y, d, wt(C.W.w_up), d);
    g.epi = mtp::EPI_STORE;
    g.out = bb(B.pq) + f;
    g.ldo = 2 * f;
    g.pdl = true;
    g.b_early = true;
    TRY(mtp::gemm_bf16_launch(g, st));
  }
  TRY(gemm_acc(M, f, d, bb(B.dhb), d, false, wt(C.W.w_down), f, true, fb(B.dgf), f, st, true));
  if (f % 8 == 0)  // workspace buffers start 16-byte aligned (256-byte offsets from an aligned base)
    swiglu_bwd_kernel<true><<<std::min(M, 16 * 152), 128, 0, st>>>(bb(B.pq), fb(B.dgf), bb(B.gb), bb(B.dpq), M, f);
  else
    swiglu_bwd_kernel<false><<<std::min(M, 16 * 152), 256, 0, st>>>(bb(B.pq), fb(B.dgf), bb(B.gb), bb(B.dpq), M, f);
  mtp::note_launch();
  if (float* gwd = gp(G->w_down)) TRY(gemm_acc(d, f, M, bb(B.dhb), d, true, bb(B.gb), f, true, gwd, f, st));
  // g = silu(y Wg^T) (y Wu^T): dWg += dp^T y; dWu += dq^T y; dy = dp Wg + dq Wu
  if (float* gg = gp(G->w_gate)) TRY(gemm_acc(f, d, M, bb(B.dpq), 2 * f, true, y, d, true, gg, d, st));
  if (float* gu = gp(G->w_up)) TRY(gemm_acc(f, d, M, bb(B.dpq) + f, 2 * f, true, y, d, true, gu, d, st));
  TRY(gemm_acc(M, d, f, bb(B.dpq), 2 * f, false, wt(C.W.w_gate), d, true, fb(B.dyf), d, st, true));
  TRY(gemm_acc(M, d, f, bb(B.dpq) + f, 2 * f, false, wt(C.W.w_up), d, true, fb(B.dyf), d, st));
  // y = RMSNorm_f(a): da = dh + RMSNorm backward (fp32, and its bf16 copy for the GEMMs)
  float* dgp = fb(T.dgp);
  rmsnorm_bwd(a, d, nullptr, wt(C.W.ffn_norm), fb(B.dyf), d, fb(B.daf), d, nullptr, gp(G->ffn_norm), dgp, M, d, D.eps,
              st, dh, true, bb(B.dab));
  // a = u + o Wo^T: dWo += da^T o; do = da Wo; du = da (+ the attention path)
  if (float* gwo = gp(G->wo)) TRY(gemm_acc(d, d, M, bb(B.dab), d, true, o, d, true, gwo, d, st));
  {  // do = da Wo, written in bf16 straight from the accumulator (the attention backward's input)
    mtp::GemmDesc g = gdesc(M, d, d, bb(B.dab), d, wt(C.W.wo), d);
    g.b_mn = true;
    g.epi = mtp::EPI_STORE;
    g.out = bb(B.dob);
    g.ldo = d;
    g.pdl = true;  // follows a GEMM or a row kernel
    g.b_early = true;
    TRY(mtp::gemm_bf16_launch(g, st));
  }
  // segment-causal attention backward (tensor cores), then RoPE backward
  TRY(mtp::attn_bwd_launch(qkv, o, bb(B.dob), reinterpret_cast<const float*>(sv + C.so.lse2),
                           C.buf<int32_t>(C.L.seg_start), C.buf<int32_t>(C.L.seg_end), fb(B.dqkvf), fb(B.adsum), D.B,
                           D.T, H, hd, st));
  rope_bwd_kernel<<<std::min(M, 16 * 152), 256, 0, st>>>(fb(B.dqkvf), C.buf<float2>(C.L.rope), C.pos, bb(B.dqkvb), M, d, hd, D.T,
                                           D.rope_base > 0.f ? 1 : 0);
  mtp::note_launch();
  // q, k, v = x W{q,k,v}^T: dW += d{q,k,v}^T x; dx = [dq dk dv] [Wq; Wk; Wv]
  float* gq[3] = {gp(G->wq), gp(G->wk), gp(G->wv)};
  const bf* wqkv[3] = {wt(C.W.wq), wt(C.W.wk), wt(C.W.wv)};
  for (int j = 0; j < 3; ++j)
    if (gq[j]) TRY(gemm_acc(d, d, M, bb(B.dqkvb) + static_cast<size_t>(j) * d, 3 * d, true, x, d, true, gq[j], d, st));
  for (int j = 0; j < 3; ++j)
    TRY(gemm_acc(M, d, d, bb(B.dqkvb) + static_cast<size_t>(j) * d, 3 * d, false, wqkv[j], d, true, fb(B.dxf), d, st,
                 j == 0));
  // x = RMSNorm_a(u): du = da + RMSNorm backward (only its bf16 copy is used)
  rmsnorm_bwd(u, d, nullptr, wt(C.W.attn_norm), fb(B.dxf), d, nullptr, d, nullptr, gp(G->attn_norm), dgp, M, d, D.eps,
              st, fb(B.daf), true, bb(B.dub));
  // u = c M^T: dM += du^T c; dc = du M
  if (float* gm = gp(G->eh_proj)) TRY(gemm_acc(d, 2 * d, M, bb(B.dub), d, true, c, 2 * d, true, gm, 2 * d, st));
  TRY(gemm_acc(M, 2 * d, d, bb(B.dub), d, false, wt(C.W.eh_proj), 2 * d, true, fb(B.dcf), 2 * d, st, true));
  // c = [RMSNorm_h(h_{k-1}); RMSNorm_e(E[x_{t+k}])]: dh_{k-1} += ..., dE[x_{t+k}] += ...
  if (k > 1) {  // dstate[k-1] is complete after this: its bf16 copy is the next backward's input
    rmsnorm_bwd(h_prev, d, nullptr, wt(C.W.hnorm), fb(B.dcf), 2 * d, dh_prev, d, nullptr, gp(G->hnorm), dgp, M, d,
                D.eps, st, nullptr, false, bb(B.dhb));
  } else {  // dL/dh^0 = (the main term's head part, in dstate[0]) + this, added into the caller's h0 gradient
    rmsnorm_bwd(h_prev, d, nullptr, wt(C.W.hnorm), fb(B.dcf), 2 * d, G->h0, d, nullptr, gp(G->hnorm), dgp, M, d, D.eps,
                st, G->h0 && with_main ? dh_prev : nullptr, false);
  }
  int32_t* tok = C.buf<int32_t>(B.tok);
  shifted_tokens_kernel<<<(M + 255) / 256, 256, 0, st>>>(C.tokens, tok, M, D.T, k, D.V);
  mtp::note_launch();
  rmsnorm_bwd(static_cast<const bf*>(C.W.embed), d, tok, wt(C.W.enorm), fb(B.dcf) + d, 2 * d, G->embed, d, tok,
              gp(G->enorm), dgp, M, d, D.eps, st);
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

}  // namespace

extern "C" size_t mtp_chain_grad_workspace_bytes(const mtp_dims* dims) {
  if (!dims || !valid_dims(*dims) || supported(*dims) != MTP_OK || dims->dtype != MTP_BF16) return 0;
  const TrainLayout T = make_train_layout(*dims);
  return make_bwd_layout(*dims, T.total, T.mp).total;
}

extern "C" mtp_status mtp_chain_loss_grad(const mtp_dims* dims, const mtp_weights* w, const int32_t* tokens,
                                          const int32_t* seg, const int32_t* pos, const void* h0, float lambda,
                                          int den, int with_main, const float* depth_weights, double* sums_counts,
                                          float* losses, const mtp_grads* grads, void* ws, size_t ws_bytes,
                                          cudaStream_t stream) {
  using bf = __nv_bfloat16;
  if (!dims) return MTP_ERR_INVALID_ARG;
  if (dims->dtype != MTP_BF16) return MTP_ERR_UNSUPPORTED;
  TRY(check_common(dims, w, tokens, seg, pos, h0, ws, ws_bytes));
  if (!sums_counts || !losses || !grads) return MTP_ERR_INVALID_ARG;
  if (!valid_den(den)) return MTP_ERR_INVALID_ARG;
  if (depth_weights && dims->D > kMaxDepthWeights) return MTP_ERR_UNSUPPORTED;
  const mtp_dims& D = *dims;
  for (const void* p : {static_cast<const void*>(grads->head), static_cast<const void*>(grads->out_norm),
                        static_cast<const void*>(grads->h0), static_cast<const void*>(grads->embed)})
    if (p && !mtp::aligned16(p)) return MTP_ERR_ALIGNMENT;
  float* const* lists[] = {grads->hnorm, grads->enorm, grads->eh_proj, grads->attn_norm, grads->wq, grads->wk,
                           grads->wv, grads->wo, grads->ffn_norm, grads->w_gate, grads->w_up, grads->w_down};
  for (float* const* l : lists)
    if (l)
      for (int k = 0; k < D.D; ++k)
        if (!l[k] || !mtp::aligned16(l[k])) return l[k] ? MTP_ERR_ALIGNMENT : MTP_ERR_INVALID_ARG;
  const TrainLayout T = make_train_layout(D);
  const BwdLayout BL = make_bwd_layout(D, T.total, T.mp);
  if (ws_bytes < BL.total) return MTP_ERR_WORKSPACE;
  Ctx C{D, *w, tokens, seg, pos, static_cast<uint8_t*>(ws), make_layout(D), stream, D.B * D.T};
  std::unique_lock<std::mutex> side_lock;
  if (SideStream* S = side_stream(side_lock)) {
    C.side = S->s;
    C.ev = S->ev;
  }
  C.lse_save = C.buf<float>(T.lse);
  C.save = C.buf<uint8_t>(T.save);
  C.so = make_save_off(D);
  bf* hs = C.buf<bf>(T.hs);
  const int M = C.M, d = D.d;
  const size_t Md = static_cast<size_t>(M) * d;
  TRY(run_chain<bf>(C, static_cast<const bf*>(h0), hs, true, lambda, den, with_main, sums_counts, losses, nullptr));
  DepthWeights W{};
  W.lambda = lambda;
  W.uniform = depth_weights ? 0 : 1;
  if (depth_weights) {
    for (int k = 0; k < D.D; ++k) W.w[k] = depth_weights[k];
    loss_assemble_kernel<<<1, 32, 0, stream>>>(sums_counts, losses, D.D, static_cast<double>(M), W, den, with_main);
    mtp::note_launch();
  }
  term_scale_kernel<<<1, 32, 0, stream>>>(sums_counts, C.buf<float>(T.scale), D.D, static_cast<double>(M), W, den,
                                          with_main);
  mtp::note_launch();
  // every term's head backward writes its dstate slice before any block adds into it (dstate[0]
  // is read only with the main term, whose head writes it); the deepest term's head also writes
  // the bf16 copy the deepest block's backward starts from
  for (int t = with_main ? 0 : 1; t <= D.D; ++t) {
    const bf* h_t = t == 0 ? static_cast<const bf*>(h0) : hs + static_cast<size_t>(t - 1) * Md;
    TRY(head_backward(C, T, t, h_t, grads->head, grads->out_norm, t == D.D ? C.buf<bf>(BL.dhb) : nullptr));
  }
  // depths D..1: each depth's state gradient is complete once the deeper depth has run; depth 1
  // adds dL/dh^0 into grads->h0
  for (int k = D.D; k >= 1; --k) {
    const bf* h_prev = k == 1 ? static_cast<const bf*>(h0) : hs + static_cast<size_t>(k - 2) * Md;
    TRY(block_backward(C, T, BL, k, h_prev, grads, with_main != 0));
  }
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}
