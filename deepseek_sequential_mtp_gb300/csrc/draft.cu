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
// Every weight-streaming product is a skinny GEMM (R <= 32 tokens): the
// tcgen05 core runs it swap-AB (weights on the 128-row side, tokens as
// N = 32) with split-K so that the weight stream covers every SM; partial
// tiles accumulate into an fp32 buffer with atomics and small "finish"
// kernels round to bf16 with the fused RoPE / residual / SwiGLU / RMSNorm.
// Attention is flash-decoding: (request, 8 heads, 512-key chunk) CTAs write
// partial (max, sum, output) records that a combine kernel merges with the
// new row's key.  The head writes logits into q_out, which a per-request
// kernel turns into probabilities in place and samples from.
#include <algorithm>
#include <cmath>

#include "gemm_tc.cuh"

MTP_DEFINE_ERROR_WORD(mtp_take_errors_draft)

namespace {

constexpr int kMaxR = 32;
constexpr int kHeadsPerCta = 8;
constexpr int kKeysPerChunk = 512;

__device__ __forceinline__ float bf(const __nv_bfloat16& v) { return __bfloat162float(v); }

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
__device__ float block_max(float v, float* sh) {
  v = mtp::warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  float t = -INFINITY;
  for (int i = 0; i < (blockDim.x >> 5); ++i) t = fmaxf(t, sh[i]);
  return t;
}

// ---------------------------------------------------------------------------
// c = [RMSNorm_h(parent_hidden); RMSNorm_e(E[frontier])], one CTA per request
// ---------------------------------------------------------------------------
__global__ void draft_prologue_kernel(const __nv_bfloat16* __restrict__ hp, const int32_t* __restrict__ frontier,
                                      const __nv_bfloat16* __restrict__ embed, const __nv_bfloat16* __restrict__ gh,
                                      const __nv_bfloat16* __restrict__ ge, __nv_bfloat16* __restrict__ c, int d, int V,
                                      float eps) {
  __shared__ float sh[32];
  const int r = blockIdx.x;
  int tok = frontier[r];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) atomicOr(&g_mtp_error_word, MTP_DEVERR_TOKEN_RANGE);
    tok = min(max(tok, 0), V - 1);
  }
  const __nv_bfloat16* h = hp + static_cast<size_t>(r) * d;
  const __nv_bfloat16* e = embed + static_cast<size_t>(tok) * d;
  float a = 0.f, b = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float x = bf(h[i]), y = bf(e[i]);
    a += x * x;
    b += y * y;
  }
  a = block_sum(a, sh);
  b = block_sum(b, sh);
  const float rh = 1.0f / sqrtf(a / d + eps), re = 1.0f / sqrtf(b / d + eps);
  __nv_bfloat16* out = c + static_cast<size_t>(r) * 2 * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    out[i] = __float2bfloat16_rn(bf(gh[i]) * (bf(h[i]) * rh));
    out[d + i] = __float2bfloat16_rn(bf(ge[i]) * (bf(e[i]) * re));
  }
}

// y = bf16(acc [+ resid]); optionally norm_out = bf16(RMSNorm_g(y)) (one CTA per row)
__global__ void finish_row_kernel(const float* __restrict__ acc, const __nv_bfloat16* __restrict__ resid,
                                  __nv_bfloat16* __restrict__ y, const __nv_bfloat16* __restrict__ g,
                                  __nv_bfloat16* __restrict__ norm_out, int d, float eps) {
  __shared__ float sh[32];
  const int r = blockIdx.x;
  const float* a = acc + static_cast<size_t>(r) * d;
  __nv_bfloat16* yr = y + static_cast<size_t>(r) * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float v = a[i];
    if (resid) v += bf(resid[static_cast<size_t>(r) * d + i]);
    const __nv_bfloat16 vb = __float2bfloat16_rn(v);
    yr[i] = vb;
    const float vf = bf(vb);
    ss += vf * vf;
  }
  if (!norm_out) return;
  ss = block_sum(ss, sh);
  const float rn = 1.0f / sqrtf(ss / d + eps);
  for (int i = threadIdx.x; i < d; i += blockDim.x)
    norm_out[static_cast<size_t>(r) * d + i] = __float2bfloat16_rn(bf(g[i]) * (bf(yr[i]) * rn));
}

// qkv = bf16(RoPE(q), RoPE(k), v) at the request's position; the angle is
// formed and reduced modulo 2*pi in double, sine/cosine taken in fp32
__global__ void finish_qkv_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ qkv,
                                  const int32_t* __restrict__ pos, int d, int hd, float base, int pos_max) {
  const int r = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // pair index over q and k, or a v column
  const int half = hd / 2;
  const float* a = acc + static_cast<size_t>(r) * 3 * d;
  __nv_bfloat16* o = qkv + static_cast<size_t>(r) * 3 * d;
  if (i < d) {  // d pairs: q and k heads, (j, j + half) within each head
    const int head = i / half, j = i % half;  // head index over 2*H (q heads then k heads)
    const int col = head * hd + j;
    const float x1 = a[col], x2 = a[col + half];
    float c = 1.f, s = 0.f;
    if (base > 0.f) {
      int p = pos[r];
      if (p < 0 || p > pos_max) {
        if (j == 0) atomicOr(&g_mtp_error_word, MTP_DEVERR_TOKEN_RANGE);
        p = min(max(p, 0), pos_max);
      }
      const double ang = static_cast<double>(p) * exp2(-2.0 * j / hd * log2(static_cast<double>(base)));
      const double two_pi = 6.283185307179586;
      sincosf(static_cast<float>(ang - rint(ang / two_pi) * two_pi), &s, &c);
    }
    o[col] = __float2bfloat16_rn(x1 * c - x2 * s);
    o[col + half] = __float2bfloat16_rn(x2 * c + x1 * s);
  }
  if (i < d) o[2 * d + i] = __float2bfloat16_rn(a[2 * d + i]);  // v
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
// flash-decoding: CTA = (request, 8 heads, 512-key chunk of the cache); warp = head
// part record: [max, sum, o(hd)] (fp32) per (r, head, chunk)
// ---------------------------------------------------------------------------
template <int HD>
__global__ void __launch_bounds__(256)
decode_attn_partial_kernel(const __nv_bfloat16* __restrict__ qkv, const __nv_bfloat16* __restrict__ kc,
                           const __nv_bfloat16* __restrict__ vc, const int32_t* __restrict__ ctx_len,
                           float* __restrict__ part, int H, int T, int n_chunks, float scale) {
  __shared__ float sq[kHeadsPerCta][HD];
  __shared__ float sp[kHeadsPerCta][kKeysPerChunk];
  const int r = blockIdx.x, chunk = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kHeadsPerCta + warp;
  const int d = H * HD;
  const int len = min(max(ctx_len[r], 0), T);
  const int s0 = chunk * kKeysPerChunk, s1 = min(s0 + kKeysPerChunk, len);
  float* rec = part + ((static_cast<size_t>(r) * H + h) * n_chunks + chunk) * (HD + 2);
  if (h >= H) return;
  for (int i = lane; i < HD; i += 32) sq[warp][i] = bf(qkv[static_cast<size_t>(r) * 3 * d + h * HD + i]) * scale;
  __syncwarp();
  if (s1 <= s0) {  // empty chunk
    if (lane == 0) {
      rec[0] = -INFINITY;
      rec[1] = 0.f;
    }
    for (int i = lane; i < HD; i += 32) rec[2 + i] = 0.f;
    return;
  }
  // scores: lane per key
  float mx = -INFINITY;
  for (int s = s0 + lane; s < s1; s += 32) {
    const uint4* k4 = reinterpret_cast<const uint4*>(kc + (static_cast<size_t>(r) * T + s) * d + h * HD);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < HD / 8; ++c) {
      const uint4 u = __ldcs(k4 + c);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(b[t]);
        acc += f.x * sq[warp][c * 8 + 2 * t] + f.y * sq[warp][c * 8 + 2 * t + 1];
      }
    }
    sp[warp][s - s0] = acc;
    mx = fmaxf(mx, acc);
  }
  mx = mtp::warp_max(mx);
  float sum = 0.f;
  for (int s = s0 + lane; s < s1; s += 32) {
    const float e = __expf(sp[warp][s - s0] - mx);
    sp[warp][s - s0] = e;
    sum += e;
  }
  sum = mtp::warp_sum(sum);
  __syncwarp();
  // P V: lane owns HD/32 consecutive dims
  constexpr int kDim = HD / 32;
  float o[kDim];
#pragma unroll
  for (int t = 0; t < kDim; ++t) o[t] = 0.f;
  const __nv_bfloat16* vbase = vc + static_cast<size_t>(r) * T * d + h * HD + lane * kDim;
#pragma unroll 4
  for (int s = s0; s < s1; ++s) {
    const float p = sp[warp][s - s0];
    const __nv_bfloat16* vr = vbase + static_cast<size_t>(s) * d;
    if constexpr (kDim == 4) {
      const uint2 u = __ldcs(reinterpret_cast<const uint2*>(vr));
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
      const float2 f0 = __bfloat1622float2(b[0]), f1 = __bfloat1622float2(b[1]);
      o[0] += p * f0.x;
      o[1] += p * f0.y;
      o[2] += p * f1.x;
      o[3] += p * f1.y;
    } else {
      const __nv_bfloat162 u = __ldcs(reinterpret_cast<const __nv_bfloat162*>(vr));
      const float2 f = __bfloat1622float2(u);
      o[0] += p * f.x;
      o[1] += p * f.y;
    }
  }
  if (lane == 0) {
    rec[0] = mx;
    rec[1] = sum;
  }
#pragma unroll
  for (int t = 0; t < kDim; ++t) rec[2 + lane * kDim + t] = o[t];
}

// merge the chunk records with the new row's own key/value; one warp per (r, head)
template <int HD>
__global__ void decode_attn_combine_kernel(const __nv_bfloat16* __restrict__ qkv, const float* __restrict__ part,
                                           __nv_bfloat16* __restrict__ out, int R, int H, int n_chunks, float scale) {
  const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (item >= R * H) return;
  const int r = item / H, h = item % H;
  const int d = H * HD;
  constexpr int kDim = HD / 32;
  const __nv_bfloat16* row = qkv + static_cast<size_t>(r) * 3 * d;
  // the new key
  float qk = 0.f;
  for (int i = lane; i < HD; i += 32) qk += bf(row[h * HD + i]) * bf(row[d + h * HD + i]);
  qk = mtp::warp_sum(qk) * scale;
  const float* rec0 = part + (static_cast<size_t>(r) * H + h) * n_chunks * (HD + 2);
  float m = qk;
  for (int c = 0; c < n_chunks; ++c) m = fmaxf(m, rec0[c * (HD + 2)]);
  float l = __expf(qk - m);
  float o[kDim];
#pragma unroll
  for (int t = 0; t < kDim; ++t) o[t] = l * bf(row[2 * d + h * HD + lane * kDim + t]);
  for (int c = 0; c < n_chunks; ++c) {
    const float* rec = rec0 + c * (HD + 2);
    if (rec[1] <= 0.f) continue;
    const float w = __expf(rec[0] - m);
    l += w * rec[1];
#pragma unroll
    for (int t = 0; t < kDim; ++t) o[t] += w * rec[2 + lane * kDim + t];
  }
  const float inv = 1.0f / l;
#pragma unroll
  for (int t = 0; t < kDim; ++t)
    out[static_cast<size_t>(r) * d + h * HD + lane * kDim + t] = __float2bfloat16_rn(o[t] * inv);
}

// ---------------------------------------------------------------------------
// q = softmax(z) in place and y ~ q by inverse CDF; one CTA (1024 threads) per request
// ---------------------------------------------------------------------------
constexpr int kSampleThreads = 1024;
constexpr int kSampleChunk = 1024;
constexpr int kMaxSampleChunks = 512;

__global__ void __launch_bounds__(kSampleThreads)
softmax_sample_kernel(float* __restrict__ q, int V, uint2 key, uint32_t off_lo, uint32_t off_hi,
                      int32_t* __restrict__ y_out) {
  __shared__ float sh[32];
  __shared__ float2 s_chunk[kMaxSampleChunks];
  __shared__ float s_w[kSampleChunk];
  __shared__ int s_cstar;
  __shared__ double s_before, s_target;
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* z = q + static_cast<size_t>(r) * V;
  float mx = -INFINITY;
  for (int v = threadIdx.x; v < V; v += kSampleThreads) mx = fmaxf(mx, z[v]);
  mx = block_max(mx, sh);
  float sum = 0.f;
  for (int v = threadIdx.x; v < V; v += kSampleThreads) sum += __expf(z[v] - mx);
  sum = block_sum(sum, sh);
  const float inv = 1.0f / sum;
  __syncthreads();
  // write q and compensated per-chunk sums (chunk c = [c*1024, c*1024+1024), warp-strided)
  const int n_chunks = (V + kSampleChunk - 1) / kSampleChunk;
  for (int c = warp; c < n_chunks; c += kSampleThreads / 32) {
    float hi = 0.f, lo = 0.f;
    for (int i = lane; i < kSampleChunk; i += 32) {
      const int v = c * kSampleChunk + i;
      if (v < V) {
        const float pv = __expf(z[v] - mx) * inv;
        z[v] = pv;
        float s, e;
        two_sum(hi, pv, s, e);
        hi = s;
        lo += e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ohi = __shfl_xor_sync(0xffffffffu, hi, o), olo = __shfl_xor_sync(0xffffffffu, lo, o);
      float s, e;
      two_sum(hi, ohi, s, e);
      hi = s;
      lo = (lo + olo) + e;
    }
    if (lane == 0) s_chunk[c] = make_float2(hi, lo);
  }
  __syncthreads();
  const uint4 w = philox4x32_10(make_uint4(0u, static_cast<uint32_t>(r), off_lo, off_hi), key);
  const double u = static_cast<double>(w.z >> 8) * (1.0 / 16777216.0);
  if (warp == 0) {
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
    }
  }
  __syncthreads();
  const int cstar = s_cstar;
  if (cstar < 0) {
    if (threadIdx.x == 0) y_out[r] = -1;
    return;
  }
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
  const double lincl = mtp::warp_inclusive_scan(lane_sum) + s_before;
  const double target = s_target;
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
    y_out[r] = eover ? base + __ffs(eover) - 1 : (epos ? base + 31 - __clz(epos) : -1);
  }
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------
inline size_t align_up(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct DraftLayout {
  size_t c, acc, u, x, qkv, o, a, g, h, part, total;
  int n_chunks;
};

DraftLayout draft_layout(const mtp_dims& D) {
  DraftLayout L{};
  const size_t R = D.B, d = D.d;
  L.n_chunks = (D.T + kKeysPerChunk - 1) / kKeysPerChunk;
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
  L.h = take(R * d * 2);
  L.part = take(R * static_cast<size_t>(D.n_heads) * L.n_chunks * (D.head_dim + 2) * 4);
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
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// out[R, ldo] (fp32, columns [col0, col0 + features)) += X[R, K] · W[features, K]^T
mtp_status skinny_gemm(const __nv_bfloat16* W, int features, int K, const __nv_bfloat16* X, int R, float* out,
                       int ldo, cudaStream_t st, bool store = false) {
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
  const int tiles = (features + 127) / 128;
  const int nk = (K + 63) / 64;
  int splits = 1;
  if (!store) {
    splits = (3 * sm_count() + tiles - 1) / tiles;
    splits = std::max(1, std::min(splits, nk / 4 > 0 ? nk / 4 : 1));
  }
  g.splits = splits;
  g.epi = store ? mtp::EPI_T_STORE : mtp::EPI_T_ATOMIC;
  return mtp::gemm_bf16_launch(g, st);
}

#define TRY(expr)                \
  do {                           \
    mtp_status s_ = (expr);      \
    if (s_ != MTP_OK) return s_; \
  } while (0)

}  // namespace

extern "C" size_t mtp_draft_workspace_bytes(const mtp_dims* dims) {
  if (!dims || !draft_dims_ok(*dims)) return 0;
  return draft_layout(*dims).total;
}

extern "C" mtp_status mtp_draft_step(const mtp_dims* dims, const mtp_weights* w, const void* parent_hidden,
                                     const int32_t* frontier, const int32_t* pos, const void* kv_k, const void* kv_v,
                                     const int32_t* ctx_len, uint64_t seed, uint64_t offset, float* q_out,
                                     int32_t* y_out, void* h_out, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (!dims || !w) return MTP_ERR_INVALID_ARG;
  const mtp_dims& D = *dims;
  if (!draft_dims_ok(D)) return D.dtype != MTP_BF16 || D.D != 1 || D.B > kMaxR ? MTP_ERR_UNSUPPORTED : MTP_ERR_SHAPE;
  if (!parent_hidden || !frontier || !pos || !kv_k || !kv_v || !ctx_len || !q_out || !y_out || !ws)
    return MTP_ERR_INVALID_ARG;
  if (!w->embed || !w->head || !w->out_norm) return MTP_ERR_INVALID_ARG;
  const void* const* lists[] = {w->hnorm, w->enorm, w->eh_proj, w->attn_norm, w->wq, w->wk, w->wv,
                                w->wo, w->ffn_norm, w->w_gate, w->w_up, w->w_down};
  for (auto l : lists)
    if (!l || !l[0] || !mtp::aligned16(l[0])) return l && l[0] ? MTP_ERR_ALIGNMENT : MTP_ERR_INVALID_ARG;
  const void* ptrs[] = {parent_hidden, kv_k, kv_v, static_cast<const void*>(q_out), ws, w->embed, w->head};
  for (const void* p : ptrs)
    if (!mtp::aligned16(p)) return MTP_ERR_ALIGNMENT;
  if (h_out && !mtp::aligned16(h_out)) return MTP_ERR_ALIGNMENT;
  const DraftLayout L = draft_layout(D);
  if (ws_bytes < L.total) return MTP_ERR_WORKSPACE;

  const int R = D.B, d = D.d, ffn = D.ffn, V = D.V, H = D.n_heads, hd = D.head_dim;
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto bfp = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(base + off); };
  float* acc = reinterpret_cast<float*>(base + L.acc);
  auto W0 = [&](const void* const* l) { return static_cast<const __nv_bfloat16*>(l[0]); };
  const __nv_bfloat16* E = static_cast<const __nv_bfloat16*>(w->embed);
  __nv_bfloat16 *c = bfp(L.c), *u = bfp(L.u), *x = bfp(L.x), *qkv = bfp(L.qkv), *o = bfp(L.o), *a = bfp(L.a),
                *g = bfp(L.g);
  __nv_bfloat16* h = h_out ? static_cast<__nv_bfloat16*>(h_out) : bfp(L.h);
  const int fin_threads = 256;

  // c, u = M c, x = RMSNorm_a(u)
  draft_prologue_kernel<<<R, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(parent_hidden), frontier, E,
                                           W0(w->hnorm), W0(w->enorm), c, d, V, D.eps);
  mtp::note_launch();
  MTP_CUDA_TRY(cudaMemsetAsync(acc, 0, static_cast<size_t>(R) * d * 4, st));
  TRY(skinny_gemm(W0(w->eh_proj), d, 2 * d, c, R, acc, d, st));
  finish_row_kernel<<<R, fin_threads, 0, st>>>(acc, nullptr, u, W0(w->attn_norm), x, d, D.eps);
  mtp::note_launch();
  // q, k, v with RoPE on q, k
  MTP_CUDA_TRY(cudaMemsetAsync(acc, 0, static_cast<size_t>(R) * 3 * d * 4, st));
  TRY(skinny_gemm(W0(w->wq), d, d, x, R, acc, 3 * d, st));
  TRY(skinny_gemm(W0(w->wk), d, d, x, R, acc + d, 3 * d, st));
  TRY(skinny_gemm(W0(w->wv), d, d, x, R, acc + 2 * d, 3 * d, st));
  finish_qkv_kernel<<<dim3((d + 255) / 256, R), 256, 0, st>>>(acc, qkv, pos, d, hd, D.rope_base, D.T);
  mtp::note_launch();
  // attention over the module's own cache plus the new row
  const float scale = 1.0f / sqrtf(static_cast<float>(hd));
  float* part = reinterpret_cast<float*>(base + L.part);
  const dim3 agrid(R, (H + kHeadsPerCta - 1) / kHeadsPerCta, L.n_chunks);
  const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(kv_k);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(kv_v);
  mtp::prof_begin(MTP_KC_ATTENTION, st);
  if (hd == 128) {
    decode_attn_partial_kernel<128><<<agrid, 256, 0, st>>>(qkv, kc, vc, ctx_len, part, H, D.T, L.n_chunks, scale);
    mtp::note_launch();
    decode_attn_combine_kernel<128><<<(R * H + 7) / 8, 256, 0, st>>>(qkv, part, o, R, H, L.n_chunks, scale);
  } else {
    decode_attn_partial_kernel<64><<<agrid, 256, 0, st>>>(qkv, kc, vc, ctx_len, part, H, D.T, L.n_chunks, scale);
    mtp::note_launch();
    decode_attn_combine_kernel<64><<<(R * H + 7) / 8, 256, 0, st>>>(qkv, part, o, R, H, L.n_chunks, scale);
  }
  mtp::note_launch();
  mtp::prof_end(MTP_KC_ATTENTION, st);
  // a = u + o Wo^T, x = RMSNorm_f(a)
  MTP_CUDA_TRY(cudaMemsetAsync(acc, 0, static_cast<size_t>(R) * d * 4, st));
  TRY(skinny_gemm(W0(w->wo), d, d, o, R, acc, d, st));
  finish_row_kernel<<<R, fin_threads, 0, st>>>(acc, u, a, W0(w->ffn_norm), x, d, D.eps);
  mtp::note_launch();
  // g = silu(x Wg^T) * (x Wu^T)
  MTP_CUDA_TRY(cudaMemsetAsync(acc, 0, static_cast<size_t>(R) * 2 * ffn * 4, st));
  TRY(skinny_gemm(W0(w->w_gate), ffn, d, x, R, acc, 2 * ffn, st));
  TRY(skinny_gemm(W0(w->w_up), ffn, d, x, R, acc + ffn, 2 * ffn, st));
  finish_swiglu_kernel<<<dim3((ffn + 255) / 256, R), 256, 0, st>>>(acc, g, ffn);
  mtp::note_launch();
  // h = a + g Wd^T, x = RMSNorm_out(h)
  MTP_CUDA_TRY(cudaMemsetAsync(acc, 0, static_cast<size_t>(R) * d * 4, st));
  TRY(skinny_gemm(W0(w->w_down), d, ffn, g, R, acc, d, st));
  finish_row_kernel<<<R, fin_threads, 0, st>>>(acc, a, h, static_cast<const __nv_bfloat16*>(w->out_norm), x, d,
                                               D.eps);
  mtp::note_launch();
  // logits into q_out, then softmax and the draw
  mtp::prof_begin(MTP_KC_HEAD_CE_GEMM, st);
  TRY(skinny_gemm(static_cast<const __nv_bfloat16*>(w->head), V, d, x, R, q_out, V, st, true));
  mtp::prof_end(MTP_KC_HEAD_CE_GEMM, st);
  const uint2 key = make_uint2(static_cast<uint32_t>(seed & 0xFFFFFFFFu), static_cast<uint32_t>(seed >> 32));
  softmax_sample_kernel<<<R, kSampleThreads, 0, st>>>(q_out, V, key, static_cast<uint32_t>(offset & 0xFFFFFFFFu),
                                                      static_cast<uint32_t>(offset >> 32), y_out);
  mtp::note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}
