// Segment-causal multi-head attention of the MTP block.
//
// "M7.6 - DeepSeek MTP" §0x03C (a = u + Attention(Norm_a u; causal)) with the
// segment rule of §0x04C: query t of a packed row sees keys
// s in [seg_start(t), t] only.  q, k, v come from the fused QKV GEMM as one
// [B*T, 3d] bf16 tensor (head h occupies columns h*hd.. of each third).
//
// bf16 path: flash-style kernel, 64 queries x one head per CTA (4 warps x 16
// rows), 64-key blocks double-buffered in shared memory with cp.async
// (16-byte chunks, XOR-swizzled rows), S = Q K^T and O += P V on
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate), online softmax in fp32 with
// exp2.  P is rounded to bf16 for the P V product.
// f32 path (small shapes): one warp per (query row, head), scores staged in
// shared memory, fp32 throughout.
#include "common.cuh"

MTP_DEFINE_ERROR_WORD(mtp_take_errors_attn)

namespace mtp {

mtp_status attn_launch(int dtype, const void* qkv, void* out, const int32_t* seg_start, int B, int T,
                       int H, int hd, cudaStream_t stream, float* lse2_out = nullptr);
mtp_status attn_bwd_launch(const __nv_bfloat16* qkv, const __nv_bfloat16* o, const __nv_bfloat16* dO,
                           const float* lse2, const int32_t* seg_start, const int32_t* seg_end, float* dqkv,
                           float* dsum, int B, int T, int H, int hd, cudaStream_t stream);

namespace {

constexpr int kBQ = 64;
constexpr int kBK = 64;
constexpr int kThreads = 128;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// byte offset of element (row, col) in a [rows][HD] bf16 tile whose 16-byte
// chunks are XOR-swizzled by (row & 7)
template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return static_cast<uint32_t>(row * HD * 2 + ((((col >> 3) ^ (row & 7))) << 4) + (col & 7) * 2);
}

// rows [row0, row0+64) of one head from the [B*T, 3d] qkv tensor (column
// offset col0 selects q/k/v and the head); rows >= T are zero-filled.
template <int HD>
__device__ __forceinline__ void load_tile(uint32_t tile, const __nv_bfloat16* qkv, int b, int T, int ld3,
                                          int row0, int col0) {
  constexpr int kChunks = kBK * HD / 8;
#pragma unroll
  for (int i = threadIdx.x; i < kChunks; i += kThreads) {
    const int r = i / (HD / 8), c = i % (HD / 8);
    const int t = row0 + r;
    const bool ok = t < T;
    const __nv_bfloat16* src = qkv + (static_cast<size_t>(b) * T + (ok ? t : 0)) * ld3 + col0 + c * 8;
    cp_async16(tile + swz<HD>(r, c * 8), src, ok);
  }
}

template <int HD>
__global__ void __launch_bounds__(kThreads)
flash_attn_bf16_kernel(const __nv_bfloat16* __restrict__ qkv, __nv_bfloat16* __restrict__ out,
                       const int32_t* __restrict__ seg_start, int T, int H, float scale_log2,
                       float* __restrict__ lse2_out) {
  pdl_trigger();  // the output projection that follows may start its setup
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + kBQ * HD * 2;
  const uint32_t sV0 = sK0 + 2 * kBK * HD * 2;
  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int d = H * HD, ld3 = 3 * d;
  const int q0 = qb * kBQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int32_t* ss = seg_start + static_cast<size_t>(b) * T;

  const int k_lo = ss[q0];
  const int k_hi = min(q0 + kBQ - 1, T - 1);
  const int kb_first = k_lo / kBK, kb_last = k_hi / kBK;

  load_tile<HD>(sQ, qkv, b, T, ld3, q0, h * HD);
  load_tile<HD>(sK0, qkv, b, T, ld3, kb_first * kBK, d + h * HD);
  load_tile<HD>(sV0, qkv, b, T, ld3, kb_first * kBK, 2 * d + h * HD);
  cp_async_commit();

  const int row_a = q0 + warp * 16 + g, row_b = row_a + 8;
  const int st_a = row_a < T ? ss[row_a] : row_a;
  const int st_b = row_b < T ? ss[row_b] : row_b;
  // a k-block at or past every row's segment start and wholly below the warp's first row
  // needs no mask (skipping invisible 16-key groups instead was measured slower: the
  // branches break the unrolled MMA schedule)
  int st_max = max(st_a, st_b);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) st_max = max(st_max, __shfl_xor_sync(0xffffffffu, st_max, o));
  const int wrow0 = q0 + warp * 16;

  uint32_t qa[HD / 16][4];
  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

  for (int kb = kb_first; kb <= kb_last; ++kb) {
    const int buf = (kb - kb_first) & 1;
    cp_async_wait_all();
    __syncthreads();
    if (kb == kb_first) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        ldsm_x4(sQ + swz<HD>(warp * 16 + (lane & 15), kk * 16 + (lane >> 4) * 8), qa[kk][0], qa[kk][1],
                qa[kk][2], qa[kk][3]);
    }
    if (kb < kb_last) {
      const int nb = buf ^ 1;
      load_tile<HD>(sK0 + nb * kBK * HD * 2, qkv, b, T, ld3, (kb + 1) * kBK, d + h * HD);
      load_tile<HD>(sV0 + nb * kBK * HD * 2, qkv, b, T, ld3, (kb + 1) * kBK, 2 * d + h * HD);
      cp_async_commit();
    }
    const uint32_t sK = sK0 + buf * kBK * HD * 2;
    const uint32_t sV = sV0 + buf * kBK * HD * 2;

    // S = Q K^T : 16 rows x 64 keys per warp
    const int kbase = kb * kBK;
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int nt = 0; nt < 8; nt += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sK + swz<HD>(nt * 8 + (lane & 7) + ((lane >> 4) << 3), kk * 16 + ((lane >> 3) & 1) * 8), b0, b1,
                b2, b3);
        mma_bf16(s[nt], qa[kk], b0, b1);
        mma_bf16(s[nt + 1], qa[kk], b2, b3);
      }
    }
    // mask, scale, online softmax
    float mx_a = -INFINITY, mx_b = -INFINITY;
    if (kbase >= st_max && kbase + kBK - 1 <= wrow0) {  // every key visible to every row of the warp
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[nt][e] *= scale_log2;
          s[nt][2 + e] *= scale_log2;
          mx_a = fmaxf(mx_a, s[nt][e]);
          mx_b = fmaxf(mx_b, s[nt][2 + e]);
        }
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = kbase + nt * 8 + 2 * tq + e;
          s[nt][e] = (key >= st_a && key <= row_a) ? s[nt][e] * scale_log2 : -INFINITY;
          s[nt][2 + e] = (key >= st_b && key <= row_b) ? s[nt][2 + e] * scale_log2 : -INFINITY;
          mx_a = fmaxf(mx_a, s[nt][e]);
          mx_b = fmaxf(mx_b, s[nt][2 + e]);
        }
      }
    }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float use_a = mn_a == -INFINITY ? 0.f : mn_a;
    const float use_b = mn_b == -INFINITY ? 0.f : mn_b;
    const float alpha_a = m_a == -INFINITY ? 0.f : exp2f(m_a - mn_a);
    const float alpha_b = m_b == -INFINITY ? 0.f : exp2f(m_b - mn_b);
    m_a = mn_a;
    m_b = mn_b;
    float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - use_a);
      s[nt][1] = exp2f(s[nt][1] - use_a);
      s[nt][2] = exp2f(s[nt][2] - use_b);
      s[nt][3] = exp2f(s[nt][3] - use_b);
      rs_a += s[nt][0] + s[nt][1];
      rs_b += s[nt][2] + s[nt][3];
    }
    l_a = l_a * alpha_a + rs_a;
    l_b = l_b * alpha_b + rs_b;
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt) {
      o[dt][0] *= alpha_a;
      o[dt][1] *= alpha_a;
      o[dt][2] *= alpha_b;
      o[dt][3] *= alpha_b;
    }
    // O += P V
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kt][0], s[2 * kt][1]);
      pa[1] = pack_bf16(s[2 * kt][2], s[2 * kt][3]);
      pa[2] = pack_bf16(s[2 * kt + 1][0], s[2 * kt + 1][1]);
      pa[3] = pack_bf16(s[2 * kt + 1][2], s[2 * kt + 1][3]);
#pragma unroll
      for (int dt = 0; dt < HD / 8; dt += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sV + swz<HD>(kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, dt * 8 + (lane >> 4) * 8), b0, b1,
                  b2, b3);
        mma_bf16(o[dt], pa, b0, b1);
        mma_bf16(o[dt + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f;
  const float inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
  if (lse2_out && tq == 0) {  // log2-domain log-sum-exp of the scaled scores, for the backward
    if (row_a < T) lse2_out[(static_cast<size_t>(b) * T + row_a) * H + h] = m_a + log2f(l_a);
    if (row_b < T) lse2_out[(static_cast<size_t>(b) * T + row_b) * H + h] = m_b + log2f(l_b);
  }
#pragma unroll
  for (int dt = 0; dt < HD / 8; ++dt) {
    const int col = h * HD + dt * 8 + 2 * tq;
    if (row_a < T)
      *reinterpret_cast<__nv_bfloat162*>(out + (static_cast<size_t>(b) * T + row_a) * d + col) =
          __floats2bfloat162_rn(o[dt][0] * inv_a, o[dt][1] * inv_a);
    if (row_b < T)
      *reinterpret_cast<__nv_bfloat162*>(out + (static_cast<size_t>(b) * T + row_b) * d + col) =
          __floats2bfloat162_rn(o[dt][2] * inv_b, o[dt][3] * inv_b);
  }
}

// ---------------------------------------------------------------------------
// Backward, flash-attention-2 form: one CTA per (64-key block, head, packed
// row).  K and V of the block stay in shared memory; every 64-query block
// that can see one of its keys streams through (Q and dO double-buffered
// with cp.async).  Warp w owns keys 16w..16w+15:
//   S^T = K_w Q^T, dP^T = V_w dO^T            (m16n8k16, K/V rows as A)
//   P = exp2(S scale_log2 - lse2[q]) on visible (key, query) pairs
//   dS^T = P (dP - D[q]),  D[q] = do_q . o_q
//   dV_w += P^T dO,  dK_w += dS^T Q           (accumulated in registers)
// dS^T goes to shared memory and each warp forms 16 rows of dQ = dS K,
// added to the fp32 dq rows with atomics (every key block contributes).
// P and dS are rounded to bf16 for the products.
// ---------------------------------------------------------------------------
template <int HD>
__global__ void attn_dsum_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
                                 float* __restrict__ dsum, int items, int H) {
  constexpr int KD = HD / 32;
  const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (item >= items) return;
  const int m = item / H, h = item % H;
  const size_t base = static_cast<size_t>(m) * H * HD + h * HD + lane * KD;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < KD; ++i) acc += __bfloat162float(o[base + i]) * __bfloat162float(dO[base + i]);
  acc = warp_sum(acc);
  if (lane == 0) dsum[item] = acc;
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
flash_attn_bwd_kernel(const __nv_bfloat16* __restrict__ qkv, const __nv_bfloat16* __restrict__ dO,
                      const float* __restrict__ lse2, const float* __restrict__ dsum,
                      const int32_t* __restrict__ seg_start, const int32_t* __restrict__ seg_end,
                      float* __restrict__ dqkv, int T, int H, float scale_log2, float scale) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kTile = kBK * HD * 2;
  const uint32_t sK = smem_u32(smem);
  const uint32_t sV = sK + kTile;
  const uint32_t sQ0 = sV + kTile;
  const uint32_t sdO0 = sQ0 + 2 * kTile;
  const uint32_t sdS = sdO0 + 2 * kTile;  // [64 keys][64 queries] bf16, rows XOR-swizzled
  uint8_t* sdS_ptr = smem + (sdS - sK);
  float* s_lse = reinterpret_cast<float*>(sdS_ptr + kBK * kBQ * 2);  // [2][64]
  float* s_D = s_lse + 2 * kBQ;
  int* s_qss = reinterpret_cast<int*>(s_D + 2 * kBQ);
  int* s_red = s_qss + 2 * kBQ;
  const int kb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int d = H * HD, ld3 = 3 * d;
  const int k0 = kb * kBK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int32_t* ss = seg_start + static_cast<size_t>(b) * T;
  const int32_t* se = seg_end + static_cast<size_t>(b) * T;

  // the last query that sees one of the block's keys
  int qhi = -1;
  for (int i = threadIdx.x; i < kBK; i += kThreads) {
    const int s = k0 + i;
    if (s < T) qhi = max(qhi, max(se[s], s + 1) - 1);
  }
  qhi = __reduce_max_sync(0xffffffffu, qhi);
  if (lane == 0) s_red[warp] = qhi;
  __syncthreads();
  qhi = max(max(s_red[0], s_red[1]), max(s_red[2], s_red[3]));
  const int qb_first = kb, qb_last = qhi / kBQ;

  auto load_params = [&](int buf, int qb) {
    for (int i = threadIdx.x; i < kBQ; i += kThreads) {
      const int q = qb * kBQ + i;
      const bool ok = q < T;
      const size_t item = (static_cast<size_t>(b) * T + (ok ? q : 0)) * H + h;
      s_lse[buf * kBQ + i] = ok ? lse2[item] : INFINITY;
      s_D[buf * kBQ + i] = ok ? dsum[item] : 0.f;
      s_qss[buf * kBQ + i] = ok ? ss[q] : 0x7fffffff;
    }
  };
  load_tile<HD>(sK, qkv, b, T, ld3, k0, d + h * HD);
  load_tile<HD>(sV, qkv, b, T, ld3, k0, 2 * d + h * HD);
  load_tile<HD>(sQ0, qkv, b, T, ld3, qb_first * kBQ, h * HD);
  load_tile<HD>(sdO0, dO, b, T, d, qb_first * kBQ, h * HD);
  cp_async_commit();
  load_params(0, qb_first);

  float dk[HD / 8][4], dv[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.f;
    dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
  }
  const int key_a = k0 + warp * 16 + g, key_b = key_a + 8;

  for (int qb = qb_first; qb <= qb_last; ++qb) {
    const int buf = (qb - qb_first) & 1;
    cp_async_wait_all();
    __syncthreads();
    if (qb < qb_last) {
      const int nb = buf ^ 1;
      load_tile<HD>(sQ0 + nb * kTile, qkv, b, T, ld3, (qb + 1) * kBQ, h * HD);
      load_tile<HD>(sdO0 + nb * kTile, dO, b, T, d, (qb + 1) * kBQ, h * HD);
      cp_async_commit();
      load_params(nb, qb + 1);
    }
    const uint32_t sQ = sQ0 + buf * kTile, sdO = sdO0 + buf * kTile;
    const float* lse_b = s_lse + buf * kBQ;
    const float* D_b = s_D + buf * kBQ;
    const int* qss_b = s_qss + buf * kBQ;

    // S^T = K_w Q^T and dP^T = V_w dO^T: 16 keys x 64 queries per warp
    float st[8][4], dp[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.f;
      dp[nt][0] = dp[nt][1] = dp[nt][2] = dp[nt][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      uint32_t ka[4], va[4];
      ldsm_x4(sK + swz<HD>(warp * 16 + (lane & 15), kk * 16 + (lane >> 4) * 8), ka[0], ka[1], ka[2], ka[3]);
      ldsm_x4(sV + swz<HD>(warp * 16 + (lane & 15), kk * 16 + (lane >> 4) * 8), va[0], va[1], va[2], va[3]);
#pragma unroll
      for (int nt = 0; nt < 8; nt += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sQ + swz<HD>(nt * 8 + (lane & 7) + ((lane >> 4) << 3), kk * 16 + ((lane >> 3) & 1) * 8), b0, b1,
                b2, b3);
        mma_bf16(st[nt], ka, b0, b1);
        mma_bf16(st[nt + 1], ka, b2, b3);
        ldsm_x4(sdO + swz<HD>(nt * 8 + (lane & 7) + ((lane >> 4) << 3), kk * 16 + ((lane >> 3) & 1) * 8), b0, b1,
                b2, b3);
        mma_bf16(dp[nt], va, b0, b1);
        mma_bf16(dp[nt + 1], va, b2, b3);
      }
    }
    // P^T (into st) and dS^T (into dp) on visible pairs: seg_start(q) <= key <= q
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int ql = nt * 8 + 2 * tq + e, q = qb * kBQ + ql;
        const float lse = lse_b[ql], Dq = D_b[ql];
        const int qss = qss_b[ql];
        const bool va_ok = key_a < T && key_a >= qss && key_a <= q;
        const bool vb_ok = key_b < T && key_b >= qss && key_b <= q;
        const float pa = va_ok ? exp2f(st[nt][e] * scale_log2 - lse) : 0.f;
        const float pb = vb_ok ? exp2f(st[nt][2 + e] * scale_log2 - lse) : 0.f;
        st[nt][e] = pa;
        st[nt][2 + e] = pb;
        dp[nt][e] = pa * (dp[nt][e] - Dq);
        dp[nt][2 + e] = pb * (dp[nt][2 + e] - Dq);
      }
    }
    // dV_w += P^T dO and dK_w += dS^T Q (k-steps of 16 queries)
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t pa[4], da[4];
      pa[0] = pack_bf16(st[2 * kt][0], st[2 * kt][1]);
      pa[1] = pack_bf16(st[2 * kt][2], st[2 * kt][3]);
      pa[2] = pack_bf16(st[2 * kt + 1][0], st[2 * kt + 1][1]);
      pa[3] = pack_bf16(st[2 * kt + 1][2], st[2 * kt + 1][3]);
      da[0] = pack_bf16(dp[2 * kt][0], dp[2 * kt][1]);
      da[1] = pack_bf16(dp[2 * kt][2], dp[2 * kt][3]);
      da[2] = pack_bf16(dp[2 * kt + 1][0], dp[2 * kt + 1][1]);
      da[3] = pack_bf16(dp[2 * kt + 1][2], dp[2 * kt + 1][3]);
#pragma unroll
      for (int dt = 0; dt < HD / 8; dt += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sdO + swz<HD>(kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, dt * 8 + (lane >> 4) * 8), b0, b1, b2,
                  b3);
        mma_bf16(dv[dt], pa, b0, b1);
        mma_bf16(dv[dt + 1], pa, b2, b3);
        ldsm_x4_t(sQ + swz<HD>(kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, dt * 8 + (lane >> 4) * 8), b0, b1, b2,
                  b3);
        mma_bf16(dk[dt], da, b0, b1);
        mma_bf16(dk[dt + 1], da, b2, b3);
      }
    }
    // dS^T to shared memory (row = key, column = query)
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = nt * 8 + 2 * tq;
      *reinterpret_cast<uint32_t*>(sdS_ptr + swz<64>(warp * 16 + g, col)) = pack_bf16(dp[nt][0], dp[nt][1]);
      *reinterpret_cast<uint32_t*>(sdS_ptr + swz<64>(warp * 16 + g + 8, col)) = pack_bf16(dp[nt][2], dp[nt][3]);
    }
    __syncthreads();
    // dQ rows 16w..16w+15 of the query block: dS (A, read transposed) times K (B, read transposed)
    float dq[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4_t(sdS + swz<64>(kk * 16 + (lane & 7) + ((lane >> 4) << 3), warp * 16 + ((lane >> 3) & 1) * 8), a[0],
                a[1], a[2], a[3]);
#pragma unroll
      for (int dt = 0; dt < HD / 8; dt += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sK + swz<HD>(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, dt * 8 + (lane >> 4) * 8), b0, b1, b2,
                  b3);
        mma_bf16(dq[dt], a, b0, b1);
        mma_bf16(dq[dt + 1], a, b2, b3);
      }
    }
    const int qa_row = qb * kBQ + warp * 16 + g, qb_row = qa_row + 8;
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt) {
      const int col = h * HD + dt * 8 + 2 * tq;
      if (qa_row < T) {
        float* dst = dqkv + (static_cast<size_t>(b) * T + qa_row) * ld3 + col;
        atomicAdd(dst, dq[dt][0] * scale);
        atomicAdd(dst + 1, dq[dt][1] * scale);
      }
      if (qb_row < T) {
        float* dst = dqkv + (static_cast<size_t>(b) * T + qb_row) * ld3 + col;
        atomicAdd(dst, dq[dt][2] * scale);
        atomicAdd(dst + 1, dq[dt][3] * scale);
      }
    }
  }
  // dK (scaled) and dV of the warp's 16 keys
#pragma unroll
  for (int dt = 0; dt < HD / 8; ++dt) {
    const int col = h * HD + dt * 8 + 2 * tq;
    if (key_a < T) {
      float* r = dqkv + (static_cast<size_t>(b) * T + key_a) * ld3;
      r[d + col] = dk[dt][0] * scale;
      r[d + col + 1] = dk[dt][1] * scale;
      r[2 * d + col] = dv[dt][0];
      r[2 * d + col + 1] = dv[dt][1];
    }
    if (key_b < T) {
      float* r = dqkv + (static_cast<size_t>(b) * T + key_b) * ld3;
      r[d + col] = dk[dt][2] * scale;
      r[d + col + 1] = dk[dt][3] * scale;
      r[2 * d + col] = dv[dt][2];
      r[2 * d + col + 1] = dv[dt][3];
    }
  }
}

// f32: one warp per (row, head); scores of the row's keys staged in smem.
__global__ void attn_f32_kernel(const float* __restrict__ qkv, float* __restrict__ out,
                                const int32_t* __restrict__ seg_start, int BT, int T, int H, int hd, float scale) {
  extern __shared__ float sc[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * (blockDim.x >> 5) + warp;
  if (item >= BT * H) return;
  const int m = item / H, h = item % H;
  const int b = m / T, t = m % T;
  const int d = H * hd;
  float* s = sc + warp * T;
  const float* q = qkv + static_cast<size_t>(m) * 3 * d + h * hd;
  const int lo = seg_start[m];
  float mx = -INFINITY;
  for (int j = lo + lane; j <= t; j += 32) {
    const float* k = qkv + (static_cast<size_t>(b) * T + j) * 3 * d + d + h * hd;
    float acc = 0.f;
    for (int i = 0; i < hd; ++i) acc += q[i] * k[i];
    acc *= scale;
    s[j] = acc;
    mx = fmaxf(mx, acc);
  }
  mx = warp_max(mx);
  float sum = 0.f;
  for (int j = lo + lane; j <= t; j += 32) {
    const float e = expf(s[j] - mx);
    s[j] = e;
    sum += e;
  }
  sum = warp_sum(sum);
  __syncwarp();
  for (int i = lane; i < hd; i += 32) {
    float acc = 0.f;
    for (int j = lo; j <= t; ++j) acc += s[j] * qkv[(static_cast<size_t>(b) * T + j) * 3 * d + 2 * d + h * hd + i];
    out[static_cast<size_t>(m) * d + h * hd + i] = acc / sum;
  }
}

}  // namespace

mtp_status attn_launch(int dtype, const void* qkv, void* out, const int32_t* seg_start, int B, int T, int H,
                       int hd, cudaStream_t stream, float* lse2_out) {
  if (B <= 0 || T <= 0) return MTP_OK;
  if (dtype == MTP_BF16) {
    const dim3 grid((T + kBQ - 1) / kBQ, H, B);
    const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
    if (hd == 64) {
      constexpr int smem = (kBQ + 4 * kBK) * 64 * 2;
      flash_attn_bf16_kernel<64><<<grid, kThreads, smem, stream>>>(
          static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(out), seg_start, T, H, scale_log2,
          lse2_out);
      mtp::note_launch();
    } else if (hd == 128) {
      constexpr int smem = (kBQ + 4 * kBK) * 128 * 2;
      static PerDevice attr;
      if (!smem_limit(attr, flash_attn_bf16_kernel<128>, smem)) return MTP_ERR_CUDA;
      flash_attn_bf16_kernel<128><<<grid, kThreads, smem, stream>>>(
          static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(out), seg_start, T, H, scale_log2,
          lse2_out);
      mtp::note_launch();
    } else {
      return MTP_ERR_UNSUPPORTED;
    }
  } else {
    const int warps = 4;
    const size_t smem = static_cast<size_t>(warps) * T * sizeof(float);
    if (smem > 200 * 1024) return MTP_ERR_UNSUPPORTED;
    static PerDevice attr;
    if (!smem_limit(attr, attn_f32_kernel, 200 * 1024)) return MTP_ERR_CUDA;
    const int items = B * T * H;
    attn_f32_kernel<<<(items + warps - 1) / warps, warps * 32, smem, stream>>>(
        static_cast<const float*>(qkv), static_cast<float*>(out), seg_start, B * T, T, H, hd,
        1.0f / sqrtf(static_cast<float>(hd)));
    mtp::note_launch();
  }
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

mtp_status attn_bwd_launch(const __nv_bfloat16* qkv, const __nv_bfloat16* o, const __nv_bfloat16* dO,
                           const float* lse2, const int32_t* seg_start, const int32_t* seg_end, float* dqkv,
                           float* dsum, int B, int T, int H, int hd, cudaStream_t stream) {
  if (B <= 0 || T <= 0) return MTP_OK;
  const int items = B * T * H;
  const dim3 grid((T + kBK - 1) / kBK, H, B);
  const float scale = 1.0f / sqrtf(static_cast<float>(hd));
  const float scale_log2 = 1.4426950408889634f * scale;
  // dq is accumulated with atomics by every key block: start from zero
  if (cudaMemsetAsync(dqkv, 0, static_cast<size_t>(B) * T * 3 * H * hd * sizeof(float), stream) != cudaSuccess)
    return MTP_ERR_CUDA;
  if (hd == 64) {
    attn_dsum_kernel<64><<<(items + 7) / 8, 256, 0, stream>>>(o, dO, dsum, items, H);
    constexpr int smem = (6 * kBK * 64 + kBK * kBQ) * 2 + 2 * kBQ * 12 + 64;
    static PerDevice attr;
    if (!smem_limit(attr, flash_attn_bwd_kernel<64>, smem)) return MTP_ERR_CUDA;
    flash_attn_bwd_kernel<64><<<grid, kThreads, smem, stream>>>(qkv, dO, lse2, dsum, seg_start, seg_end, dqkv, T, H,
                                                                scale_log2, scale);
  } else if (hd == 128) {
    attn_dsum_kernel<128><<<(items + 7) / 8, 256, 0, stream>>>(o, dO, dsum, items, H);
    constexpr int smem = (6 * kBK * 128 + kBK * kBQ) * 2 + 2 * kBQ * 12 + 64;
    static PerDevice attr;
    if (!smem_limit(attr, flash_attn_bwd_kernel<128>, smem)) return MTP_ERR_CUDA;
    flash_attn_bwd_kernel<128><<<grid, kThreads, smem, stream>>>(qkv, dO, lse2, dsum, seg_start, seg_end, dqkv, T,
                                                                 H, scale_log2, scale);
  } else {
    return MTP_ERR_UNSUPPORTED;
  }
  mtp::note_launch();
  mtp::note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

}  // namespace mtp
