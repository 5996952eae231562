// Segment-causal multi-head attention of the MTP block.
//
// "M7.6 - DeepSeek MTP" §0x03C (a = u + Attention(Norm_a u; causal)) with the
// segment rule of §0x04C: query t of a packed row sees keys
// s in [seg_start(t), t] only.  q, k, v come from the fused QKV GEMM as one
// [B*T, 3d] bf16 tensor (head h occupies columns h*hd.. of each third).
//
// bf16 forward: persistent tcgen05 kernel (attn_tc_kernel below): 128-query
// tiles, 128-key blocks fed by TMA, S = Q K^T and O += P V accumulated in
// TMEM, softmax warps reading S with tcgen05.ld; P is rounded to bf16 for
// the P V product.
// bf16 backward: flash-attention-2 form on mma.sync (flash_attn_bwd_kernel).
// f32 path (small shapes): one warp per (query row, head), scores staged in
// shared memory, fp32 throughout.
#include <cuda.h>

#include "common.cuh"
#include "gemm_tc.cuh"
#include "mbarrier.cuh"
#include "tcgen05.cuh"

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

// ---------------------------------------------------------------------------
// Forward on the tcgen05 tensor cores (bf16, head_dim 64 or 128).
//
// Persistent: one CTA per SM walks work items (128-query tile, head, packed
// row), the tiles nearest a row's end first (they see the most keys).  Six
// warps:
//   warp 4     TMA producer.  Lane 0 loads the Q tile ([128 rows x 64 cols]
//              boxes) and, per 128-key block, the K tile (same boxes) into a
//              ring of K stages; lane 1 loads the V tile as [64 keys x 64 cols]
//              boxes (the MN-major operand of P V) into its own ring.  K is
//              released as soon as S has been computed and V only after P V,
//              so K loads run further ahead than a shared K/V stage allows.
//   warp 5     allocates 512 TMEM columns (S double buffer at 0 and 128, O at
//              256); one thread issues S_j = Q K_j^T (M = 128, N = 128,
//              K = head_dim) into S buffer j % 2 and, once the softmax warps
//              have written P_j, O += P_j V_j (N = head_dim, K = 128 keys).
//              The order S_0, S_1, PV_0, S_2, PV_1, ... lets the softmax of
//              block j run while S_{j+1} and PV_{j-1} execute.
//   warps 0-3  softmax, one query row per thread (= TMEM lane): read S_j with
//              tcgen05.ld, apply the segment-causal mask and the scale (log2
//              domain), keep a running maximum m, write P = 2^(s - m) as bf16
//              into a 128-byte-swizzled K-major tile in shared memory, and sum
//              P in fp32.  m is replaced only when a block's maximum exceeds it
//              by more than 2^8 (P then stays <= 256); O, which lives in TMEM,
//              is rescaled by those rows' factor after the previous P V has
//              completed.  At the end of a tile O / l is written as bf16 (and
//              m + log2 l for the backward).
// The mask and the skipped blocks follow the segment rule: query t sees keys
// [seg_start(t), t]; a tile needs key blocks from seg_start(first query) to
// its last query.  Every wait is bounded (MTP_DEVERR_TIMEOUT, abort flag,
// drain of in-flight copies and MMAs before TMEM is freed).
// ---------------------------------------------------------------------------
constexpr int kTcQ = 128;
constexpr int kTcKeys = 128;
constexpr int kTcThreads = 192;
constexpr float kStaleMaxLog2 = 8.0f;

template <int HD>
struct TcAttn {
  static constexpr int kChunks = HD / 64;       // 64-column (128-byte) pieces of a row
  static constexpr int kTileBytes = 128 * 128;  // one [128 rows x 128 B] swizzled piece
  static constexpr int kQBytes = kTcQ * HD * 2;
  static constexpr int kKBytes = kTcKeys * HD * 2;
  static constexpr int kVBytes = kTcKeys * HD * 2;
  static constexpr int kPBytes = kTcQ * kTcKeys * 2;
  // one CTA per SM (512 TMEM columns: S double-buffered); head_dim 128 fits
  // one Q buffer and one P buffer in shared memory, head_dim 64 two of each
  static constexpr int kCtasPerSm = 1;
  static constexpr int kSBufs = 2;
  static constexpr int kQBufs = HD == 64 ? 2 : 1;
  static constexpr int kKStages = HD == 64 ? 4 : 3;
  static constexpr int kVStages = HD == 64 ? 3 : 2;
  static constexpr int kPBufs = HD == 64 ? 2 : 1;
  static constexpr int kOffK = kQBufs * kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKBytes;
  static constexpr int kOffP = kOffV + kVStages * kVBytes;
  static constexpr int kOffBar = kOffP + kPBufs * kPBytes;
  // q full/empty, k full/empty, v full/empty, s_full[2], p_full[2], pv_done[2], o_free, drain
  static constexpr int kNumBars = 2 * (kQBufs + kKStages + kVStages) + 8;
  // the dynamic shared memory starts 1024-byte aligned (no static shared memory; checked at run time)
  static constexpr int kSmemBytes = kOffBar + 8 * kNumBars + 16;
  static constexpr uint32_t kColS = 0, kColO = kSBufs * kTcKeys;
  static constexpr uint32_t kTmemCols = kSBufs == 1 ? 256 : 512;
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int HD>
__global__ void __launch_bounds__(kTcThreads, TcAttn<HD>::kCtasPerSm)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm128, const __grid_constant__ CUtensorMap tm64,
               __nv_bfloat16* __restrict__ out, const int32_t* __restrict__ seg_start, int B, int T, int H,
               float scale_log2, float* __restrict__ lse2_out) {
  using C = TcAttn<HD>;
  pdl_trigger();  // the output projection that follows may start its setup
  extern __shared__ __align__(1024) uint8_t attn_smem[];
  uint8_t* smem = attn_smem;
  const uint32_t s0 = mtp::smem_u32(smem);
  if (s0 & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(&g_mtp_error_word, MTP_DEVERR_TIMEOUT);
    return;
  }
  const uint32_t sQ = s0, sK = s0 + C::kOffK, sV = s0 + C::kOffV, sP = s0 + C::kOffP;
  const uint32_t bar0 = s0 + C::kOffBar;
  auto q_full = [&](int i) { return bar0 + 8u * i; };
  auto q_empty = [&](int i) { return bar0 + 8u * (C::kQBufs + i); };
  const uint32_t bark = bar0 + 16u * C::kQBufs;
  auto k_full = [&](int i) { return bark + 8u * i; };
  auto k_empty = [&](int i) { return bark + 8u * (C::kKStages + i); };
  const uint32_t barv = bark + 16u * C::kKStages;
  auto v_full = [&](int i) { return barv + 8u * i; };
  auto v_empty = [&](int i) { return barv + 8u * (C::kVStages + i); };
  const uint32_t barx = barv + 16u * C::kVStages;
  auto s_full = [&](uint32_t b) { return barx + 8u * b; };
  auto p_full = [&](uint32_t b) { return barx + 16u + 8u * b; };
  auto pv_done = [&](uint32_t b) { return barx + 32u + 8u * b; };
  const uint32_t o_free = barx + 48u, drain_bar = barx + 56u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned int* err = &g_mtp_error_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = H * HD;
  const int n_qb = (T + kTcQ - 1) / kTcQ;
  const int per_qb = H * B;
  const int n_tiles = n_qb * per_qb;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kQBufs; ++i) {
      mtp::mbar_init(q_full(i), 1);
      mtp::mbar_init(q_empty(i), 1);
    }
    for (int i = 0; i < C::kKStages; ++i) {
      mtp::mbar_init(k_full(i), 1);
      mtp::mbar_init(k_empty(i), 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mtp::mbar_init(v_full(i), 1);
      mtp::mbar_init(v_empty(i), 1);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mtp::mbar_init(s_full(b), 1);
      mtp::mbar_init(p_full(b), kTcQ);
      mtp::mbar_init(pv_done(b), 1);
    }
    mtp::mbar_init(o_free, kTcQ);
    mtp::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 4 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm128)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm64)) : "memory");
  }
  if (warp == 5) mtp::tmem_alloc_cols(mtp::smem_u32(tmem_slot), C::kTmemCols);
  mtp::tc_fence_before();
  __syncthreads();
  mtp::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // work item t: query tile qb (last tiles first), head h, packed row b
  auto coords = [&](int t, int& b, int& h, int& q0) {
    const int qb = n_qb - 1 - t / per_qb;
    const int r = t - (t / per_qb) * per_qb;
    h = r % H;
    b = r / H;
    q0 = qb * kTcQ;
  };
  // segment start of the tile's first query (its first key), loaded one work item ahead
  auto first_key = [&](int t) {
    if (t >= n_tiles) return 0;
    int b, h, q0;
    coords(t, b, h, q0);
    return static_cast<int>(seg_start[static_cast<size_t>(b) * T + q0]);
  };
  // key blocks [kb0, kb0 + nb) of work item t, given its first key
  auto decode = [&](int t, int key_first, int& b, int& h, int& q0, int& kb0, int& nb) {
    coords(t, b, h, q0);
    kb0 = key_first / kTcKeys;
    nb = min(q0 + kTcQ - 1, T - 1) / kTcKeys - kb0 + 1;
  };
  auto wait = [&](uint32_t bar, uint32_t parity) { return mtp::wait_phase(bar, parity, abort_flag, err); };

  if (warp == 4) {
    // ---------------- TMA producers: lane 0 Q and K, lane 1 V ----------------
    if (lane < 2) {
      const bool kside = lane == 0;
      const int stages = kside ? C::kKStages : C::kVStages;
      uint32_t g = 0, issued = 0;
      int tl = 0, q_loads = 0;
      bool ok = true;
      int key_next = first_key(blockIdx.x);
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++tl) {
        const int key_first = key_next;
        key_next = first_key(t + gridDim.x);
        int b, h, q0, kb0, nb;
        decode(t, key_first, b, h, q0, kb0, nb);
        if (kside) {
          const int qi = tl % C::kQBufs, qu = tl / C::kQBufs;
          if (qu > 0 && !wait(q_empty(qi), (qu - 1) & 1)) { ok = false; break; }
          mtp::mbar_expect_tx(q_full(qi), C::kQBytes);
          for (int c = 0; c < C::kChunks; ++c)
            mtp::tma_tile_2d(sQ + qi * C::kQBytes + c * C::kTileBytes, &tm128, h * HD + 64 * c, b * T + q0,
                             q_full(qi));
          ++q_loads;
        }
        for (int j = 0; j < nb; ++j, ++g) {
          const int st = static_cast<int>(g % stages);
          const uint32_t use = g / stages;
          const int row0 = b * T + (kb0 + j) * kTcKeys;
          if (kside) {
            if (use > 0 && !wait(k_empty(st), (use - 1) & 1)) { ok = false; break; }
            mtp::mbar_expect_tx(k_full(st), C::kKBytes);
            for (int c = 0; c < C::kChunks; ++c)
              mtp::tma_tile_2d(sK + st * C::kKBytes + c * C::kTileBytes, &tm128, d + h * HD + 64 * c, row0,
                               k_full(st));
          } else {
            if (use > 0 && !wait(v_empty(st), (use - 1) & 1)) { ok = false; break; }
            mtp::mbar_expect_tx(v_full(st), C::kVBytes);
            for (int half = 0; half < 2; ++half)
              for (int c = 0; c < C::kChunks; ++c)
                mtp::tma_tile_2d(sV + st * C::kVBytes + (half * C::kChunks + c) * 8192, &tm64,
                                 2 * d + h * HD + 64 * c, row0 + 64 * half, v_full(st));
          }
          issued = g + 1;
        }
      }
      // no copy may still be landing when the CTA leaves (matters only after an abort)
      for (uint32_t x = issued > static_cast<uint32_t>(stages) ? issued - stages : 0; x < issued; ++x)
        mtp::wait_drain(kside ? k_full(x % stages) : v_full(x % stages), (x / stages) & 1, kWaitLimitCycles);
      for (int x = q_loads > C::kQBufs ? q_loads - C::kQBufs : 0; x < q_loads; ++x)
        mtp::wait_drain(q_full(x % C::kQBufs), (x / C::kQBufs) & 1, kWaitLimitCycles);
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc_s = mtp::idesc_bf16_f32(kTcQ, kTcKeys, 0);
      constexpr uint32_t idesc_o = mtp::idesc_bf16_f32(kTcQ, HD, 2);  // V read MN-major
      uint32_t g = 0;
      int tl = 0;
      bool ok = true, any = false;
      int key_next = first_key(blockIdx.x);
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++tl) {
        const int key_first = key_next;
        key_next = first_key(t + gridDim.x);
        int b, h, q0, kb0, nb;
        decode(t, key_first, b, h, q0, kb0, nb);
        const int qi = tl % C::kQBufs;
        if (!wait(q_full(qi), (tl / C::kQBufs) & 1)) { ok = false; break; }
        const uint32_t sQt = sQ + qi * C::kQBytes;
        for (int j = 0; j <= nb; ++j) {
          if (j < nb) {  // S_j = Q K_j^T into S buffer j % 2
            const uint32_t gs = g + j;
            const int ks = static_cast<int>(gs % C::kKStages);
            if (!wait(k_full(ks), (gs / C::kKStages) & 1)) { ok = false; break; }
            // S buffer gs % kSBufs was last read by the softmax of block gs - kSBufs
            if (gs >= static_cast<uint32_t>(C::kSBufs)) {
              const uint32_t gr = gs - C::kSBufs;
              if (!wait(p_full(gr & 1), (gr >> 1) & 1)) { ok = false; break; }
            }
            mtp::tc_fence_after();
            const uint32_t sKt = sK + ks * C::kKBytes;
            const uint32_t dS = tmem + C::kColS + (gs % C::kSBufs) * kTcKeys;
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
              const uint32_t off = (k >> 2) * C::kTileBytes + (k & 3) * 32;
              mtp::umma_bf16_ss(dS, mtp::sdesc_k_sw128(sQt + off), mtp::sdesc_k_sw128(sKt + off), idesc_s, k > 0);
            }
            mtp::umma_commit(s_full(gs % C::kSBufs));
            mtp::umma_commit(k_empty(ks));
            if (j == nb - 1) mtp::umma_commit(q_empty(qi));
            any = true;
          }
          if (j >= 1) {  // O (+)= P_{j-1} V_{j-1}
            const uint32_t gp = g + j - 1;
            const int vs = static_cast<int>(gp % C::kVStages);
            if (!wait(v_full(vs), (gp / C::kVStages) & 1)) { ok = false; break; }
            if (!wait(p_full(gp & 1), (gp >> 1) & 1)) { ok = false; break; }
            if (j == 1 && tl > 0 && !wait(o_free, (tl - 1) & 1)) { ok = false; break; }
            mtp::tc_fence_after();
            const uint32_t pb = sP + (gp % C::kPBufs) * C::kPBytes;
            const uint32_t sVt = sV + vs * C::kVBytes;
#pragma unroll
            for (int k = 0; k < kTcKeys / 16; ++k) {
              const uint32_t a = pb + (k >> 2) * C::kTileBytes + (k & 3) * 32;
              const uint32_t bv = sVt + (k >> 2) * (C::kChunks * 8192) + (k & 3) * 2048;
              mtp::umma_bf16_ss(tmem + C::kColO, mtp::sdesc_k_sw128(a), mtp::sdesc_mn_sw128(bv), idesc_o,
                                (j > 1 || k > 0) ? 1u : 0u);
            }
            mtp::umma_commit(pv_done(gp & 1));
            mtp::umma_commit(v_empty(vs));
          }
        }
        g += nb;
      }
      // every issued MMA has completed before TMEM is freed
      if (any) {
        mtp::umma_commit(drain_bar);
        mtp::wait_drain(drain_bar, 0, kWaitLimitCycles);
      }
    }
  } else {
    // ---------------- softmax warps: one query row per thread ----------------
    const int row = threadIdx.x;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    // warp-uniform bounded wait: every lane waits, all must succeed
    auto wwait = [&](uint32_t bar, uint32_t parity) { return __all_sync(0xffffffffu, wait(bar, parity)); };
    uint32_t g = 0;
    // this row's segment start, loaded one work item ahead
    auto row_start = [&](int t) {
      if (t >= n_tiles) return 0;
      int b, h, q0;
      coords(t, b, h, q0);
      const int q = q0 + row;
      return q < T ? static_cast<int>(seg_start[static_cast<size_t>(b) * T + q]) : q;
    };
    int key_next = first_key(blockIdx.x), st_next = row_start(blockIdx.x);
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
      const int key_first = key_next, st_row = st_next;
      key_next = first_key(t + gridDim.x);
      st_next = row_start(t + gridDim.x);
      int b, h, q0, kb0, nb;
      decode(t, key_first, b, h, q0, kb0, nb);
      const int q = q0 + row;
      const bool live = q < T;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < nb; ++j) {
        const uint32_t gs = g + j;
        if (!wwait(s_full(gs % C::kSBufs), (gs / C::kSBufs) & 1)) { ok = false; break; }
        mtp::tc_fence_after();
        float sc[kTcKeys];
        {
          float (&lo)[64] = *reinterpret_cast<float (*)[64]>(&sc[0]);
          float (&hi)[64] = *reinterpret_cast<float (*)[64]>(&sc[64]);
          mtp::tmem_ld64(lane_base + C::kColS + (gs % C::kSBufs) * kTcKeys, lo);
          mtp::tmem_ld64(lane_base + C::kColS + (gs % C::kSBufs) * kTcKeys + 64, hi);
        }
        const int key0 = (kb0 + j) * kTcKeys;
        if (!(key0 >= st_row && key0 + kTcKeys - 1 <= q)) {  // a block the row sees only in part
#pragma unroll
          for (int i = 0; i < kTcKeys; ++i) {
            const int key = key0 + i;
            if (!(key >= st_row && key <= q)) sc[i] = -INFINITY;
          }
        }
        // row maximum of the raw scores (scale > 0), eight independent chains
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = sc[i];
#pragma unroll
        for (int i = 8; i < kTcKeys; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], sc[i]);
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * scale_log2;
        // a new running maximum only when the block's exceeds the stale one by 2^8
        const float m_new = mx > m + kStaleMaxLog2 ? mx : m;
        const bool rescale = m_new != m && m != -INFINITY;
        const float neg_use = m_new == -INFINITY ? 0.f : -m_new;
        // P = 2^(s scale - m), rounded to bf16 (packed in place: sc[i] holds pair i)
        float rs8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rs8[i] = 0.f;
#pragma unroll
        for (int i = 0; i < kTcKeys / 2; ++i) {
          const float a = ex2_approx(fmaf(sc[2 * i], scale_log2, neg_use));
          const float bb = ex2_approx(fmaf(sc[2 * i + 1], scale_log2, neg_use));
          rs8[i & 7] += a + bb;
          sc[i] = __uint_as_float(pack2_bf16(a, bb));
        }
        if (__any_sync(0xffffffffu, rescale)) {  // O holds earlier blocks' P V: wait for the last one
          if (!wwait(pv_done((gs - 1) & 1), ((gs - 1) >> 1) & 1)) { ok = false; break; }
          mtp::tc_fence_after();
          const float alpha = rescale ? ex2_approx(m - m_new) : 1.f;
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            float o[32];
            mtp::tmem_ld32(lane_base + C::kColO + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            mtp::tmem_st32(lane_base + C::kColO + 32 * c, o);
          }
          l *= alpha;
        }
        m = m_new;
        l += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        // the P buffer was last read by the P V of block gs - kPBufs
        if (gs >= static_cast<uint32_t>(C::kPBufs)) {
          const uint32_t gr = gs - C::kPBufs;
          if (!wwait(pv_done(gr & 1), (gr >> 1) & 1)) { ok = false; break; }
        }
        uint8_t* prow = smem + C::kOffP + (gs % C::kPBufs) * C::kPBytes + row * 128;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8) {
            const int i0 = 32 * c + 4 * k8;
            *reinterpret_cast<uint4*>(prow + c * C::kTileBytes + ((k8 ^ (row & 7)) << 4)) =
                make_uint4(__float_as_uint(sc[i0]), __float_as_uint(sc[i0 + 1]), __float_as_uint(sc[i0 + 2]),
                           __float_as_uint(sc[i0 + 3]));
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P visible to the tensor cores
        mtp::tc_fence_before();
        mtp::mbar_arrive1(p_full(gs & 1));
      }
      if (!ok) break;
      const uint32_t gl = g + nb - 1;
      if (!wwait(pv_done(gl & 1), (gl >> 1) & 1)) break;
      mtp::tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (live && lse2_out) lse2_out[(static_cast<size_t>(b) * T + q) * H + h] = m + log2f(l);
      __nv_bfloat16* orow = out + (static_cast<size_t>(b) * T + q) * d + h * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        mtp::tmem_ld32(lane_base + C::kColO + 32 * c, o);
        if (live) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            reinterpret_cast<uint4*>(orow + 32 * c)[v] =
                make_uint4(pack2_bf16(o[8 * v] * inv, o[8 * v + 1] * inv),
                           pack2_bf16(o[8 * v + 2] * inv, o[8 * v + 3] * inv),
                           pack2_bf16(o[8 * v + 4] * inv, o[8 * v + 5] * inv),
                           pack2_bf16(o[8 * v + 6] * inv, o[8 * v + 7] * inv));
        }
      }
      mtp::tc_fence_before();
      mtp::mbar_arrive1(o_free);
      g += nb;
    }
  }
  mtp::tc_fence_before();
  __syncthreads();
  mtp::tc_fence_after();
  if (warp == 5) mtp::tmem_free_cols(tmem, C::kTmemCols);
}

template <int HD>
mtp_status attn_tc_launch(const __nv_bfloat16* qkv, __nv_bfloat16* out, const int32_t* seg_start, int B, int T,
                          int H, float scale_log2, float* lse2_out, cudaStream_t stream) {
  using C = TcAttn<HD>;
  static PerDevice attr;
  if (!smem_limit(attr, attn_tc_kernel<HD>, C::kSmemBytes)) return MTP_ERR_CUDA;
  if (!aligned16(qkv) || !aligned16(out)) return MTP_ERR_ALIGNMENT;
  const int d = H * HD;
  const uint64_t rows = static_cast<uint64_t>(B) * T;
  if (rows > 0x7FFFFFFFull) return MTP_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
  CUtensorMap m128, m64;
  if (!tensor_map_bf16_2d(&m128, qkv, rows, 3 * d, 3 * d, 64, 128, true) ||
      !tensor_map_bf16_2d(&m64, qkv, rows, 3 * d, 3 * d, 64, 64, true))
    return MTP_ERR_CUDA;
  const long long n_tiles = static_cast<long long>((T + kTcQ - 1) / kTcQ) * H * B;
  if (n_tiles > 0x7FFFFFFFll) return MTP_ERR_UNSUPPORTED;
  const long long slots = static_cast<long long>(C::kCtasPerSm) * sm_count_current();
  const int grid = static_cast<int>(n_tiles < slots ? n_tiles : slots);
  attn_tc_kernel<HD><<<grid, kTcThreads, C::kSmemBytes, stream>>>(m128, m64, out, seg_start, B, T, H, scale_log2,
                                                                 lse2_out);
  note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

}  // namespace

mtp_status attn_launch(int dtype, const void* qkv, void* out, const int32_t* seg_start, int B, int T, int H,
                       int hd, cudaStream_t stream, float* lse2_out) {
  if (B <= 0 || T <= 0) return MTP_OK;
  if (dtype == MTP_BF16) {
    const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
    if (hd == 64)
      return attn_tc_launch<64>(static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(out), seg_start,
                                B, T, H, scale_log2, lse2_out, stream);
    if (hd == 128)
      return attn_tc_launch<128>(static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(out),
                                 seg_start, B, T, H, scale_log2, lse2_out, stream);
    return MTP_ERR_UNSUPPORTED;
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
