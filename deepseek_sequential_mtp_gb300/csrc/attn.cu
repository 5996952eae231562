// Segment-causal multi-head attention of the MTP block.
//
// "M7.6 - DeepSeek MTP" §0x03C (a = u + Attention(Norm_a u; causal)) with the
// segment rule of §0x04C: query t of a packed row sees keys
// s in [seg_start(t), t] only.  q, k, v come from the fused QKV GEMM as one
// [B*T, 3d] bf16 tensor (head h occupies columns h*hd.. of each third).
//
// bf16 forward: persistent tcgen05 kernel (attn_tc2_kernel below): work items
// of two 128-query tiles sharing 128-key blocks fed by TMA, S = Q K^T and
// O += P V accumulated in TMEM, softmax warps reading S with tcgen05.ld and
// writing P back into TMEM as bf16 for the P V product.
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

// work_ctr (bf16): a device int that is 0 on entry and is used up by the launch (one per launch)
mtp_status attn_launch(int dtype, const void* qkv, void* out, const int32_t* seg_start, int B, int T,
                       int H, int hd, cudaStream_t stream, float* lse2_out = nullptr, int* work_ctr = nullptr);
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

constexpr int kTcQ = 128;     // queries per tile (MMA M, TMEM lanes)
constexpr int kTcKeys = 128;  // keys per block (N of S = Q K^T, K of O += P V)
constexpr float kStaleMaxLog2 = 8.0f;  // a running maximum is replaced only when exceeded by 2^8

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Forward on the tcgen05 tensor cores: two query tiles per work item.
//
// A work item is 256 consecutive queries of one (packed row, head): tile A =
// queries q0..q0+127, tile B = q0+128..q0+255 (absent past T).  Both tiles
// share every K/V block they need, which halves the K/V traffic per FLOP, and
// their softmax warpgroups alternate on the tensor pipe: while warps 0-3
// turn S_A into P_A, the MMA thread runs P_B V and S_B, and the reverse.
//   warps 0-3 / 4-7  softmax of tile A / B, one query row per thread (TMEM
//              lane = row): S read with tcgen05.ld, segment-causal mask,
//              stale-by-up-to-2^8 running maximum, P = 2^(s - m) written back
//              as bf16 pairs into the first 64 columns of the tile's own S
//              (tcgen05.st), where the P V product reads it as its A operand.
//   warp 8     TMA: lane 0 loads Q_A, Q_B and the K blocks, lane 1 the V
//              blocks (MN-major [64 keys x 64 cols] boxes), each into a ring.
//   warp 9     allocates 512 TMEM columns (S_A, S_B at 0 and 128; O_A, O_B
//              at 256 and 256 + HD); one thread issues, per key block j,
//              P_A(j) V_j, S_A(j+1), P_B(j) V_j, S_B(j+1) (S of the first
//              block up front), skipping a tile outside its key range.
// Tile A needs key blocks [seg_start(q0) / 128, q0 / 128], tile B
// [seg_start(q0 + 128) / 128, (q0 + 128) / 128]: A's range is a prefix of the
// union, B's a suffix.  Work items run from the last query pairs (the longest
// key ranges) to the first; a CTA starts with item blockIdx.x and claims each
// further one from a global counter (atomicAdd) when that item's Q buffer
// frees, so CTAs whose items were short take more of them.  The TMA lane that claims an item publishes it,
// with its tiles' segment starts, in a shared-memory ring that the V lane, the
// MMA thread and the softmax warps read in the same order.  Every wait is
// bounded.
// ---------------------------------------------------------------------------
constexpr int kT2Threads = 320;

template <int HD>
struct Tc2Attn {
  static constexpr int kChunks = HD / 64;
  static constexpr int kTileBytes = 128 * 128;  // one [128 rows x 128 B] swizzled piece
  static constexpr int kQBytes = kTcQ * HD * 2;  // one tile's Q
  static constexpr int kKBytes = kTcKeys * HD * 2;
  static constexpr int kVBytes = kTcKeys * HD * 2;
  static constexpr int kQBufs = HD == 64 ? 2 : 1;  // Q of the next item loads early when it fits
  static constexpr int kKStages = HD == 64 ? 4 : 3;
  static constexpr int kVStages = HD == 64 ? 4 : 2;
  static constexpr int kOffK = kQBufs * 2 * kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKBytes;
  static constexpr int kOffBar = kOffV + kVStages * kVBytes;
  static constexpr int kRing = 4;  // claimed work items published ahead of their consumers
  // readers of a ring slot: the V lane, the MMA thread and one lane of each softmax warp
  static constexpr int kItemReaders = 10;
  // q full/empty, k full/empty, v full/empty; per tile s_full, p_full, pv_done, o_free; drain;
  // item ring full/empty
  static constexpr int kNumBars = 2 * (kQBufs + kKStages + kVStages) + 8 + 1 + 2 * kRing;
  static constexpr int kOffItems = (kOffBar + 8 * kNumBars + 15) / 16 * 16;
  static constexpr int kSmemBytes = kOffItems + 16 * kRing + 16;
  static constexpr uint32_t kColO0 = 256;
};

template <int HD>
__global__ void __launch_bounds__(kT2Threads, 1)
attn_tc2_kernel(const __grid_constant__ CUtensorMap tm128, const __grid_constant__ CUtensorMap tm64,
                __nv_bfloat16* __restrict__ out, const int32_t* __restrict__ seg_start, int B, int T, int H,
                float scale_log2, float* __restrict__ lse2_out, int* __restrict__ work_ctr) {
  using C = Tc2Attn<HD>;
  pdl_trigger();  // the output projection that follows may start its setup
  extern __shared__ __align__(1024) uint8_t attn2_smem[];
  uint8_t* smem = attn2_smem;
  const uint32_t s0 = mtp::smem_u32(smem);
  if (s0 & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(&g_mtp_error_word, MTP_DEVERR_TIMEOUT);
    return;
  }
  const uint32_t sQ = s0, sK = s0 + C::kOffK, sV = s0 + C::kOffV;
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
  auto s_full = [&](int x) { return barx + 8u * x; };
  auto p_full = [&](int x) { return barx + 16u + 8u * x; };
  auto pv_done = [&](int x) { return barx + 32u + 8u * x; };
  auto o_free = [&](int x) { return barx + 48u + 8u * x; };
  const uint32_t drain_bar = barx + 64u;
  auto it_full = [&](int i) { return barx + 72u + 8u * i; };
  auto it_empty = [&](int i) { return barx + 72u + 8u * (C::kRing + i); };
  // ring slot: (item, segment start of tile A's first query, of tile B's first query); item -1 ends
  int4* items = reinterpret_cast<int4*>(smem + C::kOffItems);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffItems + 16 * C::kRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned int* err = &g_mtp_error_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = H * HD;
  const int n_pairs = (T + 2 * kTcQ - 1) / (2 * kTcQ);
  const int per_qp = H * B;
  const int n_items = n_pairs * per_qp;

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
    for (int x = 0; x < 2; ++x) {
      mtp::mbar_init(s_full(x), 1);
      mtp::mbar_init(p_full(x), kTcQ);
      mtp::mbar_init(pv_done(x), 1);
      mtp::mbar_init(o_free(x), kTcQ);
    }
    mtp::mbar_init(drain_bar, 1);
    for (int i = 0; i < C::kRing; ++i) {
      mtp::mbar_init(it_full(i), 1);
      mtp::mbar_init(it_empty(i), C::kItemReaders);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 8 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm128)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm64)) : "memory");
  }
  if (warp == 9) mtp::tmem_alloc_cols(mtp::smem_u32(tmem_slot), 512);
  mtp::tc_fence_before();
  __syncthreads();
  mtp::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // q/k/v come from the kernel before (this launch is its programmatic dependent)

  // work item t: query pair qp (last pairs first), head h, packed row b
  auto coords = [&](int t, int& b, int& h, int& q0) {
    const int qp = n_pairs - 1 - t / per_qp;
    const int r = t - (t / per_qp) * per_qp;
    h = r % H;
    b = r / H;
    q0 = qp * 2 * kTcQ;
  };
  // segment starts of both tiles' first queries
  auto first_keys = [&](int t) {
    if (t >= n_items) return make_int2(0, 0);
    int b, h, q0;
    coords(t, b, h, q0);
    const int32_t* ss = seg_start + static_cast<size_t>(b) * T;
    return make_int2(ss[q0], q0 + kTcQ < T ? ss[q0 + kTcQ] : 0);
  };
  // key-block ranges: tile x covers blocks [lo[x], hi[x]] (empty when hi < lo); union [lo[0], u_hi]
  struct Ranges {
    int lo[2], hi[2], u_hi;
  };
  auto ranges = [&](int q0, int2 keys) {
    Ranges R;
    R.lo[0] = keys.x / kTcKeys;
    R.hi[0] = min(q0 + kTcQ - 1, T - 1) / kTcKeys;
    if (q0 + kTcQ < T) {
      R.lo[1] = keys.y / kTcKeys;
      R.hi[1] = min(q0 + 2 * kTcQ - 1, T - 1) / kTcKeys;
    } else {
      R.lo[1] = 1;
      R.hi[1] = 0;
    }
    R.u_hi = max(R.hi[0], R.hi[1]);
    return R;
  };
  auto wait = [&](uint32_t bar, uint32_t parity) { return mtp::wait_phase(bar, parity, abort_flag, err); };

  if (warp == 8) {
    // ---------------- TMA producers: lane 0 Q and K, lane 1 V ----------------
    if (lane < 2) {
      const bool kside = lane == 0;
      const int stages = kside ? C::kKStages : C::kVStages;
      uint32_t g = 0, issued = 0;
      int q_loads = 0;
      bool ok = true;
      // lane 0 claims item tl: with two Q buffers when item tl - 2 has released its Q (a CTA
      // then holds at most about one claimed item it has not started); with one, as soon as
      // item tl - 1 is published (its Q load waits for the previous item, so a later claim
      // would add the claim's latency to that wait)
      int t_next = static_cast<int>(blockIdx.x);
      for (int tl = 0; ok; ++tl) {
        const int slot = tl % C::kRing;
        const int qi = tl % C::kQBufs, qu = tl / C::kQBufs;
        int4 it;
        if (kside) {
          if (C::kQBufs > 1) {
            if (qu > 0 && !wait(q_empty(qi), (qu - 1) & 1)) { ok = false; break; }
            if (tl > 0) t_next = static_cast<int>(gridDim.x) + atomicAdd(work_ctr, 1);
          }
          const int t = t_next;
          const int2 k2 = t < n_items ? first_keys(t) : make_int2(0, 0);
          it = make_int4(t < n_items ? t : -1, k2.x, k2.y, 0);
          if (tl >= C::kRing && !wait(it_empty(slot), (tl / C::kRing - 1) & 1)) { ok = false; break; }
          items[slot] = it;
          mtp::mbar_arrive1(it_full(slot));
          if (it.x < 0) break;
          if (C::kQBufs == 1) {
            t_next = static_cast<int>(gridDim.x) + atomicAdd(work_ctr, 1);
            if (qu > 0 && !wait(q_empty(qi), (qu - 1) & 1)) { ok = false; break; }
          }
        } else {
          if (!wait(it_full(slot), (tl / C::kRing) & 1)) { ok = false; break; }
          it = items[slot];
          mtp::mbar_arrive1(it_empty(slot));
          if (it.x < 0) break;
        }
        int b, h, q0;
        coords(it.x, b, h, q0);
        const Ranges R = ranges(q0, make_int2(it.y, it.z));
        if (kside) {
          const bool has_b = R.hi[1] >= R.lo[1];
          mtp::mbar_expect_tx(q_full(qi), (has_b ? 2 : 1) * C::kQBytes);
          for (int x = 0; x < (has_b ? 2 : 1); ++x)
            for (int c = 0; c < C::kChunks; ++c)
              mtp::tma_tile_2d(sQ + (qi * 2 + x) * C::kQBytes + c * C::kTileBytes, &tm128, h * HD + 64 * c,
                               b * T + q0 + x * kTcQ, q_full(qi));
          ++q_loads;
        }
        for (int j = R.lo[0]; j <= R.u_hi; ++j, ++g) {
          const int st = static_cast<int>(g % stages);
          const uint32_t use = g / stages;
          const int row0 = b * T + j * kTcKeys;
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
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc_s = mtp::idesc_bf16_f32(kTcQ, kTcKeys, 0);
      constexpr uint32_t idesc_o = mtp::idesc_bf16_f32(kTcQ, HD, 2);  // V read MN-major, P from TMEM
      uint32_t g = 0;                  // union key blocks consumed (K/V ring position)
      uint32_t ns[2] = {0u, 0u};       // S products issued per tile (= P V products after the block)
      uint32_t no[2] = {0u, 0u};       // work items per tile whose output the softmax has read
      bool ok = true, any = false;
      for (int tl = 0; ok; ++tl) {
        const int slot = tl % C::kRing;
        if (!wait(it_full(slot), (tl / C::kRing) & 1)) { ok = false; break; }
        const int4 it = items[slot];
        mtp::mbar_arrive1(it_empty(slot));
        if (it.x < 0) break;
        int b, h, q0;
        coords(it.x, b, h, q0);
        const Ranges R = ranges(q0, make_int2(it.y, it.z));
        auto active = [&](int x, int j) { return j >= R.lo[x] && j <= R.hi[x]; };
        const int qi = tl % C::kQBufs;
        if (!wait(q_full(qi), (tl / C::kQBufs) & 1)) { ok = false; break; }
        // S_x(j) = Q_x K_j^T into tile x's S columns; its previous P was read by a P V issued before
        auto issue_s = [&](int x, uint32_t gu) -> bool {
          if (ns[x] > 0 && !wait(p_full(x), (ns[x] - 1) & 1)) return false;
          mtp::tc_fence_after();
          const uint32_t sQt = sQ + (qi * 2 + x) * C::kQBytes;
          const uint32_t sKt = sK + (gu % C::kKStages) * C::kKBytes;
#pragma unroll
          for (int k = 0; k < HD / 16; ++k) {
            const uint32_t off = (k >> 2) * C::kTileBytes + (k & 3) * 32;
            mtp::umma_bf16_ss(tmem + 128u * x, mtp::sdesc_k_sw128(sQt + off), mtp::sdesc_k_sw128(sKt + off), idesc_s,
                              k > 0);
          }
          mtp::umma_commit(s_full(x));
          ++ns[x];
          any = true;
          return true;
        };
        bool first_pv[2] = {true, true};
        const uint32_t g0 = g;
        // the first block's S products
        if (!wait(k_full(g0 % C::kKStages), (g0 / C::kKStages) & 1)) { ok = false; break; }
        for (int x = 0; x < 2 && ok; ++x)
          if (active(x, R.lo[0]) && !issue_s(x, g0)) ok = false;
        if (!ok) break;
        mtp::umma_commit(k_empty(g0 % C::kKStages));
        if (R.lo[0] == R.u_hi) mtp::umma_commit(q_empty(qi));
        for (int j = R.lo[0]; j <= R.u_hi && ok; ++j) {
          const uint32_t gu = g0 + static_cast<uint32_t>(j - R.lo[0]);
          const int vs = static_cast<int>(gu % C::kVStages);
          if (!wait(v_full(vs), (gu / C::kVStages) & 1)) { ok = false; break; }
          bool k_next_ready = false;
          for (int x = 0; x < 2; ++x) {
            if (active(x, j)) {  // O_x (+)= P_x(j) V_j, P_x in tile x's S columns
              const uint32_t n = ns[x] - 1;  // this block's S index of tile x
              if (!wait(p_full(x), n & 1)) { ok = false; break; }
              if (first_pv[x] && no[x] > 0 && !wait(o_free(x), (no[x] - 1) & 1)) { ok = false; break; }
              mtp::tc_fence_after();
              const uint32_t sVt = sV + vs * C::kVBytes;
#pragma unroll
              for (int k = 0; k < kTcKeys / 16; ++k) {
                const uint32_t bv = sVt + (k >> 2) * (C::kChunks * 8192) + (k & 3) * 2048;
                mtp::umma_bf16_ts(tmem + C::kColO0 + HD * x, tmem + 128u * x + 8u * k, mtp::sdesc_mn_sw128(bv),
                                  idesc_o, (!first_pv[x] || k > 0) ? 1u : 0u);
              }
              mtp::umma_commit(pv_done(x));
              first_pv[x] = false;
            }
            if (j < R.u_hi && active(x, j + 1)) {  // S_x(j+1)
              if (!k_next_ready) {
                if (!wait(k_full((gu + 1) % C::kKStages), ((gu + 1) / C::kKStages) & 1)) { ok = false; break; }
                k_next_ready = true;
              }
              if (!issue_s(x, gu + 1)) { ok = false; break; }
            }
          }
          if (!ok) break;
          mtp::umma_commit(v_empty(vs));
          if (k_next_ready) {
            mtp::umma_commit(k_empty((gu + 1) % C::kKStages));
            if (j + 1 == R.u_hi) mtp::umma_commit(q_empty(qi));
          }
        }
        g = g0 + static_cast<uint32_t>(R.u_hi - R.lo[0] + 1);
        for (int x = 0; x < 2; ++x)
          if (R.hi[x] >= R.lo[x]) ++no[x];
      }
      // every issued MMA has completed before TMEM is freed
      if (any) {
        mtp::umma_commit(drain_bar);
        mtp::wait_drain(drain_bar, 0, kWaitLimitCycles);
      }
    }
  } else {
    // ---------------- softmax warpgroups: tile x = warp / 4, one query row per thread ----------------
    const int x = warp >> 2;
    const int row = threadIdx.x - 128 * x;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t colS = 128u * x, colO = C::kColO0 + HD * x;
    auto wwait = [&](uint32_t bar, uint32_t parity) { return __all_sync(0xffffffffu, wait(bar, parity)); };
    uint32_t n = 0;  // S products of this tile consumed
    for (int tl = 0;; ++tl) {
      const int slot = tl % C::kRing;
      if (!wwait(it_full(slot), (tl / C::kRing) & 1)) break;
      const int4 it = items[slot];
      __syncwarp();
      if (lane == 0) mtp::mbar_arrive1(it_empty(slot));
      if (it.x < 0) break;
      int b, h, q0;
      coords(it.x, b, h, q0);
      const Ranges R = ranges(q0, make_int2(it.y, it.z));
      if (R.hi[x] < R.lo[x]) continue;  // tile B past the end of the row
      const int q = q0 + kTcQ * x + row;
      const bool live = q < T;
      // this row's segment start (first used after the item's first scores arrive)
      const int st_row = live ? static_cast<int>(seg_start[static_cast<size_t>(b) * T + q]) : q;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = R.lo[x]; j <= R.hi[x]; ++j, ++n) {
        if (!wwait(s_full(x), n & 1)) { ok = false; break; }
        mtp::tc_fence_after();
        float sc[kTcKeys];
        {
          float (&lo)[64] = *reinterpret_cast<float (*)[64]>(&sc[0]);
          float (&hi)[64] = *reinterpret_cast<float (*)[64]>(&sc[64]);
          mtp::tmem_ld64(lane_base + colS, lo);
          mtp::tmem_ld64(lane_base + colS + 64, hi);
        }
        const int key0 = j * kTcKeys;
        if (!(key0 >= st_row && key0 + kTcKeys - 1 <= q)) {  // a block the row sees only in part
#pragma unroll
          for (int i = 0; i < kTcKeys; ++i) {
            const int key = key0 + i;
            if (!(key >= st_row && key <= q)) sc[i] = -INFINITY;
          }
        }
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
        float rs8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rs8[i] = 0.f;
#pragma unroll
        for (int i = 0; i < kTcKeys / 2; ++i) {  // P pairs packed in place: sc[i] holds keys 2i, 2i+1
          const float a = ex2_approx(fmaf(sc[2 * i], scale_log2, neg_use));
          const float bb = ex2_approx(fmaf(sc[2 * i + 1], scale_log2, neg_use));
          rs8[i & 7] += a + bb;
          sc[i] = __uint_as_float(pack2_bf16(a, bb));
        }
        if (__any_sync(0xffffffffu, rescale)) {  // O holds this item's earlier P V: wait for the last one
          if (!wwait(pv_done(x), (n - 1) & 1)) { ok = false; break; }
          mtp::tc_fence_after();
          const float alpha = rescale ? ex2_approx(m - m_new) : 1.f;
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            float o[32];
            mtp::tmem_ld32(lane_base + colO + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            mtp::tmem_st32(lane_base + colO + 32 * c, o);
          }
          l *= alpha;
        }
        m = m_new;
        l += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        // P into the first 64 columns of this tile's S (the scores are in registers now; the
        // previous block's P V completed before this block's S did)
        {
          float (&p0)[32] = *reinterpret_cast<float (*)[32]>(&sc[0]);
          float (&p1)[32] = *reinterpret_cast<float (*)[32]>(&sc[32]);
          mtp::tmem_st32(lane_base + colS, p0);
          mtp::tmem_st32(lane_base + colS + 32, p1);
        }
        mtp::tc_fence_before();
        mtp::mbar_arrive1(p_full(x));
      }
      if (!ok) break;
      if (!wwait(pv_done(x), (n - 1) & 1)) break;  // the item's last P V
      mtp::tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (live && lse2_out) lse2_out[(static_cast<size_t>(b) * T + q) * H + h] = m + log2f(l);
      __nv_bfloat16* orow = out + (static_cast<size_t>(b) * T + q) * d + h * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        mtp::tmem_ld32(lane_base + colO + 32 * c, o);
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
      mtp::mbar_arrive1(o_free(x));
    }
  }
  mtp::tc_fence_before();
  __syncthreads();
  mtp::tc_fence_after();
  if (warp == 9) mtp::tmem_free_cols(tmem, 512);
}

template <int HD>
mtp_status attn_tc2_launch(const __nv_bfloat16* qkv, __nv_bfloat16* out, const int32_t* seg_start, int B, int T,
                           int H, float scale_log2, float* lse2_out, int* work_ctr, cudaStream_t stream) {
  using C = Tc2Attn<HD>;
  static PerDevice attr;
  if (!smem_limit(attr, attn_tc2_kernel<HD>, C::kSmemBytes)) return MTP_ERR_CUDA;
  if (!aligned16(qkv) || !aligned16(out)) return MTP_ERR_ALIGNMENT;
  if (!work_ctr) return MTP_ERR_INVALID_ARG;
  const int d = H * HD;
  const uint64_t rows = static_cast<uint64_t>(B) * T;
  if (rows > 0x7FFFFFFFull) return MTP_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
  CUtensorMap m128, m64;
  if (!tensor_map_bf16_2d(&m128, qkv, rows, 3 * d, 3 * d, 64, 128, true) ||
      !tensor_map_bf16_2d(&m64, qkv, rows, 3 * d, 3 * d, 64, 64, true))
    return MTP_ERR_CUDA;
  const long long n_items = static_cast<long long>((T + 2 * kTcQ - 1) / (2 * kTcQ)) * H * B;
  if (n_items > 0x7FFFFFFFll) return MTP_ERR_UNSUPPORTED;
  const int sms = sm_count_current();
  const int grid = static_cast<int>(n_items < sms ? n_items : sms);
  // the QKV projection before it releases this launch when its CTAs start their last tiles
  MTP_CUDA_TRY(launch_pdl(attn_tc2_kernel<HD>, dim3(grid), dim3(kT2Threads), C::kSmemBytes, stream, m128, m64, out,
                          seg_start, B, T, H, scale_log2, lse2_out, work_ctr));
  note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}


}  // namespace

mtp_status attn_launch(int dtype, const void* qkv, void* out, const int32_t* seg_start, int B, int T, int H,
                       int hd, cudaStream_t stream, float* lse2_out, int* work_ctr) {
  if (B <= 0 || T <= 0) return MTP_OK;
  if (dtype == MTP_BF16) {
    const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
    if (hd == 64)
      return attn_tc2_launch<64>(static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(out), seg_start,
                                B, T, H, scale_log2, lse2_out, work_ctr, stream);
    if (hd == 128)
      return attn_tc2_launch<128>(static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(out),
                                 seg_start, B, T, H, scale_log2, lse2_out, work_ctr, stream);
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
