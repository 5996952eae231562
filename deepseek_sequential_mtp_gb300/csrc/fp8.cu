// FP8 block-scaled weight GEMM for decode shapes (sm_103a, tcgen05).
//
//   out[r, n] += Σ_k x̃[r, k] · W[n, k],   W[n, k] = e4m3(q[n, k]) · s[n / 128, k / 128]
//
// Checkpoint weights are stored as FP8 with block scales while the runtime
// picks the compute representation ("M7.6 - DeepSeek MTP: Sequential Modules,
// Teacher Forcing, and Speculative Runtime" §0x03C, the layered numerical
// contract).  Weights are used as stored (e4m3 codes straight from HBM into
// the tensor cores, the block scale applied to each k-block's fp32 partial).
// The activations enter as e4m3 too, but in two terms: per token and 128-wide
// k-tile, x̃ = 2^E (hi + lo) with 2^E the smallest power of two that brings
// max|x| within 448, hi = RNE_e4m3(x / 2^E), lo = RNE_e4m3(x / 2^E - hi).  A
// bf16 value has 8 significant bits, so x̃ = x for every element of magnitude
// >= 2^(E-2); smaller ones differ by at most 2^(E-10) (below 2^-17.8 of the
// tile's largest element).
//
// Why this shape: a decode GEMM has <= 32 tokens, and a tcgen05 MMA with the
// tokens as N = 32 costs about as much issue time as a full one while covering
// only 128 x 16 weights; with the weights as N = 256 and e4m3 operands (K = 32)
// one instruction covers 256 x 32 weights.  The M = 128 side holds the
// activation terms: rows 0-31 hi, 32-63 lo, 64-127 the same again, so all four
// TMEM lane quadrants carry data and the epilogue spreads over eight warps.
//
// Persistent CTA per SM, 10 warps:
//   warp 0      TMA producer: per (row tile, k-block) the e4m3 weight box
//               [256 rows x 128 bytes] and the split-activation box [64 rows x
//               128 bytes] twice (128-byte swizzle) into a 4-stage ring.
//   warp 1      allocates 512 TMEM columns (two 256-column accumulators); one
//               thread issues tcgen05.mma.cta_group::1.kind::f8f6f4, M = 128,
//               N = 256, K = 32, four per k-block, a fresh accumulator per
//               k-block (its scale differs).
//   warps 2-9   epilogue: warp w reads TMEM lane quadrant w % 4 (term hi or
//               lo, tokens 0-31) and 64 of the 256 columns; scales the
//               partial by s[n-block, kb] * 2^E[token, kb] and accumulates in
//               registers; at the end of a row tile's run of k-blocks adds it
//               into out with fp32 atomics (hi and lo terms separately),
//               transposed through shared memory so each atomic instruction
//               covers 32 consecutive floats of one token's row.
// Work: the (row tile, k-block) pairs of all segments in order, cut into one
// contiguous range per CTA, so every SM streams the same number of weight
// bytes.  Every wait is bounded; on expiry the CTA sets MTP_DEVERR_TIMEOUT,
// every role leaves its loop, the producer waits for its copies and warp 1
// for its MMAs before TMEM is freed.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "fp8.cuh"
#include "gemm_tc.cuh"
#include "mbarrier.cuh"
#include "tcgen05.cuh"

MTP_DEFINE_ERROR_WORD(mtp_take_errors_fp8)

namespace mtp {
namespace {

constexpr int kN = 256;                            // weight rows per tile (MMA N)
constexpr int kKb = 128;                           // k per block: one weight scale, one 128-byte e4m3 row
constexpr int kTok = 32;                           // tokens; split rows: hi 0-31, lo 32-63
constexpr int kStages = 4;
constexpr int kWBytes = kN * kKb;                  // 32 KB e4m3 weight box
constexpr int kAHalf = 2 * kTok * kKb;             // 8 KB: one copy of the split-activation box
constexpr int kStageBytes = kWBytes + 2 * kAHalf;  // 48 KB
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kTmemCols = 512;                     // accumulator b: columns [256 b, 256 b + 256)
constexpr int kBarriers = 2 * kStages + 2 + 2 + 1;
constexpr int kBarBytes = 256;                     // barriers, the TMEM address and the abort flag
constexpr int kFlushLd = 33;                       // per-warp flush tile [32 tokens][33] fp32 (padded)
constexpr int kFlushBytes = kEpiWarps * 32 * kFlushLd * 4;
constexpr int kSmemBytes = kStages * kStageBytes + kFlushBytes + 1024 + kBarBytes;
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(kBarriers * 8 + 8 <= kBarBytes, "barrier block");

struct Seg {
  const float* scale;
  float* out;
  int n, tiles, sld;  // rows, 256-row tiles, scale row stride (= ceil(K / 128))
  int first;          // index of the segment's first (row tile, k-block) pair
};
struct Args {
  Seg seg[3];
  const float* xscale;  // [nkb, 32]: 2^E per (k-block, token)
  int nseg, K, nkb, R, ldo, total;
};

// D[tmem] (+)= A[smem] · B[smem]^T, kind::f8f6f4
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// kind::f8f6f4 instruction descriptor: D fp32 (bits 4-5 = 1), A and B e4m3
// (format 0 at bits 7-9 and 10-12), both K-major, N >> 3 at 17, M >> 4 at 24.
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(kN >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);

__device__ __forceinline__ void decode(const Args& P, int i, int& sg, int& nt, int& kb) {
  sg = 0;
  if (P.nseg > 1 && i >= P.seg[1].first) sg = 1;
  if (P.nseg > 2 && i >= P.seg[2].first) sg = 2;
  const int j = i - P.seg[sg].first;
  nt = j / P.nkb;
  kb = j - nt * P.nkb;
}

__global__ void __launch_bounds__(kThreads, 1)
fp8w_gemm_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                 const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmA,
                 const __grid_constant__ Args P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  float* flush_tiles = reinterpret_cast<float*>(smem + kStages * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kFlushBytes);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto dfull = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto dempty = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  const uint32_t final_bar = bar0 + 8u * (2 * kStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBarriers);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(dfull(b), 1);
      mbar_init(dempty(b), kEpiWarps);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int lo = static_cast<int>((static_cast<long long>(P.total) * blockIdx.x) / gridDim.x);
  const int hi = static_cast<int>((static_cast<long long>(P.total) * (blockIdx.x + 1)) / gridDim.x);
  const int n_local = hi - lo;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      bool issued[kStages];
      uint32_t armed[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) {
        issued[s] = false;
        armed[s] = 0;
      }
      for (int l = 0; l < n_local; ++l) {
        const int s = l % kStages;
        const uint32_t ph = (l / kStages) & 1;
        if (!wait_phase(empty(s), ph ^ 1u, abort_flag, &g_mtp_error_word)) break;
        int sg, nt, kb;
        decode(P, lo + l, sg, nt, kb);
        const uint32_t sw = base + s * kStageBytes, sa = sw + kWBytes;
        const CUtensorMap* wm = sg == 0 ? &tmW0 : (sg == 1 ? &tmW1 : &tmW2);
        mbar_expect_tx(full(s), kStageBytes);
        tma_tile_2d(sw, wm, kb * kKb, nt * kN, full(s));
        tma_tile_2d(sa, &tmA, kb * kKb, 0, full(s));
        tma_tile_2d(sa + kAHalf, &tmA, kb * kKb, 0, full(s));
        issued[s] = true;
        armed[s] = ph;
      }
      if (*abort_flag) {  // every copy this thread started lands before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) wait_drain(full(s), armed[s], 40000000ll);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      for (int l = 0; l < n_local; ++l) {
        const int s = l % kStages, b = l & 1;
        if (!wait_phase(full(s), (l / kStages) & 1, abort_flag, &g_mtp_error_word)) break;
        if (!wait_phase(dempty(b), ((l >> 1) & 1) ^ 1u, abort_flag, &g_mtp_error_word)) break;
        tc_fence_after();
        const uint32_t sw = base + s * kStageBytes;
        const uint64_t adesc = sdesc_k_sw128(sw + kWBytes), bdesc = sdesc_k_sw128(sw);
        const uint32_t d = tmem + 256 * b;
#pragma unroll
        for (int kk = 0; kk < kKb / 32; ++kk) umma_f8(d, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, kk ? 1u : 0u);
        umma_commit(empty(s));
        umma_commit(dfull(b));
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int quad = warp & 3;        // TMEM lanes 32 quad.. : term (quad & 1), tokens = lane
    const int sub = (warp - 2) >> 2;  // the two warps of a quadrant split its 128 columns
    const int col0 = 128 * (quad >> 1) + 64 * sub;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * quad) << 16) + col0;
    float acc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.f;
    // the scale of a pair, fetched one pair ahead: weight block of columns col0.. times 2^E of the token
    auto pair_scale = [&](int sg, int nt, int kb) {
      const Seg& S = P.seg[sg];
      const int nb = (nt * kN + col0) / 128;
      return __ldg(S.scale + static_cast<size_t>(nb) * S.sld + kb) * __ldg(P.xscale + kb * kTok + lane);
    };
    int sg = 0, nt = 0, kb = 0;
    float sc = 0.f;
    if (n_local > 0) {
      decode(P, lo, sg, nt, kb);
      if (nt * kN + col0 < P.seg[sg].n) sc = pair_scale(sg, nt, kb);
    }
    for (int l = 0; l < n_local; ++l) {
      const int b = l & 1;
      int sg2 = sg, nt2 = nt, kb2 = kb + 1;
      bool flush = l + 1 == n_local;
      if (kb2 == P.nkb) {
        flush = true;
        if (l + 1 < n_local) decode(P, lo + l + 1, sg2, nt2, kb2);
      }
      float sc2 = 0.f;
      if (l + 1 < n_local && nt2 * kN + col0 < P.seg[sg2].n) sc2 = pair_scale(sg2, nt2, kb2);
      const bool ok = wait_phase(dfull(b), (l >> 1) & 1, abort_flag, &g_mtp_error_word);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      float v[32];
      tmem_ld32(taddr + 256 * b, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = fmaf(sc, v[i], acc[i]);
      tmem_ld32(taddr + 256 * b + 32, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(dempty(b));
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[32 + i] = fmaf(sc, v[i], acc[32 + i]);
      if (flush) {
        // transpose 32 columns at a time through shared memory so that each
        // atomic instruction adds 32 consecutive floats of one token's row
        const Seg& S = P.seg[sg];
        const int n0 = nt * kN + col0;
        float* tile = flush_tiles + (warp - 2) * 32 * kFlushLd;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 32; ++i) tile[lane * kFlushLd + i] = acc[32 * h + i];
          __syncwarp();
          const int n = n0 + 32 * h + lane;
          if (n < S.n)
            for (int t = 0; t < P.R; ++t) atomicAdd(S.out + static_cast<size_t>(t) * P.ldo + n, tile[t * kFlushLd + lane]);
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.f;
      }
      sg = sg2;
      nt = nt2;
      kb = kb2;
      sc = sc2;
    }
  }

  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {  // every MMA of this CTA has completed before TMEM is freed
      umma_commit(final_bar);
      wait_drain(final_bar, 0, 40000000ll);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Split activations: x [R, K] bf16 -> a [64, K] e4m3 codes (rows 0-31 hi,
// 32-63 lo; tokens >= R zero) and xscale [nkb, 32] = 2^E.  One warp per
// (token, k-block), four elements a lane.
__global__ void __launch_bounds__(256) split_act_kernel(const __nv_bfloat16* __restrict__ x, int R, int K, int nkb,
                                                        uint8_t* __restrict__ a, float* __restrict__ xscale) {
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= kTok * nkb) return;
  const int t = w % kTok, kb = w / kTok;
  const int k0 = kb * kKb + 4 * lane;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (t < R) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (k0 + i < K) v[i] = __bfloat162float(x[static_cast<size_t>(t) * K + k0 + i]);
  }
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  amax = warp_max(amax);
  // smallest E with amax <= 448 2^E: amax = m 2^e, m in [0.5, 1); 448 = 0.875 2^9
  int E = 0;
  if (amax > 0.f) {
    int e;
    const float m = frexpf(amax, &e);
    E = m <= 0.875f ? e - 9 : e - 8;
  }
  uint32_t hw = 0, lw = 0;
#pragma unroll
  for (int i = 0; i < 4; i += 2) {
    const float2 s = make_float2(ldexpf(v[i], -E), ldexpf(v[i + 1], -E));
    const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(s, __NV_SATFINITE, __NV_E4M3);
    __half2 hh;
    hh = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
    const float2 hf = __half22float2(hh);
    const float2 r = make_float2(s.x - hf.x, s.y - hf.y);  // exact: both are multiples of s's last bit
    const __nv_fp8x2_storage_t lo2 = __nv_cvt_float2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3);
    hw |= static_cast<uint32_t>(h) << (8 * i);
    lw |= static_cast<uint32_t>(lo2) << (8 * i);
  }
  if (k0 + 4 <= K) {
    *reinterpret_cast<uint32_t*>(a + static_cast<size_t>(t) * K + k0) = hw;
    *reinterpret_cast<uint32_t*>(a + static_cast<size_t>(kTok + t) * K + k0) = lw;
  } else {
    for (int i = 0; i < 4 && k0 + i < K; ++i) {
      a[static_cast<size_t>(t) * K + k0 + i] = static_cast<uint8_t>(hw >> (8 * i));
      a[static_cast<size_t>(kTok + t) * K + k0 + i] = static_cast<uint8_t>(lw >> (8 * i));
    }
  }
  if (lane == 0) xscale[kb * kTok + t] = ldexpf(1.0f, E);
}

int sm_count() {
  return sm_count_current();
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t fp8w_workspace_bytes(int K) {
  if (K <= 0) return 0;
  const size_t nkb = (K + kKb - 1) / kKb;
  return align256(static_cast<size_t>(2 * kTok) * K) + align256(nkb * kTok * 4);
}

mtp_status fp8w_gemm_launch(const Fp8Seg* segs, int nseg, int K, const __nv_bfloat16* x, int R, int ldo, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  if (!segs || nseg < 1 || nseg > 3 || !x || !ws) return MTP_ERR_INVALID_ARG;
  if (K <= 0 || R <= 0 || R > kTok) return MTP_ERR_SHAPE;
  if (K % 16) return MTP_ERR_ALIGNMENT;  // 16-byte rows for the e4m3 tensor maps
  if (!aligned16(ws)) return MTP_ERR_ALIGNMENT;
  if (ws_bytes < fp8w_workspace_bytes(K)) return MTP_ERR_WORKSPACE;
  Args P{};
  P.nseg = nseg;
  P.K = K;
  P.nkb = (K + kKb - 1) / kKb;
  P.R = R;
  P.ldo = ldo;
  uint8_t* a = static_cast<uint8_t*>(ws);
  float* xs = reinterpret_cast<float*>(a + align256(static_cast<size_t>(2 * kTok) * K));
  P.xscale = xs;
  CUtensorMap tw[3], ta;
  long long total = 0;
  for (int i = 0; i < nseg; ++i) {
    const Fp8Seg& s = segs[i];
    if (!s.q || !s.scale || !s.out || s.n <= 0) return MTP_ERR_INVALID_ARG;
    if (ldo < s.n) return MTP_ERR_SHAPE;
    if (!aligned16(s.q) || (reinterpret_cast<uintptr_t>(s.scale) & 3u) || (reinterpret_cast<uintptr_t>(s.out) & 3u))
      return MTP_ERR_ALIGNMENT;
    if (!tensor_map_u8_2d(&tw[i], s.q, s.n, K, K, kKb, kN)) return MTP_ERR_CUDA;
    P.seg[i].scale = s.scale;
    P.seg[i].out = s.out;
    P.seg[i].n = s.n;
    P.seg[i].tiles = (s.n + kN - 1) / kN;
    P.seg[i].sld = P.nkb;
    P.seg[i].first = static_cast<int>(total);
    total += static_cast<long long>(P.seg[i].tiles) * P.nkb;
  }
  if (total > 0x7FFFFFFFll) return MTP_ERR_UNSUPPORTED;
  for (int i = nseg; i < 3; ++i) tw[i] = tw[0];
  if (!tensor_map_u8_2d(&ta, a, 2 * kTok, K, K, kKb, 2 * kTok)) return MTP_ERR_CUDA;
  P.total = static_cast<int>(total);
  static PerDevice attr;
  if (!smem_limit(attr, fp8w_gemm_kernel, kSmemBytes)) return MTP_ERR_CUDA;
  const int warps = kTok * P.nkb;
  split_act_kernel<<<(warps + 7) / 8, 256, 0, stream>>>(x, R, K, P.nkb, a, xs);
  note_launch();
  const int grid = static_cast<int>(total < sm_count() ? total : sm_count());
  fp8w_gemm_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tw[0], tw[1], tw[2], ta, P);
  note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

}  // namespace mtp

extern "C" size_t mtp_gemm_fp8w_workspace_bytes(int K) { return mtp::fp8w_workspace_bytes(K); }

extern "C" mtp_status mtp_gemm_fp8w(int R, int N, int K, const void* x, const void* wq, const float* scale,
                                    float* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!x || !wq || !scale || !out) return MTP_ERR_INVALID_ARG;
  mtp::Fp8Seg s;
  s.q = static_cast<const uint8_t*>(wq);
  s.scale = scale;
  s.n = N;
  s.out = out;
  return mtp::fp8w_gemm_launch(&s, 1, K, static_cast<const __nv_bfloat16*>(x), R, N, ws, ws_bytes, stream);
}
