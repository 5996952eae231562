// bf16 decode-shaped GEMM (sm_103a, tcgen05): the draft step's linear maps.
//
//   out[r, n] += Σ_k x[r, k] · W[n, k]      x: R <= 32 tokens, W: [n, K] bf16
//
// A tcgen05 MMA with the tokens as N = 32 costs about as much issue time as a
// full-width one while covering only 128 x 16 weights, so here the weights sit
// on the N = 256 side and one instruction covers 256 x 16 of them.  The M = 128
// side holds the token rows four times (rows 32q + t = token t for q = 0..3),
// so every TMEM lane quadrant carries the result and four epilogue warps each
// take 64 of the 256 columns.
//
// Persistent CTA per SM, 6 warps:
//   warp 0      TMA producer: per (256-row tile, 64-wide k-block) the weight
//               box [256 rows x 64] and the token box [32 x 64] four times
//               (128-byte swizzle) into a 4-stage ring.
//   warp 1      allocates 512 TMEM columns (two 256-column accumulators); one
//               thread issues tcgen05.mma.cta_group::1.kind::f16, M = 128,
//               N = 256, K = 16, four per k-block, accumulating over the
//               CTA's run of k-blocks of one tile.
//   warps 2-5   epilogue: at the end of a tile's run, read the accumulator
//               (lanes = tokens, 64 columns a warp) and add it into out with
//               fp32 atomics, transposed through shared memory so that each
//               atomic instruction covers 32 consecutive floats of one row.
// Work: the (tile, k-block) pairs of all segments in order, cut into one
// contiguous range per CTA (stream-K), so every SM streams the same number
// of weight bytes; a tile split between CTAs is summed by the atomics.
// Every wait is bounded; on expiry the CTA sets MTP_DEVERR_TIMEOUT, every
// role leaves its loop, the producer waits for its copies and warp 1 for its
// MMAs before TMEM is freed.
#include <cuda.h>

#include "decode_gemm.cuh"
#include "gemm_tc.cuh"
#include "mbarrier.cuh"
#include "tcgen05.cuh"

MTP_DEFINE_ERROR_WORD(mtp_take_errors_dgemm)

namespace mtp {
namespace {

constexpr int kN = 256;                            // weight rows per tile (MMA N)
constexpr int kBK = 64;                            // k per block: 128-byte bf16 rows
constexpr int kTok = 32;
constexpr int kStages = 4;
constexpr int kWBytes = kN * kBK * 2;              // 32 KB weight box
constexpr int kXBox = kTok * kBK * 2;              // 4 KB token box
constexpr int kStageBytes = kWBytes + 4 * kXBox;   // 48 KB
constexpr int kThreads = 6 * 32;
constexpr int kTmemCols = 512;                     // accumulator b: columns [256 b, 256 b + 256)
constexpr int kBarriers = 2 * kStages + 2 + 2 + 1;
constexpr int kBarBytes = 256;
constexpr int kFlushLd = 33;
constexpr int kFlushBytes = 4 * 32 * kFlushLd * 4;
constexpr int kSmemBytes = kStages * kStageBytes + kFlushBytes + 1024 + kBarBytes;
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(kBarriers * 8 + 8 <= kBarBytes, "barrier block");
// kind::f16 instruction descriptor: D fp32, A and B bf16, K-major, N = 256, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kN >> 3) << 17) |
                            (static_cast<uint32_t>(128 >> 4) << 24);

struct Seg {
  float* out;
  int n, tiles, first;
};
struct Args {
  Seg seg[3];
  int nseg, nkb, R, ldo, total;
};

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void decode(const Args& P, int i, int& sg, int& nt, int& kb) {
  sg = 0;
  if (P.nseg > 1 && i >= P.seg[1].first) sg = 1;
  if (P.nseg > 2 && i >= P.seg[2].first) sg = 2;
  const int j = i - P.seg[sg].first;
  nt = j / P.nkb;
  kb = j - nt * P.nkb;
}

__global__ void __launch_bounds__(kThreads, 1)
dgemm_bf16_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                  const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmX,
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
      mbar_init(dempty(b), 4);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc_cols(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int lo = static_cast<int>((static_cast<long long>(P.total) * blockIdx.x) / gridDim.x);
  const int hi = static_cast<int>((static_cast<long long>(P.total) * (blockIdx.x + 1)) / gridDim.x);
  const int n_local = hi - lo;
  // does local pair l end its tile's run (the last pair of the range or of the tile)?
  auto run_ends = [&](int l, int kb) { return l + 1 == n_local || kb + 1 == P.nkb; };

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
        const uint32_t sw = base + s * kStageBytes, sx = sw + kWBytes;
        const CUtensorMap* wm = sg == 0 ? &tmW0 : (sg == 1 ? &tmW1 : &tmW2);
        mbar_expect_tx(full(s), kStageBytes);
        tma_tile_2d(sw, wm, kb * kBK, nt * kN, full(s));
#pragma unroll
        for (int q = 0; q < 4; ++q) tma_tile_2d(sx + q * kXBox, &tmX, kb * kBK, 0, full(s));
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
      int run = 0;        // runs (tiles) started so far
      bool fresh = true;  // the next k-block starts a run
      for (int l = 0; l < n_local; ++l) {
        int sg, nt, kb;
        decode(P, lo + l, sg, nt, kb);
        const int s = l % kStages, b = run & 1;
        if (fresh && !wait_phase(dempty(b), ((run >> 1) & 1) ^ 1u, abort_flag, &g_mtp_error_word)) break;
        if (!wait_phase(full(s), (l / kStages) & 1, abort_flag, &g_mtp_error_word)) break;
        tc_fence_after();
        const uint32_t sw = base + s * kStageBytes;
        const uint64_t adesc = sdesc_k_sw128(sw + kWBytes), bdesc = sdesc_k_sw128(sw);
        const uint32_t d = tmem + 256 * b;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) umma_f16(d, adesc + 2 * kk, bdesc + 2 * kk, (fresh && kk == 0) ? 0u : 1u);
        umma_commit(empty(s));
        fresh = run_ends(l, kb);
        if (fresh) {
          umma_commit(dfull(b));
          ++run;
        }
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int quad = warp & 3;  // TMEM lanes 32 quad.. hold tokens 0..31; this warp takes columns 64 quad..
    const int col0 = 64 * quad;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * quad) << 16) + col0;
    float* tile = flush_tiles + (warp - 2) * 32 * kFlushLd;
    int run = 0;
    for (int l = 0; l < n_local; ++l) {
      int sg, nt, kb;
      decode(P, lo + l, sg, nt, kb);
      if (!run_ends(l, kb)) continue;
      const int b = run & 1;
      const bool ok = wait_phase(dfull(b), (run >> 1) & 1, abort_flag, &g_mtp_error_word);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      float v[2][32];
      tmem_ld32(taddr + 256 * b, v[0]);
      tmem_ld32(taddr + 256 * b + 32, v[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(dempty(b));
      const Seg& S = P.seg[sg];
      const int n0 = nt * kN + col0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32; ++i) tile[lane * kFlushLd + i] = v[h][i];
        __syncwarp();
        const int n = n0 + 32 * h + lane;
        if (n < S.n)
          for (int t = 0; t < P.R; ++t) atomicAdd(S.out + static_cast<size_t>(t) * P.ldo + n, tile[t * kFlushLd + lane]);
      }
      ++run;
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
    tmem_free_cols(tmem, kTmemCols);
  }
}

int sm_count() {
  return sm_count_current();
}

}  // namespace

mtp_status dgemm_bf16_launch(const DecSeg* segs, int nseg, int K, const __nv_bfloat16* x, int R, int ldo,
                             cudaStream_t stream) {
  if (!segs || nseg < 1 || nseg > 3 || !x) return MTP_ERR_INVALID_ARG;
  if (K <= 0 || R <= 0 || R > kTok) return MTP_ERR_SHAPE;
  if (K % 8 || !aligned16(x)) return MTP_ERR_ALIGNMENT;  // 16-byte rows for the tensor maps
  Args P{};
  P.nseg = nseg;
  P.nkb = (K + kBK - 1) / kBK;
  P.R = R;
  P.ldo = ldo;
  CUtensorMap tw[3], tx;
  long long total = 0;
  for (int i = 0; i < nseg; ++i) {
    const DecSeg& s = segs[i];
    if (!s.w || !s.out || s.n <= 0) return MTP_ERR_INVALID_ARG;
    if (ldo < s.n) return MTP_ERR_SHAPE;
    if (!aligned16(s.w) || (reinterpret_cast<uintptr_t>(s.out) & 3u)) return MTP_ERR_ALIGNMENT;
    if (!tensor_map_bf16_2d(&tw[i], s.w, s.n, K, K, kBK, kN, true)) return MTP_ERR_CUDA;
    P.seg[i].out = s.out;
    P.seg[i].n = s.n;
    P.seg[i].tiles = (s.n + kN - 1) / kN;
    P.seg[i].first = static_cast<int>(total);
    total += static_cast<long long>(P.seg[i].tiles) * P.nkb;
  }
  if (total > 0x7FFFFFFFll) return MTP_ERR_UNSUPPORTED;
  for (int i = nseg; i < 3; ++i) tw[i] = tw[0];
  if (!tensor_map_bf16_2d(&tx, x, R, K, K, kBK, kTok, true)) return MTP_ERR_CUDA;
  P.total = static_cast<int>(total);
  static PerDevice attr;
  if (!smem_limit(attr, dgemm_bf16_kernel, kSmemBytes)) return MTP_ERR_CUDA;
  const int grid = static_cast<int>(total < sm_count() ? total : sm_count());
  dgemm_bf16_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tw[0], tw[1], tw[2], tx, P);
  note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

}  // namespace mtp

extern "C" mtp_status mtp_gemm_decode_bf16(int R, int N, int K, const void* x, const void* w, float* out,
                                           cudaStream_t stream) {
  if (!x || !w || !out) return MTP_ERR_INVALID_ARG;
  mtp::DecSeg s;
  s.w = static_cast<const __nv_bfloat16*>(w);
  s.n = N;
  s.out = out;
  return mtp::dgemm_bf16_launch(&s, 1, K, static_cast<const __nv_bfloat16*>(x), R, N, stream);
}
