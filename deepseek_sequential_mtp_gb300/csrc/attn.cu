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
// bf16 backward: tcgen05 kernel (attn_bwd_tc_kernel below): one CTA per
// 128-key block, S^T and dP^T in TMEM, dV and dK accumulated in TMEM, dQ
// formed per query block in TMEM and added to global memory with atomics.
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

// D[q] = dO_q . o_q for every (query row, head): one warp per item.
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
// their softmax warps alternate on the tensor pipe: while tile A's turn S_A
// into P_A, the MMA thread runs P_B V and S_B, and the reverse.
//   softmax    tile A's warps first, then tile B's: one query row per thread
//              (TMEM lane = row) of each warpgroup; at head_dim 64 two
//              warpgroups per tile, each taking 64 of a block's 128 keys and
//              agreeing on the block maximum through shared memory.  S read
//              with tcgen05.ld, segment-causal mask, stale-by-up-to-2^8
//              running maximum, P = 2^(s - m) written back as bf16 pairs into
//              the first 64 columns of the tile's own S (tcgen05.st), where
//              the P V product reads it as its A operand.
//   TMA warp   (after the softmax warps) lane 0 loads Q_A, Q_B and the K
//              blocks, lane 1 the V blocks (MN-major [64 keys x 64 cols]
//              boxes), each into a ring.
//   MMA warp   (the last) allocates 512 TMEM columns (S_A, S_B at 0 and 128; O_A, O_B
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
template <int HD>
struct Tc2Attn {
  // softmax threads per query row: at head_dim 64 two, each taking 64 of a block's 128 keys
  static constexpr int kHalves = HD == 64 ? 2 : 1;
  static constexpr int kSoftmaxWarps = 8 * kHalves;
  static constexpr int kThreads = 32 * (kSoftmaxWarps + 2);
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
  static constexpr int kItemReaders = 2 + kSoftmaxWarps;
  // q full/empty, k full/empty, v full/empty; per tile s_full, p_full, pv_done, o_free; drain;
  // item ring full/empty; with two halves per row, per tile the block-maximum and row-sum exchanges
  static constexpr int kNumBars = 2 * (kQBufs + kKStages + kVStages) + 8 + 1 + 2 * kRing + (kHalves > 1 ? 4 : 0);
  static constexpr int kOffItems = (kOffBar + 8 * kNumBars + 15) / 16 * 16;
  // exchange between the halves of a row: block maxima [block parity][tile][half][row], row sums
  // [tile][half][row]
  static constexpr int kOffXchg = kOffItems + 16 * kRing + 16;
  static constexpr int kXchgBytes = kHalves > 1 ? 4 * (2 * 2 * kHalves * 128 + 2 * kHalves * 128) : 0;
  static constexpr int kSmemBytes = kOffXchg + kXchgBytes;
  static constexpr uint32_t kColO0 = 256;
};

template <int HD>
__global__ void __launch_bounds__(Tc2Attn<HD>::kThreads, 1)
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
  const uint32_t barh = barx + 72u + 16u * C::kRing;
  auto mx_bar = [&](int x) { return barh + 8u * x; };         // two halves: block maxima exchanged
  auto sum_bar = [&](int x) { return barh + 16u + 8u * x; };  // two halves: row sums exchanged
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
      mtp::mbar_init(p_full(x), kTcQ * C::kHalves);
      mtp::mbar_init(pv_done(x), 1);
      mtp::mbar_init(o_free(x), kTcQ * C::kHalves);
      if (C::kHalves > 1) {
        mtp::mbar_init(mx_bar(x), kTcQ * C::kHalves);
        mtp::mbar_init(sum_bar(x), kTcQ * C::kHalves);
      }
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
  constexpr int kTmaWarp = C::kSoftmaxWarps, kMmaWarp = C::kSoftmaxWarps + 1;
  if (warp == kTmaWarp && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm128)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm64)) : "memory");
  }
  if (warp == kMmaWarp) mtp::tmem_alloc_cols(mtp::smem_u32(tmem_slot), 512);
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

  if (warp == kTmaWarp) {
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
  } else if (warp == kMmaWarp) {
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
    // ---------------- softmax: one query row per thread of each half of tile x ----------------
    // With two halves (head_dim 64) half hf takes keys 64 hf .. 64 hf + 63 of every block: the
    // halves agree on each block's maximum through shared memory (both then take the same
    // running maximum), each writes its keys' P, rescales and writes half of the row's output
    // columns, and their row sums are added at the end of the item.
    constexpr int kH = C::kHalves;
    constexpr int kKeysPer = kTcKeys / kH;  // a block's scores per thread
    constexpr int kOCols = HD / kH;         // output columns per thread
    const int x = warp / (4 * kH);
    const int hf = (warp >> 2) % kH;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t colS = 128u * x, colO = C::kColO0 + HD * x + kOCols * hf;
    float* xmax = reinterpret_cast<float*>(smem + C::kOffXchg);
    float* xsum = xmax + 2 * 2 * kH * kTcQ;
    auto wwait = [&](uint32_t bar, uint32_t parity) { return __all_sync(0xffffffffu, wait(bar, parity)); };
    uint32_t n = 0;   // S products of this tile consumed
    uint32_t ns = 0;  // row-sum exchanges of this tile
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
        float sc[kKeysPer];
        if constexpr (kKeysPer == 128) {
          float (&lo)[64] = *reinterpret_cast<float (*)[64]>(&sc[0]);
          float (&hi)[64] = *reinterpret_cast<float (*)[64]>(&sc[64]);
          mtp::tmem_ld64(lane_base + colS, lo);
          mtp::tmem_ld64(lane_base + colS + 64, hi);
        } else {
          float (&v)[64] = *reinterpret_cast<float (*)[64]>(&sc[0]);
          mtp::tmem_ld64(lane_base + colS + kKeysPer * hf, v);
        }
        const int key0 = j * kTcKeys + kKeysPer * hf;
        if (!(key0 >= st_row && key0 + kKeysPer - 1 <= q)) {  // keys the row sees only in part
#pragma unroll
          for (int i = 0; i < kKeysPer; ++i) {
            const int key = key0 + i;
            if (!(key >= st_row && key <= q)) sc[i] = -INFINITY;
          }
        }
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = sc[i];
#pragma unroll
        for (int i = 8; i < kKeysPer; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], sc[i]);
        float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                         fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * scale_log2;
        if constexpr (kH > 1) {
          // the block maximum over both halves of the row; this half's scores are in registers
          // before the other half may write its P over them
          float* xm = xmax + ((n & 1) * 2 + x) * (kH * kTcQ);
          xm[hf * kTcQ + row] = mx;
          mtp::tc_fence_before();
          mtp::mbar_arrive1(mx_bar(x));
          if (!wwait(mx_bar(x), n & 1)) { ok = false; break; }
          mtp::tc_fence_after();
          mx = fmaxf(mx, xm[(hf ^ 1) * kTcQ + row]);
        }
        // a new running maximum only when the block's exceeds the stale one by 2^8
        const float m_new = mx > m + kStaleMaxLog2 ? mx : m;
        const bool rescale = m_new != m && m != -INFINITY;
        const float neg_use = m_new == -INFINITY ? 0.f : -m_new;
        float rs8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rs8[i] = 0.f;
#pragma unroll
        for (int i = 0; i < kKeysPer / 2; ++i) {  // P pairs packed in place: sc[i] holds keys 2i, 2i+1
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
          for (int c = 0; c < kOCols / 32; ++c) {
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
        // P into this tile's S columns (the pair of keys 2i, 2i + 1 of the block in column i; the
        // scores are in registers now, and the previous block's P V completed before this
        // block's S did)
#pragma unroll
        for (int c = 0; c < kKeysPer / 64; ++c) {
          float (&p)[32] = *reinterpret_cast<float (*)[32]>(&sc[32 * c]);
          mtp::tmem_st32(lane_base + colS + (kKeysPer / 2) * hf + 32 * c, p);
        }
        mtp::tc_fence_before();
        mtp::mbar_arrive1(p_full(x));
      }
      if (!ok) break;
      if (!wwait(pv_done(x), (n - 1) & 1)) break;  // the item's last P V
      mtp::tc_fence_after();
      float lt = l;
      if constexpr (kH > 1) {  // the row sum over both halves (the same sum, added in either order)
        float* xs = xsum + x * (kH * kTcQ);
        xs[hf * kTcQ + row] = l;
        mtp::mbar_arrive1(sum_bar(x));
        if (!wwait(sum_bar(x), ns & 1)) break;
        lt = l + xs[(hf ^ 1) * kTcQ + row];
        ++ns;
      }
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      if (live && lse2_out && hf == 0) lse2_out[(static_cast<size_t>(b) * T + q) * H + h] = m + log2f(lt);
      __nv_bfloat16* orow = out + (static_cast<size_t>(b) * T + q) * d + h * HD + kOCols * hf;
#pragma unroll
      for (int c = 0; c < kOCols / 32; ++c) {
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
  if (warp == kMmaWarp) mtp::tmem_free_cols(tmem, 512);
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
  MTP_CUDA_TRY(launch_pdl(attn_tc2_kernel<HD>, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, m128, m64, out,
                          seg_start, B, T, H, scale_log2, lse2_out, work_ctr));
  note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}


// ---------------------------------------------------------------------------
// Backward on the tcgen05 tensor cores (bf16, head_dim 64 or 128).
//
// One CTA per (128-key block j, head, packed row); every 128-query block i
// that can see one of the block's keys streams through.  K_j and V_j stay in
// shared memory (TMA, K-major with the 128-byte swizzle); Q_i and dO_i arrive
// by TMA into a ring, beside each query's lse2 and D = rowsum(dO * O) staged
// by the producer warp.  A key sees the queries key <= q < max(seg_end(key),
// key + 1): the forward's rule seg_start(q) <= key <= q read from the key's
// side (a pad sees only itself).  With one TMEM lane per key:
//   S^T = K_j Q_i^T, dP^T = V_j dO_i^T          (TMEM columns 0 and 128)
//   P^T = 2^(S^T scale_log2 - lse2) on the visible pairs, dS^T = P^T (dP^T - D)
//                                               (warps 0-7: two warps per lane
//                                               quadrant, one per 64 queries;
//                                               P^T and dS^T go back into the
//                                               first halves of their columns
//                                               as bf16 pairs once both warps
//                                               have read their scores, and
//                                               dS^T into shared memory)
//   dK_j += dS^T Q_i                            (A from TMEM; B = Q_i read
//                                               MN-major from its tile)
//   dQ_i = dS K_j                               (A = the staged dS^T read
//                                               MN-major, B = K_j MN-major; into
//                                               TMEM columns 128.., after dK
//                                               has read dS^T there)
//   dV_j += P^T dO_i                            (A from TMEM, B = dO_i MN-major)
// As soon as dQ_i is formed, warps 0-7 read it (a query row per thread, half
// the columns per warp group), pass it through shared memory so each access
// covers four rows of 128 bytes, and add it, scaled, to the fp32 dq rows with
// vector reductions (every key block of the segment contributes); at the end
// they store dV_j and dK_j (scaled) the same way.  Warp 8 issues the TMA loads,
// warp 9 allocates TMEM and issues the MMAs.  The MMAs of the one issuing
// thread run in order, so a product may overwrite TMEM columns that an earlier
// product read as its A operand.  P and dS are rounded to bf16 for the
// products.  Every wait is bounded.
// ---------------------------------------------------------------------------
constexpr int kBwdThreads = 320;

// two sets of 32 consecutive fp32 TMEM columns of this thread's lane, one wait
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&a)[32], float (&b)[32]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[32 + i]);
  }
}

// A warp's 32 rows x 32 fp32 columns (a row per lane, as TMEM hands them out) go
// through its own 4 KB of shared memory (16-byte chunks XOR-swizzled by row) so
// that each global access of the warp covers 4 rows x 128 contiguous bytes.
// Lane l writes row l; then lane l owns chunk l % 8 of rows l / 8 + 4k.
__device__ __forceinline__ void stage_rows32(uint8_t* wbuf, int lane, const float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<float4*>(wbuf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
        make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}
__device__ __forceinline__ float4 staged_chunk(const uint8_t* wbuf, int row, int chunk) {
  return *reinterpret_cast<const float4*>(wbuf + row * 128 + ((chunk ^ (row & 7)) << 4));
}

// *p += v element-wise (fp32, 16-byte aligned), without returning the old value
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

template <int HD>
struct TcBwd {
  static constexpr int kChunks = HD / 64;
  static constexpr int kPiece = 128 * 128;         // one [128 rows x 64 bf16] swizzled piece (16 KB)
  static constexpr int kTile = 128 * HD * 2;       // one [128 x HD] bf16 tile
  static constexpr int kSlots = HD == 64 ? 2 : 1;  // Q/dO ring (the next block loads early when it fits)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTile;
  static constexpr int kOffQ = 2 * kTile;                 // + slot * kTile
  static constexpr int kOffdO = kOffQ + kSlots * kTile;   // + slot * kTile
  static constexpr int kOffdS = kOffdO + kSlots * kTile;  // two 64-query pieces of [128 keys x 128 B]
  static constexpr int kOffPar = kOffdS + 2 * kPiece;     // per slot: lse2[128], D[128]
  static constexpr int kParFloats = 2 * 128;
  static constexpr int kOffBar = kOffPar + kSlots * kParFloats * 4;
  // kv_full, qdo_full[slots], qdo_empty[slots], sd_full, p_full, dq_ready, dq_free, mma_done, drain,
  // scores_read
  static constexpr int kNumBars = 1 + 2 * kSlots + 7;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // TMEM base, abort flag, 4 ints of scratch
  static constexpr int kSmemBytes = kOffMisc + 32;
  static constexpr uint32_t kColS = 0, kColdP = 128, kColdQ = 128, kColdV = 256, kColdK = 256 + HD;
  static_assert(kColdK + HD <= 512, "TMEM columns");
};

template <int HD>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                   const float* __restrict__ lse2, const float* __restrict__ dsum,
                   const int32_t* __restrict__ seg_end, float* __restrict__ dqkv, int T, int H, float scale_log2,
                   float scale) {
  using C = TcBwd<HD>;
  extern __shared__ __align__(1024) uint8_t bwd_smem[];
  const uint32_t s0 = mtp::smem_u32(bwd_smem);
  if (s0 & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(&g_mtp_error_word, MTP_DEVERR_TIMEOUT);
    return;
  }
  const uint32_t sK = s0 + C::kOffK, sV = s0 + C::kOffV, sdS = s0 + C::kOffdS;
  const uint32_t bar0 = s0 + C::kOffBar;
  const uint32_t kv_full = bar0;
  auto qdo_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto qdo_empty = [&](int s) { return bar0 + 8u * (1 + C::kSlots + s); };
  const uint32_t sd_full = bar0 + 8u * (1 + 2 * C::kSlots);
  const uint32_t p_full = sd_full + 8u, dq_ready = sd_full + 16u, dq_free = sd_full + 24u,
                 mma_done = sd_full + 32u, drain_bar = sd_full + 40u, scores_read = sd_full + 48u;
  float* par = reinterpret_cast<float*>(bwd_smem + C::kOffPar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bwd_smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* red = reinterpret_cast<int*>(tmem_slot + 2);
  unsigned int* err = &g_mtp_error_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int d = H * HD;
  const size_t ld3 = 3 * static_cast<size_t>(d);
  const int k0 = kb * 128;
  const int32_t* se = seg_end + static_cast<size_t>(b) * T;

  // the last query that sees one of the block's keys (keys past T see none)
  int qhi = -1;
  if (threadIdx.x < 128) {
    const int s = k0 + static_cast<int>(threadIdx.x);
    if (s < T) qhi = max(static_cast<int>(se[s]), s + 1) - 1;
  }
  qhi = __reduce_max_sync(0xffffffffu, qhi);
  if (lane == 0 && warp < 4) red[warp] = qhi;
  if (threadIdx.x == 0) {
    mtp::mbar_init(kv_full, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mtp::mbar_init(qdo_full(s), 1);
      mtp::mbar_init(qdo_empty(s), 1);
    }
    mtp::mbar_init(sd_full, 1);
    mtp::mbar_init(p_full, 256);
    mtp::mbar_init(dq_ready, 1);
    mtp::mbar_init(dq_free, 256);
    mtp::mbar_init(mma_done, 1);
    mtp::mbar_init(drain_bar, 1);
    mtp::mbar_init(scores_read, 256);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 8 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_qkv)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_do)) : "memory");
  }
  if (warp == 9) mtp::tmem_alloc_cols(mtp::smem_u32(tmem_slot), 512);
  mtp::tc_fence_before();
  __syncthreads();
  mtp::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int q_last = max(max(red[0], red[1]), max(red[2], red[3]));
  const int qb_first = kb;  // a key is seen only by queries at or after it
  const int n_blocks = q_last >= k0 ? q_last / 128 - qb_first + 1 : 0;
  auto wait = [&](uint32_t bar, uint32_t parity) { return mtp::wait_phase(bar, parity, abort_flag, err); };
  auto wwait = [&](uint32_t bar, uint32_t parity) { return __all_sync(0xffffffffu, wait(bar, parity)); };

  if (warp == 8) {
    // ---------------- TMA producer and per-query values ----------------
    int loads = 0;
    if (lane == 0) {
      mtp::mbar_expect_tx(kv_full, 2 * C::kTile);
      for (int c = 0; c < C::kChunks; ++c) {
        mtp::tma_tile_2d(sK + c * C::kPiece, &tm_qkv, d + h * HD + 64 * c, b * T + k0, kv_full);
        mtp::tma_tile_2d(sV + c * C::kPiece, &tm_qkv, 2 * d + h * HD + 64 * c, b * T + k0, kv_full);
      }
    }
    for (int i = 0; i < n_blocks; ++i) {
      const int slot = i % C::kSlots, use = i / C::kSlots;
      if (use > 0 && !wwait(qdo_empty(slot), (use - 1) & 1)) break;
      const int q0 = (qb_first + i) * 128;
      // the tiles first (the barrier counts their bytes before its one arrival), then the
      // per-query values, published by lane 0's arrival after the warp's stores
      if (lane == 0) {
        const uint32_t sQ = s0 + C::kOffQ + slot * C::kTile, sdO = s0 + C::kOffdO + slot * C::kTile;
        mtp::mbar_expect_tx_noarrive(qdo_full(slot), 2 * C::kTile);
        for (int c = 0; c < C::kChunks; ++c) {
          mtp::tma_tile_2d(sQ + c * C::kPiece, &tm_qkv, h * HD + 64 * c, b * T + q0, qdo_full(slot));
          mtp::tma_tile_2d(sdO + c * C::kPiece, &tm_do, h * HD + 64 * c, b * T + q0, qdo_full(slot));
        }
      }
      float* p = par + slot * C::kParFloats;
      for (int r = lane; r < 128; r += 32) {
        const int q = q0 + r;
        const bool live = q < T;
        const size_t item = (static_cast<size_t>(b) * T + (live ? q : 0)) * H + h;
        p[r] = live ? lse2[item] : INFINITY;
        p[128 + r] = live ? dsum[item] : 0.f;
      }
      __syncwarp();
      if (lane == 0) mtp::mbar_arrive1(qdo_full(slot));
      ++loads;
    }
    // no copy may still be landing when the CTA leaves (matters only after an abort)
    if (lane == 0) {
      mtp::wait_drain(kv_full, 0, kWaitLimitCycles);
      for (int x = loads > C::kSlots ? loads - C::kSlots : 0; x < loads; ++x)
        mtp::wait_drain(qdo_full(x % C::kSlots), (x / C::kSlots) & 1, kWaitLimitCycles);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc_s = mtp::idesc_bf16_f32(128, 128, 0);
      constexpr uint32_t idesc_kv = mtp::idesc_bf16_f32(128, HD, 2);  // A from TMEM, B MN-major
      constexpr uint32_t idesc_q = mtp::idesc_bf16_f32(128, HD, 3);   // A and B MN-major
      constexpr uint32_t kLbo = C::kPiece;                            // MN pieces of the K-major tiles
      bool ok = wait(kv_full, 0), any = false;
      for (int i = 0; i < n_blocks && ok; ++i) {
        const int slot = i % C::kSlots;
        const uint32_t sQ = s0 + C::kOffQ + slot * C::kTile, sdO = s0 + C::kOffdO + slot * C::kTile;
        if (!wait(qdo_full(slot), (i / C::kSlots) & 1)) { ok = false; break; }
        mtp::tc_fence_after();
        // S^T = K_j Q_i^T (the previous block's P^T was read by an earlier product)
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (k >> 2) * C::kPiece + (k & 3) * 32;
          mtp::umma_bf16_ss(tmem + C::kColS, mtp::sdesc_k_sw128(sK + off), mtp::sdesc_k_sw128(sQ + off), idesc_s,
                            k > 0);
        }
        any = true;
        // dP^T = V_j dO_i^T into the columns of the previous block's dQ once that has been read
        if (i > 0 && !wait(dq_free, (i - 1) & 1)) { ok = false; break; }
        mtp::tc_fence_after();
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (k >> 2) * C::kPiece + (k & 3) * 32;
          mtp::umma_bf16_ss(tmem + C::kColdP, mtp::sdesc_k_sw128(sV + off), mtp::sdesc_k_sw128(sdO + off), idesc_s,
                            k > 0);
        }
        mtp::umma_commit(sd_full);
        if (!wait(p_full, i & 1)) { ok = false; break; }
        mtp::tc_fence_after();
        // dK += dS^T Q over the block's 128 queries, then dQ = dS K over the 128 keys into
        // the columns dK has just read dS^T from, then dV += P^T dO
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mtp::umma_bf16_ts(tmem + C::kColdK, tmem + C::kColdP + 8u * k, mtp::sdesc_mn_sw128_lbo(sQ + 2048 * k, kLbo),
                            idesc_kv, (i > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mtp::umma_bf16_ss(tmem + C::kColdQ, mtp::sdesc_mn_sw128_lbo(sdS + 2048 * k, kLbo),
                            mtp::sdesc_mn_sw128_lbo(sK + 2048 * k, kLbo), idesc_q, k > 0);
        mtp::umma_commit(dq_ready);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mtp::umma_bf16_ts(tmem + C::kColdV, tmem + C::kColS + 8u * k, mtp::sdesc_mn_sw128_lbo(sdO + 2048 * k, kLbo),
                            idesc_kv, (i > 0 || k > 0) ? 1u : 0u);
        mtp::umma_commit(qdo_empty(slot));
      }
      if (ok && any) mtp::umma_commit(mma_done);  // dV and dK complete
      // every issued MMA has completed before TMEM is freed
      if (any) {
        mtp::umma_commit(drain_bar);
        mtp::wait_drain(drain_bar, 0, kWaitLimitCycles);
      }
    }
  } else {
    // ---------------- warps 0-7: P^T and dS^T, then dQ ----------------
    // Warp w serves TMEM lane quadrant w % 4 (a key row per thread for P^T and dS^T, a query
    // row per thread for dQ); warps 0-3 take queries 0-63 of each key row and columns
    // 0..HD/2 of dQ, warps 4-7 queries 64-127 and the other dQ columns.
    const int grp = warp >> 2;
    const int kr = static_cast<int>(threadIdx.x) & 127;
    const int key = k0 + kr;
    // the queries that see this key: [key, q_end) (empty for a key past T)
    const int q_end = key < T ? max(static_cast<int>(se[key]), key + 1) : key;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    uint8_t* sds_row = bwd_smem + C::kOffdS + grp * C::kPiece + (kr >> 3) * 1024 + (kr & 7) * 128;
    uint8_t* wbuf = bwd_smem + C::kOffdS + warp * 4096;  // this warp's staging area (in the dS^T tile)
    bool ok = true;
    for (int i = 0; i < n_blocks; ++i) {
      const int slot = i % C::kSlots;
      const int q0 = (qb_first + i) * 128;
      const float* p = par + slot * C::kParFloats;
      if (!wwait(qdo_full(slot), (i / C::kSlots) & 1)) { ok = false; break; }  // per-query values
      if (!wwait(sd_full, i & 1)) { ok = false; break; }
      mtp::tc_fence_after();
      uint32_t pk[2][16], dk[2][16];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {  // 32 queries per step
        const int c = 2 * grp + cc;
        const int qc = q0 + 32 * c;  // first query of the chunk
        if (!__any_sync(0xffffffffu, qc < q_end && qc + 31 >= key)) {  // the warp's keys see none of them
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[cc][j] = dk[cc][j] = 0u;
        } else {
          float sv[32], dv[32];
          tmem_ld32x2(lane_base + C::kColS + 32 * c, lane_base + C::kColdP + 32 * c, sv, dv);
          // the queries' values four at a time (every lane reads the same 16 bytes)
          const float4* lse4 = reinterpret_cast<const float4*>(p + 32 * c);
          const float4* d4 = reinterpret_cast<const float4*>(p + 128 + 32 * c);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const float4 l4 = lse4[g], dd4 = d4[g];
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dvv[4] = {dd4.x, dd4.y, dd4.z, dd4.w};
            float pp[4], dd[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int q = qc + 4 * g + t;
              const float pv = (q >= key && q < q_end) ? ex2_approx(fmaf(sv[4 * g + t], scale_log2, -lv[t])) : 0.f;
              pp[t] = pv;
              dd[t] = pv * (dv[4 * g + t] - dvv[t]);
            }
            pk[cc][2 * g] = pack2_bf16(pp[0], pp[1]);
            pk[cc][2 * g + 1] = pack2_bf16(pp[2], pp[3]);
            dk[cc][2 * g] = pack2_bf16(dd[0], dd[1]);
            dk[cc][2 * g + 1] = pack2_bf16(dd[2], dd[3]);
          }
        }
        // dS^T row into shared memory: query piece grp, 16-byte chunks cc * 4 + m
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int chunk = cc * 4 + m;
          *reinterpret_cast<uint4*>(sds_row + ((chunk ^ (kr & 7)) << 4)) =
              make_uint4(dk[cc][4 * m], dk[cc][4 * m + 1], dk[cc][4 * m + 2], dk[cc][4 * m + 3]);
        }
      }
      // both halves of every key row have read their scores before P^T and dS^T overwrite
      // them (a bounded rendezvous of warps 0-7)
      mtp::tc_fence_before();
      mtp::mbar_arrive1(scores_read);
      if (!wwait(scores_read, i & 1)) { ok = false; break; }
      mtp::tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * grp + cc;
        mtp::tmem_st16_nowait(lane_base + C::kColS + 16 * c, pk[cc]);
        mtp::tmem_st16_nowait(lane_base + C::kColdP + 16 * c, dk[cc]);
      }
      mtp::tmem_wait_st();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // dS^T for the tensor pipe
      mtp::tc_fence_before();
      mtp::mbar_arrive1(p_full);
      // dQ of this query block, half of its columns
      if (!wwait(dq_ready, i & 1)) { ok = false; break; }
      mtp::tc_fence_after();
      // (the staged dS^T was read by the dQ product: its tile is free until the next block)
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        const int col0 = grp * (HD / 2) + 32 * c;
        float v[32];
        mtp::tmem_ld32(lane_base + C::kColdQ + col0, v);
        stage_rows32(wbuf, lane, v);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = (lane >> 3) + 4 * k;  // row of the warp's 32
          const int q = q0 + (warp & 3) * 32 + r;
          const float4 x = staged_chunk(wbuf, r, lane & 7);
          if (q < T)
            red_add_v4(dqkv + (static_cast<size_t>(b) * T + q) * ld3 + h * HD + col0 + 4 * (lane & 7), x.x * scale,
                       x.y * scale, x.z * scale, x.w * scale);
        }
        __syncwarp();
      }
      mtp::tc_fence_before();
      mtp::mbar_arrive1(dq_free);
    }
    // dV_j (warps 0-3) and dK_j, scaled (warps 4-7), once every product has completed
    if (ok && n_blocks > 0 && wwait(mma_done, 0)) {
      mtp::tc_fence_after();
      const uint32_t col = grp == 0 ? C::kColdV : C::kColdK;
      const float f = grp == 0 ? 1.f : scale;
      const size_t part = (grp == 0 ? 2 * static_cast<size_t>(d) : d) + h * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        float v[32];
        mtp::tmem_ld32(lane_base + col + 32 * c, v);
        stage_rows32(wbuf, lane, v);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = (lane >> 3) + 4 * k;
          const int kk = k0 + (warp & 3) * 32 + r;  // the key of staged row r
          const float4 x = staged_chunk(wbuf, r, lane & 7);
          if (kk < T)
            *reinterpret_cast<float4*>(dqkv + (static_cast<size_t>(b) * T + kk) * ld3 + part + 32 * c +
                                       4 * (lane & 7)) = make_float4(x.x * f, x.y * f, x.z * f, x.w * f);
        }
        __syncwarp();
      }
    }
  }
  mtp::tc_fence_before();
  __syncthreads();
  mtp::tc_fence_after();
  if (warp == 9) mtp::tmem_free_cols(tmem, 512);
}

template <int HD>
mtp_status attn_bwd_tc_launch(const __nv_bfloat16* qkv, const __nv_bfloat16* dO, const float* lse2,
                              const float* dsum, const int32_t* seg_end, float* dqkv, int B,
                              int T, int H, float scale_log2, float scale, cudaStream_t stream) {
  using C = TcBwd<HD>;
  static PerDevice attr;
  if (!smem_limit(attr, attn_bwd_tc_kernel<HD>, C::kSmemBytes)) return MTP_ERR_CUDA;
  if (!aligned16(qkv) || !aligned16(dO) || !aligned16(dqkv)) return MTP_ERR_ALIGNMENT;
  const int d = H * HD;
  const uint64_t rows = static_cast<uint64_t>(B) * T;
  if (rows > 0x7FFFFFFFull) return MTP_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
  CUtensorMap mq, mdo;
  if (!tensor_map_bf16_2d(&mq, qkv, rows, 3 * d, 3 * d, 64, 128, true) ||
      !tensor_map_bf16_2d(&mdo, dO, rows, d, d, 64, 128, true))
    return MTP_ERR_CUDA;
  const dim3 grid((T + 127) / 128, H, B);
  attn_bwd_tc_kernel<HD><<<grid, kBwdThreads, C::kSmemBytes, stream>>>(mq, mdo, lse2, dsum, seg_end, dqkv, T, H,
                                                                      scale_log2, scale);
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
  const float scale = 1.0f / sqrtf(static_cast<float>(hd));
  const float scale_log2 = 1.4426950408889634f * scale;
  // dq is accumulated with reductions by every key block: its third of each row starts from
  // zero (the dk and dv thirds are stored once, by the CTA of their key block)
  const size_t d = static_cast<size_t>(H) * hd;
  if (cudaMemset2DAsync(dqkv, 3 * d * sizeof(float), 0, d * sizeof(float), static_cast<size_t>(B) * T, stream) !=
      cudaSuccess)
    return MTP_ERR_CUDA;
  if (hd == 64) {
    attn_dsum_kernel<64><<<(items + 7) / 8, 256, 0, stream>>>(o, dO, dsum, items, H);
    mtp::note_launch();
    return attn_bwd_tc_launch<64>(qkv, dO, lse2, dsum, seg_end, dqkv, B, T, H, scale_log2, scale, stream);
  }
  if (hd == 128) {
    attn_dsum_kernel<128><<<(items + 7) / 8, 256, 0, stream>>>(o, dO, dsum, items, H);
    mtp::note_launch();
    return attn_bwd_tc_launch<128>(qkv, dO, lse2, dsum, seg_end, dqkv, B, T, H, scale_log2, scale, stream);
  }
  return MTP_ERR_UNSUPPORTED;
}

}  // namespace mtp
