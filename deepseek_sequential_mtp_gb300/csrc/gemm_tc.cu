// tcgen05 GEMM core for sm_103a: acc[M,N] = A[M,K] · B[N,K]^T, bf16 operands,
// fp32 accumulation in tensor memory, fused epilogues.
//
// Persistent, warp-specialised CTA of 6 warps, one CTA per SM:
//   warp 0     TMA producer: 128x64 A box and BNx64 B box (128-byte swizzle;
//              MN-major operands as 64x64 boxes) per k-block into a
//              STAGES-deep shared-memory ring (mbarriers with transaction
//              counts).  When a tile starts it pulls the next tile's first
//              k-blocks into L2.
//   warp 1     allocates 2*BN TMEM columns; one thread issues
//              tcgen05.mma.kind::f16 (M=128, N=BN, K=16) four times per
//              k-block and tcgen05.commit's the smem slot back to the
//              producer; a whole tile's accumulator is committed to the
//              epilogue.  Two accumulators alternate so the epilogue of tile
//              i overlaps the MMAs of tile i+1.
//   warps 2-5  epilogue: tcgen05.ld 32 lanes x 32 columns per load (warp w
//              reads TMEM lanes 32*(w%4)..+31 = tile rows), applies the fused
//              operation and writes each 32-row x 64-column bf16 box into a
//              128-byte-swizzled shared-memory buffer (two per warp) that one
//              lane ships with a TMA store.  The residual epilogue has one box
//              per 64-column piece of the tile: the warp's 32 rows of the
//              residual are loaded into them by TMA while the tile's MMAs
//              still run, each thread adds its row's accumulator in place and
//              the boxes go back out by TMA.  The CE epilogue stores only
//              per-row partials.
// With more than one 128-row tile, 256-wide tiles run on CTA pairs (clusters of
// two): 256x256 tiles with tcgen05.mma.cta_group::2 issued by the leader, each
// CTA staging its 128 rows of A and half of B.
// Launches may be programmatic dependents of the previous kernel: the setup
// (barriers, TMEM, tensor-map prefetch, an optional L2 prefetch of B) runs
// before griddepcontrol.wait.
// Every mbarrier wait is bounded (and inlined: a call per wait cost ~10%):
// after ~1.5 s it sets MTP_DEVERR_TIMEOUT, raises a CTA abort flag and every
// role drains out; the producer then waits (bounded) for its in-flight copies
// and warp 1 for its MMAs before freeing TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_tc.cuh"

MTP_DEFINE_ERROR_WORD(mtp_take_errors_gemm)

namespace mtp {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 bf16 = 128 bytes = one swizzle atom row
constexpr int kGroupM = 16;
static_assert((kGroupM & (kGroupM - 1)) == 0, "tile_coords masks by kGroupM - 1");

// PAIR: a cluster of two CTAs computes a 256 x BN tile with 2-SM MMAs; each
// CTA stages its 128 rows of A and half (BN / 2 rows) of B.
template <int BN, int EPI, bool PAIR = false>
struct Cfg {
  // epilogue warps: 4, one per TMEM lane quadrant.  (Eight, two per quadrant with
  // half of the columns each, finish the CE epilogue sooner but slow the concurrent
  // MMAs of the next tile more: the head GEMM measured 3% slower with them.)
  static constexpr int kEpiWarps = 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  // the residual epilogue's boxes (a whole tile's worth) take the place of ring stages
  static constexpr int kStages = EPI == EPI_RESID ? (PAIR ? 5 : (BN == 256 ? 3 : 6))
                                                  : (PAIR ? 6 : (BN == 256 ? 4 : (BN == 128 ? 6 : 10)));
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = (PAIR ? BN / 2 : BN) * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
  // per epilogue warp: 32 x 64 bf16 boxes (4 KB each), two (one per 64-column piece of
  // the tile for the residual epilogue); none for the CE epilogue
  static constexpr int kBoxBytes = 32 * 64 * 2;
  static constexpr int kBoxesPerWarp = EPI == EPI_RESID ? BN / 64 : 2;
  static constexpr int kStagingBytes = epi_uses_staging(EPI) ? 4 * kBoxesPerWarp * kBoxBytes : 0;
  // + 1024: alignment of the stage ring; + 512: mbarriers (8 B each, 2 S + 13 slots) and the
  // TMEM address and abort flag after them (256 B did not cover the 10-stage configuration)
  static constexpr int kSmemBytes = kStages * kStageBytes + kStagingBytes + 1024 + 512;
  static_assert(8 * (2 * kStages + 13) + 8 <= 512, "barrier area");
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of `parity` to complete; false on abort or timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = cycles_now();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (cycles_now() - t0 > kWaitLimitCycles) {
        *abort_flag = 1;
        atomicOr(&g_mtp_error_word, MTP_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}
// Teardown wait that ignores the abort flag (bounded by `limit_cycles`).
__device__ __noinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, long long limit_cycles) {
  const long long t0 = cycles_now();
  while (!mbar_try_wait(bar, parity)) {
    if (cycles_now() - t0 > limit_cycles) return false;
  }
  return true;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 2-SM (CTA pair) forms.  The pair's TMEM is allocated collectively by one warp
// of each CTA; the leader (even cluster rank) issues the MMAs, which read A
// rows 0-127 and B rows 0..BN/2-1 from its own shared memory and the rest from
// the peer's at the same offsets, and write each CTA's 128 accumulator rows
// into that CTA's TMEM.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on the barrier at this offset in both CTAs of the pair when the leader's MMAs complete
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(static_cast<uint16_t>(3))
               : "memory");
}
// tiled load into this CTA's shared memory that completes its bytes on the
// leader's barrier (`bar` is a shared::cluster address)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Pull a tile of `map` at (x, y) into L2 (no shared-memory destination, no barrier).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most one committed store group may still be reading shared memory
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// generic-proxy shared-memory writes become visible to the TMA (async proxy)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane; the wait is part of
// the same asm statement so no use of the registers can precede it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major bf16 tile stored as rows of
// 128 bytes with the 128-byte swizzle (what TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B): start address >> 4 (bits 0-13), leading byte
// offset 16 B (unused for swizzled K-major), stride byte offset 1024 B
// between 8-row groups (bits 32-45), descriptor version 1 (bit 46),
// layout type 2 = 128-byte swizzle (bits 61-63).  The tile base is
// 1024-byte aligned so the base-offset field stays 0.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// Shared-memory matrix descriptor of an MN-major bf16 tile with the 128-byte
// swizzle: each 64-element (128-byte) piece of the MN extent is a TMA box of
// [64 MN x 64 k] with the k rows 128 bytes apart; leading byte offset = the
// 8 KB between those MN pieces (bits 16-29), stride byte offset = 1024 B
// between groups of 8 k rows (bits 32-45).  A K = 16 step advances the start
// by 16 rows = 2048 B.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(8192 >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), A / B MN-major when bit 15 / 16 is set (MNF bit
// 0 / 1), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, int mnf = 0) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(mnf & 1) << 15) |
         (static_cast<uint32_t>((mnf >> 1) & 1) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}
// MNF bits: 1 = A stored MN-major ([K rows][M], the M extent contiguous),
// 2 = B stored MN-major ([K rows][N]); such operands arrive as [64 x 64] boxes.
constexpr int kMnBox = 64 * 64 * 2;

struct Args {
  int M, N, K;
  int seg_rows;
  int tiles_m, tiles_n, nk;
  __nv_bfloat16* out;
  int ldo;
  const __nv_bfloat16* resid;
  int ldr;
  const int32_t* pos;
  const float2* rope;
  int rope_len, rope_cols, head_dim;
  const int32_t* labels;
  float2* ce_part;
  float* z_tgt;
  float* out_f32;
  int splits;
  int f32_overwrite;
  int ce_nparts;  // CE partials per row: one per gemm_ce_tile_n() vocabulary columns
  const float* lse;
  const float* ce_scale;
  int ce_offset;
  int trigger;  // release dependents when the last tile starts
  int b_early;  // B is read-only for the stream's earlier kernels: prefetch it before pdl_wait
};

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int per_group = kGroupM * tiles_n;
  const int group = t / per_group;
  const int first_m = group * kGroupM;
  const int gsz = min(tiles_m - first_m, kGroupM);
  const int r = t - group * per_group;
  if (gsz == kGroupM) {  // every group but a ragged last one: shifts, no division
    tm = first_m + (r & (kGroupM - 1));
    tn = r / kGroupM;
  } else {
    tm = first_m + r % gsz;
    tn = r / gsz;
  }
}

// A 32-row x 64-column bf16 box in shared memory with the 128-byte swizzle
// (what TMA reads/writes with CU_TENSOR_MAP_SWIZZLE_128B): row r occupies
// bytes [128 r, 128 r + 128) and its 16-byte chunk c sits at chunk c ^ (r & 7).
// Thread `lane` owns row `lane`; `half` selects columns [32 half, 32 half + 32).
__device__ __forceinline__ void box_write32(uint8_t* box, int lane, int half, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat162 h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
    const int c = half * 4 + q;
    *reinterpret_cast<uint4*>(box + lane * 128 + ((c ^ (lane & 7)) << 4)) = *reinterpret_cast<uint4*>(h);
  }
}
// v[i] += the residual at this lane's row, columns [32 half, 32 half + 32) of a box that TMA
// loaded with the 128-byte swizzle (the positions box_write32 then overwrites)
__device__ __forceinline__ void box_add_res32(const uint8_t* box, int lane, int half, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c = half * 4 + q;
    const uint4 w = *reinterpret_cast<const uint4*>(box + lane * 128 + ((c ^ (lane & 7)) << 4));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[8 * q + 2 * i] += f.x;
      v[8 * q + 2 * i + 1] += f.y;
    }
  }
}
// 32 (cos, sin) pairs of one RoPE table row, 16-byte loads
__device__ __forceinline__ void load_cs32(const float2* tab, float2 (&cs)[32]) {
  const float4* t4 = reinterpret_cast<const float4*>(tab);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 f = __ldg(t4 + i);
    cs[2 * i] = make_float2(f.x, f.y);
    cs[2 * i + 1] = make_float2(f.z, f.w);
  }
}
__device__ __forceinline__ void rotate32(float (&x1)[32], float (&x2)[32], const float2 (&cs)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float a = x1[i], b = x2[i];
    x1[i] = a * cs[i].x - b * cs[i].y;
    x2[i] = b * cs[i].x + a * cs[i].y;
  }
}

template <int BN, int EPI, int MNF = 0, bool PAIR = false>
__global__ void __launch_bounds__(Cfg<BN, EPI, PAIR>::kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
               const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmRes,
               const Args P) {
  using C = Cfg<BN, EPI, PAIR>;
  constexpr int S = C::kStages;
  constexpr uint32_t kIdesc = idesc_bf16(PAIR ? 2 * BM : BM, BN, MNF);
  static_assert(!PAIR || BN == 256, "CTA pairs: 256-wide tiles");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint8_t* staging = smem + S * C::kStageBytes;  // 1024-aligned: stage sizes are multiples of 1 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::kStagingBytes);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t final_bar = bar0 + 8u * (2 * S + 4);
  auto res_bar = [&](int w) { return bar0 + 8u * (2 * S + 5 + w); };  // residual boxes of epilogue warp w
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 13);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // the tensor maps are launch parameters: fetch them while an earlier kernel may still run
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB0)) : "memory");
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), (PAIR ? 2 : 1) * 32 * C::kEpiWarps);  // a pair: both CTAs' epilogue threads
    }
    mbar_init(final_bar, 1);
    for (int w = 0; w < 4; ++w) mbar_init(res_bar(w), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc2(smem_u32(tmem_slot), C::kTmemCols);
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t crank = PAIR ? cluster_ctarank() & 1u : 0u;  // 0: the leader of the pair
  // work units: (tile, K split); split s covers k-blocks [kb_lo(s), kb_lo(s+1)).  A pair
  // takes units of two M-tiles: 2 tm2 (leader) and 2 tm2 + 1 (peer) with the same N-tile.
  const int tiles_m_u = PAIR ? (P.tiles_m + 1) / 2 : P.tiles_m;
  const int ntiles = tiles_m_u * P.tiles_n * P.splits;
  const int u_first = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int u_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int nk = P.nk;
  const int splits = P.splits;  // nk * splits < 2^31: 32-bit index arithmetic throughout
  auto kb_lo = [&](int sp) { return splits == 1 ? (sp == 0 ? 0 : nk) : (nk * sp) / splits; };
  auto unit_tile = [&](int t, int& tm, int& tn) {
    tile_coords(t, tiles_m_u, P.tiles_n, tm, tn);
    if constexpr (PAIR) tm = 2 * tm + static_cast<int>(crank);
  };

  // a unit's tile coordinates and the B map and row its copies use
  auto unit_coords = [&](int u, int& tm, int& tn, int& sp, const CUtensorMap*& bmap, int& by) {
    const int t = splits == 1 ? u : u / splits;
    sp = splits == 1 ? 0 : u % splits;
    unit_tile(t, tm, tn);
    bmap = &tmB0;
    if constexpr (EPI == EPI_SWIGLU) {
      by = tn * (BN / 2);
      if constexpr (PAIR) bmap = crank ? &tmB1 : &tmB0;  // the leader stages the gate rows, the peer the up rows
    } else {
      const int n0 = tn * BN + (PAIR ? static_cast<int>(crank) * (BN / 2) : 0);  // a pair splits B's rows
      const int seg = n0 < P.seg_rows ? 0 : (n0 < 2 * P.seg_rows ? 1 : 2);  // at most three segments
      by = n0 - seg * P.seg_rows;
      bmap = seg == 0 ? &tmB0 : (seg == 1 ? &tmB1 : &tmB2);
    }
  };
  // The first k-blocks of a new tile come from DRAM with a latency close to the ring's
  // lead, so a tile boundary stalled the MMAs; the next unit's first k-blocks are pulled
  // into L2 when this unit starts, one tile's time ahead.
  constexpr int kPrefetchKb = 3;
  auto prefetch_unit = [&](int u, bool with_a) {
    int tm, tn, sp, by;
    const CUtensorMap* bmap;
    unit_coords(u, tm, tn, sp, bmap, by);
    const int kb0 = kb_lo(sp), kb1 = min(kb_lo(sp + 1), kb0 + kPrefetchKb);
    for (int kb = kb0; kb < kb1; ++kb) {
      if (with_a && tm * BM < P.M) {
        if constexpr (MNF & 1) {
#pragma unroll
          for (int c = 0; c < BM / 64; ++c) tma_prefetch_2d(&tmA, tm * BM + 64 * c, kb * BK);
        } else {
          tma_prefetch_2d(&tmA, kb * BK, tm * BM);
        }
      }
      if constexpr (MNF & 2) {
        const int n0 = tn * BN + (PAIR ? static_cast<int>(crank) * (BN / 2) : 0);
#pragma unroll
        for (int c = 0; c < (PAIR ? BN / 2 : BN) / 64; ++c) tma_prefetch_2d(&tmB0, n0 + 64 * c, kb * BK);
      } else if constexpr (EPI == EPI_SWIGLU && !PAIR) {
        tma_prefetch_2d(&tmB0, kb * BK, by);
        tma_prefetch_2d(&tmB1, kb * BK, by);
      } else {
        tma_prefetch_2d(bmap, kb * BK, by);
      }
    }
  };
  // Setup above overlaps the previous kernel (programmatic dependent launch); every access
  // to memory an earlier kernel writes follows pdl_wait().  With b_early, B's first k-blocks
  // are pulled into L2 before the wait (a prefetch into L2 stays coherent with the writes
  // that follow it; B is typically a weight matrix).  This kernel releases its own dependents
  // only by completing: with
  // an explicit early release the backward pass's results came out wrong on GB300 (cause
  // not identified), and the release bought no measurable time.
  if (P.b_early && threadIdx.x == 0 && u_first < ntiles) prefetch_unit(u_first, false);
  pdl_wait();

  if (warp == 0 && lane == 0) {
    // ------------------------------ producer ------------------------------
    int stage = 0;
    uint32_t phase = 0;
    bool issued[S];
    uint32_t armed[S];
#pragma unroll
    for (int s = 0; s < S; ++s) { issued[s] = false; armed[s] = 0; }
    bool ok = true;
    const uint32_t full_leader0 = PAIR ? map_to_rank(full_bar(0), 0) : full_bar(0);
    for (int u = u_first; ok && u < ntiles; u += u_step) {
      int tm, tn, sp, by;
      const CUtensorMap* bmap;
      unit_coords(u, tm, tn, sp, bmap, by);
      if (u + u_step < ntiles) prefetch_unit(u + u_step, true);
      const int kb_end = kb_lo(sp + 1);
      for (int kb = kb_lo(sp); kb < kb_end; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
        const uint32_t sa = base + stage * C::kStageBytes;
        const uint32_t sb = sa + C::kABytes;
        if constexpr (PAIR) {  // both CTAs' copies complete on the leader's barrier
          const uint32_t fl = full_leader0 + 8u * stage;
          if (crank == 0) mbar_expect_tx(full_bar(stage), 2 * C::kStageBytes);
          if constexpr (MNF & 1) {  // this CTA's 128 rows of A as two [64 M x 64 k] boxes
#pragma unroll
            for (int c = 0; c < BM / 64; ++c) tma_load_2d_pair(sa + c * kMnBox, &tmA, tm * BM + 64 * c, kb * BK, fl);
          } else {
            tma_load_2d_pair(sa, &tmA, kb * BK, tm * BM, fl);
          }
          if constexpr (MNF & 2) {  // this CTA's half of B's 256 columns as two [64 N x 64 k] boxes
#pragma unroll
            for (int c = 0; c < BN / 128; ++c)
              tma_load_2d_pair(sb + c * kMnBox, &tmB0, tn * BN + static_cast<int>(crank) * (BN / 2) + 64 * c, kb * BK, fl);
          } else {
            tma_load_2d_pair(sb, bmap, kb * BK, by, fl);
          }
          issued[stage] = true;
          armed[stage] = phase;
          if (++stage == S) { stage = 0; phase ^= 1u; }
          continue;
        }
        mbar_expect_tx(full_bar(stage), C::kStageBytes);
        if constexpr (MNF & 1) {
#pragma unroll
          for (int c = 0; c < BM / 64; ++c) tma_load_2d(sa + c * kMnBox, &tmA, tm * BM + 64 * c, kb * BK, full_bar(stage));
        } else {
          tma_load_2d(sa, &tmA, kb * BK, tm * BM, full_bar(stage));
        }
        if constexpr (MNF & 2) {
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) tma_load_2d(sb + c * kMnBox, &tmB0, tn * BN + 64 * c, kb * BK, full_bar(stage));
        } else if constexpr (EPI == EPI_SWIGLU) {
          tma_load_2d(sb, &tmB0, kb * BK, by, full_bar(stage));
          tma_load_2d(sb + (BN / 2) * BK * 2, &tmB1, kb * BK, by, full_bar(stage));
        } else {
          tma_load_2d(sb, bmap, kb * BK, by, full_bar(stage));
        }
        issued[stage] = true;
        armed[stage] = phase;
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
    if (*abort_flag) {  // let every copy this thread started land before the CTA exits
      if (PAIR && crank != 0) {
        // the peer's copies complete on the leader's barrier: give them a bounded time to land
        const long long t0 = cycles_now();
        while (cycles_now() - t0 < 40000000ll) __nanosleep(1000);
      } else {
        for (int s = 0; s < S; ++s)
          if (issued[s]) mbar_wait_drain(full_bar(s), armed[s], 40000000ll);
      }
    }
  } else if (warp == 1 && lane == 0 && crank == 0) {
    // ------------------------------ MMA issuer ------------------------------
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int u = u_first; ok && u < ntiles; u += u_step, ++local) {
      const int sp = splits == 1 ? 0 : u % splits;
      const int kb0 = kb_lo(sp), kb_end = kb_lo(sp + 1);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = kb0; kb < kb_end; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = base + stage * C::kStageBytes;
        // K-major: a K = 16 step is 32 bytes along the swizzled row; MN-major: 16 rows of 128 bytes
        constexpr uint64_t kStepA = (MNF & 1) ? 2048 >> 4 : 2, kStepB = (MNF & 2) ? 2048 >> 4 : 2;
        const uint64_t adesc = (MNF & 1) ? sdesc_mn_sw128(sa) : sdesc_sw128(sa);
        const uint64_t bdesc = (MNF & 2) ? sdesc_mn_sw128(sa + C::kABytes) : sdesc_sw128(sa + C::kABytes);
        if constexpr (PAIR) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16_pair(d_tmem, adesc + kStepA * kk, bdesc + kStepB * kk, kIdesc, (kb != kb0 || kk != 0) ? 1u : 0u);
          umma_commit_pair(empty_bar(stage));  // frees the stage in both CTAs
        } else {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d_tmem, adesc + kStepA * kk, bdesc + kStepB * kk, kIdesc, (kb != kb0 || kk != 0) ? 1u : 0u);
          umma_commit(empty_bar(stage));
        }
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (ok) {
        if constexpr (PAIR) umma_commit_pair(tfull_bar(acc));
        else umma_commit(tfull_bar(acc));
      }
    }
  } else if (warp >= 2) {
    // ------------------------------ epilogue ------------------------------
    const int quarter = warp & 3;  // TMEM lanes 32*quarter.. = tile rows
    const int ew = warp - 2;       // epilogue warp index: owns two staging boxes
    uint8_t* boxes = staging + ew * C::kBoxesPerWarp * C::kBoxBytes;
    int nb = 0;                        // next staging box
    int local = 0;
    bool both_pending = false;         // the last store group read both boxes
    bool res_inflight = false;         // residual boxes requested and not yet waited for
    // claim staging box nb: the store issued from it two boxes ago has read it
    auto claim = [&]() -> uint8_t* {
      if (lane == 0) {
        if (both_pending) bulk_wait_read0();
        else bulk_wait_read1();
      }
      both_pending = false;
      __syncwarp();
      return boxes + nb * C::kBoxBytes;
    };
    auto ship = [&](uint8_t* box, int col0, int row0w) {
      fence_async_smem();
      __syncwarp();
      if (lane == 0 && col0 < P.N && row0w < P.M) {
        tma_store_2d(&tmOut, col0, row0w, smem_u32(box));
        bulk_commit();
      }
      nb ^= 1;
    };
    bool ok = true;
    for (int u = u_first; ok && u < ntiles; u += u_step, ++local) {
      const int t = splits == 1 ? u : u / splits;
      int tm, tn;
      unit_tile(t, tm, tn);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (P.trigger && u + u_step >= ntiles) pdl_trigger();  // this CTA's last tile
      // residual: the warp's 32 rows of every 64-column piece of the tile are loaded by TMA into
      // its boxes while the tile's MMAs run, once the previous tile's stores have read them
      if constexpr (EPI == EPI_RESID) {
        if (lane == 0) {
          bulk_wait_read0();
          const int r0 = tm * BM + quarter * 32;
          uint32_t bytes = 0;
#pragma unroll
          for (int c = 0; c < BN / 64; ++c)
            if (r0 < P.M && tn * BN + 64 * c < P.N) bytes += C::kBoxBytes;
          if (bytes) {
            mbar_expect_tx(res_bar(ew), bytes);
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              if (r0 < P.M && tn * BN + 64 * c < P.N)
                tma_load_2d(smem_u32(boxes + c * C::kBoxBytes), &tmRes, tn * BN + 64 * c, r0, res_bar(ew));
          } else {
            mbar_arrive(res_bar(ew));
          }
        }
        __syncwarp();
        res_inflight = true;
      }
      // CE backward: the row's label, log-sum-exp and scale, fetched while the MMAs run
      // (log2 domain; a row without a label gets lse = +inf, so its exp is 0 and its scale 0)
      int ce_lab = -1;
      float ce_lse2 = INFINITY, ce_sc = 0.f;
      if constexpr (EPI == EPI_CE_GRAD) {
        const int prow = tm * BM + quarter * 32 + lane;
        if (prow < P.M) {
          ce_lab = P.labels[prow];
          if (ce_lab >= 0) {
            ce_lse2 = P.lse[prow] * 1.4426950408889634f;
            ce_sc = *P.ce_scale;
          }
        }
      }
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) break;
      tc_fence_after();
      const int row0w = tm * BM + quarter * 32;
      const int row = row0w + lane;
      const bool row_ok = row < P.M;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;

      if constexpr (EPI == EPI_STORE) {
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          const int col0 = tn * BN + c * 64;
          uint8_t* box = claim();
          float v[32];
          tmem_ld32(taddr + c * 64, v);
          box_write32(box, lane, 0, v);
          tmem_ld32(taddr + c * 64 + 32, v);
          box_write32(box, lane, 1, v);
          ship(box, col0, row0w);
        }
      } else if constexpr (EPI == EPI_RESID) {
        if (!mbar_wait(res_bar(ew), local & 1, abort_flag)) break;
        res_inflight = false;
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          uint8_t* box = boxes + c * C::kBoxBytes;
          float v[32];
          tmem_ld32(taddr + c * 64, v);
          box_add_res32(box, lane, 0, v);
          box_write32(box, lane, 0, v);
          tmem_ld32(taddr + c * 64 + 32, v);
          box_add_res32(box, lane, 1, v);
          box_write32(box, lane, 1, v);
          fence_async_smem();
          __syncwarp();
          if (lane == 0 && tn * BN + c * 64 < P.N && row0w < P.M)
            tma_store_2d(&tmOut, tn * BN + c * 64, row0w, smem_u32(box));
        }
        if (lane == 0) bulk_commit();
      } else if constexpr (EPI == EPI_ROPE) {
        const int tile_col0 = tn * BN;
        if (tile_col0 >= P.rope_cols) {
#pragma unroll 1
          for (int c = 0; c < BN / 64; ++c) {
            uint8_t* box = claim();
            float v[32];
            tmem_ld32(taddr + c * 64, v);
            box_write32(box, lane, 0, v);
            tmem_ld32(taddr + c * 64 + 32, v);
            box_write32(box, lane, 1, v);
            ship(box, tile_col0 + c * 64, row0w);
          }
        } else {
          const int hd = P.head_dim, half = hd >> 1;
          int p = row_ok ? P.pos[row] : 0;
          if (p < 0 || p >= P.rope_len) {
            if (row_ok) atomicOr(&g_mtp_error_word, MTP_DEVERR_TOKEN_RANGE);
            p = min(max(p, 0), P.rope_len - 1);
          }
          const float2* tab = P.rope + static_cast<size_t>(p) * half;
          float2 cs[32];
          if (hd == 64) {
            load_cs32(tab, cs);  // one table row serves every head of the tile
#pragma unroll 1
            for (int h0 = 0; h0 < BN; h0 += 64) {
              uint8_t* box = claim();
              float x1[32], x2[32];
              tmem_ld32(taddr + h0, x1);
              tmem_ld32(taddr + h0 + 32, x2);
              rotate32(x1, x2, cs);
              box_write32(box, lane, 0, x1);
              box_write32(box, lane, 1, x2);
              ship(box, tile_col0 + h0, row0w);
            }
          } else {  // hd == 128: columns [h0, h0+64) and [h0+64, h0+128) go to the two boxes
#pragma unroll 1
            for (int h0 = 0; h0 < BN; h0 += 128) {
              if (lane == 0) bulk_wait_read0();
              __syncwarp();
              uint8_t* box_lo = boxes;
              uint8_t* box_hi = boxes + C::kBoxBytes;
#pragma unroll 1
              for (int j = 0; j < 64; j += 32) {
                float x1[32], x2[32];
                load_cs32(tab + j, cs);
                tmem_ld32(taddr + h0 + j, x1);
                tmem_ld32(taddr + h0 + 64 + j, x2);
                rotate32(x1, x2, cs);
                box_write32(box_lo, lane, j >> 5, x1);
                box_write32(box_hi, lane, j >> 5, x2);
              }
              fence_async_smem();
              __syncwarp();
              if (lane == 0 && row0w < P.M) {
                tma_store_2d(&tmOut, tile_col0 + h0, row0w, smem_u32(box_lo));
                tma_store_2d(&tmOut, tile_col0 + h0 + 64, row0w, smem_u32(box_hi));
                bulk_commit();
              }
              both_pending = true;
            }
          }
        }
      } else if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < BN / 128; ++c) {
          const int col0 = tn * (BN / 2) + c * 64;
          uint8_t* box = claim();
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            float g[32], u[32];
            tmem_ld32(taddr + c * 64 + h * 32, g);
            tmem_ld32(taddr + BN / 2 + c * 64 + h * 32, u);
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * u[i];
            box_write32(box, lane, h, g);
          }
          ship(box, col0, row0w);
        }
      } else if constexpr (EPI == EPI_T_STORE) {
        // row = feature; TMEM columns = tokens; for a fixed token the warp's
        // 32 lanes write 32 consecutive features (128 bytes)
        float v[32];
        tmem_ld32(taddr, v);
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < P.N) {
              float* dst = P.out_f32 + static_cast<size_t>(j) * P.ldo + row;
              *dst = v[j];
            }
          }
        }
      } else if constexpr (EPI == EPI_CE_GRAD) {
        const float lse2 = ce_lse2, sc = ce_sc;
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          const int col0 = tn * BN + c * 64;
          uint8_t* box = claim();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[32];
            tmem_ld32(taddr + c * 64 + half * 32, v);
            const int off = ce_lab - (P.ce_offset + col0 + half * 32);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              v[i] = fmaf(exp2f(fmaf(v[i], 1.4426950408889634f, -lse2)), sc, i == off ? -sc : 0.f);
            box_write32(box, lane, half, v);
          }
          ship(box, col0, row0w);
        }
      } else if constexpr (EPI == EPI_F32_ACC) {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          const int col0 = tn * BN + c * 32;
          if (row_ok && col0 < P.N) {
            float* dst = P.out_f32 + static_cast<size_t>(row) * P.ldo + col0;
            if (P.splits > 1) {  // split-K partial tile: vector atomics
              if (col0 + 32 <= P.N) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  atomicAdd(reinterpret_cast<float4*>(dst + 4 * q),
                            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
              } else {
                for (int i = 0; i < 32 && col0 + i < P.N; ++i) atomicAdd(dst + i, v[i]);
              }
            } else if (P.f32_overwrite) {  // the first product into this output: no read
              if (col0 + 32 <= P.N) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  *reinterpret_cast<float4*>(dst + 4 * q) =
                      make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
              } else {
                for (int i = 0; i < 32 && col0 + i < P.N; ++i) dst[i] = v[i];
              }
            } else if (col0 + 32 <= P.N) {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                float4 o = *reinterpret_cast<float4*>(dst + 4 * q);
                o.x += v[4 * q];
                o.y += v[4 * q + 1];
                o.z += v[4 * q + 2];
                o.w += v[4 * q + 3];
                *reinterpret_cast<float4*>(dst + 4 * q) = o;
              }
            } else {
              for (int i = 0; i < 32 && col0 + i < P.N; ++i) dst[i] += v[i];
            }
          }
        }
      } else if constexpr (EPI == EPI_CE) {
        // this warp's columns: [BN/kNsub · sub, BN/kNsub · (sub + 1)) of the tile
        constexpr int kNsub = C::kEpiWarps / 4, kChunks = BN / 32 / kNsub;
        const int sub = (warp - 2) >> 2;
        const int lab = row_ok ? P.labels[row] : -1;
        float m_run = -INFINITY, s_run = 0.0f, zt = 0.0f;
        bool has_t = false;
#pragma unroll 1
        for (int c = sub * kChunks; c < (sub + 1) * kChunks; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          const int col0 = tn * BN + c * 32;
          const int valid = min(32, P.N - col0);
          if (valid < 32) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i >= valid) v[i] = -INFINITY;
          }
          // tree reductions (short dependency chains): chunk maximum, then Σ exp
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(fmaxf(v[i], v[i + 8]), fmaxf(v[i + 16], v[i + 24]));
#pragma unroll
          for (int i = 0; i < 4; ++i) mx[i] = fmaxf(mx[i], mx[i + 4]);
          const float cmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
          const float m_new = fmaxf(m_run, cmax);
          if (m_new != -INFINITY) {
            // exp(v - m) = 2^(v log2e - m log2e): one FFMA and one exp2 per element
            float e[4] = {0.f, 0.f, 0.f, 0.f};
            const float ml2 = m_new * 1.4426950408889634f;
#pragma unroll
            for (int i = 0; i < 32; ++i) e[i & 3] += exp2f(fmaf(v[i], 1.4426950408889634f, -ml2));
            s_run = s_run * exp2f((m_run - m_new) * 1.4426950408889634f) + ((e[0] + e[1]) + (e[2] + e[3]));
            m_run = m_new;
          }
          const int off = lab - col0;
          if (off >= 0 && off < 32 && off < valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i == off) zt = v[i];
            has_t = true;
          }
        }
        const int pidx = tn * kNsub + sub;
        if (row_ok && pidx * (BN / kNsub) < P.N) {
          P.ce_part[static_cast<size_t>(row) * P.ce_nparts + pidx] = make_float2(m_run, s_run);
          if (has_t) P.z_tgt[row] = zt;
        }
      }
      tc_fence_before();
      if constexpr (PAIR) {  // the leader's MMA warp waits for both CTAs' epilogues
        if (crank == 0) mbar_arrive(tempty_bar(acc));
        else mbar_arrive_remote(map_to_rank(tempty_bar(acc), 0));
      } else {
        mbar_arrive(tempty_bar(acc));
      }
    }
    // after an abort: the residual boxes still being loaded land before the CTA leaves
    if (EPI == EPI_RESID && res_inflight && lane == 0) mbar_wait_drain(res_bar(ew), local & 1, 40000000ll);
    if constexpr (EPI != EPI_CE) {
      if (lane == 0) {
        bulk_wait_all();  // every TMA store of this warp has completed
      }
      __syncwarp();
    }
  }
  if (P.trigger && warp < 2) {  // the producer and MMA warps, once their elected lane is done
    __syncwarp();
    pdl_trigger();
  }

  __syncthreads();
  if constexpr (PAIR) {
    // every MMA of the pair has completed (the leader's final commit reaches both CTAs)
    // before either CTA frees its TMEM or leaves (the MMAs read both CTAs' shared memory)
    if (warp == 1 && lane == 0) {
      if (crank == 0) umma_commit_pair(final_bar);
      mbar_wait_drain(final_bar, 0, 40000000ll);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc2(tmem_base, C::kTmemCols);
    }
  } else {
    if (warp == 1) {
      if (lane == 0) {  // every MMA this CTA issued has completed before TMEM is freed
        umma_commit(final_bar);
        mbar_wait_drain(final_bar, 0, 40000000ll);
      }
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem_base, C::kTmemCols);
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D bf16 tensor [rows, cols] with row stride `ld` elements, box 64 x box_rows.
bool make_map(CUtensorMap* m, const void* ptr, int rows, int cols, int ld, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  return sm_count_current();
}

template <int BN, int EPI, int MNF = 0, bool PAIR = false>
mtp_status launch(const GemmDesc& g, cudaStream_t stream) {
  using C = Cfg<BN, EPI, PAIR>;
  static PerDevice attr;
  if (!smem_limit(attr, gemm_tc_kernel<BN, EPI, MNF, PAIR>, C::kSmemBytes)) return MTP_ERR_CUDA;
  CUtensorMap ta, tb[3];
  const int box_b = (EPI == EPI_SWIGLU || PAIR) ? BN / 2 : BN;  // a pair stages half of B per CTA
  // MN-major operands are [K rows][M or N] in memory, loaded as [64 x 64] boxes
  if (!((MNF & 1) ? make_map(&ta, g.A, g.K, g.M, g.lda, 64) : make_map(&ta, g.A, g.M, g.K, g.lda, BM)))
    return MTP_ERR_INVALID_ARG;
  const int nmaps = EPI == EPI_SWIGLU ? 2 : g.nseg;
  const int brows = EPI == EPI_SWIGLU ? g.N : g.seg_rows;
  for (int i = 0; i < 3; ++i) {
    const void* ptr = g.B[i < nmaps ? i : 0];
    if (!((MNF & 2) ? make_map(&tb[i], ptr, g.K, g.N, g.ldb, 64) : make_map(&tb[i], ptr, brows, g.K, g.ldb, box_b)))
      return MTP_ERR_INVALID_ARG;
  }
  // output / residual boxes: 32 rows x 64 columns, 128-byte swizzle
  CUtensorMap tout = ta;
  if (epi_uses_staging(EPI) && !make_map(&tout, g.out, g.M, g.N, g.ldo, 32)) return MTP_ERR_INVALID_ARG;
  CUtensorMap tres = tout;
  if (EPI == EPI_RESID && !make_map(&tres, g.resid, g.M, g.N, g.ldr, 32)) return MTP_ERR_INVALID_ARG;
  Args a{};
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.seg_rows = g.seg_rows > 0 ? g.seg_rows : g.N;
  a.tiles_m = (g.M + BM - 1) / BM;
  a.tiles_n = (g.N + (EPI == EPI_SWIGLU ? BN / 2 : BN) - 1) / (EPI == EPI_SWIGLU ? BN / 2 : BN);
  a.nk = (g.K + BK - 1) / BK;
  a.out = g.out;
  a.ldo = g.ldo;
  a.resid = g.resid;
  a.ldr = g.ldr;
  a.pos = g.pos;
  a.rope = g.rope;
  a.rope_len = g.rope_len;
  a.rope_cols = g.rope_cols;
  a.head_dim = g.head_dim;
  a.labels = g.labels;
  a.ce_part = g.ce_part;
  a.z_tgt = g.z_tgt;
  a.out_f32 = g.out_f32;
  a.splits = g.splits > 0 ? g.splits : 1;
  a.f32_overwrite = g.f32_overwrite ? 1 : 0;
  a.ce_nparts = (g.N + BN / (C::kEpiWarps / 4) - 1) / (BN / (C::kEpiWarps / 4));
  a.lse = g.lse;
  a.ce_scale = g.ce_scale;
  a.ce_offset = g.ce_offset;
  a.b_early = g.b_early ? 1 : 0;
  a.trigger = g.trigger_early ? 1 : 0;
  if constexpr (PAIR) {  // clusters of two CTAs, one pair per two SMs
    const int units = ((a.tiles_m + 1) / 2) * a.tiles_n * a.splits;
    const int pairs = units < num_sms() / 2 ? units : num_sms() / 2;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g.pdl ? 2 : 1;
    MTP_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, EPI, MNF, PAIR>, ta, tb[0], tb[1], tb[2], tout, tres, a));
  } else {
    const int ntiles = a.tiles_m * a.tiles_n * a.splits;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ntiles < num_sms() ? ntiles : num_sms());
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g.pdl ? 1 : 0;
    MTP_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, EPI, MNF, PAIR>, ta, tb[0], tb[1], tb[2], tout, tres, a));
  }
  mtp::note_launch();
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

}  // namespace

int gemm_ce_tile_n() { return 256 / (Cfg<256, EPI_CE, true>::kEpiWarps / 4); }

bool tensor_map_bf16_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                        uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  if (!encoder()) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tensor_map_u8_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_cols,
                      uint32_t box_rows) {
  if (!encoder()) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

mtp_status gemm_bf16_launch(const GemmDesc& g, cudaStream_t stream) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return MTP_ERR_SHAPE;
  if (!g.A || !g.B[0] || g.nseg < 1 || g.nseg > 3) return MTP_ERR_INVALID_ARG;
  // B's segments must cover the N columns (the kernel picks a column's segment by comparison)
  if (g.seg_rows > 0 && static_cast<long long>(g.seg_rows) * g.nseg < g.N) return MTP_ERR_SHAPE;
  // TMA needs 16-byte row strides; a K extent that is not a multiple of the
  // k-block is zero-filled by the copies
  if (g.lda % 8 || g.ldb % 8) return MTP_ERR_ALIGNMENT;
  if ((g.a_mn || g.b_mn) && g.epi != EPI_F32_ACC && g.epi != EPI_STORE) return MTP_ERR_UNSUPPORTED;
  if (g.f32_overwrite && (g.epi != EPI_F32_ACC || g.splits > 1)) return MTP_ERR_INVALID_ARG;
  if (!aligned16(g.A)) return MTP_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i)
    if (g.B[i] && !aligned16(g.B[i])) return MTP_ERR_ALIGNMENT;
  if (epi_uses_staging(g.epi) && (!g.out || g.ldo % 8 || !aligned16(g.out))) return MTP_ERR_ALIGNMENT;
  if (!encoder()) return MTP_ERR_CUDA;
  switch (g.epi) {
    case EPI_STORE:
    case EPI_RESID: {
      if (g.epi == EPI_RESID && (!g.resid || g.ldr % 8 || !aligned16(g.resid))) return MTP_ERR_ALIGNMENT;
      const int seg = g.seg_rows > 0 ? g.seg_rows : g.N;
      if (g.nseg > 1 && seg % 128) return MTP_ERR_UNSUPPORTED;
      const bool wide = (g.nseg == 1 || seg % 256 == 0);
      if (g.epi == EPI_STORE && (g.a_mn || g.b_mn)) {  // bf16 output of a product with a transposed operand
        if (g.nseg != 1 || g.a_mn) return MTP_ERR_UNSUPPORTED;
        return g.M > BM ? launch<256, EPI_STORE, 2, true>(g, stream) : launch<256, EPI_STORE, 2>(g, stream);
      }
      const bool pair = wide && g.M > BM;
      if (g.epi == EPI_STORE)
        return pair ? launch<256, EPI_STORE, 0, true>(g, stream)
                    : (wide ? launch<256, EPI_STORE>(g, stream) : launch<128, EPI_STORE>(g, stream));
      return pair ? launch<256, EPI_RESID, 0, true>(g, stream)
                  : (wide ? launch<256, EPI_RESID>(g, stream) : launch<128, EPI_RESID>(g, stream));
    }
    case EPI_ROPE: {
      const int seg = g.seg_rows > 0 ? g.seg_rows : g.N;
      if ((g.head_dim != 64 && g.head_dim != 128) || !g.pos || !g.rope || g.rope_len <= 0) return MTP_ERR_INVALID_ARG;
      if (seg % 128 || g.rope_cols % 128) return MTP_ERR_UNSUPPORTED;
      if (seg % 256 == 0 && g.rope_cols % 256 == 0)
        return g.M > BM ? launch<256, EPI_ROPE, 0, true>(g, stream) : launch<256, EPI_ROPE>(g, stream);
      return launch<128, EPI_ROPE>(g, stream);
    }
    case EPI_SWIGLU:
      if (!g.B[1] || !aligned16(g.B[1])) return MTP_ERR_INVALID_ARG;
      return g.M > BM ? launch<256, EPI_SWIGLU, 0, true>(g, stream) : launch<256, EPI_SWIGLU>(g, stream);
    case EPI_CE:
      if (!g.labels || !g.ce_part || !g.z_tgt) return MTP_ERR_INVALID_ARG;
      return g.M > BM ? launch<256, EPI_CE, 0, true>(g, stream) : launch<256, EPI_CE>(g, stream);
    case EPI_CE_GRAD:
      if (!g.labels || !g.lse || !g.ce_scale) return MTP_ERR_INVALID_ARG;
      return g.M > BM ? launch<256, EPI_CE_GRAD, 0, true>(g, stream) : launch<256, EPI_CE_GRAD>(g, stream);
    case EPI_F32_ACC: {
      if (!g.out_f32 || g.ldo % 4 || !aligned16(g.out_f32)) return MTP_ERR_INVALID_ARG;
      const int nk = (g.K + BK - 1) / BK;
      if (g.splits < 1 || g.splits > nk || g.nseg != 1) return MTP_ERR_INVALID_ARG;
      switch ((g.a_mn ? 1 : 0) | (g.b_mn ? 2 : 0)) {
        case 0: return g.M > BM ? launch<256, EPI_F32_ACC, 0, true>(g, stream) : launch<256, EPI_F32_ACC, 0>(g, stream);
        case 1: return g.M > BM ? launch<256, EPI_F32_ACC, 1, true>(g, stream) : launch<256, EPI_F32_ACC, 1>(g, stream);
        case 2: return g.M > BM ? launch<256, EPI_F32_ACC, 2, true>(g, stream) : launch<256, EPI_F32_ACC, 2>(g, stream);
        default: return g.M > BM ? launch<256, EPI_F32_ACC, 3, true>(g, stream) : launch<256, EPI_F32_ACC, 3>(g, stream);
      }
    }
    case EPI_T_STORE:
      if (g.N > 32 || !g.out_f32 || g.nseg != 1) return MTP_ERR_UNSUPPORTED;
      if (g.splits != 1) return MTP_ERR_INVALID_ARG;
      return launch<32, EPI_T_STORE>(g, stream);
    default:
      return MTP_ERR_INVALID_ARG;
  }
}

}  // namespace mtp

extern "C" mtp_status mtp_gemm_bf16(int M, int N, int K, const void* A, const void* B, void* C,
                                    cudaStream_t stream) {
  if (!A || !B || !C) return MTP_ERR_INVALID_ARG;
  mtp::GemmDesc g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.A = static_cast<const __nv_bfloat16*>(A);
  g.lda = K;
  g.B[0] = static_cast<const __nv_bfloat16*>(B);
  g.ldb = K;
  g.nseg = 1;
  g.seg_rows = N;
  g.epi = mtp::EPI_STORE;
  g.out = static_cast<__nv_bfloat16*>(C);
  g.ldo = N;
  return mtp::gemm_bf16_launch(g, stream);
}

extern "C" mtp_status mtp_gemm_f32acc(int M, int N, int K, const void* A, int lda, int a_mn, const void* B, int ldb,
                                      int b_mn, float* out, int ldo, int splits, cudaStream_t stream) {
  if (!A || !B || !out) return MTP_ERR_INVALID_ARG;
  mtp::GemmDesc g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.A = static_cast<const __nv_bfloat16*>(A);
  g.lda = lda;
  g.a_mn = a_mn != 0;
  g.B[0] = static_cast<const __nv_bfloat16*>(B);
  g.ldb = ldb;
  g.b_mn = b_mn != 0;
  g.nseg = 1;
  g.seg_rows = N;
  g.epi = mtp::EPI_F32_ACC;
  g.out_f32 = out;
  g.ldo = ldo;
  g.splits = splits;
  return mtp::gemm_bf16_launch(g, stream);
}
