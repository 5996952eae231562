// spec_verify: exact speculative verification of gamma drafts per request.
//
// Semantics: "M7.6 - DeepSeek MTP: Sequential Modules, Teacher Forcing, and
// Speculative Runtime" §0x09 (accept with min(1, p/q), correct from the
// normalised positive residual, bonus from the next target row, EOS/budget
// truncation) generalised to gamma drafts by the left-to-right rule of the
// speculative-decoding page.  Uniforms: Philox4x32-10 (Salmon et al., SC'11).
//
// Layout on the GPU: a cluster of 2 CTAs per request, one CTA per SM (416
// threads: 12 consumer warps and one producer warp, 192 KB ring of six
// 32 KB stages), so the 64 requests of a decode batch occupy 128 SMs in one
// wave.
//   phase A  warp 0 of every CTA: lane j evaluates draft position j (two
//            scalar loads, one Philox block, an exact fp32 test of u*q < p);
//            a ballot picks the first position that ends the round.  Both
//            CTAs reach the same decision.
//   phase B  CTA `rank` owns half of the chunks of the one row pair (or bonus
//            row) the round samples from.  Its producer warp streams them
//            with one-dimensional bulk copies into a ring of shared-memory
//            stages (mbarrier-tracked); consumer warps form residuals in fp32,
//            each lane summing 32 consecutive elements of a chunk with
//            compensated (hi, lo) fp32 steps; the CTA keeps every chunk's 32
//            lane sums and its (hi, lo) total in its own shared memory.
//   phase C  warp 0 of each CTA takes the double-float prefix over its own
//            chunks and hands its half's total (and its error flags) to the
//            other CTA through distributed shared memory; after one cluster
//            barrier both know the mass and u' * mass, and the CTA whose half
//            holds it finds the chunk, then the lane's 32-element range from
//            the staged lane sums, then the element, reloading only those 32
//            elements (the row was just streamed: L2).  Nothing on phases A
//            and C uses FP64: GB300 runs it at a small fraction of the FP32
//            rate, and a short chain of FP64 additions here cost microseconds.
// The kernel is HBM-bound: it reads 2*V*4 bytes for a rejection, V*4 for a
// bonus, plus 8*gamma bytes of scalars.
// Ring invariant: a parity wait cannot tell phase u+1 from phase u-1, so no
// waiter may reach a barrier more than one phase ahead of its last completed
// phase.  With S chunks per stage and W consumer warps, consumer warp w takes
// chunks w, w+W, ..., i.e. stages w/S + (W/S) m; a ring of a multiple of W/S
// stages keeps it on the same slot(s), so it sees each slot's phases one after
// another (it waited on use u-1 itself before waiting on use u).  The producer issues use
// u of a slot only after every consumer of use u-1 released it, and waits for
// every copy it issued before it leaves.
#include <cooperative_groups.h>

#include "common.cuh"
#include "mbarrier.cuh"

namespace cg = cooperative_groups;

MTP_DEFINE_ERROR_WORD(mtp_take_errors_verify)

namespace {

constexpr int kThreads = 416;  // 12 consumer warps + 1 producer warp
constexpr int kCluster = 2;
constexpr int kConsumerWarps = 12;
constexpr int kStageChunks = 4;  // chunks per ring stage: 16 KB bulk copies per row (a copy has a fixed cost)
constexpr int kRing = 6;          // ring stages of 4 chunks x 4 KB x 2 rows (192 KB: the deeper the ring, the more bytes in flight per SM)
constexpr int kStageBytes = 2 * kStageChunks * 1024 * 4;
constexpr int kRingBytes = kRing * kStageBytes;

constexpr int kChunk = 1024;       // elements per chunk
constexpr int kMaxChunks = 512;    // V <= 524288
constexpr int kMaxGamma = 31;
// per chunk of a CTA's half: 32 lane sums and the chunk's (hi, lo) sum
constexpr int kTableBytesPerChunk = 32 * 4 + 8;
__host__ __device__ constexpr int chunks_per_cta(int V) { return ((V + kChunk - 1) / kChunk + kCluster - 1) / kCluster; }
// each consumer warp must revisit the same ring slot (see the ring invariant)
static_assert(kRing % (kConsumerWarps / kStageChunks) == 0, "ring length must be a multiple of the warp stage stride");

enum Event { EV_CONTINUE = 0, EV_STOP = 1, EV_REJECT = 2, EV_INVALID_DRAFT = 3, EV_INVALID_PROBS = 4 };

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

// u = (w >> 8) * 2^-24: a 24-bit integer times a power of two, exact in fp32
__device__ __forceinline__ float uniform24(uint32_t w) {
  return static_cast<float>(w >> 8) * (1.0f / 16777216.0f);
}

// u < min(1, p/q) for u in [0, 1) and q > 0 is u*q < p (when p >= q both hold
// for every u < 1).  u has 24 significant bits, so u*q = hi + lo exactly with
// hi = fl(u*q), lo = fma(u, q, -hi), and the test needs no division and no
// FP64 (GB300 runs FP64 at a small fraction of the FP32 rate, and this
// decision sits on the kernel's critical path).  It is the exact comparison;
// a fp64 quotient rounded first can differ only for u within one rounding of
// p/q.
__device__ __forceinline__ bool accept_draft(float u, float pj, float qj) {
  const float hi = u * qj;
  const float lo = fmaf(u, qj, -hi);
  return hi < pj || (hi == pj && lo < 0.0f);
}

__device__ __forceinline__ bool prob_ok(float v) { return isfinite(v) && v >= 0.0f; }
// prob_ok over many values at two instructions each: nanchk accumulates
// v * 0, which stays 0 for every finite v and turns NaN for a NaN or an
// infinity (no overflow is possible), and mn tracks the minimum (fminf
// ignores NaN, which nanchk catches).  Every value passed prob_ok iff
// nanchk == 0 and mn >= 0 at the end (-0.0 passes both, as it does prob_ok).
__device__ __forceinline__ void check_value4(float& nanchk, float& mn, float4 v) {
  nanchk = fmaf(v.x, 0.0f, nanchk);
  nanchk = fmaf(v.y, 0.0f, nanchk);
  nanchk = fmaf(v.z, 0.0f, nanchk);
  nanchk = fmaf(v.w, 0.0f, nanchk);
  mn = fminf(mn, fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
}

// weight of element v: residual max(p - q, 0) when q != nullptr, else p.
__device__ __forceinline__ float weight_of(float pv, float qv, bool residual) {
  return residual ? fmaxf(pv - qv, 0.0f) : pv;
}

// Error-free transformation: s + e == a + b exactly, s = fl(a + b).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
// Add x to the unevaluated sum hi + lo.
__device__ __forceinline__ void acc_add(float& hi, float& lo, float x) {
  float s, e;
  two_sum(hi, x, s, e);
  hi = s;
  lo += e;
}
// Warp-wide sum of (hi, lo) pairs with TwoSum at every level; every lane
// ends with the same pair.
__device__ __forceinline__ void warp_two_sum(float& hi, float& lo) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ohi = __shfl_xor_sync(0xffffffffu, hi, o);
    const float olo = __shfl_xor_sync(0xffffffffu, lo, o);
    float sum, err;
    two_sum(hi, ohi, sum, err);
    hi = sum;
    lo = (lo + olo) + err;
  }
}
// Double-float values (hi + lo, |lo| <= ulp(hi)/2): the running sums of
// phase C carry ~48 significant bits with FP32 instructions only.  Every
// value here is a sum of non-negative weights.
struct f2 {
  float hi, lo;
};
// renormalise hi + lo with |hi| >= |lo| (fast two-sum)
__device__ __forceinline__ f2 f2_norm(float hi, float lo) {
  const float s = hi + lo;
  return {s, lo - (s - hi)};
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  return f2_norm(s, e + (a.lo + b.lo));
}
// a > b: the difference of the high parts is exact when they are within a
// factor of two (Sterbenz) and has the right sign otherwise
__device__ __forceinline__ bool f2_gt(f2 a, f2 b) { return (a.hi - b.hi) + (a.lo - b.lo) > 0.0f; }
// u * m for a 24-bit u: the product of the high parts split exactly by FMA
__device__ __forceinline__ f2 f2_scale(float u, f2 m) {
  const float p = u * m.hi;
  return f2_norm(p, fmaf(u, m.lo, fmaf(u, m.hi, -p)));
}
__device__ __forceinline__ f2 f2_shfl(f2 v, int src) {
  return {__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}
__device__ __forceinline__ f2 f2_shfl_up(f2 v, int d) {
  return {__shfl_up_sync(0xffffffffu, v.hi, d), __shfl_up_sync(0xffffffffu, v.lo, d)};
}
__device__ __forceinline__ f2 warp_inclusive_scan_f2(f2 v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const f2 n = f2_shfl_up(v, o);
    if (lane >= o) v = f2_add(v, n);
  }
  return v;
}
// exclusive prefix from an inclusive one (lane 0 gets zero)
__device__ __forceinline__ f2 f2_exclusive(f2 incl) {
  const f2 n = f2_shfl_up(incl, 1);
  return (threadIdx.x & 31) ? n : f2{0.0f, 0.0f};
}
__device__ __forceinline__ f2 chunk_value(float2 v) { return f2_norm(v.x, v.y); }

using mtp::bulk_load;
using mtp::cluster_addr;
using mtp::mbar_arrive_cnt;
using mtp::mbar_expect_tx;
using mtp::mbar_init;
using mtp::smem_u32;
// kStarve (failure-path test only): the producer issues no copy, so every
// consumer's first ring wait runs out after `wait_limit` cycles with nothing
// in flight; the request then ends with MTP_VERIFY_DEVICE_TIMEOUT and the
// error word's MTP_DEVERR_TIMEOUT, as a real stall would.
template <bool kVec4, bool kStarve>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
spec_verify_kernel(int gamma, int V, const float* __restrict__ p, const float* __restrict__ q,
                   const int32_t* __restrict__ draft, uint2 key, uint32_t off_lo, uint32_t off_hi,
                   const int32_t* __restrict__ eos, const int32_t* __restrict__ remaining,
                   int32_t* __restrict__ accepted, int32_t* __restrict__ next_token,
                   int32_t* __restrict__ n_emit, int32_t* __restrict__ status, long long wait_limit) {
  auto mbar_wait = [wait_limit](uint32_t bar, uint32_t parity) {
    return mtp::mbar_wait_bounded(bar, parity, wait_limit);
  };
  // kRing stages of p and q chunks (with kVec4), then this CTA's lane and chunk sums
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ float2 s_tot[kCluster];  // (hi, lo) sum of each CTA's half of the row
  __shared__ __align__(8) uint64_t s_bars[2 * kRing];
  __shared__ int s_jstar, s_event, s_bad, s_timeout;
  __shared__ float s_u;
  const uint32_t s_full_bar = smem_u32(s_bars), s_empty_bar = s_full_bar + 8u * kRing;
  auto ring_p = [&](int slot) { return smem_u32(ring + slot * kStageBytes); };
  auto ring_q = [&](int slot) { return smem_u32(ring + slot * kStageBytes + kStageChunks * kChunk * 4); };

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int r = blockIdx.x / kCluster;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int budget = remaining ? remaining[r] : gamma + 1;
  const int eos_id = eos ? eos[r] : -1;

  // ---------------- phase A: the accept prefix ----------------
  if (warp == 0) {
    int ev = EV_CONTINUE;
    const int j = lane;
    if (j < gamma) {
      const int y = draft[(size_t)r * gamma + j];
      if (y < 0 || y >= V) {
        ev = EV_INVALID_DRAFT;
      } else {
        const float pj = p[((size_t)r * (gamma + 1) + j) * V + y];
        const float qj = q[((size_t)r * gamma + j) * V + y];
        if (!(prob_ok(pj) && prob_ok(qj))) {
          ev = EV_INVALID_PROBS;
        } else if (qj <= 0.0f) {
          ev = EV_INVALID_DRAFT;
        } else {
          const uint4 w = philox4x32_10(make_uint4((uint32_t)j, (uint32_t)r, off_lo, off_hi), key);
          if (!accept_draft(uniform24(w.x), pj, qj)) ev = EV_REJECT;
          else if (j + 1 == budget || y == eos_id) ev = EV_STOP;
        }
      }
    }
    const unsigned ended = __ballot_sync(0xffffffffu, ev != EV_CONTINUE);
    const int jstar = ended ? __ffs(ended) - 1 : gamma;
    const int evstar = __shfl_sync(0xffffffffu, ev, jstar & 31);
    if (lane == 0) {
      s_jstar = jstar;
      s_event = (jstar == gamma) ? EV_CONTINUE : evstar;
      s_bad = 0;
      s_timeout = 0;
      for (int i = 0; i < kRing; ++i) {
        mbar_init(s_full_bar + 8u * i, 1);
        mbar_init(s_empty_bar + 8u * i, kStageChunks);
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const uint4 w = philox4x32_10(make_uint4((uint32_t)jstar, (uint32_t)r, off_lo, off_hi), key);
      s_u = uniform24(w.y);
      if (budget < 1) s_event = -1;
    }
  }
  cluster.sync();  // publishes the barrier initialisation at cluster scope before any bulk copy
  const int jstar = s_jstar;
  const int event = s_event;

  // every CTA of the cluster takes the same branch here
  if (event != EV_CONTINUE && event != EV_REJECT) {
    if (rank == 0 && threadIdx.x == 0) {
      int st = MTP_VERIFY_OK, acc = jstar;
      if (event == -1) { st = MTP_VERIFY_INVALID_BUDGET; acc = 0; }
      else if (event == EV_STOP) acc = jstar + 1;
      else if (event == EV_INVALID_DRAFT) st = MTP_VERIFY_INVALID_DRAFT;
      else if (event == EV_INVALID_PROBS) st = MTP_VERIFY_INVALID_PROBS;
      accepted[r] = acc;
      next_token[r] = -1;
      n_emit[r] = acc;
      status[r] = st;
    }
    return;
  }

  // ---------------- phase B: lane and chunk sums of the sampled weights ----------------
  // CTA `rank` owns the contiguous chunks [c_begin, c_end).  Residual elements
  // are formed in fp32 (one rounding each, at most 2^-24 of the element); a
  // chunk's sum is accumulated as an unevaluated pair (hi, lo) of fp32 values
  // with error-free TwoSum steps, per lane and then across the warp, keeping
  // the sum of the fp32 elements to ~2^-45 relative without FP64
  // instructions (GB300 issues FP64 warp instructions at a small fraction of
  // the FP32 rate).  With 16-byte-aligned rows a producer warp streams the
  // rows with bulk copies into a ring of shared-memory stages (four chunks of
  // p and of q per stage) and the consumer warps reduce them.
  const bool residual = (event == EV_REJECT);
  const float* prow = p + ((size_t)r * (gamma + 1) + jstar) * V;
  const float* qrow = residual ? q + ((size_t)r * gamma + jstar) * V : prow;
  const int n_chunks = (V + kChunk - 1) / kChunk;
  const int npc = chunks_per_cta(V);
  const int c_begin = min(n_chunks, rank * npc);
  const int n_local = min(n_chunks, c_begin + npc) - c_begin;
  bool bad = false;
  // this CTA's tables: for each of its chunks the 32 lanes' partial sums (lane l
  // covers elements 32l .. 32l + 31 of the chunk) and the chunk's (hi, lo) sum
  float* s_lane = reinterpret_cast<float*>(ring + (kVec4 ? kRingBytes : 0));
  float2* s_chunk = reinterpret_cast<float2*>(s_lane + 32 * npc);
  if constexpr (kVec4) {
    const int n_stages = kStarve ? 0 : (n_local + kStageChunks - 1) / kStageChunks;
    if (warp == kConsumerWarps) {
      // producer warp: every lane waits, lane 0 issues the copies
      int issued_last = -1;
      for (int st = 0; st < n_stages; ++st) {
        const int slot = st % kRing, use = st / kRing;
        // warp-uniform outcome: every lane waits, all must have seen the phase
        if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(s_empty_bar + 8u * slot, (use - 1) & 1))) {
          if (lane == 0) {
            atomicOr(&g_mtp_error_word, MTP_DEVERR_TIMEOUT);
            s_timeout = 1;
          }
          break;
        }
        if (lane == 0) {
          const int chunk0 = c_begin + st * kStageChunks;
          const int nch = min(kStageChunks, n_local - st * kStageChunks);
          const uint32_t bytes = 4u * static_cast<uint32_t>(min(nch * kChunk, V - chunk0 * kChunk));
          const uint32_t full = s_full_bar + 8u * slot;
          mbar_expect_tx(full, residual ? 2u * bytes : bytes);
          const uint32_t me = static_cast<uint32_t>(rank);
          bulk_load(cluster_addr(ring_p(slot), me), prow + (size_t)chunk0 * kChunk, bytes, cluster_addr(full, me));
          if (residual) bulk_load(cluster_addr(ring_q(slot), me), qrow + (size_t)chunk0 * kChunk, bytes, cluster_addr(full, me));
        }
        issued_last = st;
        __syncwarp();
      }
      // no copy may still be landing in this CTA's shared memory when it leaves:
      // wait (bounded) for the last use of every slot that was issued
      if (lane == 0) {
        for (int st = max(0, issued_last - kRing + 1); st <= issued_last; ++st)
          if (!mbar_wait(s_full_bar + 8u * (st % kRing), (st / kRing) & 1)) {
            atomicOr(&g_mtp_error_word, MTP_DEVERR_TIMEOUT);
            s_timeout = 1;
          }
      }
      __syncwarp();
    } else {
      volatile int* timeout_flag = &s_timeout;
      for (int li = warp; li < n_local; li += kConsumerWarps) {
        const int st = li / kStageChunks, i = li % kStageChunks;
        const int slot = st % kRing, use = st / kRing;
        // warp-uniform decisions: lane 0's view of the flag, all lanes' waits
        if (__shfl_sync(0xffffffffu, *timeout_flag, 0)) break;
        if (!__all_sync(0xffffffffu, mbar_wait(s_full_bar + 8u * slot, use & 1))) {
          if (lane == 0) {
            atomicOr(&g_mtp_error_word, MTP_DEVERR_TIMEOUT);
            s_timeout = 1;
          }
          break;
        }
        const float* sp = reinterpret_cast<const float*>(ring + slot * kStageBytes) + i * kChunk;
        const float* sq = sp + kStageChunks * kChunk;
        const int base = (c_begin + li) * kChunk;
        // lane l sums its 32 consecutive elements, their eight 16-byte groups taken
        // in a rotated order (group (k + l) % 8 at step k) so that the eight lanes
        // of a quarter-warp read distinct banks; four independent compensated sums
        // per lane (one per vector component), merged after the loop
        float h0 = 0.0f, l0 = 0.0f, h1 = 0.0f, l1 = 0.0f, h2 = 0.0f, l2 = 0.0f, h3 = 0.0f, l3 = 0.0f;
        float nanchk = 0.0f, mn = 0.0f;  // see check_value
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int off = 32 * lane + 4 * ((k + lane) & 7);
          if (base + off < V) {
            const float4 pv = *reinterpret_cast<const float4*>(sp + off);
            const float4 qv = residual ? *reinterpret_cast<const float4*>(sq + off) : make_float4(0.f, 0.f, 0.f, 0.f);
            check_value4(nanchk, mn, pv);
            if (residual) check_value4(nanchk, mn, qv);
            acc_add(h0, l0, weight_of(pv.x, qv.x, residual));
            acc_add(h1, l1, weight_of(pv.y, qv.y, residual));
            acc_add(h2, l2, weight_of(pv.z, qv.z, residual));
            acc_add(h3, l3, weight_of(pv.w, qv.w, residual));
          }
        }
        bad |= !(nanchk == 0.0f) || mn < 0.0f;
        float hi = h0, lo = l0;
        acc_add(hi, lo, h1);
        acc_add(hi, lo, h2);
        acc_add(hi, lo, h3);
        lo += (l1 + l2) + l3;
        s_lane[32 * li + lane] = hi + lo;
        warp_two_sum(hi, lo);
        __syncwarp();
        if (lane == 0) {
          s_chunk[li] = make_float2(hi, lo);
          // a stage expects kStageChunks arrivals; in a partial last stage the
          // consumer of its first chunk also supplies those of the missing chunks
          const int nch = min(kStageChunks, n_local - st * kStageChunks);
          mbar_arrive_cnt(s_empty_bar + 8u * slot, i == 0 ? 1u + static_cast<uint32_t>(kStageChunks - nch) : 1u);
        }
      }
    }
  } else {
    if (warp < kConsumerWarps) {
      for (int li = warp; li < n_local; li += kConsumerWarps) {
        const int base = (c_begin + li) * kChunk + 32 * lane;  // this lane's 32 consecutive elements
        float hi = 0.0f, lo = 0.0f;
#pragma unroll 4
        for (int i = 0; i < 32; ++i) {
          const int e = base + i;
          float pv = 0.f, qv = 0.f;
          if (e < V) {
            pv = prow[e];
            if (residual) qv = qrow[e];
          }
          bad |= !prob_ok(pv) || (residual && !prob_ok(qv));
          acc_add(hi, lo, weight_of(pv, qv, residual));
        }
        s_lane[32 * li + lane] = hi + lo;
        warp_two_sum(hi, lo);
        if (lane == 0) s_chunk[li] = make_float2(hi, lo);
      }
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&s_bad, 1);
  __syncthreads();

  // ---------------- phase C: locate u' * mass ----------------
  // In double-float arithmetic (no FP64 on this latency-bound path: a chain of
  // FP64 additions here took ~4.7 us on GB300).  Warp 0 of each CTA takes the
  // prefix over its own chunks and hands its total and error flags to the other
  // CTA; after one cluster barrier both know the mass and the target, and the
  // CTA whose half holds the target finds the chunk, the lane range of 32
  // elements within it (from the staged lane sums) and, loading just those 32
  // elements of p and q again (the row was just streamed: L2), the element.
  const int per = (n_local + 31) / 32;  // lane l owns this CTA's chunks [l*per, (l+1)*per)
  const int c0 = min(n_local, lane * per), c1 = min(n_local, (lane + 1) * per);
  f2 own = {0.0f, 0.0f}, incl = {0.0f, 0.0f};
  if (warp == 0) {
    for (int c = c0; c < c1; ++c) own = f2_add(own, chunk_value(s_chunk[c]));
    incl = warp_inclusive_scan_f2(own);
    const f2 total = f2_shfl(incl, 31);
    if (lane == 0) {
      const uint32_t peer = static_cast<uint32_t>(rank ^ 1);
      s_tot[rank] = make_float2(total.hi, total.lo);
      *cluster.map_shared_rank(&s_tot[rank], peer) = make_float2(total.hi, total.lo);
      if (s_bad) atomicOr(cluster.map_shared_rank(&s_bad, peer), 1);
      if (s_timeout) atomicOr(cluster.map_shared_rank(&s_timeout, peer), 1);
    }
  }
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (warp != 0) return;
  int st = MTP_VERIFY_OK;
  const f2 S0 = chunk_value(s_tot[0]), S1 = chunk_value(s_tot[1]);
  const f2 mass = f2_add(S0, S1);
  if (s_timeout) st = MTP_VERIFY_DEVICE_TIMEOUT;
  else if (s_bad) st = MTP_VERIFY_INVALID_PROBS;
  else if (!(mass.hi > 0.0f)) st = MTP_VERIFY_ZERO_RESIDUAL;
  if (st != MTP_VERIFY_OK) {
    if (rank == 0 && lane == 0) {
      accepted[r] = jstar; next_token[r] = -1; n_emit[r] = jstar; status[r] = st;
    }
    return;
  }
  const f2 target = f2_scale(s_u, mass);
  // the half holding the target: CTA 0's when its sum exceeds it; else CTA 1's,
  // which also takes the rounding overshoot (no running sum above the target:
  // the last element with weight) unless it has no mass at all
  const int owner = f2_gt(S0, target) ? 0 : (S1.hi > 0.0f ? 1 : 0);
  if (rank != owner) return;
  const f2 base = rank == 0 ? f2{0.0f, 0.0f} : S0;  // the mass before this CTA's chunks
  int cstar = -1;  // local chunk index
  f2 before = {0.0f, 0.0f};
  {
    const f2 cum = f2_add(base, incl);
    const f2 cum_excl = f2_add(base, f2_exclusive(incl));
    const unsigned over = __ballot_sync(0xffffffffu, f2_gt(cum, target));
    const unsigned has_mass = __ballot_sync(0xffffffffu, own.hi > 0.0f);
    const int src = over ? __ffs(over) - 1 : 31 - __clz(has_mass);
    if (lane == src) {
      f2 run = cum_excl, before_last = cum_excl;
      int last_pos = -1;
      for (int c = c0; c < c1; ++c) {
        const f2 cv = chunk_value(s_chunk[c]);
        const f2 next = f2_add(run, cv);
        if (cv.hi > 0.0f) { last_pos = c; before_last = run; }
        if (over && f2_gt(next, target)) { cstar = c; before = run; break; }
        run = next;
      }
      if (cstar < 0) { cstar = last_pos; before = before_last; }
    }
    cstar = __shfl_sync(0xffffffffu, cstar, src);
    before = f2_shfl(before, src);
  }
  // the lane range of 32 elements within chunk cstar
  const float lp = s_lane[32 * cstar + lane];
  const f2 lincl = f2_add(before, warp_inclusive_scan_f2(f2{lp, 0.0f}));
  const unsigned lover = __ballot_sync(0xffffffffu, f2_gt(lincl, target));
  const unsigned lpos = __ballot_sync(0xffffffffu, lp > 0.0f);
  int pick = -1;
  if (lover || lpos) {
    const int lsrc = lover ? __ffs(lover) - 1 : 31 - __clz(lpos);
    const f2 lexcl = f2_exclusive(lincl);
    const f2 start = lsrc == 0 ? before : f2_shfl(lexcl, lsrc);  // running sum before the range
    const int e0 = (c_begin + cstar) * kChunk + 32 * lsrc;
    const int e = e0 + lane;
    const float w = e < V ? weight_of(__ldcg(prow + e), residual ? __ldcg(qrow + e) : 0.0f, residual) : 0.0f;
    const f2 cum = f2_add(start, warp_inclusive_scan_f2(f2{w, 0.0f}));
    const unsigned eover = __ballot_sync(0xffffffffu, w > 0.0f && f2_gt(cum, target));
    const unsigned epos = __ballot_sync(0xffffffffu, w > 0.0f);
    if (eover) pick = e0 + __ffs(eover) - 1;
    else if (epos) pick = e0 + 31 - __clz(epos);
  }
  if (lane == 0) {
    accepted[r] = jstar;
    next_token[r] = pick;
    n_emit[r] = pick >= 0 ? jstar + 1 : jstar;
    status[r] = pick >= 0 ? MTP_VERIFY_OK : MTP_VERIFY_ZERO_RESIDUAL;
  }
}

template <bool kStarve>
mtp_status verify_launch(int R, int gamma, int V, const float* p, const float* q, const int32_t* draft,
                         uint64_t seed, uint64_t offset, const int32_t* eos, const int32_t* remaining,
                         int32_t* accepted, int32_t* next_token, int32_t* n_emit, int32_t* status,
                         long long wait_limit, cudaStream_t stream) {
  if (R < 0 || gamma < 0 || V <= 0) return MTP_ERR_INVALID_ARG;
  if (gamma > kMaxGamma || V > kMaxChunks * kChunk) return MTP_ERR_UNSUPPORTED;
  if (R == 0) return MTP_OK;
  if (!p || (!draft && gamma > 0) || !accepted || !next_token || !n_emit || !status) return MTP_ERR_INVALID_ARG;
  if (gamma > 0 && !q) return MTP_ERR_INVALID_ARG;
  const uint2 key = make_uint2((uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32));
  const uint32_t olo = (uint32_t)(offset & 0xFFFFFFFFu), ohi = (uint32_t)(offset >> 32);
  const bool vec = (V % 4 == 0) && mtp::aligned16(p) && (gamma == 0 || mtp::aligned16(q));
  if (kStarve && !vec) return MTP_ERR_UNSUPPORTED;  // the ring exists only on the bulk-copy path
  static mtp::PerDevice attr;
  const size_t tables = static_cast<size_t>(chunks_per_cta(V)) * kTableBytesPerChunk;
  // the attribute covers the largest V this kernel takes, so it is set once per device
  constexpr size_t kMaxVecBytes = kRingBytes + static_cast<size_t>(kMaxChunks / kCluster) * kTableBytesPerChunk;
  if (vec && !mtp::smem_limit(attr, spec_verify_kernel<true, kStarve>, kMaxVecBytes)) return MTP_ERR_CUDA;
  if (!kStarve) mtp::prof_begin(MTP_KC_SPEC_VERIFY, stream);
  if (vec)
    spec_verify_kernel<true, kStarve><<<R * kCluster, kThreads, kRingBytes + tables, stream>>>(
        gamma, V, p, q, draft, key, olo, ohi, eos, remaining, accepted, next_token, n_emit, status, wait_limit);
  else
    spec_verify_kernel<false, false><<<R * kCluster, kThreads, tables, stream>>>(
        gamma, V, p, q, draft, key, olo, ohi, eos, remaining, accepted, next_token, n_emit, status, wait_limit);
  mtp::note_launch();
  if (!kStarve) mtp::prof_end(MTP_KC_SPEC_VERIFY, stream);
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}

}  // namespace

extern "C" mtp_status spec_verify(int R, int gamma, int V, const float* p, const float* q,
                                  const int32_t* draft, uint64_t seed, uint64_t offset,
                                  const int32_t* eos, const int32_t* remaining,
                                  int32_t* accepted, int32_t* next_token, int32_t* n_emit,
                                  int32_t* status, cudaStream_t stream) {
  return verify_launch<false>(R, gamma, V, p, q, draft, seed, offset, eos, remaining, accepted, next_token, n_emit,
                              status, mtp::kWaitLimitCycles, stream);
}

extern "C" mtp_status mtp_diag_verify_starved(int R, int gamma, int V, const float* p, const float* q,
                                              const int32_t* draft, uint64_t seed, uint64_t offset,
                                              int32_t* accepted, int32_t* next_token, int32_t* n_emit,
                                              int32_t* status, long long wait_limit_cycles, cudaStream_t stream) {
  if (wait_limit_cycles <= 0 || wait_limit_cycles > mtp::kWaitLimitCycles) return MTP_ERR_INVALID_ARG;
  return verify_launch<true>(R, gamma, V, p, q, draft, seed, offset, nullptr, nullptr, accepted, next_token,
                             n_emit, status, wait_limit_cycles, stream);
}
